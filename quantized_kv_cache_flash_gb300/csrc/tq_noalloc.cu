// tq_decode_attention_noalloc: decode attention for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc on the decode path: an inference server
// that carves all device memory into its own pools up front and forbids any
// other allocation, a process that runs under a hard device-memory budget, or
// code that must not create a library context (tq_decode_attention creates one
// lazily and grows its split-K workspace with cudaMalloc).  This entry point
// runs the same split-K decode and combine kernels, but their scratch (the
// per-split partial results and a status word) lives in a fixed-size,
// file-scope __device__ array that the CUDA module reserves on every GPU where
// the library is loaded, until the process exits.  The caller passes inputs
// and outputs only; the call allocates nothing.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress, once per device; make
// that first call before any stream capture.  Every call shares the array, so
// calls that overlap on the GPU (different streams, or concurrent host
// threads) race on it; serialise them.  The array keeps the previous call's
// contents; the only part that must start at zero, the internal status word,
// is cleared by each call that uses it.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "tq.h"
#include "tq_internal.h"

namespace {

constexpr int kD = 128;
constexpr int kMaxDevices = 64;
constexpr size_t kStatusBytes = 256;  // first 256 bytes: internal status word

static __device__ __align__(256) unsigned char g_tq_noalloc_scratch[TQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};  // the context the address belongs to

// The driver's cuCtxGetCurrent, looked up once per process.
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    }
    return fn;
}

// Device address of the scratch array on the current device.  Looked up once
// per device, and again if the device's context has changed since (after a
// cudaDeviceReset the module is loaded anew, possibly at another address).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_get_current();
    CUcontext cu_ctx = nullptr;
    if (get_ctx == nullptr || get_ctx(&cu_ctx) != CUDA_SUCCESS) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (cu_ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != static_cast<void*>(cu_ctx)) {
        // (the symbol lookup also makes the device's primary context current)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tq_noalloc_scratch) != cudaSuccess || p == nullptr)
            return TQ_ERR_CUDA;
        if (get_ctx(&cu_ctx) != CUDA_SUCCESS) return TQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = static_cast<void*>(cu_ctx);
    }
    *out = g_scratch_ptr[dev];
    return TQ_OK;
}

}  // namespace

extern "C" int tq_decode_attention_noalloc(const tq_cache* c, const void* q, int32_t num_q_heads,
                                           int32_t tq_rows, int32_t max_len_hint, float scale,
                                           void* out, uint32_t* status, void* stream) {
    tq::host::DecodePlan pl;
    int r = tq::host::plan_decode(c, q, out, num_q_heads, tq_rows, max_len_hint, scale, &pl);
    if (r != TQ_OK) return r;

    // decode grid, limited to what the fixed scratch holds (one slot per CTA
    // and per unit)
    const size_t slot_bytes = size_t(16) * (kD + 2) * sizeof(float);
    const size_t max_slots = (size_t(TQ_NOALLOC_SCRATCH_BYTES) - kStatusBytes) / slot_bytes;
    if (size_t(pl.units) >= max_slots) return TQ_ERR_CAPACITY;   // does not fit the fixed scratch
    if (size_t(pl.units) + size_t(pl.ctas) > max_slots) pl.ctas = int(max_slots - size_t(pl.units));

    tq::host::CodebookTables kt, vt;
    if (pl.kb != 16 && (r = tq::host::build_tables(c->codebook_k, c->codebook_k_size, pl.kb, &kt)) != TQ_OK)
        return r;
    if ((r = tq::host::build_tables(c->codebook_v, c->codebook_v_size, pl.vb, &vt)) != TQ_OK) return r;
    uint32_t signs[4];
    tq::host::make_signs(c->rot_seed, signs);
    CUtensorMap kmap;
    std::memset(&kmap, 0, sizeof(kmap));
    if (pl.kb == 16 && (r = tq::host::encode_kmap(&kmap, c)) != TQ_OK) return r;

    void* base = nullptr;
    if ((r = scratch_address(&base)) != TQ_OK) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* st_word = status;
    if (st_word == nullptr) {
        st_word = static_cast<uint32_t*>(base);
        if (cudaMemsetAsync(st_word, 0, sizeof(uint32_t), s) != cudaSuccess) return TQ_ERR_CUDA;
    }
    float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kStatusBytes);
    return tq::host::launch_decode_plan(pl, c, kt, vt, signs, &kmap, q, num_q_heads, tq_rows,
                                        max_len_hint, scale, 0.f, out, part, st_word, s, nullptr,
                                        nullptr);
}
