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

#include <cmath>
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

// Device address of the scratch array on the current device (set up once).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tq_noalloc_scratch) != cudaSuccess || p == nullptr)
            return TQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_codebook(const float* cb, int n, int bits) {
    if (cb == nullptr || n != (1 << bits)) return TQ_ERR_INVALID_ARG;
    for (int j = 0; j < n; ++j)
        if (!std::isfinite(cb[j])) return TQ_ERR_INVALID_ARG;
    for (int j = 0; j + 1 < n; ++j)
        if (!(cb[j] < cb[j + 1])) return TQ_ERR_INVALID_ARG;
    for (int j = 0; j < n; ++j)
        if (cb[j] != -cb[n - 1 - j]) return TQ_ERR_INVALID_ARG;
    return TQ_OK;
}

uint16_t half_bits(float f) {
    __half h = __float2half_rn(f);
    uint16_t b;
    std::memcpy(&b, &h, 2);
    return b;
}

// prmt byte tables of a checked codebook (same layout the kernels expect:
// 3-bit tables indexed by the sign-magnitude code, 4-bit by magnitude rank).
void tables(const float* cb, int bits, uint32_t out[4]) {
    const int h = (1 << bits) / 2;
    uint8_t lo[8] = {}, hi[8] = {};
    for (int k = 0; k < 8; ++k) {
        float v;
        if (bits == 3) v = (k & 4) ? -cb[h + (k & 3)] : cb[h + (k & 3)];
        else v = cb[h + k];
        const uint16_t hb = half_bits(v);
        lo[k] = hb & 0xFF;
        hi[k] = hb >> 8;
    }
    auto word = [](const uint8_t* b) {
        return uint32_t(b[0]) | (uint32_t(b[1]) << 8) | (uint32_t(b[2]) << 16) | (uint32_t(b[3]) << 24);
    };
    out[0] = word(lo);
    out[1] = word(lo + 4);
    out[2] = word(hi);
    out[3] = word(hi + 4);
}

void signs_of(uint64_t seed, uint32_t out[4]) {
    uint64_t st = seed;
    out[0] = out[1] = out[2] = out[3] = 0;
    for (int d = 0; d < kD; ++d) {
        st += 0x9E3779B97F4A7C15ull;
        uint64_t z = st;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        if (z >> 63) out[d >> 5] |= 1u << (d & 31);
    }
}

}  // namespace

extern "C" int tq_decode_attention_noalloc(const tq_cache* c, const void* q, int32_t num_q_heads,
                                           int32_t tq_rows, int32_t max_len_hint, float scale,
                                           void* out, uint32_t* status, void* stream) {
    int kb, vb;
    if (c == nullptr) return TQ_ERR_INVALID_ARG;
    int r = tq::mode_bits(c->mode, &kb, &vb);
    if (r != TQ_OK) return r;
    if (c->head_dim != kD) return TQ_ERR_UNSUPPORTED;
    if (c->batch <= 0 || c->num_kv_heads <= 0 || c->capacity <= 0 || (c->capacity % 16) != 0)
        return TQ_ERR_INVALID_ARG;
    const bool table = tq::mode_table(c->mode);  // table records: no norm arrays
    if (c->k_data == nullptr || c->v_data == nullptr || c->lengths == nullptr ||
        (!table && (c->v_norm == nullptr || (kb != 16 && c->k_norm == nullptr))))
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(c->k_data) || !aligned16(c->v_data) || (c->v_norm && !aligned16(c->v_norm)) ||
        (c->k_norm && !aligned16(c->k_norm)))
        return TQ_ERR_INVALID_ARG;
    if (1ll * c->batch * c->num_kv_heads * c->capacity >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;
    if (kb != 16 && (r = check_codebook(c->codebook_k, c->codebook_k_size, kb)) != TQ_OK) return r;
    if ((r = check_codebook(c->codebook_v, c->codebook_v_size, vb)) != TQ_OK) return r;
    if (q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (tq_rows <= 0 || max_len_hint <= 0 || max_len_hint > c->capacity || tq_rows > max_len_hint)
        return TQ_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale) || !std::isfinite(c->v_rescale))
        return TQ_ERR_INVALID_ARG;
    const int group = num_q_heads / c->num_kv_heads;
    const int rows = group * tq_rows;
    if (rows > 256) return TQ_ERR_UNSUPPORTED;
    const int group_rows = tq::group_rows_for(rows);
    const int row_groups = (rows + group_rows - 1) / group_rows;

    // decode grid, limited to what the fixed scratch holds (one slot per CTA
    // and per unit)
    int tokens_per_cta = 0, ctas = 0;
    r = tq_plan_splits(c->mode, c->batch, c->num_kv_heads, rows, max_len_hint, &tokens_per_cta, &ctas);
    if (r != TQ_OK) return r;
    const size_t slot_bytes = size_t(16) * (kD + 2) * sizeof(float);
    const size_t units = size_t(c->batch) * c->num_kv_heads * row_groups;
    const size_t max_slots = (size_t(TQ_NOALLOC_SCRATCH_BYTES) - kStatusBytes) / slot_bytes;
    if (units >= max_slots) return TQ_ERR_CAPACITY;   // does not fit the fixed scratch
    if (units + size_t(ctas) > max_slots) ctas = int(max_slots - units);

    void* base = nullptr;
    if ((r = scratch_address(&base)) != TQ_OK) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* st_word = status;
    if (st_word == nullptr) {
        st_word = static_cast<uint32_t*>(base);
        if (cudaMemsetAsync(st_word, 0, sizeof(uint32_t), s) != cudaSuccess) return TQ_ERR_CUDA;
    }
    float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kStatusBytes);
    const size_t slots = (units + size_t(ctas)) * 16;

    tq::DecodeParams p{};
    p.k_codes = static_cast<const uint8_t*>(c->k_data);
    p.k_norm = static_cast<const __half*>(c->k_norm);
    p.v_codes = static_cast<const uint8_t*>(c->v_data);
    p.v_norm = static_cast<const __half*>(c->v_norm);
    p.lengths = c->lengths;
    p.q = static_cast<const __half*>(q);
    p.part_o = part;
    p.part_ml = part + slots * kD;
    p.status = st_word;
    p.batch = c->batch;
    p.hkv = c->num_kv_heads;
    p.hq = num_q_heads;
    p.group = group;
    p.tq = tq_rows;
    p.rows = rows;
    p.row_groups = row_groups;
    p.group_rows = group_rows;
    p.cap = c->capacity;
    p.max_len = max_len_hint;
    p.num_ctas = ctas;
    p.table = table ? 1 : 0;
    p.scale_log2e = ((scale == 0.f) ? 1.0f / std::sqrt(float(kD)) : scale) * 1.4426950408889634f;
    if (kb != 16) tables(c->codebook_k, kb, p.ktab);
    tables(c->codebook_v, vb, p.vtab);
    signs_of(c->rot_seed, p.signs);

    CUtensorMap kmap;
    std::memset(&kmap, 0, sizeof(kmap));
    if (kb == 16) {
        cudaDriverEntryPointQueryResult qres;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &qres) != cudaSuccess ||
            qres != cudaDriverEntryPointSuccess || fn == nullptr)
            return TQ_ERR_CUDA;
        auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        const uint64_t nrows = uint64_t(c->batch) * c->num_kv_heads * c->capacity;
        cuuint64_t dims[2] = {kD, nrows};
        cuuint64_t strides[1] = {kD * 2};
        cuuint32_t box[2] = {64, 32};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, c->k_data, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TQ_ERR_CUDA;
    }
    if (tq::launch_decode(kb, vb, p, &kmap, s, nullptr, nullptr) != 0) return TQ_ERR_CUDA;

    tq::CombineParams cp{};
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.lengths = c->lengths;
    cp.out = static_cast<__half*>(out);
    cp.status = st_word;
    cp.batch = c->batch;
    cp.hkv = c->num_kv_heads;
    cp.hq = num_q_heads;
    cp.group = group;
    cp.tq = tq_rows;
    cp.row_groups = row_groups;
    cp.group_rows = group_rows;
    cp.max_len = max_len_hint;
    cp.num_ctas = ctas;
    cp.v_rescale = c->v_rescale;
    std::memcpy(cp.signs, p.signs, sizeof(cp.signs));
    return tq::launch_combine(cp, s) == 0 ? TQ_OK : TQ_ERR_CUDA;
}
