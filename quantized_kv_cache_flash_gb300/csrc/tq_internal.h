// Host <-> device parameter blocks and launcher entry points (internal).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "tq.h"

namespace tq {

// Decode (split-K) kernel parameters.  A row group is up to group_rows (4, 8
// or 16) query rows (GQA heads x Tq) of one KV head: the N dimension of the
// warp-level MMAs, whose M dimension is 16 tokens.  The CTAs split the
// context's 32-token chunks of all (batch, kv head, row group) units evenly.
struct DecodeParams {
    const uint8_t* k_codes;   // packed K codes (unused for fp16 K)
    const __half* k_norm;     // fp16 K norms (unused for fp16 K)
    const uint8_t* v_codes;   // packed V codes
    const __half* v_norm;     // fp16 V norms
    const int32_t* lengths;   // [B]
    const __half* q;          // [B, Hq, Tq, 128]
    float* part_o;            // [num_ctas + units, 16, 128], units = batch * hkv * row_groups
    float* part_ml;           // [num_ctas + units, 16, 2]  (running max in log2 units, sum)
    uint32_t* status;
    int32_t batch, hkv, hq, group, tq, rows, row_groups, group_rows, cap, max_len;
    int32_t num_ctas;         // decode grid (one wave of token-balanced CTAs)
    float scale_log2e;        // softmax scale * log2(e)
    float sparse_tau;         // sparse-V threshold on the softmax weight (0: off)
    uint32_t* sparse_tiles;   // sparse V: [0] += 16-token tiles skipped, [1] += tiles judged
    int32_t table;            // 1: records carry their centroid x norm table (no norms)
    uint32_t ktab[4];         // prmt byte tables of the K codebook (lo0, lo1, hi0, hi1)
    uint32_t vtab[4];
    uint32_t signs[4];        // bit d set <=> s_d = -1
    // K centroids' rounding residuals c - fp16(c), scaled by 2^res_shift, as
    // e4m3 bytes (3-bit: indexed by the signed code; 4-bit: by magnitude rank)
    uint32_t ktab8[2];
    int32_t res_shift;
    int32_t k_res;            // 1: the K codebook has entries that are not fp16 values
};

struct CombineParams {
    const float* part_o;
    const float* part_ml;
    const int32_t* lengths;
    __half* out;              // [B, Hq, Tq, 128]
    uint32_t* status;
    int32_t batch, hkv, hq, group, tq, row_groups, group_rows, max_len, num_ctas;
    float v_rescale;
    uint32_t signs[4];
};

struct EncodeParams {
    const __half* k_new;      // [B, Hkv, T, 128]
    const __half* v_new;
    uint8_t* k_codes;         // packed codes or fp16 K rows (fp16 K mode)
    __half* k_norm;
    uint8_t* v_codes;
    __half* v_norm;
    int32_t* lengths;
    uint32_t* status;
    uint32_t* counter;        // zero between calls; the last CTA resets it
    uint32_t* tiles_next;     // large appends: the next tile to hand out (zero between calls, reset likewise)
    int32_t batch, hkv, t_new, cap;
    // n / t_new and n / hkv for 0 <= n < 2^31 as (n * m) >> s (see div_magic)
    uint32_t div_t_m, div_h_m;
    int32_t div_t_s, div_h_s;
    uint32_t signs[4];
    // decision thresholds on |u| over the positive half of the codebook:
    // a > tau_k  <=>  a >= gt[k];   a >= tau_k  <=>  a >= ge[k]   (fp32, exact)
    float k_gt[7], k_ge[7], v_gt[7], v_ge[7];
    // table records: 48 bytes of 3-bit codes + fp16(c_j * n16), j = 0..7
    int32_t table;
    float k_cb[8], v_cb[8];
};

// Chunked-prefill attention (tcgen05) parameters.  One CTA = one (query
// tile of pos_per_tile positions x group heads, batch * kv head).
struct PrefillParams {
    const uint8_t* k_codes;   // packed K codes, or fp16 K rows (read through the tensor map)
    const __half* k_norm;
    const uint8_t* v_codes;
    const __half* v_norm;
    const int32_t* lengths;   // [B]
    const __half* q;          // [B, Hq, Tq, 128]
    __half* out;              // [B, Hq, Tq, 128]
    uint32_t* status;
    int32_t batch, hkv, hq, group, tq, cap, max_len;
    int32_t pos_per_tile;     // query positions per 128-row tile (128 / group)
    int32_t mtiles;           // tiles per kv head
    float scale_log2e, v_rescale;
    uint32_t ktab[4], vtab[4], signs[4];
};

// Division of 0 <= n < 2^31 by a constant d >= 1 as a multiply-high: with
// l = ceil(log2 d), s = 31 + l and m = ceil(2^s / d) (below 2^32),
// floor(n m / 2^s) = floor(n / d), because m d - 2^s < d <= 2^l and
// n < 2^31 keep the error term n (m d - 2^s) / (d 2^s) below 1/d.
inline void div_magic(uint32_t d, uint32_t* m, int32_t* s) {
    int l = 0;
    while ((1ull << l) < d) ++l;
    *s = 31 + l;
    *m = static_cast<uint32_t>(((1ull << *s) + d - 1) / d);
}

// Launchers (return a cudaError_t value).
// group_rows (p.group_rows) selects the 4-, 8- or 16-row variant.
int launch_decode(int kbits, int vbits, const DecodeParams& p, const CUtensorMap* kmap,
                  cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end);
int launch_combine(const CombineParams& p, cudaStream_t stream);
// Appends of more than kEncodeSmallMax vectors per stream run on the tensor
// cores and read their inputs through kmap / vmap (encode_rows_map of k_new /
// v_new); smaller ones ignore the maps.
constexpr long long kEncodeSmallMax = 4096;
int launch_encode(int kbits, int vbits, const EncodeParams& p, const CUtensorMap* kmap,
                  const CUtensorMap* vmap, cudaStream_t stream);

// Resident CTAs per SM of a decode variant (for the host split planner);
// res: the variant with the centroid residual product.
int decode_ctas_per_sm(int kbits, int vbits, int group_rows, bool table, bool res);
int launch_prefill(int kbits, int vbits, const PrefillParams& p, const CUtensorMap* kmap,
                   cudaStream_t stream);
int launch_selftest_stall(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

// Query rows per row group for `rows` query rows of one KV head: 4 when K is
// quantized and at most 4 rows share a KV head (the low halves of the rotated
// query then ride in the score MMA's spare columns), else 8, or 16 per group.
inline int group_rows_for(int rows, int kbits) {
    return (rows <= 4 && kbits != 16) ? 4 : rows <= 8 ? 8 : 16;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream finishes (every kernel of this library
// waits for its predecessor with griddep_wait() before touching memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Opt a kernel into `bytes` of dynamic shared memory (and, carveout >= 0, a
// preferred shared-memory carveout) on the current device, once per device:
// `done` keeps one bit per device ordinal (devices past 63 set it every call).
template <typename Kernel>
cudaError_t set_smem_attr_once(Kernel kernel, int bytes, std::atomic<uint64_t>& done, int carveout = -1) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && carveout >= 0)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Records that carry a centroid x norm table instead of a norm.
inline bool mode_table(int mode) { return mode == TQ_TURBO3_TABLE; }

// (K bits, V bits) of a mode; 16 = fp16 K.
inline int mode_bits(int mode, int* kb, int* vb) {
    switch (mode) {
        case TQ_TURBO4_ASYM: *kb = 16; *vb = 4; return TQ_OK;
        case TQ_TURBO3: *kb = 3; *vb = 3; return TQ_OK;
        case TQ_TURBO4: *kb = 4; *vb = 4; return TQ_OK;
        case TQ_TURBO3_ASYM: *kb = 16; *vb = 3; return TQ_OK;
        case TQ_TURBO4K_3V: *kb = 4; *vb = 3; return TQ_OK;
        case TQ_TURBO3_TABLE: *kb = 3; *vb = 3; return TQ_OK;
        default: return TQ_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------------------
// Host helpers shared by the entry points (defined in tq_api.cu)
// ---------------------------------------------------------------------------
namespace host {

// Kernel-side forms of a checked codebook.
struct CodebookTables {
    bool valid = false;
    int bits = 0;
    float cb[16] = {};
    uint32_t tab[4] = {};  // prmt byte tables of the fp16 centroids (lo0, lo1, hi0, hi1)
    float gt[7] = {}, ge[7] = {};  // encode decision thresholds (see EncodeParams)
    // e4m3 bytes of (c - fp16(c)) * 2^res_shift (3-bit: by signed code; 4-bit:
    // by magnitude rank), for the score's fp8 residual product
    uint32_t tab8[2] = {};
    int res_shift = 0;
};

int cuda_err_code(cudaError_t e);
bool aligned16(const void* p);
// Mode, shape, pointers and codebooks of a cache; *kb, *vb = its bits (16 = fp16 K).
int check_cache(const tq_cache* c, int* kb, int* vb);
// (Re)builds *t unless it already holds this codebook.
int build_tables(const float* cb, int n, int bits, CodebookTables* t);
// s_d = -1 <=> bit d of out (splitmix64 of the rotation seed).
void make_signs(uint64_t seed, uint32_t out[4]);
// Tensor map of the fp16 K rows of a cache (driver entry point looked up once).
int encode_kmap(CUtensorMap* map, const tq_cache* c);
// Tensor map of `rows` fp16 vectors of 128 dims at `base` (16-byte aligned),
// boxes of 128 rows x 64 halves (128-byte swizzle): the encode's input tiles.
int encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows);
// Whether every entry of a codebook is an fp16 value (no rounding residual).
bool codebook_is_fp16(const float* cb, int n);

// One decode call's checked arguments and the row grouping and grid derived
// from them.
struct DecodePlan {
    int kb, vb;
    bool res;          // quantized K whose codebook is not all fp16 values
    int group, rows, group_rows, row_groups;
    long long units;   // (batch, kv head, row group) units
    int ctas;          // decode grid
};
int plan_decode(const tq_cache* c, const void* q, const void* out, int num_q_heads, int tq_rows,
                int max_len_hint, float scale, DecodePlan* pl);
// Split-K scratch of a plan: (ctas + units) slots of 16 rows x (128 + 2) floats.
inline size_t decode_slots(const DecodePlan& pl) { return size_t(pl.ctas + pl.units) * 16; }
// Launch the decode and combine kernels of a plan on `stream`, the partials
// in `part` (decode_slots(pl) * 130 floats), device status bits ORed into
// `status`; ev0/ev1 (optional) bracket the decode kernel.
int launch_decode_plan(const DecodePlan& pl, const tq_cache* c, const CodebookTables& kt,
                       const CodebookTables& vt, const uint32_t signs[4], const CUtensorMap* kmap,
                       const void* q, int num_q_heads, int tq_rows, int max_len_hint, float scale,
                       float tau, void* out, float* part, uint32_t* status, cudaStream_t stream,
                       cudaEvent_t ev0, cudaEvent_t ev1, uint32_t* sparse_tiles = nullptr);

}  // namespace host

}  // namespace tq
