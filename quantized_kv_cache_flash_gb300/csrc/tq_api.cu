// Host side of the C ABI declared in include/tq.h: argument checks, codebook
// tables, sign vector, split planning, workspace, launches.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "tq.h"
#include "tq_internal.h"

namespace {

constexpr int kD = 128;

struct EventPair {
    cudaEvent_t a = nullptr, b = nullptr;
};

using tq::host::CodebookTables;

}  // namespace

namespace tq {
namespace host {

int cuda_err_code(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// splitmix64 (Steele, Lea, Flood 2014; the finaliser of Vigna's splitmix64.c)
uint64_t splitmix64_next(uint64_t& state) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void make_signs(uint64_t seed, uint32_t out[4]) {
    uint64_t st = seed;
    out[0] = out[1] = out[2] = out[3] = 0;
    for (int d = 0; d < kD; ++d) {
        const uint64_t v = splitmix64_next(st);
        if (v >> 63) out[d >> 5] |= 1u << (d & 31);
    }
}

uint16_t half_bits(float f) {
    __half h = __float2half_rn(f);
    uint16_t b;
    std::memcpy(&b, &h, 2);
    return b;
}

// A codebook must have 2^bits finite entries, strictly ascending, exactly
// symmetric (the sign-magnitude codes rely on c[j] == -c[n-1-j]).
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

// Build the prmt tables and exact decision thresholds of a checked codebook.
int build_tables(const float* cb, int n, int bits, CodebookTables* t) {
    if (t->valid && t->bits == bits && std::memcmp(t->cb, cb, n * sizeof(float)) == 0)
        return TQ_OK;
    const int h = n / 2;
    // magnitudes by rank: m[r] = cb[h + r]
    uint8_t lo[8] = {}, hi[8] = {};
    if (bits == 3) {
        // indexed by the 3-bit code kappa = sign<<2 | rank (sign 1 = negative)
        for (int k = 0; k < 8; ++k) {
            const int r = k & 3;
            const float v = (k & 4) ? -cb[h + r] : cb[h + r];
            const uint16_t hb = half_bits(v);
            lo[k] = hb & 0xFF;
            hi[k] = hb >> 8;
        }
    } else if (bits == 4) {
        // indexed by rank; the sign is applied in the kernel
        for (int r = 0; r < 8; ++r) {
            const uint16_t hb = half_bits(cb[h + r]);
            lo[r] = hb & 0xFF;
            hi[r] = hb >> 8;
        }
    } else {
        return TQ_ERR_UNSUPPORTED;
    }
    auto word = [](const uint8_t* b) {
        return uint32_t(b[0]) | (uint32_t(b[1]) << 8) | (uint32_t(b[2]) << 16) | (uint32_t(b[3]) << 24);
    };
    t->tab[0] = word(lo);
    t->tab[1] = word(lo + 4);
    t->tab[2] = word(hi);
    t->tab[3] = word(hi + 4);
    // the rounding residuals of the same 8 entries, exact in double, scaled
    // by 2^a so the largest lands in [128, 256) (e4m3 holds up to 448)
    double res[8];
    double rmax = 0.0;
    for (int k = 0; k < 8; ++k) {
        const double v = (bits == 3) ? ((k & 4) ? -double(cb[h + (k & 3)]) : double(cb[h + (k & 3)]))
                                     : double(cb[h + k]);
        res[k] = v - double(__half2float(__float2half_rn(float(v))));
        rmax = std::max(rmax, std::fabs(res[k]));
    }
    int e = 0;
    if (rmax > 0.0) (void)std::frexp(rmax, &e);
    t->res_shift = rmax > 0.0 ? 8 - e : 0;
    uint8_t r8[8];
    for (int k = 0; k < 8; ++k)
        r8[k] = static_cast<uint8_t>(
            __nv_cvt_double_to_fp8(std::ldexp(res[k], t->res_shift), __NV_SATFINITE, __NV_E4M3));
    t->tab8[0] = word(r8);
    t->tab8[1] = word(r8 + 4);
    // thresholds between positive neighbours: tau_k = (m[k] + m[k+1]) / 2 exactly
    for (int k = 0; k < 7; ++k) t->gt[k] = t->ge[k] = INFINITY;
    for (int k = 0; k + 1 < h; ++k) {
        const double tau = 0.5 * (double(cb[h + k]) + double(cb[h + k + 1]));
        const float f = float(tau);
        const float up = std::nextafter(f, INFINITY);
        if (double(f) > tau) { t->ge[k] = f; t->gt[k] = f; }
        else if (double(f) == tau) { t->ge[k] = f; t->gt[k] = up; }
        else { t->ge[k] = up; t->gt[k] = up; }
    }
    std::memcpy(t->cb, cb, n * sizeof(float));
    t->bits = bits;
    t->valid = true;
    return TQ_OK;
}

int check_cache(const tq_cache* c, int* kb, int* vb) {
    if (c == nullptr) return TQ_ERR_INVALID_ARG;
    int r = tq::mode_bits(c->mode, kb, vb);
    if (r != TQ_OK) return r;
    if (c->head_dim != kD) return TQ_ERR_UNSUPPORTED;
    if (c->batch <= 0 || c->num_kv_heads <= 0 || c->capacity <= 0 || (c->capacity % 16) != 0)
        return TQ_ERR_INVALID_ARG;
    const bool table = tq::mode_table(c->mode);  // table records: no norm arrays
    if (c->k_data == nullptr || c->v_data == nullptr || c->lengths == nullptr)
        return TQ_ERR_INVALID_ARG;
    if (!table && (c->v_norm == nullptr || (*kb != 16 && c->k_norm == nullptr)))
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(c->k_data) || !aligned16(c->v_data) || (c->v_norm && !aligned16(c->v_norm)) ||
        (c->k_norm && !aligned16(c->k_norm)))
        return TQ_ERR_INVALID_ARG;
    const long long rows = 1ll * c->batch * c->num_kv_heads * c->capacity;
    if (rows >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;
    if (*kb != 16 && (r = check_codebook(c->codebook_k, c->codebook_k_size, *kb)) != TQ_OK) return r;
    if ((r = check_codebook(c->codebook_v, c->codebook_v_size, *vb)) != TQ_OK) return r;
    return TQ_OK;
}

// The driver's tensor-map encoder, looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 get_encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool codebook_is_fp16(const float* cb, int n) {
    for (int j = 0; j < n; ++j)
        if (__half2float(__float2half_rn(cb[j])) != cb[j]) return false;
    return true;
}

// fp16 K rows [B*Hkv*cap, 128] as a 2-D tensor, boxes of 32 rows x 64 halves
// (128 bytes, 128-byte swizzle).
int encode_kmap(CUtensorMap* map, const tq_cache* c) {
    const uint64_t rows = uint64_t(c->batch) * c->num_kv_heads * c->capacity;
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_tiled();
    if (enc == nullptr) return TQ_ERR_CUDA;
    cuuint64_t dims[2] = {kD, rows};
    cuuint64_t strides[1] = {kD * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, c->k_data, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TQ_OK : TQ_ERR_CUDA;
}

int encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_tiled();
    if (enc == nullptr) return TQ_ERR_CUDA;
    cuuint64_t dims[2] = {kD, rows};
    cuuint64_t strides[1] = {kD * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TQ_OK : TQ_ERR_CUDA;
}

constexpr int kSMs = 152;  // GB300 (only used to size the split grid)
constexpr long long kMinChunks3 = 96;  // chunks per CTA below which a third wave does not pay

// Decode grid: waves of resident CTAs -- the later ones, placed wherever a
// CTA finished, even out SMs that run at different speeds, and shorter CTAs
// leave a shorter tail.  Groups of up to 8 rows: two waves, three when every
// CTA would still stream at least kMinChunks3 chunks (below that the extra
// CTAs' set-up and partials cost more than the tail saves); 16-row groups:
// one wave (their partials and query set-up are four times larger).  Fewer
// CTAs when the context (at the hint length) gives a CTA less than two
// 32-token chunks per warp.
int plan_ctas(int kb, int vb, bool table, bool res, int group_rows, long long units, int max_len) {
    const long long resident = kSMs * tq::decode_ctas_per_sm(kb, vb, group_rows, table, res);
    const long long chunks = units * ((max_len + 31) / 32);
    const long long waves = group_rows >= 16 ? 1 : (chunks >= 3 * kMinChunks3 * resident ? 3 : 2);
    const long long slots = waves * resident;
    long long ctas = std::min(slots, (chunks + 7) / 8);
    return int(std::max<long long>(ctas, 1));
}

int plan_decode(const tq_cache* c, const void* q, const void* out, int num_q_heads, int tq_rows,
                int max_len_hint, float scale, DecodePlan* pl) {
    int r = check_cache(c, &pl->kb, &pl->vb);
    if (r != TQ_OK) return r;
    if (q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (tq_rows <= 0 || max_len_hint <= 0 || max_len_hint > c->capacity) return TQ_ERR_INVALID_ARG;
    if (tq_rows > max_len_hint) return TQ_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
    if (!std::isfinite(c->v_rescale)) return TQ_ERR_INVALID_ARG;
    pl->group = num_q_heads / c->num_kv_heads;
    pl->rows = pl->group * tq_rows;
    if (pl->rows > 256) return TQ_ERR_UNSUPPORTED;
    pl->group_rows = tq::group_rows_for(pl->rows, pl->kb);
    pl->row_groups = (pl->rows + pl->group_rows - 1) / pl->group_rows;
    pl->units = 1ll * c->batch * c->num_kv_heads * pl->row_groups;
    pl->res = pl->kb != 16 && !tq::mode_table(c->mode) && !codebook_is_fp16(c->codebook_k, c->codebook_k_size);
    pl->ctas = plan_ctas(pl->kb, pl->vb, tq::mode_table(c->mode), pl->res, pl->group_rows, pl->units,
                         max_len_hint);
    return TQ_OK;
}

int launch_decode_plan(const DecodePlan& pl, const tq_cache* c, const CodebookTables& kt,
                       const CodebookTables& vt, const uint32_t signs[4], const CUtensorMap* kmap,
                       const void* q, int num_q_heads, int tq_rows, int max_len_hint, float scale,
                       float tau, void* out, float* part, uint32_t* status, cudaStream_t stream,
                       cudaEvent_t ev0, cudaEvent_t ev1, uint32_t* sparse_tiles) {
    if (tau > 0.f && sparse_tiles == nullptr) return TQ_ERR_INVALID_ARG;
    const size_t slots = decode_slots(pl);
    const float sc = (scale == 0.f) ? 1.0f / std::sqrt(float(kD)) : scale;
    tq::DecodeParams p{};
    p.k_codes = static_cast<const uint8_t*>(c->k_data);
    p.k_norm = static_cast<const __half*>(c->k_norm);
    p.v_codes = static_cast<const uint8_t*>(c->v_data);
    p.v_norm = static_cast<const __half*>(c->v_norm);
    p.lengths = c->lengths;
    p.q = static_cast<const __half*>(q);
    p.part_o = part;
    p.part_ml = part + slots * kD;
    p.status = status;
    p.batch = c->batch;
    p.hkv = c->num_kv_heads;
    p.hq = num_q_heads;
    p.group = pl.group;
    p.tq = tq_rows;
    p.rows = pl.rows;
    p.row_groups = pl.row_groups;
    p.group_rows = pl.group_rows;
    p.cap = c->capacity;
    p.max_len = max_len_hint;
    p.num_ctas = pl.ctas;
    p.scale_log2e = sc * 1.4426950408889634f;
    p.sparse_tau = tau;
    p.sparse_tiles = sparse_tiles;
    p.table = tq::mode_table(c->mode) ? 1 : 0;
    if (pl.kb != 16) {
        std::memcpy(p.ktab, kt.tab, sizeof(p.ktab));
        std::memcpy(p.ktab8, kt.tab8, sizeof(p.ktab8));
        p.res_shift = kt.res_shift;
        p.k_res = pl.res ? 1 : 0;
    }
    std::memcpy(p.vtab, vt.tab, sizeof(p.vtab));
    std::memcpy(p.signs, signs, sizeof(p.signs));
    CUtensorMap dummy;
    std::memset(&dummy, 0, sizeof(dummy));
    if (tq::launch_decode(pl.kb, pl.vb, p, pl.kb == 16 ? kmap : &dummy, stream, ev0, ev1) != 0)
        return TQ_ERR_CUDA;

    tq::CombineParams cp{};
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.lengths = c->lengths;
    cp.out = static_cast<__half*>(out);
    cp.status = status;
    cp.batch = c->batch;
    cp.hkv = c->num_kv_heads;
    cp.hq = num_q_heads;
    cp.group = pl.group;
    cp.tq = tq_rows;
    cp.row_groups = pl.row_groups;
    cp.group_rows = pl.group_rows;
    cp.max_len = max_len_hint;
    cp.num_ctas = pl.ctas;
    cp.v_rescale = c->v_rescale;
    std::memcpy(cp.signs, signs, sizeof(cp.signs));
    return cuda_err_code(static_cast<cudaError_t>(tq::launch_combine(cp, stream)));
}

}  // namespace host
}  // namespace tq

struct tq_ctx {
    int device = -1;
    uint32_t* d_words = nullptr;  // [0] status, [1] encode ticket counter, [2..3] sparse-V tiles, [4] encode tile counter
    float* d_work = nullptr;
    size_t work_bytes = 0;
    CodebookTables ktab, vtab;
    bool signs_valid = false;
    uint64_t seed = 0;
    uint32_t signs[4] = {};
    // tensor map of the fp16 K rows (rebuilt when the buffer or shape changes)
    CUtensorMap kmap;
    const void* kmap_ptr = nullptr;
    uint64_t kmap_rows = 0;
    bool timing = false;
    // stream of the most recent call that used this context (status reads
    // are ordered after it)
    cudaStream_t last_stream = nullptr;
    std::vector<EventPair> events;
    size_t events_used = 0;
};

namespace {

int cuda_err(cudaError_t e) { return tq::host::cuda_err_code(e); }
using tq::host::aligned16;
using tq::host::build_tables;
using tq::host::check_cache;
using tq::host::make_signs;

int get_ctx(tq_ctx** pctx, tq_ctx** out) {
    if (pctx == nullptr) return TQ_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (*pctx == nullptr) {
        tq_ctx* c = new (std::nothrow) tq_ctx();
        if (c == nullptr) return TQ_ERR_NOMEM;
        c->device = dev;
        if (cudaMalloc(&c->d_words, 64) != cudaSuccess) {
            delete c;
            return TQ_ERR_NOMEM;
        }
        if (cudaMemset(c->d_words, 0, 64) != cudaSuccess) {
            cudaFree(c->d_words);
            delete c;
            return TQ_ERR_CUDA;
        }
        *pctx = c;
    } else if ((*pctx)->device != dev) {
        return TQ_ERR_INVALID_ARG;
    }
    *out = *pctx;
    return TQ_OK;
}

int prepare_tables(tq_ctx* ctx, const tq_cache* c, int kb, int vb) {
    if (kb != 16) {
        int r = build_tables(c->codebook_k, c->codebook_k_size, kb, &ctx->ktab);
        if (r != TQ_OK) return r;
    }
    int r = build_tables(c->codebook_v, c->codebook_v_size, vb, &ctx->vtab);
    if (r != TQ_OK) return r;
    if (!ctx->signs_valid || ctx->seed != c->rot_seed) {
        make_signs(c->rot_seed, ctx->signs);
        ctx->seed = c->rot_seed;
        ctx->signs_valid = true;
    }
    return TQ_OK;
}

// The fp16 K tensor map, re-encoded when the buffer or its shape changes.
int prepare_kmap(tq_ctx* ctx, const tq_cache* c) {
    const uint64_t rows = uint64_t(c->batch) * c->num_kv_heads * c->capacity;
    if (ctx->kmap_ptr == c->k_data && ctx->kmap_rows == rows) return TQ_OK;
    const int r = tq::host::encode_kmap(&ctx->kmap, c);
    if (r != TQ_OK) return r;
    ctx->kmap_ptr = c->k_data;
    ctx->kmap_rows = rows;
    return TQ_OK;
}

// The event pair bracketing the next timed launch (none when timing is off).
int timing_events(tq_ctx* ctx, cudaEvent_t* e0, cudaEvent_t* e1) {
    *e0 = *e1 = nullptr;
    if (!ctx->timing) return TQ_OK;
    if (ctx->events_used == ctx->events.size()) {
        EventPair ep;
        if (cudaEventCreate(&ep.a) != cudaSuccess || cudaEventCreate(&ep.b) != cudaSuccess)
            return TQ_ERR_CUDA;
        ctx->events.push_back(ep);
    }
    *e0 = ctx->events[ctx->events_used].a;
    *e1 = ctx->events[ctx->events_used].b;
    ctx->events_used++;
    return TQ_OK;
}

int ensure_work(tq_ctx* ctx, size_t bytes) {
    if (ctx->work_bytes >= bytes) return TQ_OK;
    if (ctx->d_work) cudaFree(ctx->d_work);
    ctx->d_work = nullptr;
    ctx->work_bytes = 0;
    if (cudaMalloc(&ctx->d_work, bytes) != cudaSuccess) return TQ_ERR_NOMEM;
    ctx->work_bytes = bytes;
    return TQ_OK;
}

}  // namespace

extern "C" {

const char* tq_error_string(int32_t code) {
    switch (code) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case TQ_ERR_CAPACITY: return "capacity exceeded";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_NOMEM: return "out of device memory";
        default: return "unknown error";
    }
}

int tq_record_bytes(int32_t bits) {
    if (bits == 3) return 48;
    if (bits == 4) return 64;
    if (bits == 16) return 256;
    return TQ_ERR_UNSUPPORTED;
}

int tq_lloyd_max_codebook(int32_t bits, float* out) {
    if (out == nullptr) return TQ_ERR_INVALID_ARG;
    if (bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    const int n = 1 << bits;
    const double sigma = 1.0 / std::sqrt(double(kD));
    const double inv_sqrt2pi = 0.3989422804014327;
    double c[16], nc[16];
    for (int j = 0; j < n; ++j) c[j] = sigma * (-2.0 + 4.0 * j / (n - 1));
    // Lloyd iteration: cell boundaries at midpoints, each level at its cell's
    // conditional mean sigma * (phi(a) - phi(b)) / (Phi(b) - Phi(a)) in
    // standardised units.
    for (int it = 0; it < 200000; ++it) {
        double delta = 0.0;
        for (int j = 0; j < n; ++j) {
            const double a = (j == 0) ? -INFINITY : 0.5 * (c[j - 1] + c[j]) / sigma;
            const double b = (j == n - 1) ? INFINITY : 0.5 * (c[j] + c[j + 1]) / sigma;
            const double pa = std::isinf(a) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * a * a);
            const double pb = std::isinf(b) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * b * b);
            const double Pa = 0.5 * std::erfc(-a / std::sqrt(2.0));
            const double Pb = 0.5 * std::erfc(-b / std::sqrt(2.0));
            nc[j] = sigma * (pa - pb) / (Pb - Pa);
        }
        for (int j = 0; j < n; ++j) {
            delta = std::max(delta, std::fabs(nc[j] - c[j]));
            c[j] = nc[j];
        }
        if (delta < 1e-15) break;
    }
    // each level rounded to the nearest fp16 value (ties to the even one):
    // the candidates around the float-rounded value, compared exactly in double
    for (int j = 0; j < n; ++j) {
        const __half h0 = __float2half_rn(float(c[j]));
        uint16_t b0;
        std::memcpy(&b0, &h0, 2);
        double best_v = 0.0, best_d = INFINITY;
        uint16_t best_b = b0;
        for (int k = -1; k <= 1; ++k) {
            const uint16_t b = static_cast<uint16_t>(b0 + k);
            __half_raw raw;
            raw.x = b;
            const double v = double(__half2float(__half(raw)));
            if (!std::isfinite(v) || (v < 0) != (c[j] < 0)) continue;
            const double d = std::fabs(v - c[j]);
            if (d < best_d || (d == best_d && (b & 1u) == 0 && (best_b & 1u) != 0)) {
                best_d = d;
                best_v = v;
                best_b = b;
            }
        }
        out[j] = float(best_v);
    }
    return TQ_OK;
}

int tq_plan_splits(int32_t mode, int32_t batch, int32_t num_kv_heads, int32_t rows_per_kv_head,
                   int32_t max_len_hint, int32_t* split_tokens, int32_t* num_splits) {
    int kb, vb;
    if (tq::mode_bits(mode, &kb, &vb) != TQ_OK) return TQ_ERR_UNSUPPORTED;
    if (batch <= 0 || num_kv_heads <= 0 || rows_per_kv_head <= 0 || max_len_hint <= 0 ||
        split_tokens == nullptr || num_splits == nullptr)
        return TQ_ERR_INVALID_ARG;
    const int gr = tq::group_rows_for(rows_per_kv_head, kb);
    const long long units = 1ll * batch * num_kv_heads * ((rows_per_kv_head + gr - 1) / gr);
    const int ctas = tq::host::plan_ctas(kb, vb, tq::mode_table(mode), false, gr, units, max_len_hint);
    const long long chunks = units * ((max_len_hint + 31) / 32);
    *num_splits = ctas;
    *split_tokens = int(std::min<long long>((chunks + ctas - 1) / ctas * 32, 1ll << 30));
    return TQ_OK;
}

int tq_encode_append(tq_ctx** pctx, const tq_cache* c, const void* k_new, const void* v_new,
                     int32_t t_new, void* stream) {
    int kb, vb;
    int r = check_cache(c, &kb, &vb);
    if (r != TQ_OK) return r;
    if (t_new < 0) return TQ_ERR_INVALID_ARG;
    if (t_new == 0) return TQ_OK;
    if (k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new))
        return TQ_ERR_INVALID_ARG;
    if (t_new > c->capacity) return TQ_ERR_CAPACITY;
    tq_ctx* ctx;
    if ((r = get_ctx(pctx, &ctx)) != TQ_OK) return r;
    if ((r = prepare_tables(ctx, c, kb, vb)) != TQ_OK) return r;
    tq::EncodeParams p{};
    p.k_new = static_cast<const __half*>(k_new);
    p.v_new = static_cast<const __half*>(v_new);
    p.k_codes = static_cast<uint8_t*>(c->k_data);
    p.k_norm = static_cast<__half*>(c->k_norm);
    p.v_codes = static_cast<uint8_t*>(c->v_data);
    p.v_norm = static_cast<__half*>(c->v_norm);
    p.lengths = c->lengths;
    p.status = ctx->d_words;
    p.counter = ctx->d_words + 1;
    p.tiles_next = ctx->d_words + 4;
    p.batch = c->batch;
    p.hkv = c->num_kv_heads;
    p.t_new = t_new;
    p.cap = c->capacity;
    tq::div_magic(uint32_t(t_new), &p.div_t_m, &p.div_t_s);
    tq::div_magic(uint32_t(c->num_kv_heads), &p.div_h_m, &p.div_h_s);
    std::memcpy(p.signs, ctx->signs, sizeof(p.signs));
    if (kb != 16) {
        std::memcpy(p.k_gt, ctx->ktab.gt, sizeof(p.k_gt));
        std::memcpy(p.k_ge, ctx->ktab.ge, sizeof(p.k_ge));
    }
    std::memcpy(p.v_gt, ctx->vtab.gt, sizeof(p.v_gt));
    std::memcpy(p.v_ge, ctx->vtab.ge, sizeof(p.v_ge));
    if (tq::mode_table(c->mode)) {
        p.table = 1;
        std::memcpy(p.k_cb, c->codebook_k, sizeof(p.k_cb));
        std::memcpy(p.v_cb, c->codebook_v, sizeof(p.v_cb));
    }
    CUtensorMap kmap, vmap;
    const uint64_t nvec = uint64_t(c->batch) * c->num_kv_heads * t_new;
    if (nvec > uint64_t(tq::kEncodeSmallMax)) {
        if ((r = tq::host::encode_rows_map(&kmap, k_new, nvec)) != TQ_OK ||
            (r = tq::host::encode_rows_map(&vmap, v_new, nvec)) != TQ_OK)
            return r;
    }
    ctx->last_stream = static_cast<cudaStream_t>(stream);
    return cuda_err(static_cast<cudaError_t>(
        tq::launch_encode(kb, vb, p, &kmap, &vmap, static_cast<cudaStream_t>(stream))));
}

}  // extern "C"

namespace {

// Both decode entry points: tau = 0 is the plain decode, tau > 0 skips the V
// work of 16-token tiles whose softmax weights are all below tau.
int decode_impl(tq_ctx** pctx, const tq_cache* c, const void* q, int32_t num_q_heads,
                int32_t tq_rows, int32_t max_len_hint, float scale, float tau, void* out,
                void* stream) {
    tq::host::DecodePlan pl;
    int r = tq::host::plan_decode(c, q, out, num_q_heads, tq_rows, max_len_hint, scale, &pl);
    if (r != TQ_OK) return r;
    tq_ctx* ctx;
    if ((r = get_ctx(pctx, &ctx)) != TQ_OK) return r;
    if ((r = prepare_tables(ctx, c, pl.kb, pl.vb)) != TQ_OK) return r;
    if (pl.kb == 16 && (r = prepare_kmap(ctx, c)) != TQ_OK) return r;
    const size_t slots = tq::host::decode_slots(pl);
    if ((r = ensure_work(ctx, slots * (kD + 2) * sizeof(float))) != TQ_OK) return r;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((r = timing_events(ctx, &e0, &e1)) != TQ_OK) return r;
    ctx->last_stream = static_cast<cudaStream_t>(stream);
    return tq::host::launch_decode_plan(pl, c, ctx->ktab, ctx->vtab, ctx->signs, &ctx->kmap, q,
                                        num_q_heads, tq_rows, max_len_hint, scale, tau, out,
                                        ctx->d_work, ctx->d_words, static_cast<cudaStream_t>(stream),
                                        e0, e1, ctx->d_words + 2);
}

}  // namespace

extern "C" {

int tq_decode_attention(tq_ctx** pctx, const tq_cache* c, const void* q, int32_t num_q_heads,
                        int32_t tq_rows, int32_t max_len_hint, float scale, void* out, void* stream) {
    return decode_impl(pctx, c, q, num_q_heads, tq_rows, max_len_hint, scale, 0.f, out, stream);
}

int tq_decode_attention_sparse_v(tq_ctx** pctx, const tq_cache* c, const void* q,
                                 int32_t num_q_heads, int32_t tq_rows, int32_t max_len_hint,
                                 float scale, float tau, void* out, void* stream) {
    if (!(tau >= 0.f) || !std::isfinite(tau)) return TQ_ERR_INVALID_ARG;
    return decode_impl(pctx, c, q, num_q_heads, tq_rows, max_len_hint, scale, tau, out, stream);
}

int tq_prefill_attention(tq_ctx** pctx, const tq_cache* c, const void* q, int32_t num_q_heads,
                         int32_t tq_rows, int32_t max_len_hint, float scale, void* out,
                         void* stream) {
    int kb, vb;
    int r = check_cache(c, &kb, &vb);
    if (r != TQ_OK) return r;
    if (tq::mode_table(c->mode)) return TQ_ERR_UNSUPPORTED;
    // the prefill K tile holds fp16 centroids: exact only for fp16 levels
    if (kb != 16 && !tq::host::codebook_is_fp16(c->codebook_k, c->codebook_k_size)) return TQ_ERR_UNSUPPORTED;
    if (q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (tq_rows <= 0 || max_len_hint <= 0 || max_len_hint > c->capacity) return TQ_ERR_INVALID_ARG;
    if (tq_rows > max_len_hint) return TQ_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
    if (!std::isfinite(c->v_rescale)) return TQ_ERR_INVALID_ARG;
    const int group = num_q_heads / c->num_kv_heads;
    if (group > 128) return TQ_ERR_UNSUPPORTED;
    const long long units = 1ll * c->batch * c->num_kv_heads;
    if (units > 65535) return TQ_ERR_UNSUPPORTED;
    const int pos_per_tile = 128 / group;
    const long long mtiles = (tq_rows + pos_per_tile - 1) / pos_per_tile;
    tq_ctx* ctx;
    if ((r = get_ctx(pctx, &ctx)) != TQ_OK) return r;
    if ((r = prepare_tables(ctx, c, kb, vb)) != TQ_OK) return r;
    if (kb == 16 && (r = prepare_kmap(ctx, c)) != TQ_OK) return r;

    tq::PrefillParams p{};
    p.k_codes = static_cast<const uint8_t*>(c->k_data);
    p.k_norm = static_cast<const __half*>(c->k_norm);
    p.v_codes = static_cast<const uint8_t*>(c->v_data);
    p.v_norm = static_cast<const __half*>(c->v_norm);
    p.lengths = c->lengths;
    p.q = static_cast<const __half*>(q);
    p.out = static_cast<__half*>(out);
    p.status = ctx->d_words;
    p.batch = c->batch;
    p.hkv = c->num_kv_heads;
    p.hq = num_q_heads;
    p.group = group;
    p.tq = tq_rows;
    p.cap = c->capacity;
    p.max_len = max_len_hint;
    p.pos_per_tile = pos_per_tile;
    p.mtiles = int(mtiles);
    const float sc = (scale == 0.f) ? 1.0f / std::sqrt(float(kD)) : scale;
    p.scale_log2e = sc * 1.4426950408889634f;
    p.v_rescale = c->v_rescale;
    if (kb != 16) std::memcpy(p.ktab, ctx->ktab.tab, sizeof(p.ktab));
    std::memcpy(p.vtab, ctx->vtab.tab, sizeof(p.vtab));
    std::memcpy(p.signs, ctx->signs, sizeof(p.signs));
    CUtensorMap dummy;
    std::memset(&dummy, 0, sizeof(dummy));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ctx->last_stream = s;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((r = timing_events(ctx, &e0, &e1)) != TQ_OK) return r;
    if (e0) cudaEventRecord(e0, s);
    r = tq::launch_prefill(kb, vb, p, kb == 16 ? &ctx->kmap : &dummy, s);
    if (e1) cudaEventRecord(e1, s);
    return r == 0 ? TQ_OK : TQ_ERR_CUDA;
}

int tq_selftest_bounded_wait(tq_ctx** pctx, int32_t limit_us, void* stream) {
    if (pctx == nullptr || limit_us < 1 || limit_us > 1000000) return TQ_ERR_INVALID_ARG;
    tq_ctx* ctx;
    int r = get_ctx(pctx, &ctx);
    if (r != TQ_OK) return r;
    ctx->last_stream = static_cast<cudaStream_t>(stream);
    return cuda_err(static_cast<cudaError_t>(tq::launch_selftest_stall(
        ctx->d_words, uint64_t(limit_us) * 1000ull, static_cast<cudaStream_t>(stream))));
}

void tq_free(tq_ctx* ctx) {
    if (ctx == nullptr) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    for (auto& e : ctx->events) {
        if (e.a) cudaEventDestroy(e.a);
        if (e.b) cudaEventDestroy(e.b);
    }
    if (ctx->d_work) cudaFree(ctx->d_work);
    if (ctx->d_words) cudaFree(ctx->d_words);
    cudaSetDevice(prev);
    delete ctx;
}

int tq_get_status(tq_ctx* ctx, uint32_t* status) {
    if (status == nullptr) return TQ_ERR_INVALID_ARG;
    *status = 0;
    if (ctx == nullptr) return TQ_OK;
    // read and clear the word on the stream of the context's latest call, and
    // wait for that stream only (other streams and devices keep running)
    const cudaStream_t s = ctx->last_stream;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ctx->d_words, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaMemsetAsync(ctx->d_words, 0, 4, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
    *status = v;
    return TQ_OK;
}

int tq_get_sparse_v_tiles(tq_ctx* ctx, uint64_t* skipped, uint64_t* judged) {
    if (ctx == nullptr || skipped == nullptr || judged == nullptr) return TQ_ERR_INVALID_ARG;
    const cudaStream_t s = ctx->last_stream;
    uint32_t v[2] = {0, 0};
    if (cudaMemcpyAsync(v, ctx->d_words + 2, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaMemsetAsync(ctx->d_words + 2, 0, 8, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
    *skipped = v[0];
    *judged = v[1];
    return TQ_OK;
}

int tq_set_kernel_timing(tq_ctx* ctx, int32_t enable) {
    if (ctx == nullptr) return TQ_ERR_INVALID_ARG;
    ctx->timing = enable != 0;
    return TQ_OK;
}

int tq_get_kernel_time(tq_ctx* ctx, float* ms_total, int32_t* launches) {
    if (ctx == nullptr || ms_total == nullptr || launches == nullptr) return TQ_ERR_INVALID_ARG;
    float total = 0.f;
    for (size_t i = 0; i < ctx->events_used; ++i) {
        if (cudaEventSynchronize(ctx->events[i].b) != cudaSuccess) return TQ_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, ctx->events[i].a, ctx->events[i].b) != cudaSuccess)
            return TQ_ERR_CUDA;
        total += ms;
    }
    *ms_total = total;
    *launches = int32_t(ctx->events_used);
    ctx->events_used = 0;
    return TQ_OK;
}

}  // extern "C"
