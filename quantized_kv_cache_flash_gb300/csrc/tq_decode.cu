// Fused split-K decode attention over the packed KV cache, and the split
// combine + inverse-rotation epilogue.
//
// Scores are taken in the rotated basis: score(t) = scale * n_k(t) *
// <Rot(q), c[idx_k(t)]> for quantized K (Rot is orthogonal, so this equals the
// score against the fully dequantized key), or scale * <q, k(t)> for fp16 K.
// V is never brought back to the original basis: P.V accumulates
// p(t) * n_v(t) * c[idx_v(t)] and only the [rows, 128] result is
// inverse-rotated, in the combine kernel (mlxcel pull request #369, Change:
// the per-token inverse transform of a full V dequant is avoided by rotating
// the small output back instead).
//
// Work split: two waves of CTAs, each taking an equal share of the context's
// 32-token chunks over all (batch, kv head, row group) units.  A CTA's 4 warps
// stream their own chunks through private rings of shared-memory stages
// filled by 1-D bulk copies (tensor-map tile copies with 128-byte swizzle for
// fp16 K), dequantize in registers and run both contractions as warp MMAs
// with the 16 tokens of a tile as M and up to 8 query rows per n-tile as N.
#include <float.h>

#include <type_traits>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kChunkTokens = 32;  // tokens per warp pipeline stage (2 MMA tiles)

// TAB: 3-bit records that carry their own centroid x norm table (48 bytes of
// codes + 8 fp16 values c_j * n, 64 bytes, no norm array).
template <int KB, int VB, int NT, bool TAB = false>
struct DecCfg {
    static constexpr int kWarps = 4;
    static constexpr int kChunk = kChunkTokens;
    static constexpr int kStages = (KB == 0 || NT == 1) ? 2 : 3;
    static constexpr int kRows = 8 * NT;                    // query rows per row group
    static constexpr int kMinCtas = (NT == 1) ? 4 : 3;      // resident CTAs per SM targeted
    static constexpr int kRbK = TAB ? 64 : (KB == 0) ? 256 : KB * 16;  // bytes per K record
    static constexpr int kRbV = TAB ? 64 : VB * 16;
    static constexpr int kQuarterK = TAB ? 12 : kRbK / 4;   // a thread's 32 dims of codes
    static constexpr int kQuarterV = TAB ? 12 : kRbV / 4;
    static constexpr int kKBytes = kChunk * kRbK;
    static constexpr int kVOff = kKBytes;
    static constexpr int kVBytes = kChunk * kRbV;
    static constexpr int kKnOff = kVOff + kVBytes;
    static constexpr int kKnBytes = (KB == 0 || TAB) ? 0 : kChunk * 2;
    static constexpr int kVnOff = kKnOff + kKnBytes;
    static constexpr int kStageRaw = kVnOff + (TAB ? 0 : kChunk * 2);
    static constexpr int kStageAlign = (KB == 0) ? 1024 : 128;
    static constexpr int kStage = (kStageRaw + kStageAlign - 1) / kStageAlign * kStageAlign;
    static constexpr int kPipeBytes = kWarps * kStages * kStage;
    // fp16 query rows in MMA k order, [kRows][kQStride]: the 16-byte pad staggers
    // the rows over the banks for ldmatrix
    static constexpr int kQStride = kD + 8;
    static constexpr int kQOff = kPipeBytes;
    static constexpr int kBarOff = kQOff + kRows * kQStride * 2;
    static constexpr int kScanOff = (kBarOff + kWarps * kStages * 8 + 15) / 16 * 16;
    static constexpr int kSmem = kScanOff + kWarps * 4 * 32 * 4;  // per-warp batch scan
    static constexpr int kSmemAlloc = kSmem + 1024;          // base alignment slack
    // epilogue scratch (reuses the pipeline): per warp O[kRows][kOStride] + (m, l)[kRows]
    static constexpr int kOStride = kD + 4;
    static_assert(kWarps * kRows * kOStride * 4 + kWarps * kRows * 8 <= kPipeBytes, "scratch");
};

// A thread's quarter of a record (32 dims): 16 bytes of 4-bit codes or 12
// bytes of 3-bit codes (w[3] unused).
struct QuarterWords {
    uint32_t w[4];
};

template <int KB>
__device__ __forceinline__ QuarterWords load_quarter(const uint8_t* rec) {
    QuarterWords q;
    if constexpr (KB == 3) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(rec);
        q.w[0] = w[0]; q.w[1] = w[1]; q.w[2] = w[2]; q.w[3] = 0u;
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(rec);
        q.w[0] = v.x; q.w[1] = v.y; q.w[2] = v.z; q.w[3] = v.w;
    }
    return q;
}

// Group J (0..3) of a quarter: dim pairs 4J..4J+3 as four half2, the pairs
// the whole-quarter dequantisers put in h[4J..4J+3].  Decoding a group at a
// time lets each group's MMAs follow it, so only one group is live.
template <int KB, int J>
__device__ __forceinline__ void dequant_group(const QuarterWords& q, const Tables& t,
                                              uint32_t (&h)[4]) {
    if constexpr (KB == 3) {
        uint32_t m;
        if constexpr (J < 3) {
            m = q.w[J] & 0x77777777u;
        } else {  // the spare bits: bit k of the codes of dims 24..31 (see dequant3_quarter)
            m = (__umulhi(q.w[0], 1u << 29) & 0x11111111u) | (__umulhi(q.w[1], 1u << 30) & 0x22222222u) |
                (__umulhi(q.w[2], 1u << 31) & 0x44444444u);
        }
        lut4(m, t, h[0], h[1]);
        lut4(__umulhi(m, 1u << 16), t, h[2], h[3]);
    } else {
        dequant4_word(q.w[J], t, h[0], h[1], h[2], h[3]);
    }
}

// Work split (token-balanced): the (batch, kv head, row group) units
// are laid end to end as 32-token chunks, unit u holding ceil(min(len_b,
// max_len) / 32) chunks of batch b; CTA c of P takes the global chunks
// [c*C/P, (c+1)*C/P) of the C in total, so every CTA streams the same number
// of bytes whatever the length mix.  A CTA's range can cover the end of one
// unit and the start of the next: it writes one partial per unit it touches,
// into slot c + u (unique: a later CTA never touches an earlier unit).
__device__ __forceinline__ int unit_chunks(const int32_t* lengths, int b, int max_len) {
    const int L = min(lengths[b], max_len);
    return L > 0 ? (L + kChunkTokens - 1) / kChunkTokens : 0;
}

// Chunk bookkeeping over the batch, warp-parallel and warp-uniform in its
// results.  Lane i holds batch i of the first 32 (its length, its chunks over
// all per_b units, and the inclusive prefix of those): for batches of up to 32
// sequences one load of `lengths` per lane serves the whole kernel; larger
// batches rescan global memory block by block.  Chunk counts stay below 2^30
// (cache rows < 2^31, at most 16 row groups).
struct BatchScan {
    int* s;  // this warp's copy in shared memory: len, nch, v, inc, 32 ints each

    __device__ __forceinline__ void init(int* smem_scan, const int32_t* lengths, int batch,
                                         int per_b, int max_len, int lane) {
        s = smem_scan;
        const int len = lane < batch ? lengths[lane] : 0;
        const int nch = lane < batch ? unit_chunks(lengths, lane, max_len) : 0;
        const int v = nch * per_b;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        s[lane] = len;
        s[32 + lane] = nch;
        s[64 + lane] = v;
        s[96 + lane] = inc;
        __syncwarp();
    }

    __device__ __forceinline__ int total(const int32_t* lengths, int batch, int per_b, int max_len,
                                         int lane) const {
        const int first = s[96 + 31];  // the first 32 batches
        int sum = 0;
        for (int b = 32 + lane; b < batch; b += 32) sum += unit_chunks(lengths, b, max_len) * per_b;
        if (batch > 32) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        return first + sum;
    }

    // batch b holding global chunk pos, the chunks of all batches before it,
    // b's length and chunks per unit
    __device__ __forceinline__ void locate(const int32_t* lengths, int batch, int per_b, int max_len,
                                           int pos, int lane, int& b, int& before, int& L,
                                           int& nchunk) const {
        unsigned hit = __ballot_sync(0xffffffffu, s[96 + lane] > pos && lane < batch);
        if (hit) {
            const int l = __ffs(hit) - 1;
            b = l;
            before = s[96 + l] - s[64 + l];
            L = s[l];
            nchunk = s[32 + l];
            return;
        }
        int cum = s[96 + 31];
        for (int base = 32; base < batch; base += 32) {
            const int bb = base + lane;
            const int n = bb < batch ? unit_chunks(lengths, bb, max_len) : 0;
            const int w = n * per_b;
            int c = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, c, o);
                if (lane >= o) c += y;
            }
            hit = __ballot_sync(0xffffffffu, bb < batch && cum + c > pos);
            if (hit) {
                const int l = __ffs(hit) - 1;
                b = base + l;
                before = cum + __shfl_sync(0xffffffffu, c - w, l);
                L = lengths[b];
                nchunk = __shfl_sync(0xffffffffu, n, l);
                return;
            }
            cum += __shfl_sync(0xffffffffu, c, 31);
        }
        b = batch;  // pos past the end (not reached by the callers)
        before = cum;
        L = 0;
        nchunk = 0;
    }
};

// prmt byte tables (indexed by the 3-bit code kappa = sign << 2 | rank) from a
// record's 8 fp16 values t_0..t_7 in ascending index order: code kappa < 4 is
// index 4 + kappa, code 4 + r is index 3 - r.
__device__ __forceinline__ Tables record_tables(const uint8_t* tab16) {
    const uint4 w = *reinterpret_cast<const uint4*>(tab16);
    return Tables{prmt(w.z, w.w, 0x6420u), prmt(w.x, w.y, 0x0246u), prmt(w.z, w.w, 0x7531u),
                  prmt(w.x, w.y, 0x1357u)};
}

// V tables of a table record.  Stage slots past the end of the context hold
// stale bytes whose table could decode to inf or NaN, and a zero weight times
// inf is NaN in the MMA, so those tokens get an all-zero table.
template <bool FULL>
__device__ __forceinline__ Tables v_tables(const uint8_t* rec, bool valid) {
    if (FULL || valid) return record_tables(rec + 48);
    return Tables{0u, 0u, 0u, 0u};
}

// One CTA: 4 warps over this CTA's chunk range, one unit segment at a time.
// Per 16-token tile a warp runs
//   S^T[16 tok x 8 rows]  = C_k[16 x 128] . Rot(q)^T      (8 k-steps per row tile)
//   O^T[128 x 8 rows]    += C_v^T[128 x 16 tok] . (P n_v)^T (8 dim tiles)
// with the tokens (M = 16) dequantised in registers: a thread owns tokens g and
// g+8 of the tile and decodes its quarter t (32 dims) of both records.
template <int KB, int VB, int NT, bool TAB>
__global__ void __launch_bounds__(128, DecCfg<KB, VB, NT, TAB>::kMinCtas)
    tq_decode_kernel(const __grid_constant__ DecodeParams p,
                     const __grid_constant__ CUtensorMap kmap) {
    using C = DecCfg<KB, VB, NT, TAB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived from smem_raw by an integer offset so the
    // compiler keeps every access in the shared window (LDS, not generic loads)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    // warp index through a shuffle so the compiler treats it (and the chunk,
    // stage and copy addresses derived from it) as warp-uniform
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    griddep_wait();  // lengths, cache and q come from earlier work on the stream
    const int per_b = p.hkv * p.row_groups;
    BatchScan scan;
    scan.init(reinterpret_cast<int*>(smem + C::kScanOff) + warp * 128, p.lengths, p.batch, per_b,
              p.max_len, lane);
    // (each value the copies and masks derive from goes through a lane-0
    // shuffle, which lets the compiler keep them in uniform registers)
    const int C_all = __shfl_sync(0xffffffffu, scan.total(p.lengths, p.batch, per_b, p.max_len, lane), 0);
    // floor(c * C_all / P) in 32-bit arithmetic: c * (C_all mod P) < P^2 < 2^31
    const int P = static_cast<int>(gridDim.x), cq = C_all / P, cr = C_all - cq * P;
    const int c_me = static_cast<int>(blockIdx.x);
    const int lo = c_me * cq + (c_me * cr) / P;
    const int hi = (c_me + 1) * cq + ((c_me + 1) * cr) / P;
    if (lo >= hi) return;  // no chunks for this CTA (uniform over the CTA)

    uint8_t* wpipe = smem + warp * C::kStages * C::kStage;
    const uint32_t bar0 = smem_u32(smem + C::kBarOff) + warp * C::kStages * 8;
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
    }
    __syncwarp();
    __half* sQ = reinterpret_cast<__half*>(smem + C::kQOff);
    const uint32_t q_lds = smem_u32(sQ) + ((lane & 7) * C::kQStride + 8 * (lane >> 3)) * 2;
    const Tables kt{p.ktab[0], p.ktab[1], p.ktab[2], p.ktab[3]};
    const Tables vt{p.vtab[0], p.vtab[1], p.vtab[2], p.vtab[3]};
    const bool sparse = p.sparse_tau > 0.f;

    // the copy ring continues across segments: every copy issued in a segment
    // is consumed in it, so (stage, phase) carry over
    int stage = 0;
    uint32_t phase = 0;
    int pos = lo;
    while (pos < hi) {
        int b, before, L, nch;
        scan.locate(p.lengths, p.batch, per_b, p.max_len, pos, lane, b, before, L, nch);
        b = __shfl_sync(0xffffffffu, b, 0);
        before = __shfl_sync(0xffffffffu, before, 0);
        L = __shfl_sync(0xffffffffu, L, 0);
        nch = __shfl_sync(0xffffffffu, nch, 0);
        const int local = pos - before;
        const int ui = local / nch;  // h * row_groups + rg
        const int k0 = local - ui * nch;
        const int k1 = min(nch, k0 + (hi - pos));
        const int h = ui / p.row_groups, rg = ui - h * p.row_groups;
        const int unit = b * per_b + ui;  // global unit index, row group included
        const int t_lim = min(L, p.max_len);
        const int t_begin = k0 * C::kChunk;
        const int t_end = min(k1 * C::kChunk, t_lim);
        const int nchunks = k1 - k0;
        const size_t row0 = static_cast<size_t>(b * p.hkv + h) * p.cap;

        auto issue = [&](int c, int st_idx) {  // lane 0 only
            const int tok0 = t_begin + c * C::kChunk;
            const int nval = min(C::kChunk, t_end - tok0);
            const uint32_t dst = smem_u32(wpipe + st_idx * C::kStage);
            const uint32_t bar = bar0 + st_idx * 8;
            const uint32_t nb = static_cast<uint32_t>((nval + 7) & ~7) * 2;  // norms, 16-B multiple
            uint32_t bytes = nval * C::kRbV + (TAB ? 0u : nb);
            if (KB == 0) bytes += 2 * 4096;
            else bytes += nval * C::kRbK + (TAB ? 0u : nb);
            mbar_arrive_expect_tx(bar, bytes);
            if constexpr (KB == 0) {
                tma_g2s_2d(dst, &kmap, 0, static_cast<int32_t>(row0 + tok0), bar);
                tma_g2s_2d(dst + 4096, &kmap, 64, static_cast<int32_t>(row0 + tok0), bar);
            } else {
                bulk_g2s(dst, p.k_codes + (row0 + tok0) * C::kRbK, nval * C::kRbK, bar);
                if (!TAB) bulk_g2s(dst + C::kKnOff, p.k_norm + row0 + tok0, nb, bar);
            }
            bulk_g2s(dst + C::kVOff, p.v_codes + (row0 + tok0) * C::kRbV, nval * C::kRbV, bar);
            if (!TAB) bulk_g2s(dst + C::kVnOff, p.v_norm + row0 + tok0, nb, bar);
        };

        if (lane == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                const int c = warp + C::kWarps * s;
                int si = stage + s;
                if (si >= C::kStages) si -= C::kStages;
                if (c < nchunks) issue(c, si);
            }
        }
        __syncwarp();

        // ---- query rows of this row group -> shared (rotated for quantized K) ----
        const int rbase = rg * C::kRows;
        for (int r = warp; r < C::kRows; r += C::kWarps) {
            const int rr = rbase + r;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (rr < p.rows) {
                const int hl = rr / p.tq, j = rr - hl * p.tq;
                const __half* qp =
                    p.q + ((static_cast<size_t>(b) * p.hq + h * p.group + hl) * p.tq + j) * kD + lane * 4;
                const uint2 raw = *reinterpret_cast<const uint2*>(qp);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
                v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
                if constexpr (KB != 0) {
                    const uint32_t sn = sign_nibble(p.signs, lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = ((sn >> i) & 1u) ? -v[i] : v[i];
                    wht128_lane4(v, lane);
                    const float inv = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] *= inv;
                }
            }
            // Row r in the k order of the score MMA's B operand (k = head dims,
            // n = query rows).  Quantized K: a thread's A operand is its tokens'
            // quarter `t` in order, so k-index 16*kc + 8*hi + 2*t + e holds dim
            // 32*t + 4*kc + 2*hi + e; this lane's dims 4*lane + 2*hi + e sit at
            // k = 16*(lane & 7) + 8*hi + 2*(lane >> 3) + e.  fp16 K: k = dim.
            __half* qrow = sQ + r * C::kQStride;
            const uint32_t lo = pack_half2(v[0], v[1]), hi = pack_half2(v[2], v[3]);
            if constexpr (KB != 0) {
                const int k0 = 16 * (lane & 7) + 2 * (lane >> 3);
                *reinterpret_cast<uint32_t*>(qrow + k0) = lo;
                *reinterpret_cast<uint32_t*>(qrow + k0 + 8) = hi;
            } else {
                *reinterpret_cast<uint2*>(qrow + 4 * lane) = make_uint2(lo, hi);
            }
        }
        __syncthreads();

        // B fragments of k-steps 2*kc2 and 2*kc2 + 1 for row tile n (ldmatrix
        // matrix j = lane >> 3 covers k in [32*kc2 + 8*j, +8) of rows 8n..8n+7)
        auto load_qb = [&](int n, int kc2, uint32_t (&b)[4]) {
            ldsm_x4(q_lds + (8 * n * C::kQStride + 32 * kc2) * 2, b[0], b[1], b[2], b[3]);
        };

        // last visible token (inclusive) of the rows 8n + 2t + e this thread owns
        int lim[NT][2];
        bool row_ok[NT][2];  // real query rows (not padding of the group)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                lim[n][e] = L - p.tq + ((rbase + 8 * n + 2 * t + e) % p.tq);
                row_ok[n][e] = rbase + 8 * n + 2 * t + e < p.rows;
            }
        const int all_visible_below = L - p.tq + 1;  // tokens below this are seen by every row

        float O[NT][8][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 8; ++i) O[n][i][0] = O[n][i][1] = O[n][i][2] = O[n][i][3] = 0.f;
        // running max m, sum l, exp2 base bs (m, or 0 before the first score)
        // and growth threshold thr of the rows this thread owns
        constexpr float kSlack = 4.f;
        float m[NT][2], l[NT][2], bs[NT][2], thr[NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) m[n][e] = thr[n][e] = -INFINITY, l[n][e] = bs[n][e] = 0.f;
        bool stalled = false;

        // One 32-token chunk of this warp.  FULL: all 32 tokens valid and visible
        // to every row (no masking); otherwise the tail / causal path.
        auto process = [&](const uint8_t* st, const int tok0, auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const int nvalid = FULL ? C::kChunk : min(C::kChunk, t_end - tok0);
            const bool two = FULL || nvalid > 16;
                // ---------------- scores S^T = C_k . Rot(q)^T ----------------
                float x[2][NT][4];
        #pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
        #pragma unroll
                    for (int n = 0; n < NT; ++n) x[tile][n][0] = x[tile][n][1] = x[tile][n][2] = x[tile][n][3] = 0.f;
                    if (!FULL && tile == 1 && !two) break;
                    if constexpr (KB == 0) {
                        const int mi = lane >> 3;
                        const int row = tile * 16 + (mi & 1) * 8 + (lane & 7);
        #pragma unroll
                        for (int kc2 = 0; kc2 < 4; ++kc2) {
                            uint32_t qb[NT][4];
        #pragma unroll
                            for (int n = 0; n < NT; ++n) load_qb(n, kc2, qb[n]);
        #pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const int db = 4 * kc2 + 2 * kk + (mi >> 1);  // 16-byte chunk 0..15 of the row
                                const uint32_t addr = smem_u32(st) + (db >> 3) * 4096 + row * 128 +
                                                      (((db & 7) ^ (row & 7)) << 4);
                                uint32_t a0, a1, a2, a3;
                                ldsm_x4(addr, a0, a1, a2, a3);
        #pragma unroll
                                for (int n = 0; n < NT; ++n)
                                    mma_f16(x[tile][n], a0, a1, a2, a3, qb[n][2 * kk], qb[n][2 * kk + 1]);
                            }
                        }
                    } else {
                        // A quad of k-step kc: (token g, pair 2kc), (token g+8, pair 2kc),
                        // (token g, pair 2kc+1), (token g+8, pair 2kc+1) of the quarters;
                        // group J of both tokens feeds k-steps 2J and 2J+1
                        const uint8_t* ra = st + (tile * 16 + g) * C::kRbK;
                        const uint8_t* rb = st + (tile * 16 + g + 8) * C::kRbK;
                        const QuarterWords wa = load_quarter<KB>(ra + t * C::kQuarterK);
                        const QuarterWords wb = load_quarter<KB>(rb + t * C::kQuarterK);
                        const Tables ta = TAB ? record_tables(ra + 48) : kt;
                        const Tables tb = TAB ? record_tables(rb + 48) : kt;
                        auto kgroup = [&](auto jtag) {
                            constexpr int J = decltype(jtag)::value;
                            uint32_t ha[4], hb[4];
                            dequant_group<KB, J>(wa, ta, ha);
                            dequant_group<KB, J>(wb, tb, hb);
                            uint32_t qb[NT][4];
        #pragma unroll
                            for (int n = 0; n < NT; ++n) load_qb(n, J, qb[n]);
        #pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                mma_f16(x[tile][n], ha[0], hb[0], ha[1], hb[1], qb[n][0], qb[n][1]);
                                mma_f16(x[tile][n], ha[2], hb[2], ha[3], hb[3], qb[n][2], qb[n][3]);
                            }
                        };
                        kgroup(std::integral_constant<int, 0>{});
                        kgroup(std::integral_constant<int, 1>{});
                        kgroup(std::integral_constant<int, 2>{});
                        kgroup(std::integral_constant<int, 3>{});
                    }
                }

                // ---------------- online softmax (log2 domain) ----------------
                // thread's tokens: tile*16 + g (c0, c1) and tile*16 + g + 8 (c2, c3);
                // rows 8n + 2t (c0, c2) and 8n + 2t + 1 (c1, c3)
                float nv[2][2];
        #pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    const int ta = tile * 16 + g, tb = ta + 8;
                    float ka = p.scale_log2e, kb2 = p.scale_log2e;
                    if constexpr (KB != 0 && !TAB) {  // table records carry the norm in their values
                        ka *= __half2float(*reinterpret_cast<const __half*>(st + C::kKnOff + 2 * ta));
                        kb2 *= __half2float(*reinterpret_cast<const __half*>(st + C::kKnOff + 2 * tb));
                    }
                    if constexpr (TAB) {
                        nv[tile][0] = nv[tile][1] = 1.f;
                    } else {
                        nv[tile][0] = __half2float(*reinterpret_cast<const __half*>(st + C::kVnOff + 2 * ta));
                        nv[tile][1] = __half2float(*reinterpret_cast<const __half*>(st + C::kVnOff + 2 * tb));
                    }
                    // scaled score minus the row's exp2 base, one FFMA each
        #pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        x[tile][n][0] = fmaf(x[tile][n][0], ka, -bs[n][0]);
                        x[tile][n][1] = fmaf(x[tile][n][1], ka, -bs[n][1]);
                        x[tile][n][2] = fmaf(x[tile][n][2], kb2, -bs[n][0]);
                        x[tile][n][3] = fmaf(x[tile][n][3], kb2, -bs[n][1]);
                    }
                    if constexpr (!FULL) {
                        const int ga = tok0 + ta, gb = tok0 + tb;
                        const bool va = ga < t_end && (tile == 0 || two);
                        const bool vb = gb < t_end && (tile == 0 || two);
        #pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            x[tile][n][0] = (va && ga <= lim[n][0]) ? x[tile][n][0] : -INFINITY;
                            x[tile][n][1] = (va && ga <= lim[n][1]) ? x[tile][n][1] : -INFINITY;
                            x[tile][n][2] = (vb && gb <= lim[n][0]) ? x[tile][n][2] : -INFINITY;
                            x[tile][n][3] = (vb && gb <= lim[n][1]) ? x[tile][n][3] : -INFINITY;
                        }
                        if (!va) nv[tile][0] = 0.f;
                        if (!vb) nv[tile][1] = 0.f;
                    }
                }
                // The exp2 base of a row stays at its running max until a score exceeds
                // it by more than kSlack (log2 units); only then (warp-uniform slow
                // path) is the true max taken, O and l rescaled and the scores moved
                // to the new base.  So p <= 2^kSlack.  A row with no score yet has
                // base 0 and threshold -inf: its first finite score sets the max.
                bool grow = false;
        #pragma unroll
                for (int n = 0; n < NT; ++n)
        #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float mx = fmaxf(fmaxf(x[0][n][e], x[0][n][e + 2]), fmaxf(x[1][n][e], x[1][n][e + 2]));
                        grow |= mx > thr[n][e];
                    }
                if (__any_sync(0xffffffffu, grow)) {
        #pragma unroll
                    for (int n = 0; n < NT; ++n)
        #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float mx = fmaxf(fmaxf(x[0][n][e], x[0][n][e + 2]), fmaxf(x[1][n][e], x[1][n][e + 2]));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                            const float mn = fmaxf(m[n][e], mx + bs[n][e]);
                            const float al = (m[n][e] == -INFINITY) ? 0.f : fast_exp2(m[n][e] - mn);
                            const float nb = (mn == -INFINITY) ? 0.f : mn;
                            const float shift = bs[n][e] - nb;
        #pragma unroll
                            for (int tile = 0; tile < 2; ++tile) {
                                x[tile][n][e] += shift;
                                x[tile][n][e + 2] += shift;
                            }
                            m[n][e] = mn;
                            bs[n][e] = nb;
                            thr[n][e] = (mn == -INFINITY) ? -INFINITY : kSlack;
                            l[n][e] *= al;
        #pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                O[n][i][e] *= al;
                                O[n][i][e + 2] *= al;
                            }
                        }
                }
        #pragma unroll
                for (int n = 0; n < NT; ++n)
        #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float s = 0.f;
        #pragma unroll
                        for (int tile = 0; tile < 2; ++tile) {
                            x[tile][n][e] = fast_exp2(x[tile][n][e]);
                            x[tile][n][e + 2] = fast_exp2(x[tile][n][e + 2]);
                            s += x[tile][n][e] + x[tile][n][e + 2];
                        }
                        l[n][e] += s;
                    }

                // Sparse V: a tile whose weights are all below tau for every real row
                // skips its V dequant and P.V.  Here p = 2^(x - base) with base at
                // most the running max, so p is never below the final normalised
                // weight: only tokens the definition skips can be skipped.
                bool keep[2] = {true, true};
                if (sparse) {
        #pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        float mx = 0.f;
        #pragma unroll
                        for (int n = 0; n < NT; ++n)
        #pragma unroll
                            for (int e = 0; e < 2; ++e)
                                if (row_ok[n][e]) mx = fmaxf(mx, fmaxf(x[tile][n][e], x[tile][n][e + 2]));
                        keep[tile] = __any_sync(0xffffffffu, mx >= p.sparse_tau);
                    }
                }

                // p <= 2^kSlack = 16, so p * n_v fits fp16 for V norms up to 4094.
                // A chunk holding a larger norm (warp-uniform, rare) scales the
                // dequantised V values instead (|c| * n_v <= 0.25 * 65504) and
                // sends p itself to the MMA.
                bool bigv = false;
                if constexpr (!TAB)
                    bigv = __any_sync(0xffffffffu, fmaxf(fmaxf(nv[0][0], nv[0][1]), fmaxf(nv[1][0], nv[1][1])) > 2048.f);
                (void)bigv;

                // ---------------- O^T += C_v^T . (P n_v)^T (rotated basis) ----------------
                auto vpass = [&](auto big_tag) {
                    constexpr bool BIG = decltype(big_tag)::value;
        #pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        if (!FULL && tile == 1 && !two) break;
                        if (!keep[tile]) continue;
                        const float pa = BIG ? 1.f : nv[tile][0], pbn = BIG ? 1.f : nv[tile][1];
                        uint32_t pb0[NT], pb1[NT];
        #pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            pb0[n] = movtrans(pack_half2(x[tile][n][0] * pa, x[tile][n][1] * pa));
                            pb1[n] = movtrans(pack_half2(x[tile][n][2] * pbn, x[tile][n][3] * pbn));
                        }
                        // A quad of dim tile mt: transposed pairs 2mt, 2mt+1 of token block 0
                        // (tokens 0-7 of the tile) then of block 1 (tokens 8-15); group J of
                        // both tokens feeds dim tiles 2J and 2J+1
                        const uint8_t* rva = st + C::kVOff + (tile * 16 + g) * C::kRbV;
                        const uint8_t* rvb = st + C::kVOff + (tile * 16 + g + 8) * C::kRbV;
                        const QuarterWords va = load_quarter<VB>(rva + t * C::kQuarterV);
                        const QuarterWords vb = load_quarter<VB>(rvb + t * C::kQuarterV);
                        const Tables tva = TAB ? v_tables<FULL>(rva, tok0 + tile * 16 + g < t_end) : vt;
                        const Tables tvb = TAB ? v_tables<FULL>(rvb, tok0 + tile * 16 + g + 8 < t_end) : vt;
                        auto vgroup = [&](auto jtag) {
                            constexpr int J = decltype(jtag)::value;
                            uint32_t ha[4], hb[4];
                            dequant_group<VB, J>(va, tva, ha);
                            dequant_group<VB, J>(vb, tvb, hb);
                            if constexpr (BIG) {  // c * n_v per token (tokens g and g + 8 of the tile)
                                const __half2 sa = __float2half2_rn(nv[tile][0]);
                                const __half2 sb = __float2half2_rn(nv[tile][1]);
        #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const __half2 ca = __hmul2(*reinterpret_cast<const __half2*>(&ha[i]), sa);
                                    const __half2 cb = __hmul2(*reinterpret_cast<const __half2*>(&hb[i]), sb);
                                    ha[i] = *reinterpret_cast<const uint32_t*>(&ca);
                                    hb[i] = *reinterpret_cast<const uint32_t*>(&cb);
                                }
                            }
        #pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const uint32_t v0 = movtrans(ha[2 * e]), v1 = movtrans(ha[2 * e + 1]);
                                const uint32_t v2 = movtrans(hb[2 * e]), v3 = movtrans(hb[2 * e + 1]);
        #pragma unroll
                                for (int n = 0; n < NT; ++n) mma_f16(O[n][2 * J + e], v0, v1, v2, v3, pb0[n], pb1[n]);
                            }
                        };
                        vgroup(std::integral_constant<int, 0>{});
                        vgroup(std::integral_constant<int, 1>{});
                        vgroup(std::integral_constant<int, 2>{});
                        vgroup(std::integral_constant<int, 3>{});
                    }
                };
                if constexpr (TAB) {
                    vpass(std::false_type{});
                } else {
                    if (bigv) vpass(std::true_type{});
                    else vpass(std::false_type{});
                }
        };

        int c = warp;
        for (; c < nchunks; c += C::kWarps) {
            const bool ok = mbar_wait_bounded(bar0 + 8 * stage, phase);
            if (__any_sync(0xffffffffu, !ok)) { stalled = true; break; }
            const uint8_t* st = wpipe + stage * C::kStage;
            const int tok0 = t_begin + c * C::kChunk;
            if (tok0 + C::kChunk <= t_end && tok0 + C::kChunk <= all_visible_below)
                process(st, tok0, std::true_type{});
            else
                process(st, tok0, std::false_type{});
            __syncwarp();
            const int cn = c + C::kWarps * C::kStages;
            if (cn < nchunks && lane == 0) {
                fence_proxy_async();
                issue(cn, stage);
            }
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }

        if (pos + nchunks >= hi) griddep_launch_dependents();  // last segment: let the merge launch
        if (stalled) {
            // Drain this warp's copies still in flight (bounded), flag, and stop.
            for (int k = 0; k < C::kStages; ++k) {
                if (c + C::kWarps * k >= nchunks) break;
                (void)mbar_wait_bounded(bar0 + 8 * stage, phase);
                if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            }
            if (lane == 0) atomicOr(p.status, kStatusPipelineStall);
        }

        // ---- combine the 4 warps of the CTA, write this segment's partial ----
    #pragma unroll
        for (int n = 0; n < NT; ++n)
    #pragma unroll
            for (int e = 0; e < 2; ++e) {
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 4);
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 8);
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 16);
            }
        __syncthreads();  // every warp is done with its pipeline stages
        float* sO = reinterpret_cast<float*>(smem) + warp * C::kRows * C::kOStride;
        float* sML = reinterpret_cast<float*>(smem) + C::kWarps * C::kRows * C::kOStride;
    #pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int r0 = 8 * n + 2 * t;
    #pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int dlo = 32 * (g >> 1) + 4 * mt + (g & 1);
                sO[r0 * C::kOStride + dlo] = O[n][mt][0];
                sO[(r0 + 1) * C::kOStride + dlo] = O[n][mt][1];
                sO[r0 * C::kOStride + dlo + 2] = O[n][mt][2];
                sO[(r0 + 1) * C::kOStride + dlo + 2] = O[n][mt][3];
            }
            if (g == 0) {
                sML[(warp * C::kRows + r0) * 2 + 0] = m[n][0];
                sML[(warp * C::kRows + r0) * 2 + 1] = l[n][0];
                sML[(warp * C::kRows + r0 + 1) * 2 + 0] = m[n][1];
                sML[(warp * C::kRows + r0 + 1) * 2 + 1] = l[n][1];
            }
        }
        __syncthreads();
        {
            constexpr int kPerRow = 128 / C::kRows;      // threads per row
            constexpr int kDims = kD / kPerRow;          // dims per thread
            const int r = threadIdx.x / kPerRow;
            const int d0 = (threadIdx.x % kPerRow) * kDims;
            if (rbase + r < p.rows) {
                float mw[C::kWarps], M = -INFINITY;
    #pragma unroll
                for (int w = 0; w < C::kWarps; ++w) {
                    mw[w] = sML[(w * C::kRows + r) * 2];
                    M = fmaxf(M, mw[w]);
                }
                float sc[C::kWarps], lsum = 0.f;
    #pragma unroll
                for (int w = 0; w < C::kWarps; ++w) {
                    sc[w] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
                    lsum += sc[w] * sML[(w * C::kRows + r) * 2 + 1];
                }
                const size_t pidx = (static_cast<size_t>(blockIdx.x) + unit) * 16 + r;
                float* po = p.part_o + pidx * kD + d0;
    #pragma unroll
                for (int d = 0; d < kDims; d += 4) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    #pragma unroll
                    for (int w = 0; w < C::kWarps; ++w) {
                        const float* src = reinterpret_cast<float*>(smem) + (w * C::kRows + r) * C::kOStride + d0 + d;
                        acc.x += sc[w] * src[0];
                        acc.y += sc[w] * src[1];
                        acc.z += sc[w] * src[2];
                        acc.w += sc[w] * src[3];
                    }
                    *reinterpret_cast<float4*>(po + d) = acc;
                }
                if ((threadIdx.x % kPerRow) == 0) {
                    p.part_ml[pidx * 2 + 0] = M;
                    p.part_ml[pidx * 2 + 1] = lsum;
                }
            }
        }

        // the next segment reuses the pipeline area the epilogue just read
        if (__syncthreads_or(stalled)) break;
        pos += nchunks;
    }
}


// One CTA per output row (b, q head, query j): merge the partials of the
// CTAs that covered the row's unit with their log-sum-exp weights, apply
// v_rescale, leave the rotated basis (Rot^-1(y) = s * (H y) / sqrt(128)) and
// store fp16.  The 4 warps split the partials (warp w takes i = w mod 4), so
// a long unit's partials are read with four times the loads in flight: each
// warp merges its share against its own max, lane l holding dims 4l..4l+3,
// and warp 0 merges the four results.
__global__ void __launch_bounds__(128) tq_combine_kernel(const __grid_constant__ CombineParams p) {
    __shared__ float4 s_acc[4][32];
    __shared__ float s_m[4], s_den[4];
    griddep_wait();  // the decode kernel's partials
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int row = blockIdx.x;
    const int j = row % p.tq;
    const int hq = (row / p.tq) % p.hq;
    const int b = row / (p.tq * p.hq);
    const int kv = hq / p.group, hl = hq - kv * p.group;
    const int r = hl * p.tq + j;
    const int rg = r / p.group_rows, rl = r - rg * p.group_rows;
    const int per_b = p.hkv * p.row_groups;
    const int ui = kv * p.row_groups + rg;
    const int unit = b * per_b + ui;

    // the unit's global chunk range [k_first, k_first + nch) and the CTAs over it
    int before = 0, all = 0;
    for (int bb = lane; bb < p.batch; bb += 32) {
        const int v = unit_chunks(p.lengths, bb, p.max_len) * per_b;
        all += v;
        if (bb < b) before += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    const int nch = unit_chunks(p.lengths, b, p.max_len);
    const int P = p.num_ctas, cq = all / P, cr = all - cq * P;
    const bool some_empty = all < P;  // then some CTAs have no chunk and wrote nothing
    int c0 = 0, n = 0;
    if (nch > 0) {
        const int k_first = before + ui * nch;
        c0 = static_cast<int>((static_cast<long long>(k_first + 1) * P - 1) / all);
        const int c1 = static_cast<int>((static_cast<long long>(k_first + nch) * P - 1) / all);
        n = c1 - c0 + 1;
    }
    auto used = [&](int i) {
        const int c = c0 + i;
        return i < n && (!some_empty || c * cq + (c * cr) / P < (c + 1) * cq + ((c + 1) * cr) / P);
    };
    const size_t row0 = (static_cast<size_t>(c0) + unit) * 16 + rl;  // partial of CTA c0
    auto load_ml = [&](int i) {
        return __ldcg(reinterpret_cast<const float2*>(p.part_ml) + row0 + 16 * static_cast<size_t>(i));
    };

    // this warp's partials: i = warp + 4k; lane l reads the (m, l) pair of k = l (+32 ...)
    const int i_first = warp + 4 * lane;
    const float2 ml_first = used(i_first) ? load_ml(i_first) : make_float2(-INFINITY, 0.f);
    float M = ml_first.x;
    for (int i = i_first + 128; i < n; i += 128)
        if (used(i)) M = fmaxf(M, load_ml(i).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < n; i0 += 128) {
        const int i = i0 + i_first;
        float w = 0.f;
        const float2 ml = (i0 == 0) ? ml_first : (used(i) ? load_ml(i) : make_float2(-INFINITY, 0.f));
        if (ml.x != -INFINITY) {
            w = fast_exp2(ml.x - M);
            den += w * ml.y;
        }
        const int left = n - i0 - warp;                 // partials i0 + warp + 4k, k < nb
        const int nb = left > 0 ? min(32, (left + 3) / 4) : 0;
        for (int k0 = 0; k0 < nb; k0 += 8) {
            float wk[8];
            float4 o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                wk[k] = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);
                o[k] = (k0 + k < nb && wk[k] != 0.f)
                           ? __ldcg(reinterpret_cast<const float4*>(
                                        p.part_o + (row0 + 16 * static_cast<size_t>(i0 + warp + 4 * (k0 + k))) * kD) +
                                    lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                acc.x += wk[k] * o[k].x; acc.y += wk[k] * o[k].y;
                acc.z += wk[k] * o[k].z; acc.w += wk[k] * o[k].w;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    s_acc[warp][lane] = acc;
    if (lane == 0) {
        s_m[warp] = M;
        s_den[warp] = den;
    }
    __syncthreads();
    if (warp != 0) return;

    float Mall = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) Mall = fmaxf(Mall, s_m[w]);
    float dsum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float sc = (s_m[w] == -INFINITY) ? 0.f : fast_exp2(s_m[w] - Mall);
        const float4 x = s_acc[w][lane];
        dsum += sc * s_den[w];
        a.x += sc * x.x; a.y += sc * x.y; a.z += sc * x.z; a.w += sc * x.w;
    }
    float inv = 0.f;
    if (dsum > 0.f) inv = p.v_rescale / dsum;
    else if (lane == 0) atomicOr(p.status, kStatusShortContext);
    float v[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
    wht128_lane4(v, lane);
    const uint32_t sn = sign_nibble(p.signs, lane);
    const float nrm = 0.08838834764831845f;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ((sn >> i) & 1u) ? -v[i] * nrm : v[i] * nrm;
    uint2 out;
    out.x = pack_half2(v[0], v[1]);
    out.y = pack_half2(v[2], v[3]);
    *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(row) * kD + lane * 4) = out;
}

// Self-test of the bounded waits: one CTA waits on an mbarrier nothing ever
// arrives on, through the same wait the pipelines use, with a short limit; the
// wait must give up and leave kStatusPipelineStall in the status word.
__global__ void __launch_bounds__(32) tq_selftest_stall_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar_word;
    const uint32_t bar = smem_u32(&bar_word);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(bar, 0, limit_ns);
    if (!ok && threadIdx.x == 0) atomicOr(status, kStatusPipelineStall);
}

int launch_selftest_stall(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
    tq_selftest_stall_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

template <int KB, int VB, int NT, bool TAB = false>
static int launch_decode_t(const DecodeParams& p, const CUtensorMap* kmap, cudaStream_t stream,
                           cudaEvent_t ev0, cudaEvent_t ev1) {
    using C = DecCfg<KB, VB, NT, TAB>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tq_decode_kernel<KB, VB, NT, TAB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.num_ctas);
    if (ev0) cudaEventRecord(ev0, stream);
    cudaError_t e = launch_pdl(tq_decode_kernel<KB, VB, NT, TAB>, grid, dim3(C::kWarps * 32),
                               C::kSmemAlloc, stream, p, *kmap);
    if (ev1) cudaEventRecord(ev1, stream);
    return e;
}

template <int NT>
static int launch_decode_nt(int kbits, int vbits, const DecodeParams& p, const CUtensorMap* kmap,
                            cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    if (p.table) {
        if (kbits == 3 && vbits == 3) return launch_decode_t<3, 3, NT, true>(p, kmap, stream, ev0, ev1);
        return cudaErrorInvalidValue;
    }
    if (kbits == 16 && vbits == 4) return launch_decode_t<0, 4, NT>(p, kmap, stream, ev0, ev1);
    if (kbits == 3 && vbits == 3) return launch_decode_t<3, 3, NT>(p, kmap, stream, ev0, ev1);
    if (kbits == 4 && vbits == 4) return launch_decode_t<4, 4, NT>(p, kmap, stream, ev0, ev1);
    if (kbits == 16 && vbits == 3) return launch_decode_t<0, 3, NT>(p, kmap, stream, ev0, ev1);
    if (kbits == 4 && vbits == 3) return launch_decode_t<4, 3, NT>(p, kmap, stream, ev0, ev1);
    return cudaErrorInvalidValue;
}

int launch_decode(int kbits, int vbits, const DecodeParams& p, const CUtensorMap* kmap,
                  cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    if (p.group_rows == 8) return launch_decode_nt<1>(kbits, vbits, p, kmap, stream, ev0, ev1);
    if (p.group_rows == 16) return launch_decode_nt<2>(kbits, vbits, p, kmap, stream, ev0, ev1);
    return cudaErrorInvalidValue;
}

int launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int rows = p.batch * p.hq * p.tq;
    return launch_pdl(tq_combine_kernel, dim3(rows), dim3(128), 0, stream, p);
}

// Resident CTAs per SM: the launch bounds' target, unless shared memory
// (228 KB per SM, 1 KB of it reserved per CTA) allows fewer.
template <int KB, int VB, int NT, bool TAB = false>
static int ctas_of() {
    using C = DecCfg<KB, VB, NT, TAB>;
    const int by_smem = (228 * 1024) / (C::kSmemAlloc + 1024);
    return by_smem < C::kMinCtas ? by_smem : C::kMinCtas;
}

template <int NT>
static int ctas_nt(int kbits, int vbits, bool table) {
    if (table) return ctas_of<3, 3, NT, true>();
    if (kbits == 16) return vbits == 4 ? ctas_of<0, 4, NT>() : ctas_of<0, 3, NT>();
    if (kbits == 3) return ctas_of<3, 3, NT>();
    return vbits == 4 ? ctas_of<4, 4, NT>() : ctas_of<4, 3, NT>();
}

int decode_ctas_per_sm(int kbits, int vbits, int group_rows, bool table) {
    const int c = group_rows <= 8 ? ctas_nt<1>(kbits, vbits, table) : ctas_nt<2>(kbits, vbits, table);
    return c < 1 ? 1 : c;
}

}  // namespace tq
