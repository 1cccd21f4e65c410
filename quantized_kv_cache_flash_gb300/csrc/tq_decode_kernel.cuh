// Fused split-K decode attention over the packed KV cache: the kernel template
// (instantiated in tq_decode_f.cu, tq_decode_q.cu and tq_decode_r.cu).
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
// Work split: waves of CTAs (two or, for large contexts, three for row
// groups of up to 8 rows; one for 16-row groups), each taking an equal
// share of the context's
// 32-token chunks over all (batch, kv head, row group) units.  A CTA's 4 warps
// stream their own chunks through private rings of shared-memory stages
// filled by 1-D bulk copies (tensor-map tile copies with 128-byte swizzle for
// fp16 K), dequantize in registers and run both contractions as warp MMAs
// with the 16 tokens of a tile as M and up to 8 query rows per n-tile as N.
#pragma once

#include <float.h>

#include <type_traits>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kChunkTokens = 32;  // tokens per warp pipeline stage (2 MMA tiles)

// ROWS: query rows per row group (4, 8 or 16).  TAB: 3-bit records that carry
// their own centroid x norm table (48 bytes of codes + 8 fp16 values c_j * n,
// 64 bytes, no norm array).
//
// Score precision (quantized K).  The score MMA takes fp16 operands, but
// neither Rot(q) (fp32) nor the codebook (fp32) is an fp16 value, and a
// rounding of 2^-11 in either moves a score of 30 by ~1e-2, too much for
// peaked softmax rows.  So each score is the sum of three products, all
// accumulated in fp32:
//   C_hi . q_hi  +  C_hi . q_lo  +  (C_lo . q_8) * 2^(b - a)
// where q_hi = fp16(Rot q), q_lo = fp16(Rot q - q_hi), C_hi = fp16(c[idx]),
// C_lo = e4m3((c - fp16(c))[idx] * 2^a) and q_8 = e4m3(Rot q * 2^-b) (an fp8
// MMA; a from the codebook, b per query row).  The result is within ~2^-16 of
// the fp32 score.  With 4 rows per group (kPair) q_hi and q_lo of a row take
// the two columns of one MMA column pair; otherwise q_lo is a second B
// operand over the same dequantised A.  fp16 K needs none of this: q and K
// are fp16 inputs, their products exact.
template <int KB, int VB, int ROWS, bool TAB = false, bool RES = false>
struct DecCfg {
    static constexpr int kWarps = 4;
    static constexpr int kChunk = kChunkTokens;
    static constexpr int NT = ROWS == 16 ? 2 : 1;           // 8-column MMA n-tiles
    static constexpr bool kPair = KB != 0 && ROWS == 4;     // column 2i: q_hi of row i, 2i+1: q_lo
    static constexpr bool kQlo = KB != 0 && ROWS != 4;      // q_lo as a second B operand
    static constexpr bool kRes = RES && KB != 0 && !TAB;    // fp8 centroid residual product
    static_assert(KB == 0 || kPair || kQlo, "quantized K keeps q_lo in the pair columns or its own operand");
    static constexpr int NE = kPair ? 1 : 2;                // query rows per thread per n-tile
    // 16-token tiles per softmax pass (2: a whole chunk, 1 with two n-tiles,
    // where the scores of two tiles would not fit the registers) and whether
    // the codebook tables stay in registers
    static constexpr int kTilesPerCall = NT == 1 ? 2 : 1;
    static constexpr bool kTabRegs = NT == 1;
    static constexpr int kStages = (KB == 0 || NT == 1) ? 2 : 3;
    static constexpr int kRows = ROWS;
    static constexpr int kCols = 8 * NT;                    // B-operand columns
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
    // B-operand columns in MMA k order: fp16 [kCols][kQStride] (q_hi, or the
    // q_hi/q_lo pairs), fp16 q_lo [kCols][kQStride], e4m3 q_8 [kCols][kQ8Stride]
    // and the residual scales [kCols]; the 16-byte pads stagger the columns
    // over the banks for ldmatrix
    static constexpr int kQStride = kD + 8;
    static constexpr int kQ8Stride = kD + 16;
    static constexpr int kQOff = kPipeBytes;
    static constexpr int kQloOff = kQOff + kCols * kQStride * 2;
    static constexpr int kQ8Off = kQloOff + (kQlo ? kCols * kQStride * 2 : 0);
    static constexpr int kRsOff = kQ8Off + (kRes ? kCols * kQ8Stride : 0);
    // codebook tables (K prmt tables, V prmt tables, K fp8 residual table),
    // read from shared memory at each use so they hold no registers
    static constexpr int kTabOff = (kRsOff + (kRes ? kCols * 4 : 0) + 15) / 16 * 16;
    static constexpr int kBarOff = kTabOff + 48;
    static constexpr int kScanOff = (kBarOff + kWarps * kStages * 8 + 15) / 16 * 16;
    static constexpr int kSmem = kScanOff + kWarps * 4 * 32 * 4;  // per-warp batch scan
    static constexpr int kSmemAlloc = kSmem + 1024;          // base alignment slack
    // epilogue scratch (reuses the pipeline): per warp O[kRows][kOStride] + (m, l)[kRows]
    static constexpr int kOStride = kD + 4;
    static_assert(kWarps * kRows * kOStride * 4 + kWarps * kRows * 8 <= kPipeBytes, "scratch");

    // query row (within the group) held by this thread's slot e of n-tile n,
    // and the B-operand column of that row's q_8
    __device__ static __forceinline__ int slot_row(int n, int e, int t) {
        return kPair ? t : 8 * n + 2 * t + e;
    }
    __device__ static __forceinline__ int slot_col8(int n, int e, int t) {
        return kPair ? 2 * t : 8 * n + 2 * t + e;
    }
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

// Codes of group J (0..3) of a quarter: the 8 dims 8J..8J+7, 3-bit codes in
// the low 3 bits of each nibble (the spare bits of w0..w2 hold group 3).
__device__ __forceinline__ uint32_t group3_codes(const QuarterWords& q, int J) {
    if (J < 3) return q.w[J] & 0x77777777u;
    return (__umulhi(q.w[0], 1u << 29) & 0x11111111u) | (__umulhi(q.w[1], 1u << 30) & 0x22222222u) |
           (__umulhi(q.w[2], 1u << 31) & 0x44444444u);
}

// Group J (0..3) of a quarter: dim pairs 4J..4J+3 as four half2, the pairs
// the whole-quarter dequantisers put in h[4J..4J+3].  Decoding a group at a
// time lets each group's MMAs follow it, so only one group is live.  RES: also
// the group's fp8 centroid residuals, r[0] = dims 8J..8J+3, r[1] = 8J+4..8J+7.
template <int KB, int J, bool RES>
__device__ __forceinline__ void dequant_group(const QuarterWords& q, const Tables& t,
                                              uint32_t r8lo, uint32_t r8hi, uint32_t (&h)[4],
                                              uint32_t (&r)[2]) {
    if constexpr (KB == 3) {
        const uint32_t m = group3_codes(q, J);
        const uint32_t m2 = __umulhi(m, 1u << 16);
        lut4(m, t, h[0], h[1]);
        lut4(m2, t, h[2], h[3]);
        if constexpr (RES) {
            r[0] = prmt(r8lo, r8hi, m);
            r[1] = prmt(r8lo, r8hi, m2);
        }
    } else {
        if constexpr (RES) dequant4_word_res(q.w[J], t, r8lo, r8hi, h[0], h[1], h[2], h[3], r[0], r[1]);
        else dequant4_word(q.w[J], t, h[0], h[1], h[2], h[3]);
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
//   S^T[16 tok x 8 cols]  = C_k[16 x 128] . B_q^T          (8 k-steps per n-tile)
//   O^T[128 x 8 cols]    += C_v^T[128 x 16 tok] . (P n_v)^T (8 dim tiles)
// with the tokens (M = 16) dequantised in registers: a thread owns tokens g and
// g+8 of the tile and decodes its quarter t (32 dims) of both records.
template <int KB, int VB, int ROWS, bool TAB, bool RES>
__global__ void __launch_bounds__(128, DecCfg<KB, VB, ROWS, TAB, RES>::kMinCtas)
    tq_decode_kernel(const __grid_constant__ DecodeParams p,
                     const __grid_constant__ CUtensorMap kmap) {
    using C = DecCfg<KB, VB, ROWS, TAB, RES>;
    constexpr int NT = C::NT, NE = C::NE;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived from smem_raw by an integer offset so the
    // compiler keeps every access in the shared window (LDS, not generic loads)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    // warp index through a shuffle so the compiler treats it (and the chunk,
    // stage and copy addresses derived from it) as warp-uniform
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int per_b = p.hkv * p.row_groups;
    const int P = static_cast<int>(gridDim.x);
    const int c_me = static_cast<int>(blockIdx.x);

    // ---- set-up that reads nothing earlier work on the stream writes: it
    // overlaps the predecessor's tail under programmatic dependent launch ----
    uint8_t* wpipe = smem + warp * C::kStages * C::kStage;
    const uint32_t bar0 = smem_u32(smem + C::kBarOff) + warp * C::kStages * 8;
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
    }
    if constexpr (KB == 0)
        if (threadIdx.x == 0) prefetch_tensormap(&kmap);
    __syncwarp();

    griddep_wait();  // lengths, cache and q come from earlier work on the stream
    BatchScan scan;
    scan.init(reinterpret_cast<int*>(smem + C::kScanOff) + warp * 128, p.lengths, p.batch, per_b,
              p.max_len, lane);
    // (each value the copies and masks derive from goes through a lane-0
    // shuffle, which lets the compiler keep them in uniform registers)
    const int C_all = __shfl_sync(0xffffffffu, scan.total(p.lengths, p.batch, per_b, p.max_len, lane), 0);
    // floor(c * C_all / P) in 32-bit arithmetic: c * (C_all mod P) < P^2 < 2^31
    const int cq = C_all / P, cr = C_all - cq * P;
    const int lo = c_me * cq + (c_me * cr) / P;
    const int hi = (c_me + 1) * cq + ((c_me + 1) * cr) / P;
    if (lo >= hi) return;  // no chunks for this CTA (uniform over the CTA)
    __half* sQ = reinterpret_cast<__half*>(smem + C::kQOff);
    __half* sQlo = reinterpret_cast<__half*>(smem + C::kQloOff);
    uint8_t* sQ8 = smem + C::kQ8Off;
    float* sRS = reinterpret_cast<float*>(smem + C::kRsOff);
    const uint32_t q_lds = smem_u32(sQ) + ((lane & 7) * C::kQStride + 8 * (lane >> 3)) * 2;
    const uint32_t qlo_lds = smem_u32(sQlo) + ((lane & 7) * C::kQStride + 8 * (lane >> 3)) * 2;
    const uint32_t q8_lds = smem_u32(sQ8) + (lane & 7) * C::kQ8Stride + 16 * (lane >> 3);
    // Codebook tables: in registers for one n-tile; with two n-tiles they are
    // read from shared memory at each use, so they hold no registers
    constexpr int TPC = C::kTilesPerCall;
    uint32_t* sTab = reinterpret_cast<uint32_t*>(smem + C::kTabOff);
    if (threadIdx.x < 12) {  // visible after the first segment's __syncthreads
        const int i = threadIdx.x;
        sTab[i] = i < 4 ? p.ktab[i] : i < 8 ? p.vtab[i - 4] : i < 10 ? p.ktab8[i - 8] : 0u;
    }
    const Tables kt_r{p.ktab[0], p.ktab[1], p.ktab[2], p.ktab[3]};
    const Tables vt_r{p.vtab[0], p.vtab[1], p.vtab[2], p.vtab[3]};
    const uint2 k8_r = make_uint2(p.ktab8[0], p.ktab8[1]);
    auto tables_at = [&](int off) {
        const uint4 w = *reinterpret_cast<const uint4*>(sTab + off);
        return Tables{w.x, w.y, w.z, w.w};
    };
    auto k_tables = [&]() { return C::kTabRegs ? kt_r : tables_at(0); };
    auto v_tables_all = [&]() { return C::kTabRegs ? vt_r : tables_at(4); };
    auto k_res_table = [&]() { return C::kTabRegs ? k8_r : *reinterpret_cast<const uint2*>(sTab + 8); };
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
            const uint32_t qh0 = pack_half2(v[0], v[1]), qh1 = pack_half2(v[2], v[3]);
            if constexpr (KB != 0) {
                const int kk = 16 * (lane & 7) + 2 * (lane >> 3);
                __half* qrow = sQ + (C::kPair ? 2 * r : r) * C::kQStride;
                *reinterpret_cast<uint32_t*>(qrow + kk) = qh0;
                *reinterpret_cast<uint32_t*>(qrow + kk + 8) = qh1;
                // q_lo = Rot(q) - q_hi, exact in fp32 and rounded once more to fp16
                const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&qh0));
                const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&qh1));
                const uint32_t ql0 = pack_half2(v[0] - h0.x, v[1] - h0.y);
                const uint32_t ql1 = pack_half2(v[2] - h1.x, v[3] - h1.y);
                // (the pair column of q_hi, or the q_lo operand's own area)
                __half* lrow = C::kPair ? sQ + (2 * r + 1) * C::kQStride : sQlo + r * C::kQStride;
                *reinterpret_cast<uint32_t*>(lrow + kk) = ql0;
                *reinterpret_cast<uint32_t*>(lrow + kk + 8) = ql1;
                if constexpr (C::kRes) {
                    // q_8 = e4m3(Rot(q) * 2^-b): b puts the row's largest |value|
                    // in [128, 256) (e4m3 saturates at 448).  In the fp8 MMA's k
                    // order (group J = dims 8J..8J+7 of every quarter: k = 4t + i
                    // <-> dim 32t + 8J + i, k = 16 + 4t + i <-> dim 32t + 8J + 4 + i)
                    // this lane's 4 dims are the 4 bytes at 32J + 16 (lane & 1) + 4 t.
                    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    int eb = 0;
                    if (mx > 0.f) (void)frexpf(mx, &eb);
                    const int bsh = eb - 8;
                    const uint32_t b01 = fp8x2_e4m3(ldexpf(v[0], -bsh), ldexpf(v[1], -bsh));
                    const uint32_t b23 = fp8x2_e4m3(ldexpf(v[2], -bsh), ldexpf(v[3], -bsh));
                    const int col = C::kPair ? 2 * r : r;
                    const int off = 32 * ((lane & 7) >> 1) + 16 * (lane & 1) + 4 * (lane >> 3);
                    *reinterpret_cast<uint32_t*>(sQ8 + col * C::kQ8Stride + off) = b01 | (b23 << 16);
                    if constexpr (C::kPair)  // the odd columns of the fp8 operand stay zero
                        *reinterpret_cast<uint32_t*>(sQ8 + (col + 1) * C::kQ8Stride + off) = 0u;
                    if (lane == 0) {
                        sRS[col] = ldexpf(1.f, bsh - p.res_shift);
                        if constexpr (C::kPair) sRS[col + 1] = 0.f;
                    }
                }
            } else {
                *reinterpret_cast<uint2*>(sQ + r * C::kQStride + 4 * lane) = make_uint2(qh0, qh1);
            }
        }
        __syncthreads();

        // B fragments of k-steps 2*kc2 and 2*kc2 + 1 for n-tile n (ldmatrix
        // matrix j = lane >> 3 covers k in [32*kc2 + 8*j, +8) of columns 8n..8n+7)
        auto load_qb = [&](uint32_t base, int n, int kc2, uint32_t (&bq)[4]) {
            ldsm_x4(base + (8 * n * C::kQStride + 32 * kc2) * 2, bq[0], bq[1], bq[2], bq[3]);
        };
        // residual scale 2^(b - a) of the rows this thread's fp8 accumulators
        // hold (kept in registers for one n-tile, read from shared otherwise)
        float rs[NT][NE];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < NE; ++e) rs[n][e] = (C::kRes && NT == 1) ? sRS[C::slot_col8(n, e, t)] : 0.f;
        auto res_scale = [&](int n, int e) { return NT == 1 ? rs[n][e] : sRS[C::slot_col8(n, e, t)]; };
        // last visible token (inclusive) of a row this thread owns, and whether
        // it is a real query row (not padding of the group); only the masked
        // (tail / causal) and sparse paths ask
        auto row_lim = [&](int n, int e) { return L - p.tq + ((rbase + C::slot_row(n, e, t)) % p.tq); };
        auto row_ok = [&](int n, int e) { return rbase + C::slot_row(n, e, t) < p.rows; };
        const int all_visible_below = L - p.tq + 1;  // tokens below this are seen by every row

        float O[NT][8][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 8; ++i) O[n][i][0] = O[n][i][1] = O[n][i][2] = O[n][i][3] = 0.f;
        // running max m, sum l and exp2 base bs (m, or 0 before the first
        // score) of the rows this thread owns; a score above the base by more
        // than kSlack (once the row has a max) moves the base
        constexpr float kSlack = 4.f;
        float m[NT][NE], l[NT][NE], bs[NT][NE];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < NE; ++e) m[n][e] = -INFINITY, l[n][e] = bs[n][e] = 0.f;
        bool stalled = false;
        uint32_t tiles_seen = 0, tiles_skipped = 0;  // sparse V: this warp's tile counts

        // TPC tiles (16 tokens each) of a 32-token chunk of this warp, from
        // tile0: both tiles in one call (their K dequant interleaves, one
        // softmax bookkeeping pass) where registers allow, else one.
        // FULL: all tokens of the chunk valid and visible to every row (no
        // masking); otherwise the tail / causal path.
        // Scores of slot e: x[tt][n][e] (token g), x[tt][n][e + 2] (token g + 8).
        auto process = [&](const uint8_t* st, const int tok0, const int tile0, auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            // TPC == 2: whether tile 1 holds any token (always when FULL)
            const bool two = TPC == 1 || FULL || t_end - tok0 > 16;
            // ---------------- scores S^T = C_k . B_q^T ----------------
            float x[TPC][NT][4];
#pragma unroll
            for (int tt = 0; tt < TPC; ++tt) {
                const int tile = tile0 + tt;
#pragma unroll
                for (int n = 0; n < NT; ++n) x[tt][n][0] = x[tt][n][1] = x[tt][n][2] = x[tt][n][3] = 0.f;
                if (!FULL && tt == 1 && !two) break;
                if constexpr (KB == 0) {
                    const int mi = lane >> 3;
                    const int row = tile * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                    for (int kc2 = 0; kc2 < 4; ++kc2) {
                        uint32_t qb[NT][4];
#pragma unroll
                        for (int n = 0; n < NT; ++n) load_qb(q_lds, n, kc2, qb[n]);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const int db = 4 * kc2 + 2 * kk + (mi >> 1);  // 16-byte chunk 0..15 of the row
                            const uint32_t addr = smem_u32(st) + (db >> 3) * 4096 + row * 128 +
                                                  (((db & 7) ^ (row & 7)) << 4);
                            uint32_t a0, a1, a2, a3;
                            ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                            for (int n = 0; n < NT; ++n)
                                mma_f16(x[tt][n], a0, a1, a2, a3, qb[n][2 * kk], qb[n][2 * kk + 1]);
                        }
                    }
                } else {
                    // A quad of k-step kc: (token g, pair 2kc), (token g+8, pair 2kc),
                    // (token g, pair 2kc+1), (token g+8, pair 2kc+1) of the quarters;
                    // group J of both tokens feeds k-steps 2J and 2J+1 (fp16) and
                    // k-step J of the fp8 residual product
                    const uint8_t* ra = st + (tile * 16 + g) * C::kRbK;
                    const uint8_t* rb = st + (tile * 16 + g + 8) * C::kRbK;
                    const QuarterWords wa = load_quarter<KB>(ra + t * C::kQuarterK);
                    const QuarterWords wb = load_quarter<KB>(rb + t * C::kQuarterK);
                    const Tables kt = k_tables();
                    const uint2 k8 = k_res_table();
                    const Tables ta = TAB ? record_tables(ra + 48) : kt;
                    const Tables tb = TAB ? record_tables(rb + 48) : kt;
                    float y[NT][4];
#pragma unroll
                    for (int n = 0; n < NT; ++n) y[n][0] = y[n][1] = y[n][2] = y[n][3] = 0.f;
                    auto kgroup = [&](auto jtag) {
                        constexpr int J = decltype(jtag)::value;
                        uint32_t ha[4], hb[4], rA[2], rB[2];
                        dequant_group<KB, J, C::kRes>(wa, ta, k8.x, k8.y, ha, rA);
                        dequant_group<KB, J, C::kRes>(wb, tb, k8.x, k8.y, hb, rB);
                        // (one n-tile's B fragments live at a time: the loads and
                        // MMAs are volatile asm, issued in this order)
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            uint32_t qb[4];
                            load_qb(q_lds, n, J, qb);
                            mma_f16(x[tt][n], ha[0], hb[0], ha[1], hb[1], qb[0], qb[1]);
                            mma_f16(x[tt][n], ha[2], hb[2], ha[3], hb[3], qb[2], qb[3]);
                            if constexpr (C::kQlo) {
                                load_qb(qlo_lds, n, J, qb);
                                mma_f16(x[tt][n], ha[0], hb[0], ha[1], hb[1], qb[0], qb[1]);
                                mma_f16(x[tt][n], ha[2], hb[2], ha[3], hb[3], qb[2], qb[3]);
                            }
                        }
                        if constexpr (C::kRes) {
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                uint32_t b8[2];
                                ldsm_x2(q8_lds + 8 * n * C::kQ8Stride + 32 * J, b8[0], b8[1]);
                                mma_e4m3(y[n], rA[0], rB[0], rA[1], rB[1], b8[0], b8[1]);
                            }
                        }
                    };
                    kgroup(std::integral_constant<int, 0>{});
                    kgroup(std::integral_constant<int, 1>{});
                    kgroup(std::integral_constant<int, 2>{});
                    kgroup(std::integral_constant<int, 3>{});
                    // fold: q_lo column into q_hi (pairs), fp8 residual at its scale
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        if constexpr (C::kPair) {
                            x[tt][n][0] += x[tt][n][1];
                            x[tt][n][2] += x[tt][n][3];
                        }
                        if constexpr (C::kRes) {
#pragma unroll
                            for (int e = 0; e < NE; ++e) {
                                const float sc = res_scale(n, e);
                                x[tt][n][e] = fmaf(y[n][e], sc, x[tt][n][e]);
                                x[tt][n][e + 2] = fmaf(y[n][e + 2], sc, x[tt][n][e + 2]);
                            }
                        }
                    }
                }
            }

            // ---------------- online softmax (log2 domain) ----------------
            float nv[TPC][2];
#pragma unroll
            for (int tt = 0; tt < TPC; ++tt) {
                const int ta = (tile0 + tt) * 16 + g, tb = ta + 8;
                float ka = p.scale_log2e, kb2 = p.scale_log2e;
                if constexpr (KB != 0 && !TAB) {  // table records carry the norm in their values
                    ka *= __half2float(*reinterpret_cast<const __half*>(st + C::kKnOff + 2 * ta));
                    kb2 *= __half2float(*reinterpret_cast<const __half*>(st + C::kKnOff + 2 * tb));
                }
                if constexpr (TAB) {
                    nv[tt][0] = nv[tt][1] = 1.f;
                } else {
                    nv[tt][0] = __half2float(*reinterpret_cast<const __half*>(st + C::kVnOff + 2 * ta));
                    nv[tt][1] = __half2float(*reinterpret_cast<const __half*>(st + C::kVnOff + 2 * tb));
                }
                // scaled score minus the row's exp2 base, one FFMA each (two rows
                // of a token in one packed instruction)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if constexpr (NE == 2) {
                        const float2 nb = make_float2(-bs[n][0], -bs[n][1]);
                        const float2 ya = __ffma2_rn(make_float2(x[tt][n][0], x[tt][n][1]), make_float2(ka, ka), nb);
                        const float2 yb = __ffma2_rn(make_float2(x[tt][n][2], x[tt][n][3]), make_float2(kb2, kb2), nb);
                        x[tt][n][0] = ya.x;
                        x[tt][n][1] = ya.y;
                        x[tt][n][2] = yb.x;
                        x[tt][n][3] = yb.y;
                    } else {
#pragma unroll
                        for (int e = 0; e < NE; ++e) {
                            x[tt][n][e] = fmaf(x[tt][n][e], ka, -bs[n][e]);
                            x[tt][n][e + 2] = fmaf(x[tt][n][e + 2], kb2, -bs[n][e]);
                        }
                    }
                }
                if constexpr (!FULL) {
                    const int ga = tok0 + ta, gb = tok0 + tb;
                    const bool va = ga < t_end && (tt == 0 || two);
                    const bool vb = gb < t_end && (tt == 0 || two);
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < NE; ++e) {
                            const int lim = row_lim(n, e);
                            x[tt][n][e] = (va && ga <= lim) ? x[tt][n][e] : -INFINITY;
                            x[tt][n][e + 2] = (vb && gb <= lim) ? x[tt][n][e + 2] : -INFINITY;
                        }
                    if (!va) nv[tt][0] = 0.f;
                    if (!vb) nv[tt][1] = 0.f;
                }
            }
            // The exp2 base of a row stays at its running max until a score exceeds
            // it by more than kSlack (log2 units); only then (warp-uniform slow
            // path) is the true max taken, O and l rescaled and the scores moved
            // to the new base.  So p <= 2^kSlack.  A row with no score yet has
            // base 0 and threshold -inf: its first finite score sets the max.
            auto row_max = [&](int n, int e) {
                float mx = fmaxf(x[0][n][e], x[0][n][e + 2]);
#pragma unroll
                for (int tt = 1; tt < TPC; ++tt) mx = fmaxf(mx, fmaxf(x[tt][n][e], x[tt][n][e + 2]));
                return mx;
            };
            bool grow = false;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < NE; ++e)
                    grow |= row_max(n, e) > (m[n][e] == -INFINITY ? -INFINITY : kSlack);
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < NE; ++e) {
                        float mx = row_max(n, e);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float mn = fmaxf(m[n][e], mx + bs[n][e]);
                        const float al = (m[n][e] == -INFINITY) ? 0.f : fast_exp2(m[n][e] - mn);
                        const float nb = (mn == -INFINITY) ? 0.f : mn;
                        const float shift = bs[n][e] - nb;
#pragma unroll
                        for (int tt = 0; tt < TPC; ++tt) {
                            x[tt][n][e] += shift;
                            x[tt][n][e + 2] += shift;
                        }
                        m[n][e] = mn;
                        bs[n][e] = nb;
                        l[n][e] *= al;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            O[n][i][e] *= al;
                            O[n][i][e + 2] *= al;
                        }
                    }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if constexpr (NE == 2) {  // the two rows' sums as one packed pair
                    float2 s = make_float2(0.f, 0.f);
#pragma unroll
                    for (int tt = 0; tt < TPC; ++tt) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) x[tt][n][e] = fast_exp2(x[tt][n][e]);
                        s = __fadd2_rn(s, __fadd2_rn(make_float2(x[tt][n][0], x[tt][n][1]),
                                                     make_float2(x[tt][n][2], x[tt][n][3])));
                    }
                    const float2 ln = __fadd2_rn(make_float2(l[n][0], l[n][1]), s);
                    l[n][0] = ln.x;
                    l[n][1] = ln.y;
                } else {
#pragma unroll
                    for (int e = 0; e < NE; ++e) {
                        float s = 0.f;
#pragma unroll
                        for (int tt = 0; tt < TPC; ++tt) {
                            x[tt][n][e] = fast_exp2(x[tt][n][e]);
                            x[tt][n][e + 2] = fast_exp2(x[tt][n][e + 2]);
                            s += x[tt][n][e] + x[tt][n][e + 2];
                        }
                        l[n][e] += s;
                    }
                }
            }

            // Sparse V: a tile whose weights are all below tau for every real row
            // skips its V dequant and P.V.  Here p = 2^(x - base) with base at
            // most the running max, so p is never below the final normalised
            // weight: only tokens the definition skips can be skipped.
            bool keep[TPC];
#pragma unroll
            for (int tt = 0; tt < TPC; ++tt) keep[tt] = true;
            if (sparse) {
#pragma unroll
                for (int tt = 0; tt < TPC; ++tt) {
                    float mx = 0.f;
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < NE; ++e)
                            if (row_ok(n, e)) mx = fmaxf(mx, fmaxf(x[tt][n][e], x[tt][n][e + 2]));
                    keep[tt] = __any_sync(0xffffffffu, mx >= p.sparse_tau);
                    if (FULL || tt == 0 || two) {
                        ++tiles_seen;
                        tiles_skipped += keep[tt] ? 0u : 1u;
                    }
                }
            }

            // p <= 2^kSlack = 16, so p * n_v fits fp16 for V norms up to 4094.
            // A chunk holding a larger norm (warp-uniform, rare) scales the
            // dequantised V values instead (|c| * n_v <= 0.25 * 65504) and
            // sends p itself to the MMA.
            bool bigv = false;
            if constexpr (!TAB) {
                float nmax = fmaxf(nv[0][0], nv[0][1]);
#pragma unroll
                for (int tt = 1; tt < TPC; ++tt) nmax = fmaxf(nmax, fmaxf(nv[tt][0], nv[tt][1]));
                bigv = __any_sync(0xffffffffu, nmax > 2048.f);
            }
            (void)bigv;

            // ---------------- O^T += C_v^T . (P n_v)^T (rotated basis) ----------------
            // B columns: slot e of thread t is column 2t + e (one row per thread
            // with 4-row groups: its column 2t + 1 carries 0)
            auto vpass = [&](auto big_tag) {
                constexpr bool BIG = decltype(big_tag)::value;
#pragma unroll
                for (int tt = 0; tt < TPC; ++tt) {
                    if (!FULL && tt == 1 && !two) break;
                    if (!keep[tt]) continue;
                    const int tile = tile0 + tt;
                    const float pa = BIG ? 1.f : nv[tt][0], pbn = BIG ? 1.f : nv[tt][1];
                    uint32_t pb0[NT], pb1[NT];
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        if constexpr (NE == 2) {
                            const float2 wa = __fmul2_rn(make_float2(x[tt][n][0], x[tt][n][1]), make_float2(pa, pa));
                            const float2 wb = __fmul2_rn(make_float2(x[tt][n][2], x[tt][n][3]), make_float2(pbn, pbn));
                            pb0[n] = movtrans(pack_half2(wa.x, wa.y));
                            pb1[n] = movtrans(pack_half2(wb.x, wb.y));
                        } else {
                            pb0[n] = movtrans(pack_half2(x[tt][n][0] * pa, 0.f));
                            pb1[n] = movtrans(pack_half2(x[tt][n][2] * pbn, 0.f));
                        }
                    }
                    // A quad of dim tile mt: transposed pairs 2mt, 2mt+1 of token block 0
                    // (tokens 0-7 of the tile) then of block 1 (tokens 8-15); group J of
                    // both tokens feeds dim tiles 2J and 2J+1
                    const uint8_t* rva = st + C::kVOff + (tile * 16 + g) * C::kRbV;
                    const uint8_t* rvb = st + C::kVOff + (tile * 16 + g + 8) * C::kRbV;
                    const QuarterWords va = load_quarter<VB>(rva + t * C::kQuarterV);
                    const QuarterWords vb = load_quarter<VB>(rvb + t * C::kQuarterV);
                    const Tables vt = v_tables_all();
                    const Tables tva = TAB ? v_tables<FULL>(rva, tok0 + tile * 16 + g < t_end) : vt;
                    const Tables tvb = TAB ? v_tables<FULL>(rvb, tok0 + tile * 16 + g + 8 < t_end) : vt;
                    auto vgroup = [&](auto jtag) {
                        constexpr int J = decltype(jtag)::value;
                        uint32_t ha[4], hb[4], unused[2];
                        dequant_group<VB, J, false>(va, tva, 0u, 0u, ha, unused);
                        dequant_group<VB, J, false>(vb, tvb, 0u, 0u, hb, unused);
                        if constexpr (BIG) {  // c * n_v per token (tokens g and g + 8 of the tile)
                            const __half2 sa = __float2half2_rn(nv[tt][0]);
                            const __half2 sb = __float2half2_rn(nv[tt][1]);
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
            if (tok0 + C::kChunk <= t_end && tok0 + C::kChunk <= all_visible_below) {
                process(st, tok0, 0, std::true_type{});
                if constexpr (TPC == 1) process(st, tok0, 1, std::true_type{});
            } else {
                process(st, tok0, 0, std::false_type{});
                if constexpr (TPC == 1)
                    if (t_end - tok0 > 16) process(st, tok0, 1, std::false_type{});
            }
            __syncwarp();
            const int cn = c + C::kWarps * C::kStages;
            if (cn < nchunks && lane == 0) {
                fence_proxy_async();
                issue(cn, stage);
            }
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }

        if (pos + nchunks >= hi) griddep_launch_dependents();  // last segment: let the merge launch
        if (sparse && lane == 0 && tiles_seen) {
            atomicAdd(p.sparse_tiles, tiles_skipped);
            atomicAdd(p.sparse_tiles + 1, tiles_seen);
        }
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
            for (int e = 0; e < NE; ++e) {
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 4);
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 8);
                l[n][e] += __shfl_xor_sync(0xffffffffu, l[n][e], 16);
            }
        __syncthreads();  // every warp is done with its pipeline stages
        float* sO = reinterpret_cast<float*>(smem) + warp * C::kRows * C::kOStride;
        float* sML = reinterpret_cast<float*>(smem) + C::kWarps * C::kRows * C::kOStride;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                const int r = C::slot_row(n, e, t);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int dlo = 32 * (g >> 1) + 4 * mt + (g & 1);
                    sO[r * C::kOStride + dlo] = O[n][mt][e];
                    sO[r * C::kOStride + dlo + 2] = O[n][mt][e + 2];
                }
                if (g == 0) {
                    sML[(warp * C::kRows + r) * 2 + 0] = m[n][e];
                    sML[(warp * C::kRows + r) * 2 + 1] = l[n][e];
                }
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


template <int KB, int VB, int ROWS, bool TAB, bool RES>
int launch_decode_t(const DecodeParams& p, const CUtensorMap* kmap, cudaStream_t stream,
                    cudaEvent_t ev0, cudaEvent_t ev1) {
    using C = DecCfg<KB, VB, ROWS, TAB, RES>;
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t e = set_smem_attr_once(tq_decode_kernel<KB, VB, ROWS, TAB, RES>, C::kSmemAlloc, attr_done);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_ctas);
    if (ev0) cudaEventRecord(ev0, stream);
    e = launch_pdl(tq_decode_kernel<KB, VB, ROWS, TAB, RES>, grid, dim3(C::kWarps * 32),
                               C::kSmemAlloc, stream, p, *kmap);
    if (ev1) cudaEventRecord(ev1, stream);
    return e;
}

// Resident CTAs per SM: the launch bounds' target, unless shared memory
// (228 KB per SM, 1 KB of it reserved per CTA) allows fewer.
template <int KB, int VB, int ROWS, bool TAB, bool RES>
int ctas_of() {
    using C = DecCfg<KB, VB, ROWS, TAB, RES>;
    const int by_smem = (228 * 1024) / (C::kSmemAlloc + 1024);
    return by_smem < C::kMinCtas ? by_smem : C::kMinCtas;
}

// The variants of one translation unit: launch (ev0/ev1 may be null) or, with
// launch == false, the resident CTAs per SM; cudaErrorInvalidValue / 0 when
// the unit does not hold the variant.
#define TQ_DECODE_VARIANT(KB_, VB_, ROWS_, TAB_, RES_)                                             \
    if (kb == KB_ && vb == VB_ && rows == ROWS_ && table == TAB_ && res == RES_)                   \
        return launch ? launch_decode_t<KB_, VB_, ROWS_, TAB_, RES_>(p, kmap, stream, ev0, ev1)    \
                      : ctas_of<KB_, VB_, ROWS_, TAB_, RES_>();

}  // namespace tq
