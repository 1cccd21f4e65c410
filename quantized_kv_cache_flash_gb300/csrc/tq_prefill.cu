// Chunked-prefill attention over the packed KV cache on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Same result as the decode kernels -- query j of a Tq block attends to
// tokens [0, L - Tq + j] of its sequence, scores and P.V in the rotated basis,
// only the output inverse-rotated (mlxcel pull request #369, Change) -- for
// blocks of many queries (a prefill chunk), where every K/V tile serves 128
// query rows and the two products are dense GEMMs:
//   S[128 rows x 128 tok]  = Q'[128 x 128] . K^T     (8 or 16 MMAs of K = 16, fp32 in TMEM)
//   O[128 rows x 128 dim] += P[128 x 128 tok] . V    (8 MMAs, fp32 in TMEM)
// Q' = Rot(q) (quantized K) or q (fp16 K); the softmax scale * log2(e) and
// the K norm are applied to the fp32 scores.  fp16 K: q and K are fp16
// inputs, their products exact.  Quantized K: Rot(q) is not an fp16 value,
// so it is split into q_hi = fp16(Rot q) and q_lo = fp16(Rot q - q_hi) and S
// takes both products (16 MMAs of K = 16 per query tile instead of 8); the K
// tile holds the fp16 centroids c[idx], exact for a codebook of fp16 values
// (other codebooks are not taken by this kernel).  K and V are dequantised
// once per tile into shared memory (the 128-byte-swizzled K-major layout the
// MMA descriptors read); V transposed, [dim][token], as fp16 c[idx] * n_v (a
// tile has half as many V values as P values, so the norm goes there).
//
// CTA = 256 threads on one (batch, kv head, pair of 128-row query tiles):
// thread = one query row (tensor-memory lane) of one tile, so each K/V tile is
// dequantised once for 256 rows.  Tensor memory holds, per query tile, S (128
// columns, whose first 64 take P back as fp16 pairs for the P.V MMA) and O
// (128 columns): all 512.  The MMAs overlap the CUDA-core work and the two
// query tiles take turns on the tensor core: S(n) runs while tile 1's warps
// dequantise V(n), S_1(n) during tile 0's softmax, P.V_0(n) during tile 1's,
// and tile 0's warps dequantise K(n + 1) during tile 1's softmax and
// P.V_1(n).  Packed records of the next tiles
// stream into two staging slots by bulk copies (fp16 K by 2-D tensor-map
// copies straight into the MMA layout); every mbarrier wait is bounded.
#include <float.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

template <int KB, int VB>
struct PreCfg {
    static constexpr int kTile = 128;                           // tokens per tile = rows per CTA
    static constexpr int kRbK = (KB == 0) ? 256 : KB * 16;
    static constexpr int kRbV = VB * 16;
    static constexpr int kQOff = 0;                             // fp16 Q' (q_hi) of the two query tiles (64 KB)
    static constexpr int kVtOff = 65536;                        // fp16 V^T [dim][token] (32 KB)
    static constexpr int kKOff = 98304;                         // fp16 K [token][dim] (quantized K)
    static constexpr int kQloOff = kKOff + 32768;               // fp16 q_lo of the two tiles (quantized K, 64 KB)
    static constexpr int kStgOff = (KB == 0) ? kKOff : kQloOff + 65536;
    // staging slot: K (fp16 K: the MMA tile itself, 32 KB; else records), K norms, V records, V norms
    static constexpr int kSK = (KB == 0) ? 32768 : kTile * kRbK;
    static constexpr int kSKn = (KB == 0) ? 0 : kTile * 2;
    static constexpr int kSV = kTile * kRbV;
    static constexpr int kSVn = kTile * 2;
    static constexpr int kSlotRaw = kSK + kSKn + kSV + kSVn;
    // (fp16 K is read by the MMA straight from the slot: 1024-byte aligned)
    static constexpr int kSlotAlign = (KB == 0) ? 1024 : 128;
    static constexpr int kSlot = (kSlotRaw + kSlotAlign - 1) / kSlotAlign * kSlotAlign;
    static constexpr int kColOff = kStgOff + 2 * kSlot;         // fp32 n_k * scale * log2(e) [128]
    // mbarriers stg[2], S[2], O[2] (one per query tile), V^T stored, K stored,
    // tile 1's softmax done; TMEM slot; last tile copied
    static constexpr int kBarOff = kColOff + kTile * 4;
    static constexpr int kSmem = kBarOff + 80;
    static constexpr int kSmemAlloc = kSmem + 1024;             // base alignment slack
    static constexpr uint32_t kIdesc = umma_idesc_f16_f32(128, 128);
};

template <int BITS>
__device__ __forceinline__ void dequant_q32(const uint8_t* rec, const Tables& t, uint32_t (&h)[16]) {
    if constexpr (BITS == 3) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(rec);
        dequant3_quarter(w[0], w[1], w[2], t, h);
    } else {
        dequant4_quarter(*reinterpret_cast<const uint4*>(rec), t, h);
    }
}

// Four 8x8 b16 matrices stored transposed: register i of lane 4r + c holds
// elements (r, 2c) and (r, 2c+1) of matrix i; matrix i's row k lands at the
// address given by lane 8i + k as elements (0..7, k).
__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                              uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// In-thread 128-point Walsh-Hadamard transform (unnormalised).  From stride
// 2 on, a butterfly's elements i, i + 1 pair with i + h, i + h + 1, so those
// stages run on packed fp32 pairs (a - b as fma(b, -1, a), exact).
__device__ __forceinline__ void wht128_thread(float (&x)[128]) {
#pragma unroll
    for (int i = 0; i < 128; i += 2) {
        const float a = x[i], b = x[i + 1];
        x[i] = a + b;
        x[i + 1] = a - b;
    }
    const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int h = 2; h < 128; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
            if (i & h) continue;
            const float2 a = make_float2(x[i], x[i + 1]), b = make_float2(x[i + h], x[i + h + 1]);
            const float2 sum = __fadd2_rn(a, b), dif = __ffma2_rn(b, m1, a);
            x[i] = sum.x;
            x[i + 1] = sum.y;
            x[i + h] = dif.x;
            x[i + h + 1] = dif.y;
        }
    }
}

template <int KB, int VB>
__global__ void __launch_bounds__(256, 1)
    tq_prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap kmap) {
    using C = PreCfg<KB, VB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    // thread = (query tile tl of the CTA's two, row r = TMEM lane): warps 0-3
    // hold the rows of the first tile, warps 4-7 those of the second
    const int tl = tid >> 7, r = tid & 127;

    // heaviest (latest) query tiles first
    const int npairs = (p.mtiles + 1) / 2;
    const int pair = npairs - 1 - static_cast<int>(blockIdx.x);
    const int mt = 2 * pair + tl;
    const int unit = blockIdx.y;  // b * hkv + h
    const int b = unit / p.hkv, h = unit - b * p.hkv;
    griddep_wait();  // cache, lengths and q come from earlier work on the stream
    const int L = p.lengths[b];
    const int t_lim = min(L, p.max_len);
    // row r of tile mt: query position j, head hl of the group
    const int jl = r / p.group, hl = r - jl * p.group;
    const int j = mt * p.pos_per_tile + jl;
    const bool row_ok = mt < p.mtiles && jl < p.pos_per_tile && j < p.tq;
    const int lim = row_ok ? min(L - p.tq + j, t_lim - 1) : -1;  // last visible token
    // this tile's rows see every token up to lim_lo; the CTA's tiles end at `last`
    const int lim_lo = mt < p.mtiles ? min(L - p.tq + mt * p.pos_per_tile, t_lim - 1) : -1;
    const int j_hi = min(p.tq - 1, (2 * pair + 2) * p.pos_per_tile - 1);
    const int last = min(L - p.tq + j_hi, t_lim - 1);
    const int ntiles = last >= 0 ? last / C::kTile + 1 : 0;
    const size_t row0 = static_cast<size_t>(unit) * p.cap;

    uint8_t* sQ = smem + C::kQOff;       // [2][128 x 128] fp16
    uint8_t* sVt = smem + C::kVtOff;
    // n_k * scale * log2(e) per token (quantized K), written with K's dequant
    float* colK = reinterpret_cast<float*>(smem + C::kColOff);
    const uint32_t bar_stg = smem_u32(smem + C::kBarOff);       // 2 x 8 bytes
    const uint32_t bar_s = bar_stg + 16, bar_o = bar_stg + 32, bar_v = bar_stg + 48;
    const uint32_t bar_kr = bar_stg + 56, bar_sm1 = bar_stg + 64;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 72);
    int* last_issued = reinterpret_cast<int*>(smem + C::kBarOff + 76);  // last tile whose copy was issued

    auto issue = [&](int n) {  // one thread: tile n into staging slot n & 1
        const int tok0 = n * C::kTile;
        const int nval = min(C::kTile, t_lim - tok0);
        uint8_t* slot = smem + C::kStgOff + (n & 1) * C::kSlot;
        const uint32_t bar = bar_stg + 8 * (n & 1);
        const uint32_t nb = static_cast<uint32_t>((nval + 7) & ~7) * 2;
        uint32_t bytes = nval * C::kRbV + nb;
        bytes += (KB == 0) ? 32768u : nval * C::kRbK + nb;
        mbar_arrive_expect_tx(bar, bytes);
        if constexpr (KB == 0) {
            // 128 rows x 128 dims in four 32-row boxes per 64-dim half (rows past
            // the tensor's end are zero-filled; masked below)
            for (int half = 0; half < 2; ++half)
                for (int rb = 0; rb < 4; ++rb)
                    tma_g2s_2d(smem_u32(slot) + half * 16384 + rb * 4096, &kmap, half * 64,
                               static_cast<int32_t>(row0 + tok0 + rb * 32), bar);
        } else {
            bulk_g2s(smem_u32(slot), p.k_codes + (row0 + tok0) * C::kRbK, nval * C::kRbK, bar);
            bulk_g2s(smem_u32(slot + C::kSK), p.k_norm + row0 + tok0, nb, bar);
        }
        bulk_g2s(smem_u32(slot + C::kSK + C::kSKn), p.v_codes + (row0 + tok0) * C::kRbV,
                 nval * C::kRbV, bar);
        bulk_g2s(smem_u32(slot + C::kSK + C::kSKn + C::kSV), p.v_norm + row0 + tok0, nb, bar);
    };

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(bar_stg + 8 * i, 1);  // stg[2], S[2], O[2]
        mbar_init(bar_v, 128);  // the V dequant's threads
        mbar_init(bar_kr, 1);
        mbar_init(bar_sm1, 1);
        fence_barrier_init();
        for (int n = 0; n < 2 && n < ntiles; ++n) issue(n);
        *last_issued = min(ntiles, 2) - 1;
    }
    // tensor memory: tile t at columns 256 t: S (128, its first 64 reused for
    // P as fp16 pairs), then O (128)
    if (warp == 0) tmem_alloc(smem_u32(tslot), 512);

    // ---- Q' = Rot(q) as q_hi + q_lo (quantized K) or q (fp16 K) ----
    uint8_t* sQt = sQ + tl * 32768;
    uint8_t* sQlt = smem + C::kQloOff + tl * 32768;
    {
        float x[128];
        if (row_ok) {
            const __half* qp = p.q + ((static_cast<size_t>(b) * p.hq + h * p.group + hl) * p.tq + j) * kD;
#pragma unroll
            for (int k = 0; k < 128; k += 8) {
                const uint4 w = *reinterpret_cast<const uint4*>(qp + k);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
                    x[k + 2 * e] = f.x;
                    x[k + 2 * e + 1] = f.y;
                }
            }
            if constexpr (KB != 0) {
#pragma unroll
                for (int k = 0; k < 128; ++k) x[k] = ((p.signs[k >> 5] >> (k & 31)) & 1u) ? -x[k] : x[k];
                wht128_thread(x);
#pragma unroll
                for (int k = 0; k < 128; k += 2) {  // 1/sqrt(128)
                    const float2 v = __fmul2_rn(make_float2(x[k], x[k + 1]),
                                                make_float2(0.08838834764831845f, 0.08838834764831845f));
                    x[k] = v.x;
                    x[k + 1] = v.y;
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 128; ++k) x[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 128; k += 8) {
            uint32_t hv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) hv[e] = pack_half2(x[k + 2 * e], x[k + 2 * e + 1]);
            *reinterpret_cast<uint4*>(sQt + sw128_offset(r, k)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            if constexpr (KB != 0) {  // q_lo = Rot(q) - q_hi (exact in fp32), rounded once more
                uint32_t lv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hv[e]));
                    lv[e] = pack_half2(x[k + 2 * e] - hf.x, x[k + 2 * e + 1] - hf.y);
                }
                *reinterpret_cast<uint4*>(sQlt + sw128_offset(r, k)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
            }
        }
    }
    fence_proxy_async();  // the MMAs read Q' through the async proxy
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + 256 * tl + lane_off;         // this row of S (and of P)
    const uint32_t t_o = tmem + 256 * tl + 128 + lane_off;   // this row of O

    float m_base = -INFINITY, l_sum = 0.f;
    bool stalled = false;  // once set, waits return at once and no MMA or copy is issued
    int issued_o = 0;      // P.V batches of this thread's query tile
    const uint32_t bar_st = bar_s + 8 * tl, bar_ot = bar_o + 8 * tl;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!stalled && !mbar_wait_bounded(bar, parity)) stalled = true;
    };

    // K(n) -> sK, one token per thread of query tile 0's warps (fp16 K: the
    // tile is read in place from the staging slot)
    auto k_dequant = [&](int n) {
        if constexpr (KB != 0) {
            // (tables from the parameters at each use: none held across the loop)
            const Tables kt{p.ktab[0], p.ktab[1], p.ktab[2], p.ktab[3]};
            const uint8_t* rec = smem + C::kStgOff + (n & 1) * C::kSlot + r * C::kRbK;
            uint8_t* sK = smem + C::kKOff;
#pragma unroll 1
            for (int quarter = 0; quarter < 4; ++quarter) {
                uint32_t hh[16];
                dequant_q32<KB>(rec + quarter * (C::kRbK / 4), kt, hh);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    *reinterpret_cast<uint4*>(sK + sw128_offset(r, 32 * quarter + 8 * m)) =
                        make_uint4(hh[4 * m], hh[4 * m + 1], hh[4 * m + 2], hh[4 * m + 3]);
            }
            fence_proxy_async();
        }
    };
    // colK of tile n (n_k * scale * log2 e per token, 0 past the end)
    auto k_scales = [&](int n) {
        if constexpr (KB != 0) {
            const uint8_t* slot = smem + C::kStgOff + (n & 1) * C::kSlot;
            const float nk = __half2float(reinterpret_cast<const __half*>(slot + C::kSK)[r]);
            colK[r] = n * C::kTile + r < t_lim ? nk * p.scale_log2e : 0.f;
        }
    };
    // S_t(n) = Q'_t . K(n)^T into tile t's S columns
    auto issue_s = [&](int n, int t2) {
        const uint32_t kbase = (KB == 0) ? smem_u32(smem + C::kStgOff + (n & 1) * C::kSlot) : smem_u32(smem + C::kKOff);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_f16(tmem + 256 * t2, umma_desc_sw128(smem_u32(sQ) + t2 * 32768 + koff),
                     umma_desc_sw128(kbase + koff), C::kIdesc, kk > 0 ? 1u : 0u);
            if constexpr (KB != 0)  // + q_lo . K^T
                umma_f16(tmem + 256 * t2, umma_desc_sw128(smem_u32(smem + C::kQloOff) + t2 * 32768 + koff),
                         umma_desc_sw128(kbase + koff), C::kIdesc, 1u);
        }
        umma_commit(bar_s + 8 * t2);
    };
    // O_t += P_t(n) . V(n), P from tensor memory over S_t
    auto issue_pv = [&](int n, int t2) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_f16_ts(tmem + 256 * t2 + 128, tmem + 256 * t2 + 8 * kk,
                        umma_desc_sw128(smem_u32(sVt) + koff), C::kIdesc, (n > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar_o + 8 * t2);
    };
    // V(n)^T for the 16 tokens 16 vw .. 16 vw + 15 (query tile 1's warps take
    // vw = warp - 4 and vw = warp): thread (g, t) = lane 4g + t dequantises
    // quarter t of tokens 16vw+g and 16vw+g+8 (the MMA fragment layout, so
    // stmatrix.trans writes [dim][token] rows); V^T rows are stored in the order
    // pi(d) = d ^ 2(d >> 5), which puts the 8 rows of each stored 8x8 matrix in
    // 8 different 16-byte bank groups (the epilogue reads O's columns back
    // through the same pi)
    auto v_dequant = [&](int n, int vw) {
        const Tables vt{p.vtab[0], p.vtab[1], p.vtab[2], p.vtab[3]};
        const uint8_t* slot = smem + C::kStgOff + (n & 1) * C::kSlot;
        const int tok0 = n * C::kTile;
        const int lane = tid & 31, g = lane >> 2, tq4 = lane & 3;
        const int ta = 16 * vw + g, tb = ta + 8;
        const uint8_t* vrec = slot + C::kSK + C::kSKn;
        const __half* vnorm = reinterpret_cast<const __half*>(slot + C::kSK + C::kSKn + C::kSV);
        // tokens past the end: stale records still decode to finite
        // centroids, and their norm (and weight) is 0
        uint32_t ha[16], hb[16];
        dequant_q32<VB>(vrec + ta * C::kRbV + tq4 * (C::kRbV / 4), vt, ha);
        dequant_q32<VB>(vrec + tb * C::kRbV + tq4 * (C::kRbV / 4), vt, hb);
        // n_v scales the stored values, so P itself goes to the MMA: 128 x
        // 128 multiplies a tile instead of the 256 x 128 of scaling P
        const __half2 na = tok0 + ta < t_lim ? __half2half2(vnorm[ta]) : __float2half2_rn(0.f);
        const __half2 nb = tok0 + tb < t_lim ? __half2half2(vnorm[tb]) : __float2half2_rn(0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const __half2 a = __hmul2(*reinterpret_cast<const __half2*>(&ha[k]), na);
            const __half2 b = __hmul2(*reinterpret_cast<const __half2*>(&hb[k]), nb);
            ha[k] = *reinterpret_cast<const uint32_t*>(&a);
            hb[k] = *reinterpret_cast<const uint32_t*>(&b);
        }
        // stmatrix k2 stores dim pairs 2k2 (matrices 0, 1: tokens A, B) and
        // 2k2+1 (matrices 2, 3); lane 8j + c gives row c of matrix j: dim
        // d = 32(c>>1) + 2(2k2 + (j>>1)) + (c&1), tokens 16vw + 8(j&1) .. + 7
        const int sj = lane >> 3, sc = lane & 7;
        const int tokc = 2 * (vw & 3) + (sj & 1);  // 16-byte chunk of the tokens in their row
        uint32_t vaddr[2];
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            const int row = 32 * (sc >> 1) + 2 * ((((par << 1) | (sj >> 1)) ^ (sc >> 1)) & 3) + (sc & 1);
            vaddr[par] = smem_u32(sVt) + (vw >> 2) * 16384 + row * 128 + ((tokc ^ (row & 7)) << 4);
        }
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2)
            stsm_x4_trans(vaddr[k2 & 1] + 1024 * (k2 >> 1), ha[2 * k2], hb[2 * k2], ha[2 * k2 + 1],
                          hb[2 * k2 + 1]);
    };
    // softmax_t(n) of this thread's row (log2 domain): P over S_t's first 64
    // columns as fp16 pairs; O_t rescaled in place when the row's base moves
    auto softmax = [&](int n) {
        const int tok0 = n * C::kTile;
        float x[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(t_s + 32 * c, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(v[e]);
        }
        // t = s * n_k * scale * log2(e) - base in one FFMA per score; the base moves only when a
        // score passes it by more than 4 (so p <= 16 in fp16)
        const bool fresh = (m_base == -INFINITY);
        const float base0 = fresh ? 0.f : m_base;
        // (packed pairs: one instruction per two scores)
        const float2 nb2 = make_float2(-base0, -base0);
#pragma unroll
        for (int e = 0; e < 128; e += 4) {
            const float sl = p.scale_log2e;
            float4 nk = make_float4(sl, sl, sl, sl);
            if constexpr (KB != 0) nk = *reinterpret_cast<const float4*>(colK + e);
            const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), make_float2(nk.x, nk.y), nb2);
            const float2 b = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), make_float2(nk.z, nk.w), nb2);
            x[e] = a.x;
            x[e + 1] = a.y;
            x[e + 2] = b.x;
            x[e + 3] = b.y;
        }
        if (tok0 + C::kTile - 1 > lim_lo) {  // a tile some row of this query tile sees in part
#pragma unroll
            for (int e = 0; e < 128; ++e)
                if (tok0 + e > lim) x[e] = -INFINITY;
        }
        // row max over four independent chains (16 deep instead of 64)
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 128; e += 8)
#pragma unroll
            for (int j = 0; j < 4; ++j) mq[j] = fmaxf(mq[j], fmaxf(x[e + 2 * j], x[e + 2 * j + 1]));
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        const bool grow = fresh ? (mx > -INFINITY) : (mx > 4.f);
        if (__any_sync(0xffffffffu, grow)) {
            // rows that grow move their base up by mx (t -= mx below); the others keep it
            const float shift = grow ? mx : 0.f;
            const float alpha = grow ? (fresh ? 0.f : fast_exp2(-mx)) : 1.f;
            l_sum *= alpha;
            if (grow) m_base = base0 + mx;  // a row that saw no token yet keeps no base
#pragma unroll
            for (int e = 0; e < 128; ++e) x[e] -= shift;
            if (issued_o > 0) {  // rescale this row of O in tensor memory (P.V(n-1) is done)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_o + 32 * c, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(t_o + 32 * c, v);
                }
            }
        }
        // row sum as four independent packed pairs (chains 16 deep instead of 64)
        float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int k = 64 * c + 2 * e;
                const float p0 = fast_exp2(x[k]), p1 = fast_exp2(x[k + 1]);
                s2[e & 3] = __fadd2_rn(s2[e & 3], make_float2(p0, p1));
                pk[e] = pack_half2(p0, p1);
            }
            tmem_st32(t_s + 32 * c, pk);  // P over S columns 0..63 (tokens 64c..64c+63)
        }
        const float2 sa = __fadd2_rn(s2[0], s2[1]), sb = __fadd2_rn(s2[2], s2[3]);
        const float2 st = __fadd2_rn(sa, sb);
        l_sum += st.x + st.y;
    };

    // Query tile 0's warps (0-3) dequantise K and its scales and issue S_0 and
    // P.V_0 (thread 0); query tile 1's warps (4-7) dequantise V and issue S_1,
    // P.V_1 and the copies (thread 128).  Per K/V tile n the tensor core takes
    // S_0(n), S_1(n) (named barrier 3 keeps that order), P.V_0(n), P.V_1(n):
    // tile 0's softmax runs under S_1, tile 1's under P.V_0 and the K(n+1)
    // dequant.  The two groups hand over through mbarriers: bar_kr (K(n) and
    // its scales stored), bar_v (V(n)^T stored), bar_sm1 (tile 1's softmax(n)
    // is past its reads of the scales).  No thread leaves the loop early, so
    // every named barrier is met; after a wait times out the thread's later
    // waits return at once and it issues nothing more.
    if (tl == 0 && ntiles > 0) {
        wait(bar_stg, 0);
        k_dequant(0);
        k_scales(0);
    }
    for (int n = 0; n < ntiles; ++n) {
        if (tl == 0) {
            tc_fence_before();
            named_bar_sync(1, 128);  // K(n) and its scales are stored
            tc_fence_after();
            if (r == 0) {
                mbar_arrive(bar_kr);
                if (n > 0) wait(bar_o, (n - 1) & 1);  // P.V_0(n-1) has read P_0
                tc_fence_after();
                if (!stalled) issue_s(n, 0);
            }
            __syncwarp();
            if (warp == 0) named_bar_arrive(3, 64);  // S_0(n) is queued: S_1(n) may follow
            if (n > 0) wait(bar_o, (n - 1) & 1);    // O_0 and the P_0 columns are free
        } else {
            // V(n), once its records landed and both P.V(n-1) have read V(n-1)^T
            wait(bar_stg + 8 * (n & 1), (n >> 1) & 1);
            if (n > 0) {
                wait(bar_o, (n - 1) & 1);
                wait(bar_o + 8, (n - 1) & 1);
            }
            v_dequant(n, warp - 4);
            v_dequant(n, warp);
            fence_proxy_async();
            mbar_arrive(bar_v);
            if (warp == 4) {
                named_bar_sync(3, 64);
                if (r == 0) {
                    tc_fence_after();
                    if (!stalled) issue_s(n, 1);
                }
                __syncwarp();
            }
            wait(bar_kr, n & 1);  // the scales of tile n are stored
        }
        wait(bar_st, n & 1);
        tc_fence_after();
        softmax(n);
        tc_fence_before();
        if (named_bar_or(1 + tl, 128, stalled)) stalled = true;  // P_tl(n) is stored
        tc_fence_after();
        if (tl == 0) {
            if (r == 0) {
                wait(bar_v, n & 1);  // V(n)^T is stored
                tc_fence_after();
                if (!stalled) issue_pv(n, 0);
            }
            if (n + 1 < ntiles) {  // K(n+1), under tile 1's softmax(n)
                wait(bar_stg + 8 * ((n + 1) & 1), ((n + 1) >> 1) & 1);
                wait(bar_s + 8, n & 1);  // S_1(n) has read K(n)
                k_dequant(n + 1);
                wait(bar_sm1, n & 1);    // tile 1's softmax(n) is done with the scales
                k_scales(n + 1);
            }
        } else if (r == 0) {
            // P.V_1(n) first: S_0(n+1) queues behind it on the tensor core
            mbar_arrive(bar_sm1);   // tile 1's softmax(n) is past its reads of the scales
            tc_fence_after();
            if (!stalled) issue_pv(n, 1);
            wait(bar_s, n & 1);     // S_0(n) is done (fp16 K reads it from the slot)
            if (!stalled && n + 2 < ntiles) {  // tile n's staging slot is consumed
                issue(n + 2);
                *last_issued = n + 2;
            }
        }
        ++issued_o;
    }

    // ---- epilogue: O / l, v_rescale, inverse rotation, fp16 ----
    bool ok = !stalled;
    if (issued_o > 0 && !mbar_wait_bounded(bar_ot, (issued_o - 1) & 1)) ok = false;
    ok = __syncthreads_and(ok) != 0;  // one decision for the whole CTA
    tc_fence_after();
    if (!ok) {
        if (tid == 0) atomicOr(p.status, kStatusPipelineStall);
    } else {
        float o[128];
        if (issued_o > 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // every lane: the loads are warp-collective
                uint32_t v[32];
                tmem_ld32(t_o + 32 * c, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[32 * c + e] = __uint_as_float(v[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 128; ++e) o[e] = 0.f;
        }
        if (row_ok) {
            float inv = 0.f;
            if (l_sum > 0.f) inv = p.v_rescale / l_sum;
            else atomicOr(p.status, kStatusShortContext);
            // 1/l, v_rescale and the rotation's 1/sqrt(128), applied after the
            // (linear) transform in one packed multiply
            const float g = inv * 0.08838834764831845f;
            // O's column pi(d) holds dim d (V^T rows were stored in pi order)
            float od[128];
#pragma unroll
            for (int d = 0; d < 128; ++d) od[d] = o[d ^ (2 * (d >> 5))];
#pragma unroll
            for (int d = 0; d < 128; ++d) o[d] = od[d];
            wht128_thread(o);
            __half* op = p.out + ((static_cast<size_t>(b) * p.hq + h * p.group + hl) * p.tq + j) * kD;
#pragma unroll
            for (int k = 0; k < 128; k += 8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 v = __fmul2_rn(make_float2(o[k + e], o[k + e + 1]), make_float2(g, g));
                    y[e] = ((p.signs[(k + e) >> 5] >> ((k + e) & 31)) & 1u) ? -v.x : v.x;
                    y[e + 1] = ((p.signs[(k + e + 1) >> 5] >> ((k + e + 1) & 31)) & 1u) ? -v.y : v.y;
                }
                *reinterpret_cast<uint4*>(op + k) = make_uint4(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]),
                                                               pack_half2(y[4], y[5]), pack_half2(y[6], y[7]));
            }
        }  // padding rows write nothing
    }
    if (!ok) {
        // let the copies still in flight land before the shared memory goes away
        const int li = *last_issued;
        for (int m = li > 0 ? li - 1 : 0; m <= li; ++m)
            (void)mbar_wait_bounded(bar_stg + 8 * (m & 1), (m >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KB, int VB>
static int launch_prefill_t(const PrefillParams& p, const CUtensorMap* kmap, cudaStream_t stream) {
    using C = PreCfg<KB, VB>;
    static std::atomic<uint64_t> attr_done{0};
    const cudaError_t e = set_smem_attr_once(tq_prefill_kernel<KB, VB>, C::kSmemAlloc, attr_done);
    if (e != cudaSuccess) return e;
    return launch_pdl(tq_prefill_kernel<KB, VB>, dim3((p.mtiles + 1) / 2, p.batch * p.hkv), dim3(256),
                      C::kSmemAlloc, stream, p, *kmap);
}

int launch_prefill(int kbits, int vbits, const PrefillParams& p, const CUtensorMap* kmap,
                   cudaStream_t stream) {
    if (kbits == 16 && vbits == 4) return launch_prefill_t<0, 4>(p, kmap, stream);
    if (kbits == 16 && vbits == 3) return launch_prefill_t<0, 3>(p, kmap, stream);
    if (kbits == 3 && vbits == 3) return launch_prefill_t<3, 3>(p, kmap, stream);
    if (kbits == 4 && vbits == 4) return launch_prefill_t<4, 4>(p, kmap, stream);
    if (kbits == 4 && vbits == 3) return launch_prefill_t<4, 3>(p, kmap, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tq
