// Fused split-K decode attention over the packed KV cache, and the split
// combine + inverse-rotation epilogue.
//
// Scores are taken in the rotated basis: score(t) = scale * n_k(t) *
// <Rot(q), c[idx_k(t)]> for quantized K (Rot is orthogonal, so this equals the
// score against the fully dequantized key), or scale * <q, k(t)> for fp16 K.
// V is never brought back to the original basis: P.V accumulates
// p(t) * n_v(t) * c[idx_v(t)] and only the [rows, 128] result is
// inverse-rotated, in the combine kernel (mlxcel pull request #369, Change:
// "inverse-rotates only the small [B, Hq, Tq, D] output").
//
// Work split: CTA = 4 warps on one (split of the context, batch*kv-head, row
// group).  Each warp streams its own 32-token chunks through a private ring
// of shared-memory stages filled by 1-D bulk copies (tensor-map tile copies
// with 128-byte swizzle for fp16 K), dequantizes in registers and runs the
// two contractions as warp MMAs with the query rows as M = 16:
//   S[16 x 8 tok]   = Rot(q)[16 x 128] . C_k^T            (8 k-steps)
//   O[16 x 128]    += (P * n_v)[16 x 16 tok] . C_v[16 x 128] (16 n-tiles)
// The K operand of a thread is its own token's quarter record (32 dims); the
// V operand comes from the same dequant followed by an 8x8 transpose.
#include <float.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

template <int KB, int VB>
struct DecCfg {
    static constexpr int kWarps = 4;
    static constexpr int kChunk = 32;                       // tokens per warp stage
    static constexpr int kStages = (KB == 0) ? 3 : 4;
    static constexpr int kRbK = (KB == 0) ? 256 : KB * 16;  // bytes per K record
    static constexpr int kRbV = VB * 16;
    static constexpr int kKBytes = kChunk * kRbK;
    static constexpr int kVOff = kKBytes;
    static constexpr int kVBytes = kChunk * kRbV;
    static constexpr int kKnOff = kVOff + kVBytes;
    static constexpr int kKnBytes = (KB == 0) ? 0 : kChunk * 2;
    static constexpr int kVnOff = kKnOff + kKnBytes;
    static constexpr int kStageRaw = kVnOff + kChunk * 2;
    static constexpr int kStageAlign = (KB == 0) ? 1024 : 128;
    static constexpr int kStage = (kStageRaw + kStageAlign - 1) / kStageAlign * kStageAlign;
    static constexpr int kPipeBytes = kWarps * kStages * kStage;
    static constexpr int kQOff = kPipeBytes;                 // fp32 [16][128] query rows
    static constexpr int kBarOff = kQOff + 16 * kD * 4;
    static constexpr int kSmem = kBarOff + kWarps * kStages * 8;
    static constexpr int kSmemAlloc = kSmem + 1024;          // base alignment slack
    // epilogue scratch (reuses the pipeline): per warp O[16][kOStride] + (m, l)[16]
    static constexpr int kOStride = kD + 8;
    static_assert(kWarps * 16 * kOStride * 4 + kWarps * 16 * 8 <= kPipeBytes, "scratch");
};

template <int KB, int VB>
__global__ void __launch_bounds__(128)
    tq_decode_kernel(const __grid_constant__ DecodeParams p,
                     const __grid_constant__ CUtensorMap kmap) {
    using C = DecCfg<KB, VB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int split = blockIdx.x, unit = blockIdx.y, rg = blockIdx.z;
    const int b = unit / p.hkv, h = unit - b * p.hkv;
    const int L = p.lengths[b];
    const int t_lim = min(L, p.max_len);
    const int t_begin = split * p.split_tokens;
    const int t_end = min(t_begin + p.split_tokens, t_lim);
    if (t_begin >= t_end) return;  // no tokens in this split (uniform over the CTA)
    const int nchunks = (t_end - t_begin + C::kChunk - 1) / C::kChunk;
    const size_t row0 = static_cast<size_t>(unit) * p.cap;

    uint8_t* wpipe = smem + warp * C::kStages * C::kStage;
    const uint32_t bar0 = smem_u32(smem + C::kBarOff) + warp * C::kStages * 8;

    auto issue = [&](int c, int stage) {  // lane 0 only
        const int tok0 = t_begin + c * C::kChunk;
        const int nval = min(C::kChunk, t_end - tok0);
        const uint32_t dst = smem_u32(wpipe + stage * C::kStage);
        const uint32_t bar = bar0 + stage * 8;
        const uint32_t nb = static_cast<uint32_t>((nval + 7) & ~7) * 2;  // norms, 16-B multiple
        uint32_t bytes = nval * C::kRbV + nb;
        if (KB == 0) bytes += 2 * 4096;
        else bytes += nval * C::kRbK + nb;
        mbar_arrive_expect_tx(bar, bytes);
        if constexpr (KB == 0) {
            tma_g2s_2d(dst, &kmap, 0, static_cast<int32_t>(row0 + tok0), bar);
            tma_g2s_2d(dst + 4096, &kmap, 64, static_cast<int32_t>(row0 + tok0), bar);
        } else {
            bulk_g2s(dst, p.k_codes + (row0 + tok0) * C::kRbK, nval * C::kRbK, bar);
            bulk_g2s(dst + C::kKnOff, p.k_norm + row0 + tok0, nb, bar);
        }
        bulk_g2s(dst + C::kVOff, p.v_codes + (row0 + tok0) * C::kRbV, nval * C::kRbV, bar);
        bulk_g2s(dst + C::kVnOff, p.v_norm + row0 + tok0, nb, bar);
    };

    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
        for (int s = 0; s < C::kStages; ++s) {
            const int c = warp + C::kWarps * s;
            if (c < nchunks) issue(c, s);
        }
    }
    __syncwarp();

    // ---- query rows of this row group -> shared (rotated for quantized K) ----
    float* sQ = reinterpret_cast<float*>(smem + C::kQOff);
    const int rbase = rg * 16;
    for (int r = warp; r < 16; r += C::kWarps) {
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
        *reinterpret_cast<float4*>(sQ + r * kD + lane * 4) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();

    // A fragments of the score MMA.  Quantized K: a thread's B operand is its
    // token's quarter `tig` (dims 32*tig .. +31) in order, so logical k-index
    // 16*kc + 2*tig + e maps to dim 32*tig + 4*kc + e (and +8 -> +2).
    uint32_t qa[8][4];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
        int d0, d1;
        if constexpr (KB != 0) { d0 = 32 * tig + 4 * kc; d1 = d0 + 2; }
        else { d0 = 16 * kc + 2 * tig; d1 = d0 + 8; }
        qa[kc][0] = pack_half2(sQ[g * kD + d0], sQ[g * kD + d0 + 1]);
        qa[kc][1] = pack_half2(sQ[(g + 8) * kD + d0], sQ[(g + 8) * kD + d0 + 1]);
        qa[kc][2] = pack_half2(sQ[g * kD + d1], sQ[g * kD + d1 + 1]);
        qa[kc][3] = pack_half2(sQ[(g + 8) * kD + d1], sQ[(g + 8) * kD + d1 + 1]);
    }

    const Tables kt{p.ktab[0], p.ktab[1], p.ktab[2], p.ktab[3]};
    const Tables vt{p.vtab[0], p.vtab[1], p.vtab[2], p.vtab[3]};
    // last visible token (inclusive) of the two rows this thread owns
    const int lim0 = L - p.tq + ((rbase + g) % p.tq);
    const int lim1 = L - p.tq + ((rbase + g + 8) % p.tq);

    float O[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool stalled = false;
    int it = 0;

    for (;; ++it) {
        const int c = warp + C::kWarps * it;
        if (c >= nchunks) break;
        const int stage = it % C::kStages;
        const uint32_t parity = (it / C::kStages) & 1;
        const bool ok = mbar_wait_bounded(bar0 + 8 * stage, parity);
        if (__any_sync(0xffffffffu, !ok)) { stalled = true; break; }
        const uint8_t* st = wpipe + stage * C::kStage;
        const int tok0 = t_begin + c * C::kChunk;

#pragma unroll 1
        for (int so = 0; so < C::kChunk; so += 16) {
            if (tok0 + so >= t_end) break;
            // ---------------- scores S = Rot(q) . C_k^T ----------------
            float S[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
                if constexpr (KB == 0) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int row = so + nt * 8 + (lane & 7);
                        const int db = 4 * jj + (lane >> 3);  // 16-byte chunk 0..15 of the row
                        const uint32_t addr = smem_u32(st) + (db >> 3) * 4096 + row * 128 +
                                              ((((db & 7) ^ (row & 7))) << 4);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(addr, r0, r1, r2, r3);
                        mma_f16(S[nt], qa[2 * jj][0], qa[2 * jj][1], qa[2 * jj][2], qa[2 * jj][3], r0, r1);
                        mma_f16(S[nt], qa[2 * jj + 1][0], qa[2 * jj + 1][1], qa[2 * jj + 1][2],
                                qa[2 * jj + 1][3], r2, r3);
                    }
                } else {
                    uint32_t hk[16];
                    const uint8_t* rec = st + (so + nt * 8 + g) * C::kRbK + tig * (C::kRbK / 4);
                    if constexpr (KB == 3) {
                        const uint32_t* w = reinterpret_cast<const uint32_t*>(rec);
                        dequant3_quarter(w[0], w[1], w[2], kt, hk);
                    } else {
                        dequant4_quarter(*reinterpret_cast<const uint4*>(rec), kt, hk);
                    }
#pragma unroll
                    for (int kc = 0; kc < 8; ++kc)
                        mma_f16(S[nt], qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], hk[2 * kc],
                                hk[2 * kc + 1]);
                }
            }

            // ---------------- online softmax (log2 domain) ----------------
            // this thread's tokens: so + {2tig, 2tig+1, 8+2tig, 9+2tig}
            const int ta = so + 2 * tig, tb = so + 8 + 2 * tig;
            float ks[4];
            if constexpr (KB == 0) {
                ks[0] = ks[1] = ks[2] = ks[3] = p.scale_log2e;
            } else {
                const float2 na = __half22float2(*reinterpret_cast<const __half2*>(st + C::kKnOff + 2 * ta));
                const float2 nb = __half22float2(*reinterpret_cast<const __half2*>(st + C::kKnOff + 2 * tb));
                ks[0] = na.x * p.scale_log2e; ks[1] = na.y * p.scale_log2e;
                ks[2] = nb.x * p.scale_log2e; ks[3] = nb.y * p.scale_log2e;
            }
            const float2 va = __half22float2(*reinterpret_cast<const __half2*>(st + C::kVnOff + 2 * ta));
            const float2 vb = __half22float2(*reinterpret_cast<const __half2*>(st + C::kVnOff + 2 * tb));
            const float nv[4] = {va.x, va.y, vb.x, vb.y};
            const int tg[4] = {tok0 + ta, tok0 + ta + 1, tok0 + tb, tok0 + tb + 1};
            float x0[4] = {S[0][0], S[0][1], S[1][0], S[1][1]};
            float x1[4] = {S[0][2], S[0][3], S[1][2], S[1][3]};
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool valid = tg[i] < t_end;
                x0[i] = (valid && tg[i] <= lim0) ? x0[i] * ks[i] : -INFINITY;
                x1[i] = (valid && tg[i] <= lim1) ? x1[i] * ks[i] : -INFINITY;
                mx0 = fmaxf(mx0, x0[i]);
                mx1 = fmaxf(mx1, x1[i]);
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
            const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
            m0 = mn0;
            m1 = mn1;
            float p0[4], p1[4], s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p0[i] = fast_exp2(x0[i] - base0);
                p1[i] = fast_exp2(x1[i] - base1);
                s0 += p0[i];
                s1 += p1[i];
            }
            l0 = l0 * al0 + s0;
            l1 = l1 * al1 + s1;
            if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    O[i][0] *= al0; O[i][1] *= al0;
                    O[i][2] *= al1; O[i][3] *= al1;
                }
            }
            float w0[4], w1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool valid = tg[i] < t_end;
                w0[i] = valid ? p0[i] * nv[i] : 0.f;
                w1[i] = valid ? p1[i] * nv[i] : 0.f;
            }
            const uint32_t a0 = pack_half2(w0[0], w0[1]);
            const uint32_t a1 = pack_half2(w1[0], w1[1]);
            const uint32_t a2 = pack_half2(w0[2], w0[3]);
            const uint32_t a3 = pack_half2(w1[2], w1[3]);

            // ---------------- O += (P n_v) . C_v (rotated basis) ----------------
            uint32_t bv0[16], bv1[16];
            {
                const uint8_t* rec = st + C::kVOff + (so + g) * C::kRbV + tig * (C::kRbV / 4);
                if constexpr (VB == 3) {
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(rec);
                    dequant3_quarter(w[0], w[1], w[2], vt, bv0);
                } else {
                    dequant4_quarter(*reinterpret_cast<const uint4*>(rec), vt, bv0);
                }
            }
            {
                const uint8_t* rec = st + C::kVOff + (so + 8 + g) * C::kRbV + tig * (C::kRbV / 4);
                if constexpr (VB == 3) {
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(rec);
                    dequant3_quarter(w[0], w[1], w[2], vt, bv1);
                } else {
                    dequant4_quarter(*reinterpret_cast<const uint4*>(rec), vt, bv1);
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                bv0[i] = movtrans(bv0[i]);
                bv1[i] = movtrans(bv1[i]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) mma_f16(O[i], a0, a1, a2, a3, bv0[i], bv1[i]);
        }

        __syncwarp();
        if (lane == 0) {
            const int cn = c + C::kWarps * C::kStages;
            if (cn < nchunks) {
                fence_proxy_async();
                issue(cn, stage);
            }
        }
    }

    if (stalled) {
        // Drain this warp's copies still in flight (bounded), flag, and stop.
        for (int k = 0; k < C::kStages; ++k) {
            const int c = warp + C::kWarps * (it + k);
            if (c >= nchunks) break;
            const int stage = (it + k) % C::kStages;
            (void)mbar_wait_bounded(bar0 + 8 * stage, ((it + k) / C::kStages) & 1);
        }
        if (lane == 0) atomicOr(p.status, kStatusPipelineStall);
    }

    // ---- combine the 4 warps of the CTA, write this split's partial ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();  // every warp is done with its pipeline stages
    float* sO = reinterpret_cast<float*>(smem) + warp * 16 * C::kOStride;
    float* sML = reinterpret_cast<float*>(smem) + C::kWarps * 16 * C::kOStride;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int d = 32 * tig + 2 * i;
        *reinterpret_cast<float2*>(sO + g * C::kOStride + d) = make_float2(O[i][0], O[i][1]);
        *reinterpret_cast<float2*>(sO + (g + 8) * C::kOStride + d) = make_float2(O[i][2], O[i][3]);
    }
    if (tig == 0) {
        sML[(warp * 16 + g) * 2 + 0] = m0;
        sML[(warp * 16 + g) * 2 + 1] = l0;
        sML[(warp * 16 + g + 8) * 2 + 0] = m1;
        sML[(warp * 16 + g + 8) * 2 + 1] = l1;
    }
    __syncthreads();
    {
        const int r = threadIdx.x >> 3;
        const int d0 = (threadIdx.x & 7) * 16;
        if (rbase + r < p.rows) {
            float mw[C::kWarps], M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                mw[w] = sML[(w * 16 + r) * 2];
                M = fmaxf(M, mw[w]);
            }
            float sc[C::kWarps], lsum = 0.f;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                sc[w] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
                lsum += sc[w] * sML[(w * 16 + r) * 2 + 1];
            }
            const size_t pidx =
                ((static_cast<size_t>(unit) * p.row_groups + rg) * p.nsplit + split) * 16 + r;
            float* po = p.part_o + pidx * kD + d0;
#pragma unroll
            for (int d = 0; d < 16; d += 4) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < C::kWarps; ++w) {
                    const float* src = reinterpret_cast<float*>(smem) + (w * 16 + r) * C::kOStride + d0 + d;
                    acc.x += sc[w] * src[0];
                    acc.y += sc[w] * src[1];
                    acc.z += sc[w] * src[2];
                    acc.w += sc[w] * src[3];
                }
                *reinterpret_cast<float4*>(po + d) = acc;
            }
            if ((threadIdx.x & 7) == 0) {
                p.part_ml[pidx * 2 + 0] = M;
                p.part_ml[pidx * 2 + 1] = lsum;
            }
        }
    }
}

// One warp per output row (b, q head, query j): merge the split partials with
// their log-sum-exp weights, apply v_rescale, leave the rotated basis
// (Rot^-1(y) = s * (H y) / sqrt(128)) and store fp16.
__global__ void __launch_bounds__(128) tq_combine_kernel(const __grid_constant__ CombineParams p) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int total = p.batch * p.hq * p.tq;
    if (row >= total) return;
    const int j = row % p.tq;
    const int hq = (row / p.tq) % p.hq;
    const int b = row / (p.tq * p.hq);
    const int kv = hq / p.group, hl = hq - kv * p.group;
    const int r = hl * p.tq + j;
    const int rg = r >> 4, rl = r & 15;
    const int unit = b * p.hkv + kv;
    const int L = min(p.lengths[b], p.max_len);
    const int ns = min(p.nsplit, (L + p.split_tokens - 1) / p.split_tokens);
    const size_t base = (static_cast<size_t>(unit) * p.row_groups + rg) * p.nsplit * 16 + rl;

    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p.part_ml[(base + s * 16) * 2]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
        const size_t pi = base + s * 16;
        const float m = p.part_ml[pi * 2];
        const float w = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
        den += w * p.part_ml[pi * 2 + 1];
        const float4 o = *reinterpret_cast<const float4*>(p.part_o + pi * kD + lane * 4);
        acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
    float inv = 0.f;
    if (den > 0.f) inv = p.v_rescale / den;
    else if (lane == 0) atomicOr(p.status, kStatusShortContext);
    float v[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
    wht128_lane4(v, lane);
    const uint32_t sn = sign_nibble(p.signs, lane);
    const float nrm = 0.08838834764831845f;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ((sn >> i) & 1u) ? -v[i] * nrm : v[i] * nrm;
    uint2 o;
    o.x = pack_half2(v[0], v[1]);
    o.y = pack_half2(v[2], v[3]);
    *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(row) * kD + lane * 4) = o;
}

template <int KB, int VB>
static int launch_decode_t(const DecodeParams& p, const CUtensorMap* kmap, cudaStream_t stream,
                           cudaEvent_t ev0, cudaEvent_t ev1) {
    using C = DecCfg<KB, VB>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tq_decode_kernel<KB, VB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(p.nsplit, p.batch * p.hkv, p.row_groups);
    if (ev0) cudaEventRecord(ev0, stream);
    tq_decode_kernel<KB, VB><<<grid, C::kWarps * 32, C::kSmemAlloc, stream>>>(p, *kmap);
    cudaError_t e = cudaGetLastError();
    if (ev1) cudaEventRecord(ev1, stream);
    return e;
}

int launch_decode(int kbits, int vbits, const DecodeParams& p, const CUtensorMap* kmap,
                  cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    if (kbits == 16 && vbits == 4) return launch_decode_t<0, 4>(p, kmap, stream, ev0, ev1);
    if (kbits == 3 && vbits == 3) return launch_decode_t<3, 3>(p, kmap, stream, ev0, ev1);
    if (kbits == 4 && vbits == 4) return launch_decode_t<4, 4>(p, kmap, stream, ev0, ev1);
    return cudaErrorInvalidValue;
}

int launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int rows = p.batch * p.hq * p.tq;
    tq_combine_kernel<<<(rows + 3) / 4, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

int decode_ctas_per_sm(int kbits, int vbits) {
    int smem = 0;
    if (kbits == 16) smem = DecCfg<0, 4>::kSmemAlloc;
    else if (kbits == 3) smem = DecCfg<3, 3>::kSmemAlloc;
    else smem = DecCfg<4, 4>::kSmemAlloc;
    int by_smem = (228 * 1024) / (smem + 1024);  // 1 KB per CTA is reserved
    if (by_smem < 1) by_smem = 1;
    return by_smem < 3 ? by_smem : 3;
}

}  // namespace tq
