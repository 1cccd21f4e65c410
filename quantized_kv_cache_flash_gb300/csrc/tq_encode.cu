// Encode/append: fp16 K/V vectors -> (fp16 norm, packed b-bit codes) written
// at each sequence's current length, then lengths[b] += t_new.
//
// Per vector (four lanes of a warp, lane q holds dims 32q .. 32q+31):
//   n16  = fp16 round-to-nearest-even of the exact L2 norm: fp32 sum of the
//          exact squares, certified against the rounding midpoints; if it is
//          too close to call, the sum of squares is formed exactly as a
//          128-bit integer (every fp16 value is an integer multiple of 2^-24)
//          and the candidate corrected with exact integer comparisons.
//   u    = Rot(x) / n = H (s * x) / (sqrt(128) n), in fp32.
//   code = sign-magnitude index of the nearest codebook entry to u, decided
//          with thresholds that make the fp32 comparison exact against the
//          true midpoints of neighbouring centroids (ties to the lower index).
// (The encode of mlxcel pull request #369, Change: seeded sign flip, Walsh-
// Hadamard rotation, nearest codebook entry, bit packing; turboquant_plus
// smem-dequant experiment, Hypothesis 1: a 128-element rotation group with
// one norm per group.)
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

struct U128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ U128 add128(U128 a, U128 b) {
    U128 r;
    r.lo = a.lo + b.lo;
    r.hi = a.hi + b.hi + (r.lo < a.lo ? 1ull : 0ull);
    return r;
}

__device__ __forceinline__ U128 sq_u128(long long m) {
    const unsigned long long a = m < 0 ? static_cast<unsigned long long>(-m)
                                       : static_cast<unsigned long long>(m);
    U128 r;
    r.lo = a * a;
    r.hi = __umul64hi(a, a);
    return r;
}

__device__ __forceinline__ int cmp128(U128 a, U128 b) {
    if (a.hi != b.hi) return a.hi < b.hi ? -1 : 1;
    if (a.lo != b.lo) return a.lo < b.lo ? -1 : 1;
    return 0;
}

// k * k for k < 2^63.
__device__ __forceinline__ U128 square_u64(unsigned long long k) {
    U128 r;
    r.lo = k * k;
    r.hi = __umul64hi(k, k);
    return r;
}

// x (fp16, finite) -> x * 2^24 as an exact integer.
__device__ __forceinline__ long long fp16_scaled_int(float x) {
    return __float2ll_rn(x * 16777216.0f);
}

// fp16 value of a non-negative finite half, and its neighbours on the grid
// (in units of 2^-25 as exact integers).
__device__ __forceinline__ unsigned long long half_units25(unsigned short bits) {
    // value * 2^25; for the overflow neighbour of 65504 use 2^16.
    if (bits >= 0x7C00u) return 65536ull << 25;
    const float f = __half2float(__ushort_as_half(bits));
    return static_cast<unsigned long long>(f * 33554432.0f);
}

// Round sqrt(S * 2^-48) (S exact) to fp16, nearest-even.  S4 = 4*S is the
// square of the target in units of 2^-50, midpoints m (units of 2^-25) compare
// as S4 <=> m^2.
__device__ __forceinline__ unsigned short norm_to_half(U128 S) {
    if (S.hi == 0 && S.lo == 0) return 0;
    U128 S4;
    S4.lo = S.lo << 2;
    S4.hi = (S.hi << 2) | (S.lo >> 62);
    // candidate from an fp32 square root
    const float sf = static_cast<float>(S.hi) * 18446744073709551616.0f + static_cast<float>(S.lo);
    const float n = sqrtf(sf) * (1.0f / 16777216.0f);
    unsigned short hb = __half_as_ushort(__float2half_rn(n));
    if (hb > 0x7C00u) hb = 0x7C00u;
    // walk at most a few steps until the candidate is the correctly rounded value
    for (int step = 0; step < 4; ++step) {
        if (hb < 0x7C00u) {
            // midpoint with the next value up
            const unsigned long long up = (half_units25(hb) + half_units25(hb + 1)) >> 1;
            const int cu = cmp128(S4, square_u64(up));
            if (cu > 0 || (cu == 0 && (hb & 1u))) { ++hb; continue; }
        }
        if (hb > 0) {
            const unsigned short dn_bits = (hb == 0x7C00u) ? 0x7BFFu : static_cast<unsigned short>(hb - 1);
            const unsigned long long lo_mid = (half_units25(dn_bits) + half_units25(hb)) >> 1;
            const int cd = cmp128(S4, square_u64(lo_mid));
            // below the lower midpoint, or on it with the lower value even
            if (cd < 0 || (cd == 0 && !(dn_bits & 1u))) { hb = dn_bits; continue; }
        }
        break;
    }
    return hb;
}

// Exact fp16 norm of one vector whose 4 lanes each hold 32 dims; reloads the
// lane's 32 fp16 values from src (out of line: it is the rare path of
// norm_fp16 below).  gmask = the group's lanes.
__device__ __noinline__ unsigned short norm_exact_group(const __half* src, int q, bool valid,
                                                        unsigned gmask) {
    U128 S;
    S.lo = 0;
    S.hi = 0;
    if (valid) {
        const __half* x = src + q * 32;
        for (int i = 0; i < 32; ++i) S = add128(S, sq_u128(fp16_scaled_int(__half2float(x[i]))));
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        U128 o;
        o.lo = __shfl_xor_sync(gmask, S.lo, m);
        o.hi = __shfl_xor_sync(gmask, S.hi, m);
        S = add128(S, o);
    }
    return norm_to_half(S);
}

__device__ __forceinline__ float half_bits_to_float(unsigned short b) {
    return (b >= 0x7C00u) ? 65536.f : __half2float(__ushort_as_half(b));
}

// norm_fp16: fp16 round-to-nearest-even of the exact norm sqrt(sum x^2).  Fast path: the
// fp32 sum of the (exact) squares is within 2^-17 (relative) of the exact sum,
// so the candidate rounding of its square root is certain unless the sum lies
// within 2^-16 of the square of a rounding midpoint (midpoints have 12
// significant bits, so their squares are exact in fp32); then the exact
// 128-bit integer path decides.
// Candidate fp16 rounding of sqrt(S32) and whether it is certain (see norm_fp16).
__device__ __forceinline__ unsigned short norm_candidate(float S32, bool& certain) {
    certain = true;
    if (S32 == 0.f) return 0;
    const float n = sqrtf(S32);
    unsigned short hb = __half_as_ushort(__float2half_rn(n));
    if (hb > 0x7C00u) hb = 0x7C00u;
    const float margin = S32 * (1.0f / 65536.0f);
    const float hf = half_bits_to_float(hb);
    if (hb < 0x7C00u) {
        const float up = 0.5f * (hf + half_bits_to_float(hb + 1));
        certain = certain && (S32 < up * up - margin);
    }
    if (hb > 0) {
        const unsigned short db = (hb == 0x7C00u) ? 0x7BFFu : static_cast<unsigned short>(hb - 1);
        const float dn = 0.5f * (half_bits_to_float(db) + ((hb == 0x7C00u) ? 65536.f : hf));
        certain = certain && (S32 > dn * dn + margin);
    }
    return hb;
}

__device__ __forceinline__ unsigned short norm_fp16(const __half* src, int q, bool valid,
                                                    float S32, unsigned gmask) {
    bool ok;
    const unsigned short hb = norm_candidate(S32, ok);
    const bool all_ok = __all_sync(gmask, ok);   // the group decides together
    return all_ok ? hb : norm_exact_group(src, q, valid, gmask);
}

// Sign-magnitude code of the centroid nearest to u: rank = #{tau_k < |u|} for
// u > 0 and #{tau_k <= |u|} for u <= 0, with gt[k] / ge[k] the smallest fp32
// values above / at-or-above the exact midpoint tau_k (ascending).  gt and ge
// differ only when tau_k is itself an fp32 value, so the search runs on gt and
// a negative u sitting exactly on such a tau_k moves one rank up.  Binary
// search: BITS-1 comparisons.
template <int BITS>
__device__ __forceinline__ uint32_t quantize_code(float u, const float* gt, const float* ge,
                                                  bool any_tie) {
    constexpr int H = 1 << (BITS - 1);
    const float a = fabsf(u);
    const bool neg = !(u > 0.f);
    uint32_t rank;
    if constexpr (BITS == 3) {
        const bool b1 = a >= gt[1];
        const bool b0 = a >= (b1 ? gt[2] : gt[0]);
        rank = (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
    } else {
        const bool b2 = a >= gt[3];
        const bool b1 = a >= (b2 ? gt[5] : gt[1]);
        const float t0 = b2 ? (b1 ? gt[6] : gt[4]) : (b1 ? gt[2] : gt[0]);
        const bool b0 = a >= t0;
        rank = (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
    }
    if (any_tie && neg && rank < H - 1) {
        // a in [ge[rank], gt[rank]) means a == tau_rank: the tie goes down (more negative)
        if (a >= ge[rank] && a < gt[rank]) rank += 1;
    }
    return (neg ? static_cast<uint32_t>(H) : 0u) | rank;
}

// Encode the vectors of one warp: 8 vectors, 4 lanes each; lane quarter q
// holds dims 32q .. 32q+31.  `valid` marks lanes whose vector exists.
// The record's norm (norm format) or, for table records (tcb != nullptr), the
// eight fp16 values c_j * n16 after the 48 code bytes: c_j (fp32) times n16
// (fp16) is exact in double, so each value is one rounding of the exact
// product.
__device__ __forceinline__ void store_norm(__half* dst_norm, uint8_t* dst, const float* tcb,
                                           unsigned short nb) {
    if (tcb == nullptr) {
        dst_norm[0] = __ushort_as_half(nb);
        return;
    }
    const double n = static_cast<double>(__half2float(__ushort_as_half(nb)));
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t a = __half_as_ushort(__double2half(static_cast<double>(tcb[2 * k]) * n));
        const uint32_t b = __half_as_ushort(__double2half(static_cast<double>(tcb[2 * k + 1]) * n));
        w[k] = a | (b << 16);
    }
    *reinterpret_cast<uint4*>(dst + 48) = make_uint4(w[0], w[1], w[2], w[3]);
}

// XOR masks that apply a lane's 32 signs to its dims as fp16 pairs: word k
// flips dim 2k with bit 15 and dim 2k+1 with bit 31.
__device__ __forceinline__ void sign_masks(uint32_t sg, uint32_t (&hm)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) hm[k] = (((sg >> (2 * k)) & 1u) << 15) | (((sg >> (2 * k + 1)) & 1u) << 31);
}

// Encode one vector per 4 lanes (8 per warp); lane quarter q holds dims
// 32q .. 32q+31.  `valid` marks lanes whose vector exists.  The codes compare
// the unnormalised rotated value y = H (s * x) / sqrt(128) ... scaled back:
// u = y / n > tau_k  <=>  y > tau_k * sqrt(128) * n  for the fp32 norm n, so
// the thresholds are scaled once per vector instead of every u divided.  The
// fp32 rotation and scaling are within ~1e-7 (relative) of the exact u;
// elements that close to a midpoint may round either way (a zero u is
// negative: the tie goes to the lower index).
// The lane's 32 fp16 inputs (64 bytes), or zeros for a lane without a vector.
struct QuarterIn {
    uint4 w[4];
};

__device__ __forceinline__ QuarterIn load_quarter_in(const __half* src, int q, bool valid) {
    QuarterIn r;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + q * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) r.w[i] = valid ? s4[i] : make_uint4(0u, 0u, 0u, 0u);
    return r;
}

template <int BITS>
__device__ __forceinline__ void encode_group(const QuarterIn& in, const __half* src, uint8_t* dst,
                                             __half* dst_norm, const float* tcb,
                                             const uint32_t (&hm)[16], const float* gt, bool valid,
                                             uint32_t* status, int q, unsigned gmask) {
    float x[32];  // s * x for the lane's dims
    {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = in.w[i];
            const uint32_t ww[4] = {w.x ^ hm[4 * i], w.y ^ hm[4 * i + 1], w.z ^ hm[4 * i + 2],
                                    w.w ^ hm[4 * i + 3]};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[k]));
                x[8 * i + 2 * k] = f.x;
                x[8 * i + 2 * k + 1] = f.y;
            }
        }
    }
    if (!valid) {  // a lane without a vector takes part in the shuffles with zeros
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.f;
    }

    // norm: squares of fp16 values are exact in fp32 (the signs do not matter)
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = fmaf(x[i], x[i], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float S32 = __shfl_sync(0xffffffffu, ss, 0, 4);   // one rounding order per group
    const unsigned short nb = norm_fp16(src, q, valid, S32, gmask);
    if (valid && q == 0) {
        store_norm(dst_norm, dst, tcb, nb);
        if (nb >= 0x7C00u) atomicOr(status, kStatusNormOverflow);
    }

    // rotate: H (s * x), 5 in-lane stages + 2 across the group's lanes
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (i & h) continue;
            const float a = x[i], b = x[i + h];
            x[i] = a + b;
            x[i + h] = a - b;
        }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const float sgn = (q & m) ? -1.f : 1.f;   // upper half of the pair: o - x
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = fmaf(sgn, x[i], o);
        }
    }

    constexpr int H = 1 << (BITS - 1);
    const float scale = sqrtf(S32) * 11.313708498984761f;   // sqrt(128) n
    float T[H - 1];
#pragma unroll
    for (int k = 0; k < H - 1; ++k) T[k] = gt[k] * scale;
    if (!valid) return;
    if constexpr (BITS == 4) {
        // word k = dims 8k..8k+7: rank of dim 8k+j in bits 4j..4j+2; sign of dim
        // 8k+j (j < 4) in bit 8j+7, of dim 8k+4+j in bit 8j+3
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t v = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float y = x[8 * k + j];
                const float a = fabsf(y);
                const bool b2 = a > T[3];
                const bool b1 = a > (b2 ? T[5] : T[1]);
                const float t0 = b2 ? (b1 ? T[6] : T[4]) : (b1 ? T[2] : T[0]);
                const bool b0 = a > t0;
                const uint32_t rank = (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
                v |= rank << (4 * j);
                if (!(y > 0.f)) v |= 1u << (j < 4 ? 8 * j + 7 : 8 * (j - 4) + 3);
            }
            w[k] = v;
        }
        *reinterpret_cast<uint4*>(dst + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        // sign-magnitude code kappa = sign << 2 | rank; quarter q: word k (k < 3):
        // bits 4j..4j+2 = code(8k+j), bit 4j+3 = bit k of code(24+j).  The
        // comparisons give 0.0 / 1.0 and the words are summed in fp32 as two
        // 16-bit halves (exact: every partial sum is an integer below 2^16).
        float h[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float y = x[i];
            const float a = fabsf(y);
            const bool b1 = a > T[1];
            const float f1 = b1 ? 1.f : 0.f;
            const float f0 = (a > (b1 ? T[2] : T[0])) ? 1.f : 0.f;
            const float fn = (y > 0.f) ? 0.f : 1.f;
            if (i < 24) {
                const int j = i & 7;
                const float unit = static_cast<float>(1u << (4 * (j & 3)));  // nibble j of the half
                float& acc = h[i >> 3][j >> 2];
                acc = fmaf(fn, 4.f * unit, acc);
                acc = fmaf(f1, 2.f * unit, acc);
                acc = fmaf(f0, unit, acc);
            } else {
                const int j = i - 24;
                const float bit = static_cast<float>(1u << (4 * (j & 3) + 3));
                h[0][j >> 2] = fmaf(f0, bit, h[0][j >> 2]);
                h[1][j >> 2] = fmaf(f1, bit, h[1][j >> 2]);
                h[2][j >> 2] = fmaf(fn, bit, h[2][j >> 2]);
            }
        }
        uint32_t d[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
            d[k] = static_cast<uint32_t>(h[k][0]) | (static_cast<uint32_t>(h[k][1]) << 16);
        uint32_t* o = reinterpret_cast<uint32_t*>(dst + q * 12);
        o[0] = d[0];
        o[1] = d[1];
        o[2] = d[2];
    }
}

// Advance lengths[] after the last CTA of the launch has read it: one ticket
// per CTA, taken once every thread of the CTA has read lengths[] for the last
// time (so none sees an advanced length); the counter is back at zero for the
// next launch.
__device__ __forceinline__ void finish_append(const EncodeParams& p, int lane) {
    __shared__ unsigned int s_ticket;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_ticket = atomicAdd(p.counter, 1u);
    }
    __syncthreads();
    if (s_ticket == gridDim.x - 1 && threadIdx.x < 32) {
        __threadfence();
        for (int bb = lane; bb < p.batch; bb += 32) {
            const int Lb = *((volatile int32_t*)p.lengths + bb);
            if (Lb >= 0 && Lb + p.t_new <= p.cap) p.lengths[bb] = Lb + p.t_new;
        }
        if (lane == 0) *((volatile uint32_t*)p.counter) = 0u;
        __threadfence();
    }
}

// grid: [K blocks | V blocks]; a CTA of 4 warps encodes 128 vectors of one
// stream (K or V): each warp takes 8 vectors at a time, 4 lanes each, for 4
// passes, so a lane's sign masks (its quarter of s) serve 4 vectors.
// KB = 0 copies fp16 K rows.
constexpr int kEncWarps = 4;
constexpr int kEncPasses = 4;
constexpr int kEncVecs = 8 * kEncWarps * kEncPasses;

template <int KB, int VB>
__global__ void __launch_bounds__(32 * kEncWarps)
    tq_encode_kernel(const __grid_constant__ EncodeParams p, int k_blocks) {
    __shared__ unsigned long long s_pos[kEncPasses][32 * kEncWarps];
    griddep_wait();                // inputs and lengths come from earlier work on the stream
    griddep_launch_dependents();   // the decode that follows may start launching
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int q = lane & 3;
    const unsigned gmask = 0xFu << (lane & ~3);
    const bool is_v = static_cast<int>(blockIdx.x) >= k_blocks;
    const int blk = is_v ? static_cast<int>(blockIdx.x) - k_blocks : static_cast<int>(blockIdx.x);
    // vector counts stay below 2^31 (the host checks), so 32-bit index math
    const int nvec = p.batch * p.hkv * p.t_new;
    auto vec_of = [&](int pass) { return blk * kEncVecs + (pass * kEncWarps + warp) * 8 + (lane >> 2); };

    // Every lane first reads the lengths its passes write at and keeps the
    // record positions (or ~0 for no vector); then the CTA takes its ticket,
    // so the last CTA advances lengths[] while the others are still encoding
    // (they no longer read it).
    constexpr unsigned long long kNone = ~0ull;
#pragma unroll
    for (int r = 0; r < kEncPasses; ++r) {
        const int v = vec_of(r);
        unsigned long long pos = kNone;
        if (v < nvec) {
            const int bh = v / p.t_new;
            const int t = v - bh * p.t_new;
            const int L = p.lengths[bh / p.hkv];
            if (L < 0 || L + p.t_new > p.cap) {
                if (q == 0 && !is_v && t == 0 && (bh % p.hkv) == 0) atomicOr(p.status, kStatusCapacity);
            } else {
                pos = static_cast<unsigned long long>(bh) * p.cap + L + t;
            }
        }
        s_pos[r][threadIdx.x] = pos;
    }
    finish_append(p, lane);

    uint32_t hm[16];
    sign_masks(p.signs[q], hm);

    // pass r's vector for this lane, whether it exists, and where it goes
    struct Slot {
        const __half* src;
        size_t pos;
        bool valid;
    };
    const __half* const in_base = is_v ? p.v_new : p.k_new;
    auto slot = [&](int pass) {
        Slot sl;
        const unsigned long long pos = s_pos[pass][threadIdx.x];
        sl.valid = pos != kNone;
        sl.pos = sl.valid ? static_cast<size_t>(pos) : 0;
        sl.src = in_base + static_cast<size_t>(sl.valid ? vec_of(pass) : 0) * kD;
        return sl;
    };
    // the stream this CTA encodes (one code path serves both when K and V have
    // the same bits)
    uint8_t* const codes = is_v ? p.v_codes : p.k_codes;
    __half* const norms = is_v ? p.v_norm : p.k_norm;
    const float* const tcb = p.table ? (is_v ? p.v_cb : p.k_cb) : nullptr;
    const float* const gt = is_v ? p.v_gt : p.k_gt;
    const int rec = is_v ? (p.table ? 64 : VB * 16) : (KB == 0 ? 256 : (p.table ? 64 : KB * 16));

    // the next pass's inputs are loaded before this pass is encoded
    Slot cur = slot(0);
    QuarterIn in = load_quarter_in(cur.src, q, cur.valid);
#pragma unroll 1
    for (int pass = 0; pass < kEncPasses; ++pass) {
        Slot nxt = cur;
        QuarterIn in_next = in;
        if (pass + 1 < kEncPasses) {
            nxt = slot(pass + 1);
            in_next = load_quarter_in(nxt.src, q, nxt.valid);
        }
        uint8_t* const dst = codes + cur.pos * rec;
        if constexpr (KB == VB) {
            encode_group<KB>(in, cur.src, dst, norms + cur.pos, tcb, hm, gt, cur.valid, p.status, q,
                             gmask);
        } else if (!is_v) {
            if constexpr (KB == 0) {
                if (cur.valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + q * 64);
#pragma unroll
                    for (int i = 0; i < 4; ++i) d4[i] = in.w[i];
                }
            } else {
                encode_group<KB>(in, cur.src, dst, norms + cur.pos, tcb, hm, gt, cur.valid,
                                 p.status, q, gmask);
            }
        } else {
            encode_group<VB>(in, cur.src, dst, norms + cur.pos, tcb, hm, gt, cur.valid, p.status,
                             q, gmask);
        }
        cur = nxt;
        in = in_next;
    }
}

// Small appends (a few tokens per sequence): one warp per vector, lane l holds
// dims 4l .. 4l+3, so every vector gets its own warp and the dependent chain
// per lane is short.  The same output as encode_group, except that elements
// within ~1e-7 of a midpoint may round the other way: here u itself is formed
// and compared exactly against the fp32 midpoints.
template <int BITS>
__device__ __forceinline__ void encode_vector_warp(const __half* src, uint8_t* dst,
                                                   __half* dst_norm, const float* tcb,
                                                   const uint32_t (&signs)[4], const float* gt,
                                                   const float* ge, uint32_t* status, int lane) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    float x[4] = {f0.x, f0.y, f1.x, f1.y};

    float ss = fmaf(x[0], x[0], x[1] * x[1]) + fmaf(x[2], x[2], x[3] * x[3]);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float S32 = __shfl_sync(0xffffffffu, ss, 0);
    bool ok;
    unsigned short nb = norm_candidate(S32, ok);
    if (!__all_sync(0xffffffffu, ok)) {
        // exact sum of squares (units of 2^-48) as a 128-bit integer
        U128 S = sq_u128(fp16_scaled_int(x[0]));
#pragma unroll
        for (int i = 1; i < 4; ++i) S = add128(S, sq_u128(fp16_scaled_int(x[i])));
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            U128 o;
            o.lo = __shfl_xor_sync(0xffffffffu, S.lo, m);
            o.hi = __shfl_xor_sync(0xffffffffu, S.hi, m);
            S = add128(S, o);
        }
        nb = norm_to_half(S);
    }
    if (lane == 0) {
        store_norm(dst_norm, dst, tcb, nb);
        if (nb >= 0x7C00u) atomicOr(status, kStatusNormOverflow);
    }

    // rotate: u = H (s * x) / (sqrt(128) n)
    const uint32_t sn = sign_nibble(signs, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = ((sn >> i) & 1u) ? -x[i] : x[i];
    wht128_lane4(x, lane);
    const float n = sqrtf(S32);
    const float inv = (n > 0.f) ? 1.0f / (n * 11.313708498984761f) : 0.f;
    constexpr int H = 1 << (BITS - 1);
    bool any_tie = false;
#pragma unroll
    for (int k = 0; k < H - 1; ++k) any_tie |= ge[k] != gt[k];
    uint32_t code[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) code[i] = quantize_code<BITS>(x[i] * inv, gt, ge, any_tie);

    if constexpr (BITS == 4) {
        // word k = dims 8k..8k+7 (lanes 2k, 2k+1): rank of dim 8k+j in bits
        // 4j..4j+2; sign of dim 8k+j (j < 4) in bit 8j+7, of dim 8k+4+j in bit 8j+3
        const bool upper = (lane & 1) != 0;
        uint32_t part = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            part |= (code[i] & 7u) << (4 * i + (upper ? 16 : 0));
            part |= (code[i] >> 3) << (8 * i + (upper ? 3 : 7));
        }
        const uint32_t other = __shfl_down_sync(0xffffffffu, part, 1);
        if (!upper) reinterpret_cast<uint32_t*>(dst)[lane >> 1] = part | other;
    } else {
        // quarter q = lanes 8q..8q+7; lanes 8q+2k, 8q+2k+1 carry dims 32q+8k..+7
        // (word k's nibbles); lanes 8q+6, 8q+7 carry dims 32q+24..31, whose
        // code bit k goes to bit 4j+3 of word k.
        const uint32_t nib = (code[0] & 7u) | ((code[1] & 7u) << 4) | ((code[2] & 7u) << 8) |
                             ((code[3] & 7u) << 12);
        uint32_t sp[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
            sp[k] = (((code[0] >> k) & 1u) << 3) | (((code[1] >> k) & 1u) << 7) |
                    (((code[2] >> k) & 1u) << 11) | (((code[3] >> k) & 1u) << 15);
        const int qb = lane & ~7;
        const uint32_t up = __shfl_down_sync(0xffffffffu, nib, 1);
        uint32_t spw[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint32_t s6 = __shfl_sync(0xffffffffu, sp[k], qb + 6);
            const uint32_t s7 = __shfl_sync(0xffffffffu, sp[k], qb + 7);
            spw[k] = s6 | (s7 << 16);
        }
        const int sub = lane & 7;
        if (sub < 6 && (sub & 1) == 0) {
            const int k = sub >> 1;
            const uint32_t word = nib | (up << 16) | (k == 0 ? spw[0] : (k == 1 ? spw[1] : spw[2]));
            reinterpret_cast<uint32_t*>(dst)[(lane >> 3) * 3 + k] = word;
        }
    }
}

// grid: 4 warps per CTA, warp = (K-or-V, vector).  KB = 0 copies fp16 K rows.
template <int KB, int VB>
__global__ void __launch_bounds__(128) tq_encode_small_kernel(const __grid_constant__ EncodeParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const long long nvec = static_cast<long long>(p.batch) * p.hkv * p.t_new;
    if (gw < 2 * nvec) {
        const int which = static_cast<int>(gw & 1);  // 0 = K, 1 = V
        const long long v = gw >> 1;
        const int t = static_cast<int>(v % p.t_new);
        const long long bh = v / p.t_new;
        const int b = static_cast<int>(bh / p.hkv);
        const int L = p.lengths[b];
        if (L < 0 || L + p.t_new > p.cap) {
            if (lane == 0 && which == 0 && t == 0 && (bh % p.hkv) == 0)
                atomicOr(p.status, kStatusCapacity);
        } else {
            const size_t pos = static_cast<size_t>(bh) * p.cap + L + t;
            const __half* src = (which ? p.v_new : p.k_new) + v * kD;
            if (which == 0) {
                if constexpr (KB == 0) {
                    reinterpret_cast<uint2*>(p.k_codes + pos * 256)[lane] =
                        reinterpret_cast<const uint2*>(src)[lane];
                } else {
                    encode_vector_warp<KB>(src, p.k_codes + pos * (p.table ? 64 : KB * 16),
                                           p.k_norm + pos, p.table ? p.k_cb : nullptr, p.signs,
                                           p.k_gt, p.k_ge, p.status, lane);
                }
            } else {
                encode_vector_warp<VB>(src, p.v_codes + pos * (p.table ? 64 : VB * 16),
                                       p.v_norm + pos, p.table ? p.v_cb : nullptr, p.signs,
                                       p.v_gt, p.v_ge, p.status, lane);
            }
        }
    }
    finish_append(p, lane);
}

int launch_encode(int kbits, int vbits, const EncodeParams& p, cudaStream_t stream) {
    const long long nvec = 1ll * p.batch * p.hkv * p.t_new;
    if (nvec <= 4096) {   // a warp per vector: short chains for small appends
        const dim3 grid(static_cast<unsigned int>((2 * nvec + 3) / 4)), block(128);
        if (kbits == 16 && vbits == 4) return launch_pdl(tq_encode_small_kernel<0, 4>, grid, block, 0, stream, p);
        if (kbits == 3 && vbits == 3) return launch_pdl(tq_encode_small_kernel<3, 3>, grid, block, 0, stream, p);
        if (kbits == 4 && vbits == 4) return launch_pdl(tq_encode_small_kernel<4, 4>, grid, block, 0, stream, p);
        if (kbits == 16 && vbits == 3) return launch_pdl(tq_encode_small_kernel<0, 3>, grid, block, 0, stream, p);
        if (kbits == 4 && vbits == 3) return launch_pdl(tq_encode_small_kernel<4, 3>, grid, block, 0, stream, p);
        return cudaErrorInvalidValue;
    }
    const int kblocks = static_cast<int>((nvec + kEncVecs - 1) / kEncVecs);
    const dim3 grid(static_cast<unsigned int>(2 * kblocks)), block(32 * kEncWarps);
    if (kbits == 16 && vbits == 4) return launch_pdl(tq_encode_kernel<0, 4>, grid, block, 0, stream, p, kblocks);
    if (kbits == 3 && vbits == 3) return launch_pdl(tq_encode_kernel<3, 3>, grid, block, 0, stream, p, kblocks);
    if (kbits == 4 && vbits == 4) return launch_pdl(tq_encode_kernel<4, 4>, grid, block, 0, stream, p, kblocks);
    if (kbits == 16 && vbits == 3) return launch_pdl(tq_encode_kernel<0, 3>, grid, block, 0, stream, p, kblocks);
    if (kbits == 4 && vbits == 3) return launch_pdl(tq_encode_kernel<4, 3>, grid, block, 0, stream, p, kblocks);
    return cudaErrorInvalidValue;
}

}  // namespace tq
