// Encode/append: fp16 K/V vectors -> (fp16 norm, packed b-bit codes) written
// at each sequence's current length, then lengths[b] += t_new.
//
// Per vector (one warp, lane l holds dims 4l .. 4l+3):
//   n16  = fp16 round-to-nearest-even of the exact L2 norm.  The sum of
//          squares is formed exactly as a 128-bit integer (every fp16 value is
//          an integer multiple of 2^-24), an fp32 square root gives a
//          candidate, and the candidate is corrected against the neighbouring
//          rounding midpoints with exact integer comparisons.
//   u    = Rot(x) / n = H (s * x) / (sqrt(128) n), in fp32.
//   code = sign-magnitude index of the nearest codebook entry to u, decided
//          with thresholds that make the fp32 comparison exact against the
//          true midpoints of neighbouring centroids (ties to the lower index).
// ("seeded sign flip + WHT + nearest centroid + bit-pack": mlxcel pull request
// #369, Change; turboquant_plus smem-dequant experiment, Hypothesis 1, for the
// 128-element rotation group with one norm per group.)
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

template <int BITS>
__device__ __forceinline__ uint32_t quantize_code(float u, const float* gt, const float* ge) {
    constexpr int H = 1 << (BITS - 1);
    const float a = fabsf(u);
    const bool neg = !(u > 0.f);
    uint32_t rank = 0;
#pragma unroll
    for (int k = 0; k < H - 1; ++k) rank += (a >= (neg ? ge[k] : gt[k])) ? 1u : 0u;
    return (neg ? static_cast<uint32_t>(H) : 0u) | rank;
}

// Encode one fp16 vector with the warp; returns nothing, writes codes + norm.
template <int BITS>
__device__ __forceinline__ void encode_vector(const __half* src, uint8_t* dst, __half* dst_norm,
                                              const uint32_t (&signs)[4], const float* gt,
                                              const float* ge, uint32_t* status, int lane) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    float x[4] = {f0.x, f0.y, f1.x, f1.y};

    // exact sum of squares (units of 2^-48)
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
    const unsigned short nb = norm_to_half(S);
    const float sf = static_cast<float>(S.hi) * 18446744073709551616.0f + static_cast<float>(S.lo);
    const float n = sqrtf(sf) * (1.0f / 16777216.0f);   // unrounded norm (fp32)
    if (lane == 0) {
        dst_norm[0] = __ushort_as_half(nb);
        if (nb >= 0x7C00u) atomicOr(status, kStatusNormOverflow);
    }

    // rotate: u = H (s * x) / (sqrt(128) n)
    const uint32_t sn = sign_nibble(signs, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = ((sn >> i) & 1u) ? -x[i] : x[i];
    wht128_lane4(x, lane);
    const float inv = (n > 0.f) ? 1.0f / (n * 11.313708498984761f) : 0.f;
    uint32_t code[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) code[i] = quantize_code<BITS>(x[i] * inv, gt, ge);

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

// grid: 8 warps per CTA, warp = (vector, K-or-V).  KB = 0 copies fp16 K rows.
template <int KB, int VB>
__global__ void __launch_bounds__(256) tq_encode_kernel(const __grid_constant__ EncodeParams p) {
    const int lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
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
                    encode_vector<KB>(src, p.k_codes + pos * (KB * 16), p.k_norm + pos, p.signs,
                                      p.k_gt, p.k_ge, p.status, lane);
                }
            } else {
                encode_vector<VB>(src, p.v_codes + pos * (VB * 16), p.v_norm + pos, p.signs, p.v_gt,
                                  p.v_ge, p.status, lane);
            }
        }
    }
    // The last CTA to finish advances the lengths.  Every CTA read lengths[]
    // before its ticket, so no CTA can see an advanced length.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned int ticket = atomicAdd(p.counter, 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            for (int b = 0; b < p.batch; ++b) {
                const int L = *((volatile int32_t*)p.lengths + b);
                if (L >= 0 && L + p.t_new <= p.cap) p.lengths[b] = L + p.t_new;
            }
            *((volatile uint32_t*)p.counter) = 0u;
            __threadfence();
        }
    }
}

int launch_encode(int kbits, int vbits, const EncodeParams& p, cudaStream_t stream) {
    const long long warps = 2ll * p.batch * p.hkv * p.t_new;
    const unsigned int blocks = static_cast<unsigned int>((warps + 7) / 8);
    if (kbits == 16 && vbits == 4) tq_encode_kernel<0, 4><<<blocks, 256, 0, stream>>>(p);
    else if (kbits == 3 && vbits == 3) tq_encode_kernel<3, 3><<<blocks, 256, 0, stream>>>(p);
    else if (kbits == 4 && vbits == 4) tq_encode_kernel<4, 4><<<blocks, 256, 0, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace tq
