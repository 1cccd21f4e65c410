// Device-side building blocks for the quantized-KV kernels (sm_103a).
//
// Inline PTX wrappers (byte permute, warp-level MMA, 8x8 transpose, shared
// memory matrix loads, mbarrier, bulk and tensor copies) and the register
// dequantisers that turn packed b-bit codes into fp16 pairs.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

constexpr int kD = 128;

// ---------------------------------------------------------------------------
// status bits (mirrors include/tq.h)
// ---------------------------------------------------------------------------
constexpr uint32_t kStatusCapacity = 1u;
constexpr uint32_t kStatusNormOverflow = 2u;
constexpr uint32_t kStatusShortContext = 4u;
constexpr uint32_t kStatusPipelineStall = 8u;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
// prmt.b32 in its default mode: result byte n is byte (sel[4n+2:4n]) of the
// pair {b, a} (a = bytes 0..3), or, when sel bit 4n+3 is set, that byte's top
// bit replicated over 8 bits.  Only sel[15:0] is read.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                        uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 fp16 matrix held one row pair per lane (lane = 4*row + colpair).
__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier + bulk / tensor copies ---------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream still runs;
// griddep_wait() blocks until that predecessor has completed and its memory
// is visible (a no-op without the launch attribute), and
// griddep_launch_dependents() lets the successor start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier, giving up after ~2 s of wall time.
// Returns false on time-out (the caller raises kStatusPipelineStall).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) return false;
    }
}

// 1-D bulk copy global -> shared (bytes and both addresses multiples of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];\n" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tensor-map tile copy global -> shared.  x (innermost) in elements.
__device__ __forceinline__ void tma_g2s_2d(uint32_t dst, const void* tmap, int32_t x,
                                           int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// 128-point Walsh-Hadamard transform across a warp
// ---------------------------------------------------------------------------
__device__ __forceinline__ void wht128_lane4(float (&v)[4], int lane) {
    // Sylvester-order fast Walsh-Hadamard transform of the 128 values held
    // 4 per lane (lane l holds elements 4l .. 4l+3), unnormalised.
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[2] = a0 - a2;
    v[1] = a1 + a3;
    v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = (lane & m) ? (o - v[i]) : (v[i] + o);
        }
    }
}

__device__ __forceinline__ uint32_t sign_nibble(const uint32_t (&signs)[4], int lane) {
    return (signs[lane >> 3] >> ((lane & 7) * 4)) & 0xFu;
}

// ---------------------------------------------------------------------------
// Register dequantisers.
//
// A centroid value is an fp16 whose low and high bytes are looked up with
// prmt from 8-byte tables held in two registers each, so no lookup touches
// memory (a constant-memory table would serialise on divergent indices).
// Output: fp16 pairs in ascending dimension order, h[i] = (dim 2i, dim 2i+1).
// ---------------------------------------------------------------------------
struct Tables {
    uint32_t lo0, lo1, hi0, hi1;
};

// Four elements from a selector whose nibbles n0..n3 index both tables.
__device__ __forceinline__ void lut4(uint32_t sel, const Tables& t, uint32_t& h01,
                                     uint32_t& h23) {
    const uint32_t L = prmt(t.lo0, t.lo1, sel);
    const uint32_t H = prmt(t.hi0, t.hi1, sel);
    h01 = prmt(L, H, 0x5140);
    h23 = prmt(L, H, 0x7362);
}

// 3-bit quarter (32 dims, 12 bytes = w0..w2).  Tables are indexed by the
// 3-bit code itself (8 entries, sign included).  Nibble j of (wk & 0x7777...)
// is the code of dim 8k+j; the spare bit 4j+3 of wk is bit k of the code of
// dim 24+j, gathered into nibbles by three masked shifts.
__device__ __forceinline__ void dequant3_quarter(uint32_t w0, uint32_t w1, uint32_t w2,
                                                 const Tables& t, uint32_t (&h)[16]) {
    // right shifts as multiply-high (FMA pipe) to leave the ALU pipe to prmt
    const uint32_t m0 = w0 & 0x77777777u;
    const uint32_t m1 = w1 & 0x77777777u;
    const uint32_t m2 = w2 & 0x77777777u;
    const uint32_t sp = (__umulhi(w0, 1u << 29) & 0x11111111u) |
                        (__umulhi(w1, 1u << 30) & 0x22222222u) |
                        (__umulhi(w2, 1u << 31) & 0x44444444u);
    lut4(m0, t, h[0], h[1]);
    lut4(__umulhi(m0, 1u << 16), t, h[2], h[3]);
    lut4(m1, t, h[4], h[5]);
    lut4(__umulhi(m1, 1u << 16), t, h[6], h[7]);
    lut4(m2, t, h[8], h[9]);
    lut4(__umulhi(m2, 1u << 16), t, h[10], h[11]);
    lut4(sp, t, h[12], h[13]);
    lut4(__umulhi(sp, 1u << 16), t, h[14], h[15]);
}

// 4-bit: eight dims of one word w.  Bits 4j..4j+2 = magnitude rank of dim j;
// the tables hold the 8 magnitudes (indexed by rank).  The sign of dim j < 4
// sits in bit 8j+7 and that of dim 4+j in bit 8j+3, i.e. exactly where the
// fp16 sign bit of the gathered high byte goes (directly for dims 0..3, after
// a shift by 4 for dims 4..7), so one logic op applies four signs.
__device__ __forceinline__ void dequant4_word(uint32_t w, const Tables& t, uint32_t& h0,
                                              uint32_t& h1, uint32_t& h2, uint32_t& h3) {
    const uint32_t rk = w & 0x77777777u;
    {
        const uint32_t L = prmt(t.lo0, t.lo1, rk);
        const uint32_t H = prmt(t.hi0, t.hi1, rk) | (w & 0x80808080u);
        h0 = prmt(L, H, 0x5140);
        h1 = prmt(L, H, 0x7362);
    }
    {
        const uint32_t r2 = __umulhi(rk, 1u << 16);  // rk >> 16, on the FMA pipe
        const uint32_t w4 = w << 4;
        const uint32_t L = prmt(t.lo0, t.lo1, r2);
        const uint32_t H = prmt(t.hi0, t.hi1, r2) | (w4 & 0x80808080u);
        h2 = prmt(L, H, 0x5140);
        h3 = prmt(L, H, 0x7362);
    }
}

// Quarter dequantisers that write pair i straight into slot q[i/2][COL + 2*(i%2)]
// of an 8 x 4 array of MMA operand quads (no register copies to form quads).
template <int COL>
__device__ __forceinline__ void dequant3_quarter_q(uint32_t w0, uint32_t w1, uint32_t w2,
                                                   const Tables& t, uint32_t (&q)[8][4]) {
    const uint32_t m0 = w0 & 0x77777777u;
    const uint32_t m1 = w1 & 0x77777777u;
    const uint32_t m2 = w2 & 0x77777777u;
    const uint32_t sp = (__umulhi(w0, 1u << 29) & 0x11111111u) |
                        (__umulhi(w1, 1u << 30) & 0x22222222u) |
                        (__umulhi(w2, 1u << 31) & 0x44444444u);
    lut4(m0, t, q[0][COL], q[0][COL + 2]);
    lut4(__umulhi(m0, 1u << 16), t, q[1][COL], q[1][COL + 2]);
    lut4(m1, t, q[2][COL], q[2][COL + 2]);
    lut4(__umulhi(m1, 1u << 16), t, q[3][COL], q[3][COL + 2]);
    lut4(m2, t, q[4][COL], q[4][COL + 2]);
    lut4(__umulhi(m2, 1u << 16), t, q[5][COL], q[5][COL + 2]);
    lut4(sp, t, q[6][COL], q[6][COL + 2]);
    lut4(__umulhi(sp, 1u << 16), t, q[7][COL], q[7][COL + 2]);
}

template <int COL>
__device__ __forceinline__ void dequant4_quarter_q(uint4 w, const Tables& t, uint32_t (&q)[8][4]) {
    dequant4_word(w.x, t, q[0][COL], q[0][COL + 2], q[1][COL], q[1][COL + 2]);
    dequant4_word(w.y, t, q[2][COL], q[2][COL + 2], q[3][COL], q[3][COL + 2]);
    dequant4_word(w.z, t, q[4][COL], q[4][COL + 2], q[5][COL], q[5][COL + 2]);
    dequant4_word(w.w, t, q[6][COL], q[6][COL + 2], q[7][COL], q[7][COL + 2]);
}

__device__ __forceinline__ void dequant4_quarter(uint4 w, const Tables& t,
                                                 uint32_t (&h)[16]) {
    dequant4_word(w.x, t, h[0], h[1], h[2], h[3]);
    dequant4_word(w.y, t, h[4], h[5], h[6], h[7]);
    dequant4_word(w.z, t, h[8], h[9], h[10], h[11]);
    dequant4_word(w.w, t, h[12], h[13], h[14], h[15]);
}

}  // namespace tq
