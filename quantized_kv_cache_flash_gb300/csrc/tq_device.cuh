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

// D += A(16x32, row) * B(32x8, col), e4m3 inputs (four per register), fp32
// accumulate.  A: a0 = row g, k 4t..4t+3; a1 = row g+8, same k; a2, a3 the same
// rows at k 16+4t..16+4t+3.  B: b0 = column g, k 4t..4t+3; b1 = k 16+4t...
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
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

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 values as e4m3 (round to nearest even, saturating at +-448) in the
// low 16 bits: lo in byte 0, hi in byte 1.
__device__ __forceinline__ uint32_t fp8x2_e4m3(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
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

// Named barriers (ids 1..15; 0 is __syncthreads) over n threads, whole warps.
// Every thread that takes part must reach each use: callers place them on
// paths no thread leaves early.
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t n) {
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
// named_bar_sync that also returns whether any participant passed pred.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
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

// Non-blocking probe of phase `parity` (try_wait may suspend the thread for a
// while when the phase is not complete; test_wait returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier, giving up after limit_ns of wall
// time (2 s by default).  Returns false on time-out (the caller raises
// kStatusPipelineStall).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
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

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(tmap) : "memory");
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

// dequant4_word plus the centroids' fp8 residuals (e4m3 bytes of
// (c - fp16(c)) * 2^a looked up from the 8-byte table r8lo:r8hi by rank, the
// element's sign XORed into bit 7): q0 = dims 0..3, q1 = dims 4..7.
__device__ __forceinline__ void dequant4_word_res(uint32_t w, const Tables& t, uint32_t r8lo,
                                                  uint32_t r8hi, uint32_t& h0, uint32_t& h1,
                                                  uint32_t& h2, uint32_t& h3, uint32_t& q0,
                                                  uint32_t& q1) {
    const uint32_t rk = w & 0x77777777u;
    const uint32_t s0 = w & 0x80808080u;
    {
        const uint32_t L = prmt(t.lo0, t.lo1, rk);
        const uint32_t H = prmt(t.hi0, t.hi1, rk) | s0;
        h0 = prmt(L, H, 0x5140);
        h1 = prmt(L, H, 0x7362);
        q0 = prmt(r8lo, r8hi, rk) ^ s0;
    }
    {
        const uint32_t r2 = __umulhi(rk, 1u << 16);  // rk >> 16, on the FMA pipe
        const uint32_t s1 = (w << 4) & 0x80808080u;
        const uint32_t L = prmt(t.lo0, t.lo1, r2);
        const uint32_t H = prmt(t.hi0, t.hi1, r2) | s1;
        h2 = prmt(L, H, 0x5140);
        h3 = prmt(L, H, 0x7362);
        q1 = prmt(r8lo, r8hi, r2) ^ s1;
    }
}

__device__ __forceinline__ void dequant4_quarter(uint4 w, const Tables& t,
                                                 uint32_t (&h)[16]) {
    dequant4_word(w.x, t, h[0], h[1], h[2], h[3]);
    dequant4_word(w.y, t, h[4], h[5], h[6], h[7]);
    dequant4_word(w.z, t, h[8], h[9], h[10], h[11]);
    dequant4_word(w.w, t, h[12], h[13], h[14], h[15]);
}


// ---- tcgen05: 5th-generation tensor cores, accumulators in tensor memory ----
// Operands come from shared memory through 64-bit matrix descriptors; the
// accumulator D lives in tensor memory (TMEM: 128 lanes x 512 32-bit columns
// per SM; row i of an M = 128 tile is lane i).  One thread issues the MMAs;
// tcgen05.commit arrives on an mbarrier when they have completed.

// Byte offset of element (row, k) of a [128][128] fp16 tile in the K-major
// 128-byte-swizzle layout: two 64-element column blocks of 128 rows x 128 B
// (16 KB each), the 16-byte chunk index XORed with (row & 7) (the layout TMA's
// 128-byte swizzle writes).  The tile base must be 1024-byte aligned.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
    return static_cast<uint32_t>((k >> 6) * 16384 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                                 (k & 7) * 2);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// The alloc, dealloc, ld and st forms are warp-collective (.sync.aligned):
// every lane of the warp executes them together, so each starts by
// reconverging the warp.
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {  // one warp
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 ::"r"(slot_smem), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // one warp
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T  (M x N x 16)
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]^T  (M x N x 16); A: lane = row, two fp16 per column
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 ::"r"(bar) : "memory");
}
// 32 consecutive columns of this warp's 32 lanes (thread = lane), then wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// tmem_ld32 without its wait: the registers are valid only after
// tmem_ld_wait on them (which also keeps their uses behind the wait).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
// Waits for this thread's outstanding tensor-memory loads; a and b (the
// registers they fill) are threaded through so no use moves above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
                   "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]),
                   "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]),
                   "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]),
                   "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31])
                 :
                 : "memory");
    asm volatile(""
                 : "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                   "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                   "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]),
                   "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]),
                   "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    __syncwarp();
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

}  // namespace tq
