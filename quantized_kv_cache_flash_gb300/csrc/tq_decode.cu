// Split-K decode: the combine + inverse-rotation kernel, the bounded-wait
// self-test, and the dispatch over the decode kernel's variants (those are
// instantiated in tq_decode_f.cu (fp16 K), tq_decode_q.cu (quantized K) and
// tq_decode_r.cu (quantized K with the centroid residual product), compiled
// in parallel).
#include "tq_decode_kernel.cuh"  // chunk arithmetic shared with the decode kernel

namespace tq {

// Per-unit variant tables (tq_decode_f.cu / _q.cu / _r.cu).
int decode_variant_f(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1);
int decode_variant_q(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1);
int decode_variant_r(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1);

namespace {
// kb: 0 = fp16 K; rows: 4 (quantized K only), 8 or 16
int decode_variant(bool launch, int kbits, int vbits, int group_rows, bool table, bool res,
                   const DecodeParams& p, const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0,
                   cudaEvent_t ev1) {
    const int kb = kbits == 16 ? 0 : kbits;
    if (kb == 0) return decode_variant_f(launch, 0, vbits, group_rows < 8 ? 8 : group_rows, false, false, p,
                                         kmap, stream, ev0, ev1);
    if (res && !table) return decode_variant_r(launch, kb, vbits, group_rows, false, true, p, kmap, stream, ev0, ev1);
    return decode_variant_q(launch, kb, vbits, group_rows, table, false, p, kmap, stream, ev0, ev1);
}
}  // namespace

// One CTA per output row (b, q head, query j): merge the partials of the
// CTAs that covered the row's unit with their log-sum-exp weights, apply
// v_rescale, leave the rotated basis (Rot^-1(y) = s * (H y) / sqrt(128)) and
// store fp16.  The W warps split the partials (warp w takes i = w mod W) in
// passes of 8 per warp: a pass's (m, l) pairs and O rows are loaded
// together, so a unit of up to 8W partials is one trip to L2.  Each
// warp merges its share against a running max (lane l holding dims
// 4l..4l+3), and warp 0 merges the W results.
template <int W>
__global__ void __launch_bounds__(32 * W) tq_combine_kernel(const __grid_constant__ CombineParams p) {
    __shared__ float4 s_acc[W][32];
    __shared__ float s_m[W], s_den[W];
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

    // The unit's global chunk range [k_first, k_first + nch) and the CTAs over
    // it.  `lengths` may be read before the dependency wait: this grid follows
    // the decode kernel, whose CTAs each waited for the work that wrote
    // `lengths` before any of them let this grid launch.
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
    griddep_wait();  // the decode kernel's partials

    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = warp; i0 < n; i0 += 8 * W) {
        // this pass: partials i0 + W k, k < 8; lane k < 8 holds partial k's (m, l)
        const bool mine = lane < 8 && used(i0 + W * lane);
        const unsigned used_mask = __ballot_sync(0xffffffffu, mine);  // bit k: partial i0 + W k
        const float2 ml = mine ? __ldcg(reinterpret_cast<const float2*>(p.part_ml) + row0 +
                                        16 * static_cast<size_t>(i0 + W * lane))
                               : make_float2(-INFINITY, 0.f);
        float4 o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            o[k] = ((used_mask >> k) & 1u)
                       ? __ldcg(reinterpret_cast<const float4*>(
                                    p.part_o + (row0 + 16 * static_cast<size_t>(i0 + W * k)) * kD) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        float mr = ml.x;
#pragma unroll
        for (int o2 = 4; o2 > 0; o2 >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o2));
        mr = __shfl_sync(0xffffffffu, mr, 0);
        const float Mn = fmaxf(M, mr);
        if (Mn == -INFINITY) continue;  // (warp-uniform) no partial of this pass saw a token
        if (M != Mn) {  // rescale what earlier passes merged
            const float sc = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
            acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
            den *= sc;
            M = Mn;
        }
        const float w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
        den += w * ml.y;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (wk != 0.f) {   // (a partial whose rows saw no token adds nothing, whatever its O)
                acc.x += wk * o[k].x; acc.y += wk * o[k].y;
                acc.z += wk * o[k].z; acc.w += wk * o[k].w;
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
    for (int w = 0; w < W; ++w) Mall = fmaxf(Mall, s_m[w]);
    float dsum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
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

int launch_decode(int kbits, int vbits, const DecodeParams& p, const CUtensorMap* kmap,
                  cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    return decode_variant(true, kbits, vbits, p.group_rows, p.table != 0, p.k_res != 0, p, kmap, stream, ev0,
                          ev1);
}

// Eight warps where units average more than 16 partials (few units over many
// CTAs), four otherwise.
int launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int rows = p.batch * p.hq * p.tq;
    const long long units = 1ll * p.batch * p.hkv * p.row_groups;
    if (p.num_ctas > 16 * units) return launch_pdl(tq_combine_kernel<8>, dim3(rows), dim3(256), 0, stream, p);
    return launch_pdl(tq_combine_kernel<4>, dim3(rows), dim3(128), 0, stream, p);
}

int decode_ctas_per_sm(int kbits, int vbits, int group_rows, bool table, bool res) {
    DecodeParams dummy{};
    const int c = decode_variant(false, kbits, vbits, group_rows, table, res, dummy, nullptr, nullptr, nullptr,
                                 nullptr);
    return c < 1 ? 1 : c;
}

}  // namespace tq
