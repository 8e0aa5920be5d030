// Split-KV (flash-decoding) causal decode attention over the temporal KV ring
// ("PersonaPlex native LM audit", section 3: 32 query / key / value heads of width 128,
// keys allowed where 0 <= query_position - key_position < 3000; section 6: the cache
// holds keys after RoPE, values without).
//
// For batch row b at position p the visible keys are positions max(0, p-ctx+1) .. p,
// stored at ring slots position mod ctx.  Grid (S, H, B): CTA (s, h, b) takes the s-th
// contiguous chunk of those positions.  128 threads = 4 warps; within a warp, lane group
// g (8 lanes) handles one key at a time and lane i of the group 16 of the 128 head
// coordinates, so a key row is one coalesced 256-byte read.  Scores use the base-2
// exponential with the query pre-scaled by log2(e)/sqrt(128) (same softmax), running
// max / sum per group, merged across groups and warps, then across the S chunks by the
// last CTA of the head to finish (completion counter, no waiting).
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;

struct Run {
    float m, l;
    float acc[16];
};

__device__ __forceinline__ void merge_run(Run& a, float m2, float l2, const float* acc2) {
    const float mn = fmaxf(a.m, m2);
    const float fa = (a.m == -INFINITY) ? 0.f : exp2f(a.m - mn);
    const float fb = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
    a.l = a.l * fa + l2 * fb;
#pragma unroll
    for (int e = 0; e < 16; ++e) a.acc[e] = a.acc[e] * fa + acc2[e] * fb;
    a.m = mn;
}

__global__ void __launch_bounds__(128) k_attn(const AttnParams p) {
    __shared__ float s_m[4], s_l[4];
    __shared__ float s_acc[4][DH];
    __shared__ int s_last;
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;

    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 3, sub = lane & 7;
    const int pos = p.st.pos[b];
    const int n = min(pos + 1, p.ctx);
    const int lo = pos - n + 1;
    const int chunk = (n + p.S - 1) / p.S;
    const int k0 = lo + s * chunk;
    const int k1 = min(k0 + chunk, pos + 1);

    float q[16];
    {
        const float4* qp = reinterpret_cast<const float4*>(p.q + (size_t)b * p.D + h * DH + 16 * sub);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float4 t = qp[v];
            q[4 * v + 0] = t.x * p.scale_log2;
            q[4 * v + 1] = t.y * p.scale_log2;
            q[4 * v + 2] = t.z * p.scale_log2;
            q[4 * v + 3] = t.w * p.scale_log2;
        }
    }
    Run run;
    run.m = -INFINITY;
    run.l = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) run.acc[e] = 0.f;

    const size_t head_base = ((size_t)b * p.H + h) * (size_t)p.ctx * DH;
    const uint16_t* kbase = p.kc + head_base + 16 * sub;
    const uint16_t* vbase = p.vc + head_base + 16 * sub;

    // warp-uniform trip count: every lane of the warp runs the same iterations
    for (int base = k0 + warp * 4; base < k1; base += 16) {
        const int kk = base + g;
        const bool valid = kk < k1;
        const int slot = valid ? (kk % p.ctx) : 0;
        uint4 ka = make_uint4(0, 0, 0, 0), kb = ka, va = ka, vb = ka;
        if (valid) {
            const uint4* kp = reinterpret_cast<const uint4*>(kbase + (size_t)slot * DH);
            const uint4* vp = reinterpret_cast<const uint4*>(vbase + (size_t)slot * DH);
            ka = __ldg(kp);
            kb = __ldg(kp + 1);
            va = __ldg(vp);
            vb = __ldg(vp + 1);
        }
        float sc = dot8(ka, q) + dot8(kb, q + 8);
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc += __shfl_xor_sync(0xffffffffu, sc, 4);
        if (valid) {
            const float mn = fmaxf(run.m, sc);
            const float corr = (run.m == -INFINITY) ? 0.f : exp2f(run.m - mn);
            const float pe = exp2f(sc - mn);
            run.l = run.l * corr + pe;
            const float v[16] = {bf16lo(va.x), bf16hi(va.x), bf16lo(va.y), bf16hi(va.y),
                                 bf16lo(va.z), bf16hi(va.z), bf16lo(va.w), bf16hi(va.w),
                                 bf16lo(vb.x), bf16hi(vb.x), bf16lo(vb.y), bf16hi(vb.y),
                                 bf16lo(vb.z), bf16hi(vb.z), bf16lo(vb.w), bf16hi(vb.w)};
#pragma unroll
            for (int e = 0; e < 16; ++e) run.acc[e] = run.acc[e] * corr + pe * v[e];
            run.m = mn;
        }
    }
    // merge the 4 key groups of the warp (lanes with equal `sub` hold the same coordinates)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, run.m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, run.l, off);
        float a2[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, run.acc[e], off);
        merge_run(run, m2, l2, a2);
    }
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) s_acc[warp][16 * sub + e] = run.acc[e];
        if (sub == 0) {
            s_m[warp] = run.m;
            s_l[warp] = run.l;
        }
    }
    __syncthreads();
    // thread t owns coordinate t
    const int t = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, A = 0.f;
    for (int w = 0; w < 4; ++w) {
        const float f = (s_m[w] == -INFINITY) ? 0.f : exp2f(s_m[w] - M);
        L += s_l[w] * f;
        A += s_acc[w][t] * f;
    }
    float* ob = p.o + (size_t)b * p.D + h * DH;
    if (p.S == 1) {
        ob[t] = A / L;
        return;
    }
    float* part = p.part + (((size_t)b * p.H + h) * p.S + s) * (DH + 2);
    part[t] = A;
    if (t == 0) {
        part[DH] = M;
        part[DH + 1] = L;
    }
    __threadfence();
    __syncthreads();
    if (t == 0) {
        const uint32_t done = atomicAdd(&p.count[(size_t)b * p.H + h], 1u);
        s_last = (done == (uint32_t)p.S - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* pb = p.part + ((size_t)b * p.H + h) * p.S * (DH + 2);
    float M2 = -INFINITY;
    for (int i = 0; i < p.S; ++i) M2 = fmaxf(M2, __ldcg(pb + (size_t)i * (DH + 2) + DH));
    float L2 = 0.f, A2 = 0.f;
    for (int i = 0; i < p.S; ++i) {
        const float mi = __ldcg(pb + (size_t)i * (DH + 2) + DH);
        const float f = (mi == -INFINITY) ? 0.f : exp2f(mi - M2);
        L2 += __ldcg(pb + (size_t)i * (DH + 2) + DH + 1) * f;
        A2 += __ldcg(pb + (size_t)i * (DH + 2) + t) * f;
    }
    ob[t] = A2 / L2;
    if (t == 0) p.count[(size_t)b * p.H + h] = 0u;
}

}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.S, (unsigned)p.H, (unsigned)p.B);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attn, p);
}

}  // namespace pm
