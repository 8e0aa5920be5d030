// Split-KV (flash-decoding) causal decode attention over the temporal KV ring
// ("PersonaPlex native LM audit", section 3: 32 query / key / value heads of width 128,
// keys allowed where 0 <= query_position - key_position < 3000; section 6: the cache
// holds keys after RoPE, values without).
//
// For batch row b at position p the visible keys are positions max(0, p-ctx+1) .. p,
// stored at ring slots position mod ctx.  Grid (S_max, H, B) with S_max = ceil(ctx / 64):
// CTA (s, h, b) owns keys lo + 64 s .. lo + 64 s + 63 of that window; CTAs past the
// window's last chunk exit at once.  128 threads = 4 warps; in a warp, lane group g
// (8 lanes) takes one key per step and lane i of the group 16 of the 128 coordinates, so
// a key row is one coalesced 256-byte read; four steps cover the CTA's 64 keys.
//
// Keys and values of positions before p were written by earlier frames, so each lane
// loads its four keys' K and V rows into registers before griddepcontrol.wait: with
// programmatic dependent launch this overlaps the fused-QKV kernel that writes the
// current position's K/V and the query.  After the wait only the query, the current
// position's row (if this CTA owns it) and the softmax remain.  Scores use the base-2
// exponential with the query pre-scaled by log2(e)/sqrt(128) (the same softmax).  Chunk
// results (running max, sum, weighted values) merge across groups, warps and finally
// across chunks in the last CTA of the head to finish (completion counter; no waiting).
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;
constexpr int KPC = 64;     // keys per CTA
constexpr int STEPS = 4;    // KPC / 16 keys per step (4 warps x 4 lane groups)

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float* v) {
    v[0] = bf16lo(a.x); v[1] = bf16hi(a.x); v[2] = bf16lo(a.y); v[3] = bf16hi(a.y);
    v[4] = bf16lo(a.z); v[5] = bf16hi(a.z); v[6] = bf16lo(a.w); v[7] = bf16hi(a.w);
    v[8] = bf16lo(b.x); v[9] = bf16hi(b.x); v[10] = bf16lo(b.y); v[11] = bf16hi(b.y);
    v[12] = bf16lo(b.z); v[13] = bf16hi(b.z); v[14] = bf16lo(b.w); v[15] = bf16hi(b.w);
}

__global__ void __launch_bounds__(128) k_attn(const AttnParams p) {
    __shared__ float s_m[4], s_l[4];
    __shared__ float s_acc[4][DH];
    __shared__ int s_last;
    pdl_trigger();
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    // positions do not change within a frame (only the final text-head kernel advances
    // them), so the window is known before the wait
    const int pos = p.st.pos[b];
    const int n = min(pos + 1, p.ctx);
    const int lo = pos - n + 1;
    const int n_split = (n + KPC - 1) / KPC;
    if (s >= n_split) return;
    const int k0 = lo + s * KPC;
    const int k1 = min(k0 + KPC, pos + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 3, sub = lane & 7;
    const size_t head_base = ((size_t)b * p.H + h) * (size_t)p.ctx * DH;
    const uint16_t* kbase = p.kc + head_base + 16 * sub;
    const uint16_t* vbase = p.vc + head_base + 16 * sub;

    uint4 kr[STEPS][2], vr[STEPS][2];
#pragma unroll
    for (int it = 0; it < STEPS; ++it) {
        const int kk = k0 + warp * 4 + g + 16 * it;
        kr[it][0] = kr[it][1] = vr[it][0] = vr[it][1] = make_uint4(0, 0, 0, 0);
        if (kk < k1 && kk != pos) {
            const int slot = kk % p.ctx;
            const uint4* kp = reinterpret_cast<const uint4*>(kbase + (size_t)slot * DH);
            const uint4* vp = reinterpret_cast<const uint4*>(vbase + (size_t)slot * DH);
            kr[it][0] = __ldg(kp);
            kr[it][1] = __ldg(kp + 1);
            vr[it][0] = __ldg(vp);
            vr[it][1] = __ldg(vp + 1);
        }
    }

    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
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
    // the current position's row is written by the kernel this one waited for
    const int kcur = pos - k0 - warp * 4 - g;  // step that holds `pos` for this lane group, if any
    if (kcur >= 0 && kcur % 16 == 0 && kcur / 16 < STEPS) {
        const int it = kcur / 16;
        const int slot = pos % p.ctx;
        const uint4* kp = reinterpret_cast<const uint4*>(kbase + (size_t)slot * DH);
        const uint4* vp = reinterpret_cast<const uint4*>(vbase + (size_t)slot * DH);
#pragma unroll
        for (int j = 0; j < STEPS; ++j)
            if (j == it) {
                kr[j][0] = __ldcg(kp);
                kr[j][1] = __ldcg(kp + 1);
                vr[j][0] = __ldcg(vp);
                vr[j][1] = __ldcg(vp + 1);
            }
    }

    float sc[STEPS];
    float m = -INFINITY;
#pragma unroll
    for (int it = 0; it < STEPS; ++it) {
        const int kk = k0 + warp * 4 + g + 16 * it;
        float kv[16];
        unpack16(kr[it][0], kr[it][1], kv);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) d = fmaf(q[e], kv[e], d);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        sc[it] = (kk < k1) ? d : -INFINITY;
        m = fmaxf(m, sc[it]);
    }
    float l = 0.f, acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    if (m != -INFINITY) {
#pragma unroll
        for (int it = 0; it < STEPS; ++it) {
            const float w = exp2f(sc[it] - m);  // exp2(-inf) = 0 for keys past the window
            l += w;
            float vv[16];
            unpack16(vr[it][0], vr[it][1], vv);
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = fmaf(w, vv[e], acc[e]);
        }
    }
    // merge the 4 lane groups of the warp (lanes with equal `sub` hold the same coordinates)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, m2);
        const float fa = (m == -INFINITY) ? 0.f : exp2f(m - mn);
        const float fb = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float a2 = __shfl_xor_sync(0xffffffffu, acc[e], off);
            acc[e] = acc[e] * fa + a2 * fb;
        }
        l = l * fa + l2 * fb;
        m = mn;
    }
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) s_acc[warp][16 * sub + e] = acc[e];
        if (sub == 0) {
            s_m[warp] = m;
            s_l[warp] = l;
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
    uint16_t* obb = p.ob ? p.ob + (size_t)b * p.D + h * DH : nullptr;
    if (n_split == 1) {
        ob[t] = A / L;
        if (obb) obb[t] = f32_to_bf16_rne(A / L);
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
        s_last = (done == (uint32_t)n_split - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* pb = p.part + ((size_t)b * p.H + h) * p.S * (DH + 2);
    float M2 = -INFINITY;
    for (int i = 0; i < n_split; ++i) M2 = fmaxf(M2, __ldcg(pb + (size_t)i * (DH + 2) + DH));
    float L2 = 0.f, A2 = 0.f;
    for (int i = 0; i < n_split; ++i) {
        const float mi = __ldcg(pb + (size_t)i * (DH + 2) + DH);
        const float f = (mi == -INFINITY) ? 0.f : exp2f(mi - M2);
        L2 += __ldcg(pb + (size_t)i * (DH + 2) + DH + 1) * f;
        A2 += __ldcg(pb + (size_t)i * (DH + 2) + t) * f;
    }
    ob[t] = A2 / L2;
    if (obb) obb[t] = f32_to_bf16_rne(A2 / L2);
    if (t == 0) p.count[(size_t)b * p.H + h] = 0u;
}

}  // namespace

int attn_max_splits(int ctx) { return (ctx + KPC - 1) / KPC; }

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.S < attn_max_splits(p.ctx)) return cudaErrorInvalidValue;
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
