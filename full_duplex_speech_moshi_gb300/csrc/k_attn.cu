// Split-KV (flash-decoding) causal decode attention over the temporal KV ring
// ("PersonaPlex native LM audit", section 3: 32 query / key / value heads of width 128,
// keys allowed where 0 <= query_position - key_position < 3000; section 6: the cache
// holds keys after RoPE, values without).
//
// For batch row b at position p the visible keys are positions max(0, p-win+1) .. p,
// stored at ring slots position mod ctx (win = ctx for the declared mask, ctx - 1 for the
// pinned ring's labels, which hide the oldest key of a full ring).  Work item (b, h, c) is the 64 keys
// lo + 64c .. lo + 64c + 63 of row b's window for head h.  The items of all rows form one
// list whose length follows the device-resident positions; a fixed grid of CTAs walks it
// with a grid stride, so the launch does not grow with the context.  128 threads = 4
// warps; in a warp, lane group g (8 lanes) takes 4 keys and lane i of the group 16 of
// the 128 coordinates, so a key row is one coalesced 256-byte read.
//
// Keys and values of positions before p were written by earlier frames, so each lane
// loads its first item's K and V rows into registers before griddepcontrol.wait: with
// programmatic dependent launch this overlaps the fused-QKV kernel that writes the
// current position's K/V and the query.  Scores use the base-2 exponential with the
// query pre-scaled by log2(e)/sqrt(128) (the same softmax).  Running (max, sum, weighted
// values) merge across lane groups (shuffles), warps (shared memory) and finally across
// the chunks of a (b, h) in the CTA that finishes last (completion counter, nothing
// waits), which stages the chunk maxima in shared memory and reads the partial vectors
// with independent loads.
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;
constexpr int KPC = 64;    // keys per CTA item
constexpr int KPG = 4;     // keys per lane group (4 warps x 4 groups x 4 keys = 64)
constexpr int MAX_CHUNKS = 64;  // chunks per (b, h) the merge stages in shared memory (ctx <= 4096)

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float* v) {
    v[0] = bf16lo(a.x); v[1] = bf16hi(a.x); v[2] = bf16lo(a.y); v[3] = bf16hi(a.y);
    v[4] = bf16lo(a.z); v[5] = bf16hi(a.z); v[6] = bf16lo(a.w); v[7] = bf16hi(a.w);
    v[8] = bf16lo(b.x); v[9] = bf16hi(b.x); v[10] = bf16lo(b.y); v[11] = bf16hi(b.y);
    v[12] = bf16lo(b.z); v[13] = bf16hi(b.z); v[14] = bf16lo(b.w); v[15] = bf16hi(b.w);
}

__device__ __forceinline__ int n_chunks(int pos, int ctx) { return (min(pos + 1, ctx) + KPC - 1) / KPC; }

__global__ void __launch_bounds__(128) k_attn(const AttnParams p) {
    __shared__ int s_first[PM_MAX_B_DEV + 1];  // prefix of chunk counts over batch rows
    __shared__ float s_m[4], s_l[4];
    __shared__ float s_acc[4][DH];
    __shared__ float s_pm[MAX_CHUNKS], s_pl[MAX_CHUNKS];
    __shared__ int s_last;
    pdl_trigger();
    // positions do not change within a frame (only the final text-head kernel advances
    // them), so every row's window, and the whole work list, is known before the wait
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int bb = 0; bb < p.B; ++bb) {
            s_first[bb] = acc;
            acc += p.H * n_chunks(p.st.pos[bb], p.win);
        }
        s_first[p.B] = acc;
    }
    __syncthreads();
    const int total = s_first[p.B];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 3, sub = lane & 7;
    const int t = threadIdx.x;
    bool waited = false;

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        int b = 0;
        while (item >= s_first[b + 1]) ++b;
        const int pos = p.st.pos[b];
        const int n = min(pos + 1, p.win);
        const int lo = pos - n + 1;
        const int nc = (n + KPC - 1) / KPC;
        const int h = (item - s_first[b]) / nc;
        const int ci = (item - s_first[b]) % nc;
        const int k0 = lo + ci * KPC + warp * 16 + g * KPG;  // this lane group's first key
        const int k1 = pos + 1;

        const size_t head_base = ((size_t)b * p.H + h) * (size_t)p.ctx * DH;
        const uint16_t* kbase = p.kc + head_base + 16 * sub;
        const uint16_t* vbase = p.vc + head_base + 16 * sub;
        uint4 kr[KPG][2], vr[KPG][2];
#pragma unroll
        for (int it = 0; it < KPG; ++it) {
            const int kk = k0 + it;
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
        if (!waited) {
            pdl_wait();
            waited = true;
            if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
        }
        float q[16];
        {
            const float4* qp = reinterpret_cast<const float4*>(p.q + (size_t)b * p.D + h * DH + 16 * sub);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 tq = qp[v];
                q[4 * v + 0] = tq.x * p.scale_log2;
                q[4 * v + 1] = tq.y * p.scale_log2;
                q[4 * v + 2] = tq.z * p.scale_log2;
                q[4 * v + 3] = tq.w * p.scale_log2;
            }
        }
        // the current position's row is written by the kernel this one waited for
#pragma unroll
        for (int it = 0; it < KPG; ++it)
            if (k0 + it == pos) {
                const int slot = pos % p.ctx;
                const uint4* kp = reinterpret_cast<const uint4*>(kbase + (size_t)slot * DH);
                const uint4* vp = reinterpret_cast<const uint4*>(vbase + (size_t)slot * DH);
                kr[it][0] = __ldcg(kp);
                kr[it][1] = __ldcg(kp + 1);
                vr[it][0] = __ldcg(vp);
                vr[it][1] = __ldcg(vp + 1);
            }

        float sc[KPG];
        float m = -INFINITY;
#pragma unroll
        for (int it = 0; it < KPG; ++it) {
            float kv[16];
            unpack16(kr[it][0], kr[it][1], kv);
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) d = fmaf(q[e], kv[e], d);
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            d += __shfl_xor_sync(0xffffffffu, d, 4);
            sc[it] = (k0 + it < k1) ? d : -INFINITY;
            m = fmaxf(m, sc[it]);
        }
        float l = 0.f, acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        if (m != -INFINITY) {
#pragma unroll
            for (int it = 0; it < KPG; ++it) {
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
        // merge the 4 warps in shared memory; thread t owns coordinate t
        if (g == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) s_acc[warp][16 * sub + e] = acc[e];
            if (sub == 0) {
                s_m[warp] = m;
                s_l[warp] = l;
            }
        }
        __syncthreads();
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
        if (nc == 1) {
            ob[t] = A / L;
            if (obb) obb[t] = f32_to_bf16_rne(A / L);
            __syncthreads();  // shared partials are reused by the next item
            continue;
        }
        float* part = p.part + (((size_t)b * p.H + h) * p.S + ci) * (DH + 2);
        part[t] = A;
        if (t == 0) {
            part[DH] = M;
            part[DH + 1] = L;
        }
        __threadfence();
        __syncthreads();
        if (t == 0) {
            const uint32_t done = atomicAdd(&p.count[(size_t)b * p.H + h], 1u);
            s_last = (done == (uint32_t)nc - 1u) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) continue;
        // last chunk of (b, h): merge every chunk in slot order with loads in parallel
        __threadfence();
        const float* pb = p.part + ((size_t)b * p.H + h) * p.S * (DH + 2);
        for (int i = t; i < nc; i += 128) {
            s_pm[i] = __ldcg(pb + (size_t)i * (DH + 2) + DH);
            s_pl[i] = __ldcg(pb + (size_t)i * (DH + 2) + DH + 1);
        }
        __syncthreads();
        float Mx = -INFINITY;
        for (int i = 0; i < nc; ++i) Mx = fmaxf(Mx, s_pm[i]);
        float Lx = 0.f, Ax = 0.f;
#pragma unroll 8
        for (int i = 0; i < nc; ++i) {
            const float f = (s_pm[i] == -INFINITY) ? 0.f : exp2f(s_pm[i] - Mx);
            Lx += s_pl[i] * f;
            Ax += __ldcg(pb + (size_t)i * (DH + 2) + t) * f;
        }
        ob[t] = Ax / Lx;
        if (obb) obb[t] = f32_to_bf16_rne(Ax / Lx);
        if (t == 0) p.count[(size_t)b * p.H + h] = 0u;
        __syncthreads();
    }
}

}  // namespace

int attn_max_splits(int ctx) { return (ctx + KPC - 1) / KPC; }

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.S < attn_max_splits(p.ctx) || p.S > MAX_CHUNKS || p.B > PM_MAX_B_DEV || p.grid < 1 || p.win < 1 ||
        p.win > p.ctx)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
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
