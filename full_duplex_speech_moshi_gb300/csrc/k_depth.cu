// Depformer helpers ("PersonaPlex native LM audit", section 4 "Native depth
// computation"): the per-frame set-up kernel and the depth self-attention.
//
// k_dep_begin resolves and validates the conditioning text token (caller's, or the
// context's last greedy text token) and the supplied codes (-1 = greedy), copies the
// caller's hidden state into the buffer the chain reads, and raises the abort flag on
// an invalid value.  Invalid values are replaced by 0 / -1 so that every later index
// stays in range; an aborted frame writes no feedback tokens.
//
// k_dep_attn: one warp per (head, batch row).  Position q attends to depth positions
// max(0, q - dep_ctx + 1) .. q of this frame (no positional encoding); lane l owns
// coordinates 2l, 2l+1 of the 64-wide head.
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

__global__ void __launch_bounds__(256) k_dep_begin(const DepBeginParams p) {
    pdl_trigger();
    pdl_wait();
    int bad = 0;
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        int tok = p.dio->text_tok ? p.dio->text_tok[i] : p.st.sel[(size_t)i * PM_MAX_STREAMS_DEV + 0];
        if (tok < 0 || tok >= p.text_rows) {
            bad = 1;
            tok = 0;
        }
        p.st.dep_tok[i] = tok;
    }
    for (int i = threadIdx.x; i < p.B * p.Q; i += blockDim.x) {
        int sup = p.dio->supplied ? p.dio->supplied[i] : -1;
        if (sup < -1 || sup >= p.card) {
            bad = 1;
            sup = -1;
        }
        p.st.dep_sup[i] = sup;
    }
    if (p.dio->hidden != p.h_internal) {
        const int n4 = p.B * p.D / 4;
        const float4* src = reinterpret_cast<const float4*>(p.dio->hidden);
        float4* dst = reinterpret_cast<float4*>(p.h_internal);
        for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        p.st.status[1] = bad ? 1u : 0u;
        if (bad) set_status(p.st.status, PM_DEV_ERR_INVALID_ID);
    }
}

__global__ void __launch_bounds__(32) k_dep_attn(const DepAttnParams p) {
    pdl_trigger();
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
    const int qpos = p.q_pos;
    const int lo = max(0, qpos - p.dep_ctx + 1);
    const int n = qpos - lo + 1;
    const float2 qv = *reinterpret_cast<const float2*>(p.q + (size_t)b * p.Dd + h * p.dhd + 2 * lane);
    const size_t hb = ((size_t)b * p.Hd + h) * p.Q * p.dhd;
    float sc[16];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        sc[i] = -INFINITY;
        if (i < n) {
            const uint32_t kk = *reinterpret_cast<const uint32_t*>(p.kc + hb + (size_t)(lo + i) * p.dhd + 2 * lane);
            float d = qv.x * bf16lo(kk) + qv.y * bf16hi(kk);
            d = warp_sum(d) * p.scale_log2;
            sc[i] = d;
            m = fmaxf(m, d);
        }
    }
    float l = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (i < n) {
            const float e = exp2f(sc[i] - m);
            l += e;
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(p.vc + hb + (size_t)(lo + i) * p.dhd + 2 * lane);
            o0 += e * bf16lo(vv);
            o1 += e * bf16hi(vv);
        }
    }
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    *reinterpret_cast<float2*>(p.o + (size_t)b * p.Dd + h * p.dhd + 2 * lane) = make_float2(o0 / l, o1 / l);
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, bool pdl, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

}  // namespace

cudaError_t launch_dep_begin(const DepBeginParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(256), s, pdl, attr);
    return cudaLaunchKernelEx(&cfg, k_dep_begin, p);
}

cudaError_t launch_dep_attn(const DepAttnParams& p, cudaStream_t s, bool pdl) {
    if (p.dhd != 64 || p.dep_ctx > 16) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)p.Hd, (unsigned)p.B), dim3(32), s, pdl, attr);
    return cudaLaunchKernelEx(&cfg, k_dep_attn, p);
}

}  // namespace pm
