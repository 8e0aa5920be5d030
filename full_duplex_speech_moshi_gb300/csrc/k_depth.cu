// Depformer set-up ("PersonaPlex native LM audit", section 4 "Native depth
// computation").  The depth self-attention itself runs in the prologue of the W_o
// projection (k_gemv, PRO_DEPATTN).
//
// k_dep_begin resolves and validates the conditioning text token (caller's, or the
// context's last greedy text token) and the supplied codes (-1 = greedy; a supplied code
// is a row of the next position's depth embedding, so 0..dep_audio_in-1), copies the
// caller's hidden state into the buffer the chain reads, and raises the abort flag on
// an invalid value.  Invalid values are replaced by 0 / -1 so that every later index
// stays in range; an aborted frame writes no feedback tokens.
//
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
        // depth-head accumulators start cleared, also after a call whose head did not finish
        p.st.dep_amax[i] = 0ull;
        p.st.dep_count[i] = 0u;
    }
    for (int i = threadIdx.x; i < p.B * p.Q; i += blockDim.x) {
        int sup = p.dio->supplied ? p.dio->supplied[i] : -1;
        if (sup < -1 || sup >= p.sup_rows) {
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


}  // namespace pm
