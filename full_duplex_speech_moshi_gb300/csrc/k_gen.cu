// Generator step kernels ("PersonaPlex native LM audit", section 7 "One exact generator
// step"; the rings of section 6 "Generator delayed-code cache").
//
// Per stream b the context keeps a token ring and a provided ring of 4 columns for each of
// the streams (stride PM_MAX_STREAMS_DEV), and the generator offset s (separate from the
// temporal position).  One generator call is
//   k_gen_begin   steps 1-3: place the provided codes at (s + delay[k]) mod 4 (provided),
//                 insert the initial IDs at s mod 4 while s <= delay[k] (provided), hand the
//                 frame the input column (s - 1) mod 4 (initial IDs at s = 0, whose frame
//                 is undone afterwards);
//   frame         step 4: the temporal frame on those inputs as given (FrameIO.direct);
//   k_gen_mid     steps 4-5: the depth conditioning token (the provided text target, else
//                 the frame's selection) and the provided depth targets (-1: select);
//   depformer     step 5;
//   k_gen_end     steps 6-7: selections into unprovided target slots, the input column's
//                 provided flags cleared, the aligned output (s - max_delay + delay[k]) mod 4
//                 once s > max_delay, s advanced.
// One CTA per stream, one thread per token stream (or depth position): every thread
// touches only its own stream's ring slots, so no thread waits on another except where
// noted.
#include "pm_kernels.h"

namespace pm {
namespace {

__device__ __forceinline__ int32_t* slot(int32_t* base, int b, int k) {
    return base + ((size_t)b * PM_MAX_STREAMS_DEV + k) * 4;
}

__global__ void __launch_bounds__(32) k_gen_begin(const GenParams p) {
    const int b = blockIdx.x, k = threadIdx.x;
    // the stream's position and selections, restored if this call's frame is undone
    if (k == 0) p.pos_save[b] = p.st.pos[b];
    p.sel_save[(size_t)b * PM_MAX_STREAMS_DEV + k] = p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + k];
    if (k >= p.S) return;
    const int s = p.off[b];
    int32_t* R = slot(p.ring, b, k);
    int32_t* P = slot(p.prov, b, k);
    const int d = p.delays[k];
    // 1. provided codes (the user's codebooks, forced text / agent codes)
    if (p.provided) {
        const int32_t code = p.provided[(size_t)b * p.S + k];
        if (code >= 0) {
            R[(s + d) & 3] = code;
            P[(s + d) & 3] = 1;
        }
    }
    // 2. the initial calls insert the native initial tokens
    if (s <= d) {
        R[s & 3] = p.init[k];
        P[s & 3] = 1;
    }
    // 3. the temporal input column (a call at s = 0 runs no model step of its own; if the
    // batch's frame runs anyway, it is handed the initial IDs and undone in k_gen_end)
    p.in[(size_t)b * p.S + k] = (s == 0) ? p.init[k] : R[(s - 1) & 3];
}

__global__ void __launch_bounds__(32) k_gen_mid(const GenParams p) {
    const int b = blockIdx.x, q = threadIdx.x;
    const int s = p.off[b];
    const int tgt = s & 3;
    if (q < p.Q) {
        const int k = q + 1;
        p.dep_sup[(size_t)b * p.Q + q] = (s > 0 && slot(p.prov, b, k)[tgt]) ? slot(p.ring, b, k)[tgt] : -1;
    }
    if (q == 0) {
        int32_t tok = (s > 0 && slot(p.prov, b, 0)[tgt]) ? slot(p.ring, b, 0)[tgt]
                                                         : p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 0];
        p.dep_tok[b] = tok < 0 ? 0 : tok;  // a row at s = 0 only needs some valid token
    }
}

__global__ void __launch_bounds__(32) k_gen_end(const GenParams p) {
    const int b = blockIdx.x, k = threadIdx.x;
    const int s = p.off[b];
    __syncthreads();  // every thread has read the offset before thread 0 advances it
    if (s == 0) {
        // the first call: nothing selected, no output; a frame run for the batch is undone
        if (p.ran) {
            if (k == 0) p.st.pos[b] = p.pos_save[b];
            p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + k] = p.sel_save[(size_t)b * PM_MAX_STREAMS_DEV + k];
        }
        if (k < p.S && p.out) p.out[(size_t)b * p.S + k] = -1;
        if (k == 0) {
            if (p.valid) p.valid[b] = 0;
            p.off[b] = 1;
        }
        return;
    }
    if (k < p.S) {
        int32_t* R = slot(p.ring, b, k);
        int32_t* P = slot(p.prov, b, k);
        const int tgt = s & 3;
        // 6. selections into unprovided target slots; the consumed input's flags cleared
        if (!P[tgt])
            R[tgt] = (k == 0) ? p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 0] : p.st.dep_codes[(size_t)b * p.Q + k - 1];
        P[(s - 1) & 3] = 0;
        // 7. the aligned output once the initial delay padding is over
        if (p.out) p.out[(size_t)b * p.S + k] = (s > p.max_delay) ? R[(s - p.max_delay + p.delays[k]) & 3] : -1;
    }
    if (k == 0) {
        if (p.valid) p.valid[b] = s > p.max_delay ? 1 : 0;
        p.off[b] = s + 1;
    }
}

}  // namespace

cudaError_t launch_gen(int phase, const GenParams& p, cudaStream_t s) {
    const dim3 grid((unsigned)p.B), block(32);
    if (phase == 0)
        k_gen_begin<<<grid, block, 0, s>>>(p);
    else if (phase == 1)
        k_gen_mid<<<grid, block, 0, s>>>(p);
    else
        k_gen_end<<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pm
