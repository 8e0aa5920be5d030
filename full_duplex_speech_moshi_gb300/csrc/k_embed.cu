// Delay assembly, ID validation and the 17-stream embedding gather-sum
// ("PersonaPlex native LM audit": section 3 "Input embedding sum" -- x is the sum of the
// 17 table rows, ID -1 is an exact zero vector, -2 never a valid input; section 7 "One
// exact generator step" -- stream delays and initial IDs).
//
// Grid (ceil(D / 1024), B), 128 threads; thread t of CTA (cx, b) sums columns
// cx*1024 + 8t .. +7 of the 17 selected rows with 16-byte loads.
//
// Per stream k of batch row b at position p = pos[b]:
//   id_k    = ids[b][k], or the stream's last selected token when ids[b][k] == -3;
//   in[k]   = id_k                          if delay_k == 0,
//             resolved id of frame p-delay_k (ring slot (p - delay_k) & 3)
//                                           if p - delay_k >= first_pos[b],
//             the stream's initial ID       otherwise.
// If any resolved ID of any row (including one read back from the delay ring) is outside
// -1..rows-1 the frame is aborted: the status
// word records PM_DEV_ERR_INVALID_ID, the abort flag is raised for the rest of the frame,
// and no state changes.
#include "pm_kernels.h"

namespace pm {
namespace {

__global__ void __launch_bounds__(128) k_embed(const EmbedParams p) {
    __shared__ int s_in[PM_MAX_STREAMS_DEV];
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int S = p.n_streams;
    const bool seq = p.resolved != nullptr;  // prefill: rows are frames of one stream

    int bad = 0;
    const bool direct = !seq && p.io->direct != 0;  // inputs already delayed (generator step)
    if (seq) {
        bad = *(volatile uint32_t*)&p.st.status[1] != 0u;  // set by k_seq_prepare
    } else {
        // validate every row's IDs (cheap: B * 17 values) so all CTAs agree on the abort;
        // a delayed stream's input comes from the delay ring, which is checked the same way
        // (the ring only ever holds validated IDs unless a restored snapshot was corrupt)
        for (int i = tid; i < p.B * S; i += blockDim.x) {
            const int bb = i / S, k = i % S;
            int id = p.io->ids[i];
            if (id == -3) id = p.st.sel[(size_t)bb * PM_MAX_STREAMS_DEV + k];
            if (id < -1 || id >= p.rows[k]) bad = 1;
            const int src = p.st.pos[bb] - p.delays[k];
            if (!direct && p.delays[k] != 0 && src >= p.st.first_pos[bb]) {
                const int in = p.st.ring[((size_t)bb * 4 + (src & 3)) * PM_MAX_STREAMS_DEV + k];
                if (in < -1 || in >= p.rows[k]) bad = 1;
            }
        }
        bad = __syncthreads_or(bad);
    }

    if (seq) {
        if (tid < S) s_in[tid] = p.resolved[(size_t)b * S + tid];
    } else if (tid < S) {
        const int k = tid;
        int id = p.io->ids[(size_t)b * S + k];
        if (id == -3) id = p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + k];
        const int pos = p.st.pos[b];
        const int src = pos - p.delays[k];
        int in;
        if (direct || p.delays[k] == 0)
            in = id;
        else if (src >= p.st.first_pos[b])
            in = p.st.ring[((size_t)b * 4 + (src & 3)) * PM_MAX_STREAMS_DEV + k];
        else
            in = p.init_id[k];
        s_in[k] = in;
        if (!bad && !direct && blockIdx.x == 0) p.st.ring[((size_t)b * 4 + (pos & 3)) * PM_MAX_STREAMS_DEV + k] = id;
    }
    if (!seq && blockIdx.x == 0 && b == 0 && tid == 0) {
        p.st.status[1] = bad ? 1u : 0u;
        if (bad) set_status(p.st.status, PM_DEV_ERR_INVALID_ID);
    }
    if (!seq && blockIdx.x == 0 && tid == 0) {
        // the text head's argmax accumulator and completion counter start every frame
        // cleared, also after a frame whose head did not finish (a wait that ran out)
        p.st.amax[b] = 0ull;
        p.st.head_count[b] = 0u;
    }
    __syncthreads();
    if (bad) return;
    if (blockIdx.x == 0 && tid < p.dh / 2) {
        // RoPE angles of this frame: position (integer) times frequency, in double
        const int pos = seq ? p.st.pos[p.io->seq_stream] + b : p.st.pos[b];
        double sn, cs;
        sincos((double)pos * p.rope_freq[tid], &sn, &cs);
        p.rope_tab[(size_t)b * (p.dh / 2) + tid] = make_float2((float)cs, (float)sn);
    }

    const int col = blockIdx.x * 1024 + 8 * tid;
    __shared__ float s_ss[4];
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int k = 0; k < S && col < p.D; ++k) {
        const int id = s_in[k];
        if (id < 0) continue;  // -1: exact zero contribution
        const uint4 w = *reinterpret_cast<const uint4*>(p.tables[k] + (size_t)id * p.D + col);
        acc[0] += bf16lo(w.x); acc[1] += bf16hi(w.x);
        acc[2] += bf16lo(w.y); acc[3] += bf16hi(w.y);
        acc[4] += bf16lo(w.z); acc[5] += bf16hi(w.z);
        acc[6] += bf16lo(w.w); acc[7] += bf16hi(w.w);
    }
    if (col < p.D) {
        float4* dst = reinterpret_cast<float4*>(p.x + (size_t)b * p.D + col);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    if (p.xb) {
        // tensor-core operand bf16(alpha * x) and this CTA's share of sum(x^2)
        float ss = 0.f;
        if (col < p.D) {
            const uint4 av = *reinterpret_cast<const uint4*>(p.alpha + col);
            const float al[8] = {bf16lo(av.x), bf16hi(av.x), bf16lo(av.y), bf16hi(av.y),
                                 bf16lo(av.z), bf16hi(av.z), bf16lo(av.w), bf16hi(av.w)};
            uint32_t w[4], wl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v0 = acc[2 * e] * al[2 * e], v1 = acc[2 * e + 1] * al[2 * e + 1];
                const uint16_t h0 = f32_to_bf16_rne(v0), h1 = f32_to_bf16_rne(v1);
                w[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                wl[e] = (uint32_t)bf16_lo_part(v0, h0) | ((uint32_t)bf16_lo_part(v1, h1) << 16);
                ss = fmaf(acc[2 * e], acc[2 * e], ss);
                ss = fmaf(acc[2 * e + 1], acc[2 * e + 1], ss);
            }
            *reinterpret_cast<uint4*>(p.xb + (size_t)b * p.D + col) = make_uint4(w[0], w[1], w[2], w[3]);
            if (p.xb_lo_rows)
                *reinterpret_cast<uint4*>(p.xb + ((size_t)b + p.xb_lo_rows) * p.D + col) =
                    make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) s_ss[tid >> 5] = ss;
        __syncthreads();
        if (tid == 0) p.ss[(size_t)blockIdx.x * p.npad + b] = s_ss[0] + s_ss[1] + s_ss[2] + s_ss[3];
    }
}

}  // namespace

cudaError_t launch_embed(const EmbedParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.D + 1023) / 1024), (unsigned)p.B);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_embed, p);
}

}  // namespace pm
