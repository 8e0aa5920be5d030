// Prefill: T consecutive frames of one stream as the rows of one batched pass
// ("PersonaPlex native LM audit", section 9: the startup voice prompt, silence frames and
// text prompt each advance one model step with provided codes; section 7: delays).
// Every result is that of T sequential frames; the projections run as T-row tensor-core
// GEMMs (k_gemm_tc with `seq`), and these two kernels supply the sequential parts:
//
// k_seq_prepare (one CTA): validates the T x n_streams IDs, resolves each frame's delayed
// inputs (frame t of stream k reads the ID given at frame t - delay_k: from this chunk,
// from the delay ring for frames before it, or the stream's initial ID before its first
// frame), then writes the last frames' IDs into the ring.  One thread per stream walks
// the frames in order, so every ring read precedes the write of the same slot.
//
// k_attn_seq: causal windowed attention of T query rows (frames p0 .. p0+T-1) over the
// keys they can see (positions max(0, p0 - win + 1) .. p0 + T - 1): positions before p0
// from the ring, the pass's own from the kv_new rows its QKV projection wrote (a full
// ring's slots are reused by the pass's positions, so they are committed only afterwards
// by k_seq_commit: the last row of each slot).  Work item = (head,
// 256-key chunk): the chunk's K and V rows are staged once in shared memory (64 keys at a
// time) and used by every row; per row a running (max, sum, weighted values) is kept in
// registers; chunks merge in the CTA that finishes a head last (completion counter).
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;
constexpr int KSUB = 64;                   // keys staged at a time
constexpr int SEQ_NT = 256;                // threads of k_attn_seq (8 warps)
constexpr int ROWS_PER_WARP = PM_SEQ_MAX_ROWS / (SEQ_NT / 32);
constexpr int PSTRIDE = PM_SEQ_PART_STRIDE;  // floats per partial: DH values, max, sum (16-byte rows)

__global__ void __launch_bounds__(32) k_seq_prepare(const SeqPrepParams p) {
    pdl_trigger();
    pdl_wait();
    const int k = threadIdx.x;
    const int S = p.n_streams;
    const int s = p.io->seq_stream;
    const int pos0 = p.st.pos[s], first = p.st.first_pos[s];
    int bad = 0;
    if (k < S) {
        for (int t = 0; t < p.T; ++t) {
            const int id = p.io->ids[(size_t)t * S + k];
            if (id < -1 || id >= p.rows[k]) bad = 1;  // no feedback ID in a prefill
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (k < S) {
        const int d = p.delays[k];
        for (int t = 0; t < p.T; ++t) {
            const int src = pos0 + t - d;
            int in;
            if (d == 0)
                in = p.io->ids[(size_t)t * S + k];
            else if (src < first)
                in = p.init_id[k];
            else if (src >= pos0)
                in = p.io->ids[(size_t)(src - pos0) * S + k];
            else
                in = p.st.ring[((size_t)s * 4 + (src & 3)) * PM_MAX_STREAMS_DEV + k];
            p.resolved[(size_t)t * S + k] = in;
        }
        if (!bad)
            for (int t = p.T > 4 ? p.T - 4 : 0; t < p.T; ++t)
                p.st.ring[((size_t)s * 4 + ((pos0 + t) & 3)) * PM_MAX_STREAMS_DEV + k] = p.io->ids[(size_t)t * S + k];
    }
    if (k == 0) {
        p.st.status[1] = bad ? 1u : 0u;
        if (bad) set_status(p.st.status, PM_DEV_ERR_INVALID_ID);
    }
}

__global__ void __launch_bounds__(SEQ_NT) k_attn_seq(const AttnSeqParams p) {
    extern __shared__ float sm[];
    float* s_q = sm;                                   // [T][DH]
    float* s_kt = s_q + (size_t)PM_SEQ_MAX_ROWS * DH;   // [DH][KSUB + 1] keys, transposed
    float* s_v = s_kt + (size_t)DH * (KSUB + 1);        // [KSUB][DH]
    __shared__ int s_last;
    __shared__ float s_pm[SEQ_NT / 32][PM_SEQ_MAX_CHUNKS], s_pl[SEQ_NT / 32][PM_SEQ_MAX_CHUNKS];
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = p.io->seq_stream;
    const int p0 = p.st.pos[s];
    const int T = p.T;
    const int lo_all = max(0, p0 - p.win + 1), hi_all = p0 + T - 1;
    const int C = (hi_all - lo_all + 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC;
    const int items = p.H * C;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int h = item / C, c = item % C;
        const int c0 = lo_all + c * PM_SEQ_KPC;
        const int c1 = min(c0 + PM_SEQ_KPC, hi_all + 1);
        for (int i = tid; i < T * DH; i += SEQ_NT)
            s_q[i] = p.q[(size_t)(i / DH) * p.D + h * DH + (i % DH)] * p.scale_log2;
        float m[ROWS_PER_WARP], l[ROWS_PER_WARP], acc[ROWS_PER_WARP][4];
#pragma unroll
        for (int r = 0; r < ROWS_PER_WARP; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
        }
        const size_t head_base = ((size_t)s * p.H + h) * (size_t)p.ctx * DH;
        for (int k0 = c0; k0 < c1; k0 += KSUB) {
            const int nk = min(KSUB, c1 - k0);
            __syncthreads();  // previous sub-chunk (and q) fully used / written
            // stage K (transposed) and V of keys k0 .. k0+nk-1 as fp32
            for (int i = tid; i < KSUB * (DH / 8); i += SEQ_NT) {
                const int j = i / (DH / 8), d0 = (i % (DH / 8)) * 8;
                float kv[8], vv[8];
                if (j < nk) {
                    const int kp = k0 + j;
                    const uint16_t *ksrc, *vsrc;
                    if (kp >= p0) {
                        const size_t off = ((size_t)(kp - p0) * p.H + h) * DH + d0;
                        ksrc = p.kv_new + off;
                        vsrc = p.kv_new + (size_t)T * p.H * DH + off;
                    } else {
                        const size_t off = head_base + (size_t)(kp % p.ctx) * DH + d0;
                        ksrc = p.kc + off;
                        vsrc = p.vc + off;
                    }
                    const uint4 a = *reinterpret_cast<const uint4*>(ksrc);
                    const uint4 bv = *reinterpret_cast<const uint4*>(vsrc);
                    kv[0] = bf16lo(a.x); kv[1] = bf16hi(a.x); kv[2] = bf16lo(a.y); kv[3] = bf16hi(a.y);
                    kv[4] = bf16lo(a.z); kv[5] = bf16hi(a.z); kv[6] = bf16lo(a.w); kv[7] = bf16hi(a.w);
                    vv[0] = bf16lo(bv.x); vv[1] = bf16hi(bv.x); vv[2] = bf16lo(bv.y); vv[3] = bf16hi(bv.y);
                    vv[4] = bf16lo(bv.z); vv[5] = bf16hi(bv.z); vv[6] = bf16lo(bv.w); vv[7] = bf16hi(bv.w);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kv[e] = vv[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    s_kt[(size_t)(d0 + e) * (KSUB + 1) + j] = kv[e];
                    s_v[(size_t)j * DH + d0 + e] = vv[e];
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < ROWS_PER_WARP; ++r) {
                const int t = warp + r * (SEQ_NT / 32);
                if (t >= T) break;
                const int qpos = p0 + t, klo = qpos - p.win + 1;
                // scores of keys lane and lane + 32 (base-2 scaled)
                const float* qr = s_q + (size_t)t * DH;
                float d0 = 0.f, d1 = 0.f;
#pragma unroll 16
                for (int d = 0; d < DH; ++d) {
                    const float qv = qr[d];
                    d0 = fmaf(qv, s_kt[(size_t)d * (KSUB + 1) + lane], d0);
                    d1 = fmaf(qv, s_kt[(size_t)d * (KSUB + 1) + lane + 32], d1);
                }
                const int kp0 = k0 + lane, kp1 = k0 + lane + 32;
                const bool v0 = lane < nk && kp0 >= klo && kp0 <= qpos;
                const bool v1 = lane + 32 < nk && kp1 >= klo && kp1 <= qpos;
                float sc0 = v0 ? d0 : -INFINITY, sc1 = v1 ? d1 : -INFINITY;
                float mx = fmaxf(sc0, sc1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (mx == -INFINITY) continue;  // no visible key in this sub-chunk
                const float mn = fmaxf(m[r], mx);
                const float fo = (m[r] == -INFINITY) ? 0.f : exp2f(m[r] - mn);
                const float w0 = v0 ? exp2f(sc0 - mn) : 0.f, w1 = v1 ? exp2f(sc1 - mn) : 0.f;
                float ws = w0 + w1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
                l[r] = l[r] * fo + ws;
                m[r] = mn;
                float a[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) a[e] = acc[r][e] * fo;
                // weighted values: lane owns coordinates 4*lane .. 4*lane+3
                for (int j = 0; j < nk; ++j) {
                    const float w = __shfl_sync(0xffffffffu, j < 32 ? w0 : w1, j & 31);
                    const float4 vv = *reinterpret_cast<const float4*>(s_v + (size_t)j * DH + 4 * lane);
                    a[0] = fmaf(w, vv.x, a[0]);
                    a[1] = fmaf(w, vv.y, a[1]);
                    a[2] = fmaf(w, vv.z, a[2]);
                    a[3] = fmaf(w, vv.w, a[3]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[r][e] = a[e];
            }
        }
        // this chunk's partial of every row
#pragma unroll
        for (int r = 0; r < ROWS_PER_WARP; ++r) {
            const int t = warp + r * (SEQ_NT / 32);
            if (t >= T) break;
            float* part = p.part + (((size_t)t * p.H + h) * PM_SEQ_MAX_CHUNKS + c) * PSTRIDE;
            *reinterpret_cast<float4*>(part + 4 * lane) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            if (lane == 0) {
                part[DH] = m[r];
                part[DH + 1] = l[r];
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const uint32_t done = atomicAdd(&p.count[h], 1u);
            s_last = (done == (uint32_t)C - 1u) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) continue;
        // last chunk of head h: merge every row's chunks in chunk order
        __threadfence();
        for (int t = warp; t < T; t += SEQ_NT / 32) {
            const float* pb = p.part + ((size_t)t * p.H + h) * PM_SEQ_MAX_CHUNKS * PSTRIDE;
            float* wm = s_pm[warp];
            float* wl = s_pl[warp];
            for (int i = lane; i < C; i += 32) {
                wm[i] = __ldcg(pb + (size_t)i * PSTRIDE + DH);
                wl[i] = __ldcg(pb + (size_t)i * PSTRIDE + DH + 1);
            }
            __syncwarp();
            float M = -INFINITY;
            for (int i = 0; i < C; ++i) M = fmaxf(M, wm[i]);
            float L = 0.f, A[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < C; ++i) {
                const float f = (wm[i] == -INFINITY) ? 0.f : exp2f(wm[i] - M);
                L += wl[i] * f;
                const float4 a = __ldcg(reinterpret_cast<const float4*>(pb + (size_t)i * PSTRIDE + 4 * lane));
                A[0] += a.x * f;
                A[1] += a.y * f;
                A[2] += a.z * f;
                A[3] += a.w * f;
            }
            __syncwarp();
            float* ob = p.o + (size_t)t * p.D + h * DH + 4 * lane;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = A[e] / L;
                ob[e] = v;
                if (p.ob) p.ob[(size_t)t * p.D + h * DH + 4 * lane + e] = f32_to_bf16_rne(v);
            }
        }
        if (tid == 0) p.count[h] = 0u;
        __syncthreads();
    }
}

}  // namespace

// CTA t copies row t's K and V (all heads) into the ring slot (p0 + t) mod ctx unless a
// later row of the pass owns the same slot
__global__ void __launch_bounds__(128) k_seq_commit(const AttnSeqParams p) {
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    const int t = blockIdx.x;
    if (t + p.ctx < p.T) return;
    const int s = p.io->seq_stream;
    const int slot = (p.st.pos[s] + t) % p.ctx;
    const int n16 = p.H * DH / 8;  // 16-byte pieces per row
    for (int i = threadIdx.x; i < 2 * n16; i += blockDim.x) {
        const int kv = i / n16, j = i % n16;
        const int h = (j * 8) / DH, d = (j * 8) % DH;
        const uint4 v = *reinterpret_cast<const uint4*>(p.kv_new + (((size_t)kv * p.T + t) * p.H + h) * DH + d);
        uint16_t* dst = const_cast<uint16_t*>(kv ? p.vc : p.kc) + (((size_t)s * p.H + h) * p.ctx + slot) * DH + d;
        *reinterpret_cast<uint4*>(dst) = v;
    }
}

cudaError_t launch_seq_commit(const AttnSeqParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.T);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_seq_commit, p);
}

cudaError_t launch_seq_prepare(const SeqPrepParams& p, cudaStream_t s, bool pdl) {
    if (p.n_streams > 32 || p.T < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_seq_prepare, p);
}

size_t attn_seq_smem() { return sizeof(float) * ((size_t)PM_SEQ_MAX_ROWS * DH + (size_t)DH * (KSUB + 1) + (size_t)KSUB * DH); }

cudaError_t attn_seq_prepare() {
    return cudaFuncSetAttribute(k_attn_seq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_seq_smem());
}

int attn_seq_max_chunks(int win) { return (win + PM_SEQ_MAX_ROWS - 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC; }

cudaError_t launch_attn_seq(const AttnSeqParams& p, cudaStream_t s, bool pdl) {
    if (p.T < 1 || p.T > PM_SEQ_MAX_ROWS || attn_seq_max_chunks(p.win) > PM_SEQ_MAX_CHUNKS || p.win < 1 ||
        p.win > p.ctx)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(SEQ_NT);
    cfg.dynamicSmemBytes = attn_seq_smem();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attn_seq, p);
}

}  // namespace pm
