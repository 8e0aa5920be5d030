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
// by k_seq_commit: the last row of each slot).  Work item = (head, 256-key chunk): 64 keys
// at a time are staged in shared memory (K as rows, V transposed) and every warp -- 16
// query rows -- computes its scores and weighted values with warp-wide m16n8k16 tensor
// core MMAs (bf16 operands, fp32 accumulation), keeping the running (max, sum, weighted
// values) of its rows in registers; chunks merge in the CTA that finishes a head last
// (completion counter).
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;
constexpr int KSUB = 64;                   // keys staged at a time
constexpr int SEQ_NT = 128;                // threads of k_attn_seq: 4 warps x 16 query rows
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
            if (in < -1 || in >= p.rows[k]) {  // a ring entry from a corrupt restored snapshot
                bad = 1;
                in = -1;
            }
            p.resolved[(size_t)t * S + k] = in;
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (k < S) {
        if (!bad)
            for (int t = p.T > 4 ? p.T - 4 : 0; t < p.T; ++t)
                p.st.ring[((size_t)s * 4 + ((pos0 + t) & 3)) * PM_MAX_STREAMS_DEV + k] = p.io->ids[(size_t)t * S + k];
    }
    if (k == 0) {
        p.st.status[1] = bad ? 1u : 0u;
        if (bad) set_status(p.st.status, PM_DEV_ERR_INVALID_ID);
    }
}

// D += A * B on the tensor cores, warp-wide m16n8k16 (bf16 in, fp32 accumulate).
// Fragments (g = lane / 4, t = lane % 4): a[0] = A[g][2t..2t+1], a[1] = A[g+8][2t..],
// a[2] = A[g][2t+8..], a[3] = A[g+8][2t+8..]; b[0] = B[2t..2t+1][g], b[1] = B[2t+8..][g];
// d[0..1] = D[g][2t..2t+1], d[2..3] = D[g+8][2t..2t+1].
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)f32_to_bf16_rne(lo) | ((uint32_t)f32_to_bf16_rne(hi) << 16);
}

constexpr int KS_STRIDE = DH + 8;    // bf16 per staged key row (conflict-free fragment loads)
constexpr int VT_STRIDE = KSUB + 8;  // bf16 per staged value column

__global__ void __launch_bounds__(SEQ_NT) k_attn_seq(const AttnSeqParams p) {
    __shared__ __align__(16) uint16_t s_k[KSUB * KS_STRIDE];  // [key][dim]
    __shared__ __align__(16) uint16_t s_vt[DH * VT_STRIDE];   // [dim][key]
    __shared__ int s_last;
    __shared__ float s_pm[SEQ_NT / 32][PM_SEQ_MAX_CHUNKS], s_pl[SEQ_NT / 32][PM_SEQ_MAX_CHUNKS];
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int s = p.io->seq_stream;
    const int p0 = p.st.pos[s];
    const int T = p.T;
    const int lo_all = max(0, p0 - p.win + 1), hi_all = p0 + T - 1;
    const int C = (hi_all - lo_all + 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC;
    const int items = p.H * C;
    // this thread's two query rows (the warp owns rows 16 * warp .. 16 * warp + 15)
    const int r0 = 16 * warp + g, r1 = r0 + 8;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int h = item / C, c = item % C;
        const int c0 = lo_all + c * PM_SEQ_KPC;
        const int c1 = min(c0 + PM_SEQ_KPC, hi_all + 1);
        // query fragments, pre-scaled by log2(e) / sqrt(dh), bf16
        uint32_t qf[DH / 16][4];
        {
            const float* q0 = p.q + (size_t)r0 * p.D + h * DH;
            const float* q1 = p.q + (size_t)r1 * p.D + h * DH;
            const bool v0 = r0 < T, v1 = r1 < T;
#pragma unroll
            for (int ks = 0; ks < DH / 16; ++ks) {
                const int d = 16 * ks + 2 * tq;
                const float2 a = v0 ? *reinterpret_cast<const float2*>(q0 + d) : make_float2(0.f, 0.f);
                const float2 b = v1 ? *reinterpret_cast<const float2*>(q1 + d) : make_float2(0.f, 0.f);
                const float2 a8 = v0 ? *reinterpret_cast<const float2*>(q0 + d + 8) : make_float2(0.f, 0.f);
                const float2 b8 = v1 ? *reinterpret_cast<const float2*>(q1 + d + 8) : make_float2(0.f, 0.f);
                qf[ks][0] = pack_bf16(a.x * p.scale_log2, a.y * p.scale_log2);
                qf[ks][1] = pack_bf16(b.x * p.scale_log2, b.y * p.scale_log2);
                qf[ks][2] = pack_bf16(a8.x * p.scale_log2, a8.y * p.scale_log2);
                qf[ks][3] = pack_bf16(b8.x * p.scale_log2, b8.y * p.scale_log2);
            }
        }
        float o[DH / 8][4];
#pragma unroll
        for (int d = 0; d < DH / 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
        float m_0 = -INFINITY, m_1 = -INFINITY, l_0 = 0.f, l_1 = 0.f;
        const size_t head_base = ((size_t)s * p.H + h) * (size_t)p.ctx * DH;
        for (int k0 = c0; k0 < c1; k0 += KSUB) {
            const int nk = min(KSUB, c1 - k0);
            __syncthreads();  // the previous sub-chunk's K / V fully used
            for (int i = tid; i < KSUB * (DH / 8); i += SEQ_NT) {
                const int j = i / (DH / 8), d0 = (i % (DH / 8)) * 8;
                uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
                if (j < nk) {
                    const int kp = k0 + j;
                    if (kp >= p0) {
                        const size_t off = ((size_t)(kp - p0) * p.H + h) * DH + d0;
                        kv = *reinterpret_cast<const uint4*>(p.kv_new + off);
                        vv = *reinterpret_cast<const uint4*>(p.kv_new + (size_t)T * p.H * DH + off);
                    } else {
                        const size_t off = head_base + (size_t)(kp % p.ctx) * DH + d0;
                        kv = *reinterpret_cast<const uint4*>(p.kc + off);
                        vv = *reinterpret_cast<const uint4*>(p.vc + off);
                    }
                }
                *reinterpret_cast<uint4*>(s_k + (size_t)j * KS_STRIDE + d0) = kv;
                const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s_vt[(size_t)(d0 + 2 * e) * VT_STRIDE + j] = (uint16_t)(vw[e] & 0xFFFFu);
                    s_vt[(size_t)(d0 + 2 * e + 1) * VT_STRIDE + j] = (uint16_t)(vw[e] >> 16);
                }
            }
            __syncthreads();
            // S = Q K^T for the warp's 16 rows and the 64 staged keys (8 tiles of 8 keys)
            float sc[KSUB / 8][4];
#pragma unroll
            for (int j = 0; j < KSUB / 8; ++j) {
                sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                const uint16_t* kr = s_k + (size_t)(8 * j + g) * KS_STRIDE + 2 * tq;
#pragma unroll
                for (int ks = 0; ks < DH / 16; ++ks) {
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks + 8);
                    mma16816(sc[j], qf[ks], b0, b1);
                }
            }
            // mask (window, causality, pass rows) and the running softmax of both rows
            const int qp0 = p0 + r0, qp1 = p0 + r1;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < KSUB / 8; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kp = k0 + 8 * j + 2 * tq + e;
                    const bool in = kp < k0 + nk;
                    const bool ok0 = in && r0 < T && kp <= qp0 && kp > qp0 - p.win;
                    const bool ok1 = in && r1 < T && kp <= qp1 && kp > qp1 - p.win;
                    sc[j][e] = ok0 ? sc[j][e] : -INFINITY;
                    sc[j][2 + e] = ok1 ? sc[j][2 + e] : -INFINITY;
                    mx0 = fmaxf(mx0, sc[j][e]);
                    mx1 = fmaxf(mx1, sc[j][2 + e]);
                }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_0, mx0), mn1 = fmaxf(m_1, mx1);
            const float f0 = (m_0 == -INFINITY) ? 0.f : exp2f(m_0 - mn0);
            const float f1 = (m_1 == -INFINITY) ? 0.f : exp2f(m_1 - mn1);
            float sum0 = 0.f, sum1 = 0.f;
            uint32_t pf[KSUB / 16][4];
#pragma unroll
            for (int j = 0; j < KSUB / 8; ++j) {
                const float e0 = sc[j][0] == -INFINITY ? 0.f : exp2f(sc[j][0] - mn0);
                const float e1 = sc[j][1] == -INFINITY ? 0.f : exp2f(sc[j][1] - mn0);
                const float e2 = sc[j][2] == -INFINITY ? 0.f : exp2f(sc[j][2] - mn1);
                const float e3 = sc[j][3] == -INFINITY ? 0.f : exp2f(sc[j][3] - mn1);
                sum0 += e0 + e1;
                sum1 += e2 + e3;
                // P as the A operand of P V: keys 16 kk .. 16 kk + 15 are tiles 2 kk, 2 kk + 1
                const int kk = j >> 1, hi = j & 1;
                pf[kk][hi ? 2 : 0] = pack_bf16(e0, e1);
                pf[kk][hi ? 3 : 1] = pack_bf16(e2, e3);
            }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                sum0 += __shfl_xor_sync(0xffffffffu, sum0, off);
                sum1 += __shfl_xor_sync(0xffffffffu, sum1, off);
            }
            l_0 = l_0 * f0 + sum0;
            l_1 = l_1 * f1 + sum1;
            m_0 = mn0;
            m_1 = mn1;
#pragma unroll
            for (int d = 0; d < DH / 8; ++d) {
                o[d][0] *= f0;
                o[d][1] *= f0;
                o[d][2] *= f1;
                o[d][3] *= f1;
            }
            // O += P V (16 tiles of 8 output coordinates)
#pragma unroll
            for (int d = 0; d < DH / 8; ++d) {
                const uint16_t* vr = s_vt + (size_t)(8 * d + g) * VT_STRIDE + 2 * tq;
#pragma unroll
                for (int kk = 0; kk < KSUB / 16; ++kk) {
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vr + 16 * kk);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vr + 16 * kk + 8);
                    mma16816(o[d], pf[kk], b0, b1);
                }
            }
        }
        // this chunk's partial of the thread's rows
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = hr ? r1 : r0;
            if (r >= T) continue;
            float* part = p.part + (((size_t)r * p.H + h) * PM_SEQ_MAX_CHUNKS + c) * PSTRIDE;
#pragma unroll
            for (int d = 0; d < DH / 8; ++d)
                *reinterpret_cast<float2*>(part + 8 * d + 2 * tq) = make_float2(o[d][2 * hr], o[d][2 * hr + 1]);
            if (tq == 0) {
                part[DH] = hr ? m_1 : m_0;
                part[DH + 1] = hr ? l_1 : l_0;
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

cudaError_t attn_seq_prepare() { return cudaSuccess; }

int attn_seq_max_chunks(int win) { return (win + PM_SEQ_MAX_ROWS - 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC; }

cudaError_t launch_attn_seq(const AttnSeqParams& p, cudaStream_t s, bool pdl) {
    if (p.T < 1 || p.T > PM_SEQ_MAX_ROWS || attn_seq_max_chunks(p.win) > PM_SEQ_MAX_CHUNKS || p.win < 1 ||
        p.win > p.ctx)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(SEQ_NT);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attn_seq, p);
}

}  // namespace pm
