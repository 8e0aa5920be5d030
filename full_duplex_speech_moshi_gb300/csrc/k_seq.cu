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
// by k_seq_commit: the last row of each slot).  Work item = (head, 256-key chunk): the
// chunk's keys stream through a ring of three 64-key stages in shared memory (K and V as
// rows, filled by cp.async while the previous stage is in use), and every warp -- 16 query
// rows -- computes its scores and weighted values with warp-wide m16n8k16 tensor-core MMAs
// (bf16 operands from ldmatrix, V through its transposing form; fp32 accumulation),
// keeping the running (max, sum, weighted values) of its rows in registers.  A head whose
// keys fit one chunk writes its output directly; otherwise every chunk leaves a partial
// and k_seq_commit, one CTA per row, merges the row's partials of all heads.
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

// shared-memory stage ring of k_attn_seq: K rows then V rows of 64 keys, 272 B per row
// (16-byte aligned rows for cp.async and ldmatrix; 8 rows of a fragment land in 8
// distinct 4-bank groups)
constexpr int NSTAGE = 3;
constexpr int KROW = DH + 8;                               // bf16 per staged row
constexpr uint32_t HALF_BYTES = KSUB * KROW * 2;           // K (or V) of one stage
constexpr uint32_t STAGE_BYTES = 2 * HALF_BYTES;
constexpr size_t SEQ_SMEM = (size_t)NSTAGE * STAGE_BYTES;  // 104,448 B: two CTAs per SM

// 16-byte global -> shared copy; when !valid the destination is zero-filled and nothing is read
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// four 8x8 b16 matrices; lanes 8q .. 8q+7 give the row addresses of matrix q
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// the pass's key range and its chunking (k_attn_seq and k_seq_commit agree on it)
struct SeqChunks {
    int lo, hi, C;
};
__device__ __forceinline__ SeqChunks seq_chunks(int p0, int T, int win) {
    SeqChunks k;
    k.lo = max(0, p0 - win + 1);
    k.hi = p0 + T - 1;
    k.C = (k.hi - k.lo + 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC;
    return k;
}

__global__ void __launch_bounds__(SEQ_NT) k_attn_seq(const AttnSeqParams p) {
    extern __shared__ __align__(128) uint8_t seq_smem[];
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int s = p.io->seq_stream;
    const int p0 = p.st.pos[s];
    const int T = p.T;
    const SeqChunks ch = seq_chunks(p0, T, p.win);
    const int C = ch.C;
    const int items = p.H * C;
    // this thread's two query rows (the warp owns rows 16 * warp .. 16 * warp + 15)
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const uint32_t sbase = smem_u32(seq_smem);
    // ldmatrix row of this lane: matrix q = lane / 8, row lane % 8
    const int lq = lane >> 3, lr = lane & 7;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int h = item / C, c = item % C;
        const int c0 = ch.lo + c * PM_SEQ_KPC;
        const int c1 = min(c0 + PM_SEQ_KPC, ch.hi + 1);
        const int nsub = (c1 - c0 + KSUB - 1) / KSUB;
        const size_t head_base = ((size_t)s * p.H + h) * (size_t)p.ctx * DH;
        // K and V of keys k0 .. k0+63 into stage `buf`; keys past the chunk are zeros
        auto stage = [&](int sub, int buf) {
            const int k0 = c0 + sub * KSUB;
            const uint32_t sk = sbase + (uint32_t)buf * STAGE_BYTES;
            for (int i = tid; i < KSUB * (DH / 8); i += SEQ_NT) {
                const int j = i >> 4, d0 = (i & 15) * 8;
                const int kp = k0 + j;
                const bool ok = kp < c1;
                const uint16_t* ks = p.kv_new;
                const uint16_t* vs = p.kv_new;
                if (ok) {
                    if (kp >= p0) {
                        const size_t off = ((size_t)(kp - p0) * p.H + h) * DH + d0;
                        ks = p.kv_new + off;
                        vs = p.kv_new + (size_t)T * p.H * DH + off;
                    } else {
                        const size_t off = head_base + (size_t)(kp % p.ctx) * DH + d0;
                        ks = p.kc + off;
                        vs = p.vc + off;
                    }
                }
                const uint32_t o = (uint32_t)(j * KROW + d0) * 2u;
                cp_async16(sk + o, ks, ok);
                cp_async16(sk + HALF_BYTES + o, vs, ok);
            }
        };
#pragma unroll
        for (int i = 0; i < NSTAGE - 1; ++i) {
            if (i < nsub) stage(i, i);
            cp_async_commit();
        }
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
        for (int sub = 0; sub < nsub; ++sub) {
            cp_async_wait<NSTAGE - 2>();  // this thread's copies of stage `sub` landed
            __syncthreads();              // everyone's did, and stage sub-1 is no longer read
            if (sub + NSTAGE - 1 < nsub) stage(sub + NSTAGE - 1, (sub + NSTAGE - 1) % NSTAGE);
            cp_async_commit();
            const uint32_t sk = sbase + (uint32_t)(sub % NSTAGE) * STAGE_BYTES;
            const uint32_t sv = sk + HALF_BYTES;
            const int k0 = c0 + sub * KSUB;
            // S = Q K^T for the warp's 16 rows and the 64 staged keys (8 tiles of 8 keys);
            // matrices q = 0..3 of one ldmatrix: dims 16 ks + 8 q .. +7 of keys 8 j .. 8 j + 7
            float sc[KSUB / 8][4];
#pragma unroll
            for (int j = 0; j < KSUB / 8; ++j) {
                sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                const uint32_t kr = sk + (uint32_t)((8 * j + lr) * KROW + 8 * lq) * 2u;
#pragma unroll
                for (int ks = 0; ks < DH / 16; ks += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kr + 32u * ks, b0, b1, b2, b3);
                    mma16816(sc[j], qf[ks], b0, b1);
                    mma16816(sc[j], qf[ks + 1], b2, b3);
                }
            }
            // mask (window, causality, pass rows, chunk end) and the running softmax of both rows
            const int qp0 = p0 + r0, qp1 = p0 + r1;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < KSUB / 8; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kp = k0 + 8 * j + 2 * tq + e;
                    const bool in = kp < c1;
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
            // O += P V: transposed 8x8 loads of V give the B fragments; matrices q = 0..3 are
            // keys 16 kk + 8 (q & 1) .. +7 of dims 8 d + 8 (q >> 1) .. +7 (tiles d, d + 1)
#pragma unroll
            for (int kk = 0; kk < KSUB / 16; ++kk) {
                const uint32_t vr = sv + (uint32_t)((16 * kk + 8 * (lq & 1) + lr) * KROW + 8 * (lq >> 1)) * 2u;
#pragma unroll
                for (int d = 0; d < DH / 8; d += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vr + 16u * d, b0, b1, b2, b3);
                    mma16816(o[d], pf[kk], b0, b1);
                    mma16816(o[d + 1], pf[kk], b2, b3);
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // the stages are free for the next item
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = hr ? r1 : r0;
            if (r >= T) continue;
            if (C == 1) {
                // the whole window in one chunk: the normalised output
                const float inv = 1.0f / (hr ? l_1 : l_0);
                float* ob = p.o + (size_t)r * p.D + h * DH;
#pragma unroll
                for (int d = 0; d < DH / 8; ++d) {
                    const float a = o[d][2 * hr] * inv, b = o[d][2 * hr + 1] * inv;
                    *reinterpret_cast<float2*>(ob + 8 * d + 2 * tq) = make_float2(a, b);
                    if (p.ob)
                        *reinterpret_cast<uint32_t*>(p.ob + (size_t)r * p.D + h * DH + 8 * d + 2 * tq) = pack_bf16(a, b);
                }
            } else {
                // this chunk's partial of the row: unnormalised values, max, sum
                float* part = p.part + (((size_t)r * p.H + h) * PM_SEQ_MAX_CHUNKS + c) * PSTRIDE;
#pragma unroll
                for (int d = 0; d < DH / 8; ++d)
                    *reinterpret_cast<float2*>(part + 8 * d + 2 * tq) = make_float2(o[d][2 * hr], o[d][2 * hr + 1]);
                if (tq == 0) {
                    part[DH] = hr ? m_1 : m_0;
                    part[DH + 1] = hr ? l_1 : l_0;
                }
            }
        }
    }
}

}  // namespace

// CTA (t, j) handles row t for heads 8j .. 8j+7: (1) when the window took several chunks,
// merges the row's chunk partials of those heads, out = sum_c exp2(m_c - M) o_c / L with
// M = max_c m_c and L = sum_c exp2(m_c - M) l_c (chunks in order); (2) copies the row's K
// and V of those heads into the ring slot (p0 + t) mod ctx unless a later row of the pass
// owns the same slot.
constexpr int CM_HEADS = 8;  // heads per k_seq_commit CTA: 16 threads per head, 8 coordinates each

__global__ void __launch_bounds__(128) k_seq_commit(const AttnSeqParams p) {
    __shared__ float s_w[CM_HEADS * PM_SEQ_MAX_CHUNKS];
    __shared__ float s_m[CM_HEADS * PM_SEQ_MAX_CHUNKS];
    pdl_trigger();
    pdl_wait();
    if (*(volatile uint32_t*)&p.st.status[1] != 0u) return;
    const int t = blockIdx.x, h0 = blockIdx.y * CM_HEADS;
    const int nh = min(CM_HEADS, p.H - h0);
    const int tid = threadIdx.x;
    const int s = p.io->seq_stream;
    const int p0 = p.st.pos[s];
    const int C = seq_chunks(p0, p.T, p.win).C;
    if (C > 1) {
        const float* pr = p.part + ((size_t)t * p.H + h0) * PM_SEQ_MAX_CHUNKS * PSTRIDE;
        for (int i = tid; i < nh * C; i += blockDim.x) {
            const int hh = i / C, c = i % C;
            const float* pc = pr + ((size_t)hh * PM_SEQ_MAX_CHUNKS + c) * PSTRIDE;
            s_m[hh * PM_SEQ_MAX_CHUNKS + c] = __ldcg(pc + DH);
            s_w[hh * PM_SEQ_MAX_CHUNKS + c] = __ldcg(pc + DH + 1);
        }
        __syncthreads();
        if (tid < nh) {
            float* m = s_m + tid * PM_SEQ_MAX_CHUNKS;
            float* w = s_w + tid * PM_SEQ_MAX_CHUNKS;
            float M = -INFINITY;
            for (int c = 0; c < C; ++c) M = fmaxf(M, m[c]);
            float L = 0.f;
            for (int c = 0; c < C; ++c) {
                const float f = (m[c] == -INFINITY) ? 0.f : exp2f(m[c] - M);
                m[c] = f;
                L += w[c] * f;
            }
            const float inv = 1.0f / L;
            for (int c = 0; c < C; ++c) w[c] = m[c] * inv;
        }
        __syncthreads();
        const int hh = tid >> 4, d0 = (tid & 15) * 8;
        if (hh < nh) {
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            const float* ph = pr + (size_t)hh * PM_SEQ_MAX_CHUNKS * PSTRIDE + d0;
            // eight chunks' loads in flight, then their weighted sums in chunk order
            for (int c0 = 0; c0 < C; c0 += 8) {
                float4 a[8][2];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const bool in = c0 + j < C;
                    const float4* pc = reinterpret_cast<const float4*>(ph + (size_t)(c0 + j) * PSTRIDE);
                    a[j][0] = in ? __ldcg(pc) : make_float4(0.f, 0.f, 0.f, 0.f);
                    a[j][1] = in ? __ldcg(pc + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (c0 + j >= C) break;
                    const float wt = s_w[hh * PM_SEQ_MAX_CHUNKS + c0 + j];
                    acc[0] += a[j][0].x * wt;
                    acc[1] += a[j][0].y * wt;
                    acc[2] += a[j][0].z * wt;
                    acc[3] += a[j][0].w * wt;
                    acc[4] += a[j][1].x * wt;
                    acc[5] += a[j][1].y * wt;
                    acc[6] += a[j][1].z * wt;
                    acc[7] += a[j][1].w * wt;
                }
            }
            const size_t ob = (size_t)t * p.D + (size_t)(h0 + hh) * DH + d0;
            reinterpret_cast<float4*>(p.o + ob)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            reinterpret_cast<float4*>(p.o + ob)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (p.ob)
                *reinterpret_cast<uint4*>(p.ob + ob) = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                                                                  pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
        }
    }
    if (t + p.ctx < p.T) return;
    const int slot = (p0 + t) % p.ctx;
    const int n16 = nh * DH / 8;  // 16-byte pieces of the CTA's heads in one row
    for (int i = tid; i < 2 * n16; i += blockDim.x) {
        const int kv = i / n16, j = i % n16;
        const int h = h0 + (j * 8) / DH, d = (j * 8) % DH;
        const uint4 v = *reinterpret_cast<const uint4*>(p.kv_new + (((size_t)kv * p.T + t) * p.H + h) * DH + d);
        uint16_t* dst = const_cast<uint16_t*>(kv ? p.vc : p.kc) + (((size_t)s * p.H + h) * p.ctx + slot) * DH + d;
        *reinterpret_cast<uint4*>(dst) = v;
    }
}

cudaError_t launch_seq_commit(const AttnSeqParams& p, cudaStream_t s, bool pdl) {
    if (p.H < 1 || p.T < 1 || p.T > PM_SEQ_MAX_ROWS) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.T, (unsigned)((p.H + CM_HEADS - 1) / CM_HEADS));
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

cudaError_t attn_seq_prepare() {
    return cudaFuncSetAttribute(k_attn_seq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SEQ_SMEM);
}

int attn_seq_max_chunks(int win) { return (win + PM_SEQ_MAX_ROWS - 1 + PM_SEQ_KPC - 1) / PM_SEQ_KPC; }

cudaError_t launch_attn_seq(const AttnSeqParams& p, cudaStream_t s, bool pdl) {
    if (p.T < 1 || p.T > PM_SEQ_MAX_ROWS || attn_seq_max_chunks(p.win) > PM_SEQ_MAX_CHUNKS || p.win < 1 ||
        p.win > p.ctx)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(SEQ_NT);
    cfg.dynamicSmemBytes = SEQ_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_attn_seq, p);
}

}  // namespace pm
