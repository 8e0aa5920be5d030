// Weight-streaming GEMV for the batch-1 decode step: y = W x with W bf16 [rows][K]
// (PyTorch [out, in]), x fp32, fp32 accumulation.  Every projection of the temporal
// block and of the depformer runs through this kernel ("PersonaPlex native LM audit",
// sections 3 and 4: fused QKV, W_O, SwiGLU linear_in / linear_out, text head, depth
// projections and heads).
//
// Design (HBM-bound: each weight byte is read once, ~1 flop per byte):
//  * One CTA per SM per batch row.  CTA c owns a contiguous, balanced range of units
//    (rows, or row pairs when the epilogue needs two rows together), so its weights are
//    one or two contiguous byte ranges.
//  * A producer thread streams the range through a ring of shared-memory stages with 1-D
//    bulk copies (cp.async.bulk, TMA engine, L2 evict-first).  It issues the first ring's
//    worth of copies before griddepcontrol.wait, so with programmatic dependent launch the
//    weights of kernel i+1 are already in flight while kernel i finishes.
//  * Consumer warps split each row's K dimension P ways; each lane keeps its fixed slice
//    of the (normalised) input vector in registers, so shared memory carries only weights.
//    Per stage a warp reduces its row slice with shuffles and leaves one partial per
//    (row, slice) in shared memory; the epilogue adds the P partials per row.
//  * Prologue: optional RMSNorm of x (fp32 arithmetic, eps inside the sqrt, learned
//    scale), computed per CTA from the full vector.  Epilogues fuse what follows the
//    projection: residual add, SwiGLU, RoPE + KV-ring append, text-head argmax, ...
#include <math.h>

#include "pm_kernels.h"

// Tiling policy (compile-time tuning constants, chosen by measurement on GB300):
//  stage bytes   - target size of one shared-memory stage (whole rows, rounded down)
//  ring bytes    - target size of the stage ring per CTA
//  CTAs per SM   - resident GEMV CTAs per SM for one kernel
//  max warps     - consumer warps per CTA (each reduces one K-slice of one row per stage)
#ifndef PM_GEMV_STAGE_BYTES
#define PM_GEMV_STAGE_BYTES 16384
#endif
#ifndef PM_GEMV_RING_BYTES
#define PM_GEMV_RING_BYTES 81920
#endif
#ifndef PM_GEMV_CTAS_PER_SM
#define PM_GEMV_CTAS_PER_SM 2
#endif
#ifndef PM_GEMV_MAX_WARPS
#define PM_GEMV_MAX_WARPS 16
#endif

namespace pm {

namespace {

__device__ __forceinline__ void consumer_bar(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int CH, int PRO, int EPI, int UNIT>
__global__ void __launch_bounds__(32 * (PM_GEMV_MAX_WARPS + 1), 1) k_gemv(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RPU = (UNIT == U_ROW) ? 1 : 2;
    constexpr bool NORM = PRO == PRO_RMSNORM || PRO == PRO_RMSNORM_EMB;
    const int W = p.warps;
    const int P = p.P;
    const int K = p.K;
    const uint32_t row_bytes = (uint32_t)K * 2u;
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.nst * p.stage_bytes);
    uint64_t* empty = full + p.nst;
    float* partial = reinterpret_cast<float*>(empty + p.nst);
    float* red = partial + (size_t)p.units_cta_max * RPU * P;  // [32] scratch
    __shared__ int s_flags[4];  // [0] timeout seen, [1] abort, [2] stages issued

    const int b = blockIdx.x % p.B;
    const int c = blockIdx.x / p.B;
    const int u0 = (int)((long long)c * p.n_units / p.grid_per_b);
    const int u1 = (int)((long long)(c + 1) * p.n_units / p.grid_per_b);
    const int nu = u1 - u0;
    const int nstages = (nu + p.upst - 1) / p.upst;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // poll budget of the ring waits (the drain after a timeout keeps the full budget)
    const uint32_t budget = wait_budget(p.st);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], (uint32_t)W);
        }
        fence_barrier_init();
        s_flags[0] = 0;
        s_flags[1] = 0;
        s_flags[2] = 0;
    }
    __syncthreads();
    pdl_trigger();

    float ep_res = 0.f;                          // E_RESIDUAL: y of the first row
    int ep_pos = 0;                              // E_QKV_ROPE: position and (cos, sin) of the first pair
    float2 ep_cs = make_float2(1.f, 0.f);
    if (warp == W) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            // a CTA's range lies in one segment (the plan makes the grid a multiple of nseg)
            const uint16_t* Wb = p.W;
            int ub = 0;
            if (p.nseg > 1) {
                const int seg = u0 / p.seg_units;
                Wb = p.Wseg[seg];
                ub = seg * p.seg_units;
            }
            int slot = 0, round = 0;  // k % nst, k / nst without a division per stage
            for (int k = 0; k < nstages; ++k) {
                if (k >= p.nst) {
                    if (!mbar_wait_n(&empty[slot], (uint32_t)(round - 1) & 1u, budget)) {
                        s_flags[0] = 1;
                        timeout_abort(p.st);
                        break;
                    }
                }
                const int ua = u0 + k * p.upst;
                const int n = min(p.upst, u1 - ua);
                uint8_t* dst = stages + (size_t)slot * p.stage_bytes;
                if (UNIT == U_PAIR_SPLIT) {
                    const uint32_t bytes = (uint32_t)n * row_bytes;
                    mbar_arrive_expect_tx(&full[slot], 2u * bytes);
                    bulk_g2s(dst, Wb + (size_t)(ua - ub) * K, bytes, &full[slot], pol);
                    bulk_g2s(dst + (size_t)p.upst * row_bytes, Wb + (size_t)(ua - ub + p.split_rows) * K, bytes,
                             &full[slot], pol);
                } else {
                    const uint32_t bytes = (uint32_t)(n * RPU) * row_bytes;
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    bulk_g2s(dst, Wb + (size_t)(ua - ub) * RPU * K, bytes, &full[slot], pol);
                }
                s_flags[2] = k + 1;
                if (++slot == p.nst) {
                    slot = 0;
                    ++round;
                }
            }
        }
    } else {
        // ------------------------------ consumers ------------------------------
        const int r = warp / P;   // stage row this warp reduces
        const int pp = warp % P;  // K slice
        const int kslice = K / P;
        // the norm scale does not depend on the previous kernel: in flight before the wait
        uint4 alv[CH];
        if (NORM) {
            const uint16_t* al = p.alpha + (size_t)pp * kslice;
#pragma unroll
            for (int ci = 0; ci < CH; ++ci) alv[ci] = *reinterpret_cast<const uint4*>(al + 8 * (lane + 32 * ci));
        }
        pdl_wait();
        const bool abort_frame = *(volatile uint32_t*)&p.st.status[1] != 0u;
        if (threadIdx.x == 0) s_flags[1] = abort_frame ? 1 : 0;
        // epilogue operands of this thread's first row, loaded with the input vector rather
        // than after the last stage
        if (EPI == E_RESIDUAL && (int)threadIdx.x < nu) ep_res = p.y[(size_t)b * p.y_stride + u0 + threadIdx.x];
        if (EPI == E_QKV_ROPE && (int)threadIdx.x < nu) {
            ep_pos = p.st.pos[b];
            const int row = 2 * (u0 + (int)threadIdx.x), sec = row / p.D;
            if (sec < 2) ep_cs = p.rope_tab[(size_t)b * (p.dh / 2) + (((row - sec * p.D) % p.dh) >> 1)];
        }
        float xr[CH * 8];
        const float* xb = p.x + (size_t)b * p.x_stride + (size_t)pp * kslice;
        if (PRO == PRO_DEPATTN) {
            // Depth self-attention of position q over positions max(0, q-ctx+1)..q of this
            // frame (no positional encoding), recomputed by every CTA from q and the depth
            // cache: warp w takes heads w, w + W, ...; lane l coordinates 2l, 2l+1 of 64.
            float* xs = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(red + 32) + 15) & ~(uintptr_t)15);
            const int lo = max(0, p.q - p.dep_ctx + 1), nk = p.q - lo + 1;
            for (int hh = warp; hh < p.H; hh += W) {
                const size_t hb = ((size_t)b * p.H + hh) * p.Q * 64 + 2 * lane;
                // all loads first (q, then every K and V row of the window), then arithmetic
                const float2 qv = __ldcg(reinterpret_cast<const float2*>(p.x + (size_t)b * p.x_stride + hh * 64 +
                                                                        2 * lane));
                uint32_t kr[16], vr[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    kr[i] = vr[i] = 0u;
                    if (i < nk) {
                        kr[i] = __ldcg(reinterpret_cast<const unsigned int*>(p.dkc + hb + (size_t)(lo + i) * 64));
                        vr[i] = __ldcg(reinterpret_cast<const unsigned int*>(p.dvc + hb + (size_t)(lo + i) * 64));
                    }
                }
                float sc[16];
                float m = -INFINITY;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    sc[i] = -INFINITY;
                    if (i < nk) {
                        const float d = warp_sum(qv.x * bf16lo(kr[i]) + qv.y * bf16hi(kr[i])) * p.dep_scale_log2;
                        sc[i] = d;
                        m = fmaxf(m, d);
                    }
                }
                float l = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (i < nk) {
                        const float e = exp2f(sc[i] - m);
                        l += e;
                        o0 = fmaf(e, bf16lo(vr[i]), o0);
                        o1 = fmaf(e, bf16hi(vr[i]), o1);
                    }
                }
                xs[hh * 64 + 2 * lane] = o0 / l;
                xs[hh * 64 + 2 * lane + 1] = o1 / l;
            }
            consumer_bar(32 * W);
            xb = xs + (size_t)pp * kslice;
        }
#pragma unroll
        for (int ci = 0; ci < CH; ++ci) {
            const float4* src = reinterpret_cast<const float4*>(xb + 8 * (lane + 32 * ci));
            float4 a = src[0], bb = src[1];
            xr[8 * ci + 0] = a.x; xr[8 * ci + 1] = a.y; xr[8 * ci + 2] = a.z; xr[8 * ci + 3] = a.w;
            xr[8 * ci + 4] = bb.x; xr[8 * ci + 5] = bb.y; xr[8 * ci + 6] = bb.z; xr[8 * ci + 7] = bb.w;
        }
        if (PRO == PRO_RMSNORM_EMB) {
            // depformer layer 0: the input projection (computed for every position at the
            // start of the call) plus the embedding of the previous position's code, or of
            // the text token at position 0 -- decided by the kernel this one waited for
            const int tok = (p.q == 0) ? p.st.dep_tok[b] : p.st.dep_codes[(size_t)b * p.Q + p.q - 1];
            const uint16_t* eb = p.emb + (size_t)tok * K + (size_t)pp * kslice;
#pragma unroll
            for (int ci = 0; ci < CH; ++ci) {
                const uint4 e = *reinterpret_cast<const uint4*>(eb + 8 * (lane + 32 * ci));
                xr[8 * ci + 0] += bf16lo(e.x); xr[8 * ci + 1] += bf16hi(e.x);
                xr[8 * ci + 2] += bf16lo(e.y); xr[8 * ci + 3] += bf16hi(e.y);
                xr[8 * ci + 4] += bf16lo(e.z); xr[8 * ci + 5] += bf16hi(e.z);
                xr[8 * ci + 6] += bf16lo(e.w); xr[8 * ci + 7] += bf16hi(e.w);
            }
            if (c == 0 && r == 0 && !abort_frame) {
                // the residual stream of the position: warps of stage row 0 cover every column once
                float* xo = p.x_out + (size_t)b * K + (size_t)pp * kslice;
#pragma unroll
                for (int ci = 0; ci < CH; ++ci) {
                    float4* d4 = reinterpret_cast<float4*>(xo + 8 * (lane + 32 * ci));
                    d4[0] = make_float4(xr[8 * ci + 0], xr[8 * ci + 1], xr[8 * ci + 2], xr[8 * ci + 3]);
                    d4[1] = make_float4(xr[8 * ci + 4], xr[8 * ci + 5], xr[8 * ci + 6], xr[8 * ci + 7]);
                }
            }
        }
        if (NORM) {
            // warps of stage row 0 cover every column exactly once
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < CH * 8; ++i) ss = fmaf(xr[i], xr[i], ss);
            ss = warp_sum(ss);
            if (r == 0 && lane == 0) red[pp] = ss;
            consumer_bar(32 * W);
            float tot = 0.f;
            for (int i = 0; i < P; ++i) tot += red[i];
            const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
            for (int ci = 0; ci < CH; ++ci) {
                const uint4 av = alv[ci];
                xr[8 * ci + 0] *= inv * bf16lo(av.x); xr[8 * ci + 1] *= inv * bf16hi(av.x);
                xr[8 * ci + 2] *= inv * bf16lo(av.y); xr[8 * ci + 3] *= inv * bf16hi(av.y);
                xr[8 * ci + 4] *= inv * bf16lo(av.z); xr[8 * ci + 5] *= inv * bf16hi(av.z);
                xr[8 * ci + 6] *= inv * bf16lo(av.w); xr[8 * ci + 7] *= inv * bf16hi(av.w);
            }
            if (EPI == E_HEAD && c == 0 && r == 0) {
                // the normalised vector is the hidden state h: publish it once per batch row
                float* dsts[2] = {p.h_internal ? p.h_internal + (size_t)b * K : nullptr,
                                  p.io->hidden ? p.io->hidden + (size_t)b * K : nullptr};
                for (int t = 0; t < 2; ++t) {
                    if (!dsts[t] || abort_frame) continue;
                    float* hb = dsts[t] + (size_t)pp * kslice;
#pragma unroll
                    for (int ci = 0; ci < CH; ++ci) {
                        float4* d4 = reinterpret_cast<float4*>(hb + 8 * (lane + 32 * ci));
                        d4[0] = make_float4(xr[8 * ci + 0], xr[8 * ci + 1], xr[8 * ci + 2], xr[8 * ci + 3]);
                        d4[1] = make_float4(xr[8 * ci + 4], xr[8 * ci + 5], xr[8 * ci + 6], xr[8 * ci + 7]);
                    }
                }
            }
        }
        int i_unit, j_row;
        if (UNIT == U_PAIR_SPLIT) {
            j_row = r / p.upst;
            i_unit = r % p.upst;
        } else {
            i_unit = r / RPU;
            j_row = r % RPU;
        }
        int slot = 0, round = 0;  // k % nst, k / nst without a division per stage
        for (int k = 0; k < nstages; ++k) {
            if (k > 0 && ++slot == p.nst) {
                slot = 0;
                ++round;
            }
            if (!mbar_wait_n(&full[slot], (uint32_t)round & 1u, budget)) {
                s_flags[0] = 1;
                timeout_abort(p.st);
                break;
            }
            const int n = min(p.upst, u1 - (u0 + k * p.upst));
            if (i_unit < n) {
                const uint4* wrow = reinterpret_cast<const uint4*>(stages + (size_t)slot * p.stage_bytes +
                                                                   (size_t)r * row_bytes + (size_t)pp * kslice * 2);
                float acc = 0.f;
#pragma unroll
                for (int ci = 0; ci < CH; ++ci) acc += dot8(wrow[lane + 32 * ci], xr + 8 * ci);
                acc = warp_sum(acc);
                if (lane == 0) partial[((size_t)(k * p.upst + i_unit) * RPU + j_row) * P + pp] = acc;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    __syncthreads();

    if (s_flags[0]) {
        // a wait ran out: let any copy still in flight land before the CTA exits
        if (threadIdx.x == 0) {
            const int issued = s_flags[2];
            for (int k = issued - p.nst < 0 ? 0 : issued - p.nst; k < issued; ++k)
                (void)mbar_wait(&full[k % p.nst], (uint32_t)(k / p.nst) & 1u);
        }
        return;
    }
    const bool aborted = s_flags[1] != 0;
    const int nthr = 32 * W;
    const int tid = threadIdx.x;

    // ------------------------------ epilogues ------------------------------
    auto rowsum = [&](int lu, int j) -> float {
        const float* pr = partial + ((size_t)lu * RPU + j) * P;
        float s = 0.f;
        for (int i = 0; i < P; ++i) s += pr[i];
        return s;
    };

    if (EPI == E_STORE || EPI == E_RESIDUAL) {
        if (aborted || tid >= nthr) return;
        float* yb = p.y + (size_t)b * p.y_stride;
        for (int lu = tid; lu < nu; lu += nthr) {
            const int row = u0 + lu;
            float v = rowsum(lu, 0);
            if (EPI == E_RESIDUAL) v += (lu == tid) ? ep_res : yb[row];
            yb[row] = v;
        }
    } else if (EPI == E_SWIGLU) {
        if (aborted || tid >= nthr) return;
        float* yb = p.y + (size_t)b * p.y_stride;
        for (int lu = tid; lu < nu; lu += nthr) {
            const float g = rowsum(lu, 0);
            const float z = rowsum(lu, 1);
            yb[u0 + lu] = g / (1.0f + expf(-g)) * z;
        }
    } else if (EPI == E_QKV_ROPE) {
        if (aborted || tid >= nthr) return;
        const int pos = tid < nu ? ep_pos : p.st.pos[b];
        const int slot = pos % p.ctx;
        for (int lu = tid; lu < nu; lu += nthr) {
            const int row = 2 * (u0 + lu);
            float a = rowsum(lu, 0), bb = rowsum(lu, 1);
            const int sec = row / p.D;
            const int idx = row - sec * p.D;
            const int h = idx / p.dh, d = idx % p.dh;
            if (sec < 2) {
                const float2 t2 = (lu == tid) ? ep_cs : p.rope_tab[(size_t)b * (p.dh / 2) + (d >> 1)];
                const float c = t2.x, s = t2.y;
                const float ra = a * c - bb * s;
                const float rb = a * s + bb * c;
                a = ra;
                bb = rb;
            }
            if (sec == 0) {
                *reinterpret_cast<float2*>(p.y + (size_t)b * p.y_stride + idx) = make_float2(a, bb);
            } else {
                uint16_t* cache = (sec == 1) ? p.kc : p.vc;
                const size_t off = (((size_t)b * p.H + h) * p.ctx + slot) * p.dh + d;
                const uint32_t packed = (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(bb) << 16);
                *reinterpret_cast<uint32_t*>(cache + off) = packed;
            }
        }
    } else if (EPI == E_DEP_QKV) {
        if (aborted || tid >= nthr) return;
        const int Dd = p.D, dhd = p.dh;
        for (int lu = tid; lu < nu; lu += nthr) {
            const int row = u0 + lu;
            const float v = rowsum(lu, 0);
            const int sec = row / Dd;
            const int idx = row - sec * Dd;
            if (sec == 0) {
                p.y[(size_t)b * p.y_stride + idx] = v;
            } else {
                const int h = idx / dhd, d = idx % dhd;
                uint16_t* cache = (sec == 1) ? p.dkc : p.dvc;
                cache[(((size_t)b * p.H + h) * p.Q + p.q) * dhd + d] = f32_to_bf16_rne(v);
            }
        }
    } else if (EPI == E_HEAD || EPI == E_DEP_HEAD) {
        if (aborted) return;
        float* out = nullptr;
        if (EPI == E_HEAD) {
            if (p.io->logits) out = p.io->logits + (size_t)b * p.y_stride;
        } else {
            if (p.dio->logits) out = p.dio->logits + ((size_t)b * p.Q + p.q) * p.y_stride;
        }
        unsigned long long best = 0ull;
        if (tid < nthr) {
            for (int lu = tid; lu < nu; lu += nthr) {
                const int row = u0 + lu;
                const float v = rowsum(lu, 0);
                if (out) out[row] = v;
                if (p.logits_copy) p.logits_copy[(size_t)b * p.y_stride + row] = v;
                best = umax64(best, pack_argmax(v, (uint32_t)row));
            }
        }
        // CTA max of the packed keys
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
        __shared__ unsigned long long s_best[32];
        if (lane == 0) s_best[warp] = best;
        __syncthreads();
        if (tid == 0) {
            unsigned long long m = 0ull;
            for (int i = 0; i < W + 1; ++i) m = umax64(m, s_best[i]);
            unsigned long long* acc = (EPI == E_HEAD) ? &p.st.amax[b] : &p.st.dep_amax[b];
            uint32_t* cnt = (EPI == E_HEAD) ? &p.st.head_count[b] : &p.st.dep_count[b];
            atomicMax(acc, m);
            __threadfence();
            const uint32_t done = atomicAdd(cnt, 1u);
            if (done == (uint32_t)p.grid_per_b - 1u) {
                __threadfence();
                const unsigned long long key = atomicExch(acc, 0ull);
                *cnt = 0u;
                const int32_t am = (int32_t)unpack_argmax_index(key);
                if (EPI == E_HEAD) {
                    if (p.io->token) p.io->token[b] = am;
                    p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 0] = am;
                    p.st.pos[b] += 1;
                } else {
                    const int32_t sup = p.st.dep_sup[(size_t)b * p.Q + p.q];
                    const int32_t code = sup >= 0 ? sup : am;
                    p.st.dep_codes[(size_t)b * p.Q + p.q] = code;
                    if (p.dio->codes) p.dio->codes[(size_t)b * p.Q + p.q] = code;
                    if (p.q == p.Q - 1) {
                        // feedback slots: stream k = 1 + q' takes depth code q'
                        for (int qq = 0; qq < p.Q && 1 + qq < p.n_streams; ++qq)
                            p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 1 + qq] =
                                p.st.dep_codes[(size_t)b * p.Q + qq];
                    }
                }
            }
        }
    }
}

template <int PRO, int EPI, int UNIT>
cudaError_t launch_t(const GemvParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.grid_per_b * p.B));
    cfg.blockDim = dim3((unsigned)(32 * (p.warps + 1)));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (p.CH) {
        case 4: return cudaLaunchKernelEx(&cfg, k_gemv<4, PRO, EPI, UNIT>, p);
        case 2: return cudaLaunchKernelEx(&cfg, k_gemv<2, PRO, EPI, UNIT>, p);
        case 1: return cudaLaunchKernelEx(&cfg, k_gemv<1, PRO, EPI, UNIT>, p);
        default: return cudaErrorInvalidValue;
    }
}

template <int PRO, int EPI, int UNIT>
cudaError_t prepare_t() {
    const int mx = 220 * 1024;  // opt-in limit minus room for static shared memory
    cudaError_t e = cudaFuncSetAttribute(k_gemv<4, PRO, EPI, UNIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemv<2, PRO, EPI, UNIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemv<1, PRO, EPI, UNIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
}

#define PM_GEMV_VARIANTS(X)                      \
    X(PRO_RMSNORM, E_QKV_ROPE, U_PAIR_ADJ)       \
    X(PRO_PLAIN, E_RESIDUAL, U_ROW)              \
    X(PRO_RMSNORM, E_SWIGLU, U_PAIR_SPLIT)       \
    X(PRO_RMSNORM, E_HEAD, U_ROW)                \
    X(PRO_RMSNORM_EMB, E_DEP_QKV, U_ROW)         \
    X(PRO_RMSNORM, E_DEP_QKV, U_ROW)             \
    X(PRO_PLAIN, E_DEP_HEAD, U_ROW)              \
    X(PRO_PLAIN, E_STORE, U_ROW)                 \
    X(PRO_DEPATTN, E_RESIDUAL, U_ROW)

}  // namespace

bool plan_gemv(GemvParams& p, int rpu, int num_sms) {
    const int K = p.K;
    if (K <= 0 || K % 256 != 0 || p.n_units <= 0) return false;
    p.CH = (K % 1024 == 0) ? 4 : (K % 512 == 0) ? 2 : 1;
    p.P = K / (256 * p.CH);
    if (rpu * p.P > PM_GEMV_MAX_WARPS) return false;
    const int row_bytes = 2 * K;
    int upst = PM_GEMV_STAGE_BYTES / (row_bytes * rpu);
    if (upst < 1) upst = 1;
    while (upst > 1 && upst * rpu * p.P > PM_GEMV_MAX_WARPS) --upst;
    p.upst = upst;
    p.warps = upst * rpu * p.P;
    p.stage_bytes = (uint32_t)(upst * rpu * row_bytes);
    int nst = (int)(PM_GEMV_RING_BYTES / p.stage_bytes);
    if (nst < 2) nst = 2;
    if (nst > 16) nst = 16;
    p.nst = nst;
    const int ctas = PM_GEMV_CTAS_PER_SM * num_sms;
    p.grid_per_b = p.n_units < ctas ? p.n_units : ctas;
    if (p.nseg > 1) {
        // consecutive matrices of seg_units units each: a multiple of nseg CTAs keeps every
        // CTA's range inside one of them
        if (p.nseg > PM_GEMV_MAX_SEG || p.seg_units <= 0 || p.n_units != p.nseg * p.seg_units) return false;
        p.grid_per_b = (p.grid_per_b / p.nseg) * p.nseg;
        if (p.grid_per_b < p.nseg) p.grid_per_b = p.nseg;
    }
    p.units_cta_max = (p.n_units + p.grid_per_b - 1) / p.grid_per_b;
    p.smem = (size_t)nst * p.stage_bytes + 16u * (size_t)nst + (size_t)p.units_cta_max * rpu * p.P * 4u + 32u * 4u;
    if (p.x_in_smem) p.smem += 4u * (size_t)K + 16u;  // the input vector built by the prologue
    if (p.smem > 220u * 1024u) return false;
    return true;
}

cudaError_t gemv_prepare() {
    cudaError_t e = cudaSuccess;
#define PM_PREP(PR, EP, UN) \
    if (e == cudaSuccess) e = prepare_t<PR, EP, UN>();
    PM_GEMV_VARIANTS(PM_PREP)
#undef PM_PREP
    return e;
}

cudaError_t launch_gemv(int pro, int epi, int unit, const GemvParams& p, cudaStream_t s, bool pdl) {
#define PM_CASE(PR, EP, UN) \
    if (pro == PR && epi == EP && unit == UN) return launch_t<PR, EP, UN>(p, s, pdl);
    PM_GEMV_VARIANTS(PM_CASE)
#undef PM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pm
