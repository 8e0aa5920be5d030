// Persistent frame program for batch 1: the whole temporal frame ("PersonaPlex native LM
// audit", section 3: embedding sum, 32 x [RMSNorm, fused QKV, RoPE + KV append, causal
// windowed attention, W_O + residual, RMSNorm, SwiGLU FFN + residual], final RMSNorm,
// text head, greedy token) in one cooperative launch.
//
// Why: every step of the frame is bound by streaming weights from HBM, and each
// dependency between steps is a whole-vector reduction.  As separate kernels, each step
// boundary drains and refills the memory pipeline.  Here one CTA per SM runs the steps as
// phases separated by grid-wide barriers (a per-phase arrival counter, bounded spins),
// while a producer warp in every CTA keeps issuing bulk copies for the *following*
// phases -- the next matrix's rows, or the attention phase's cached K/V rows, none of
// which depends on the phase in progress -- into a six-slot shared-memory ring.  The
// weight stream therefore runs across phase boundaries; consumers only wait for the
// small activation vectors.
//
// Roles in a CTA (544 threads): warps 0-15 consume, warp 16 produces.
//  * GEMV phase (units = rows or row pairs of a matrix, balanced contiguous ranges per
//    CTA): a stage holds R = 16 / (K/1024) rows; consumer warp w reduces row w / nsl over
//    K-slice w % nsl (1024 columns, 32 per lane, the input slice held in registers), the
//    per-row partials meet in shared memory, then the fused epilogue runs: RMSNorm scale
//    (prologue), RoPE + bf16 KV append, residual add, SwiGLU, or logits + argmax.
//  * attention phase: items (head, 64-key chunk) of the window, a grid-stride list per
//    CTA; the producer copies each item's K and V rows (16 KB + 16 KB, ring wrap split in
//    two copies, the current position excluded) into one slot; consumer warp group
//    g (4 warps) takes items g, g+4, ...; chunk results merge in the last CTA to finish
//    the head (completion counter).
//  * embed phase: IDs validated by every CTA before anything starts (an invalid frame
//    is a no-op), 256-column slices of the 17-row sum, RoPE table of the position.
//  * final phase (CTA 0): greedy token, feedback slot, position advance, counter reset.
#include <math.h>
#include <string.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int NCW = 16;             // consumer warps
constexpr int NTH = 32 * (NCW + 1);  // threads per CTA
constexpr int NSLOT = 6;
constexpr uint32_t SLOT_BYTES = 32768;
constexpr int DH = 128;
constexpr int KPC = 64;

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ void group_bar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory"); }

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t cnt) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(cnt) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float* v) {
    v[0] = bf16lo(a.x); v[1] = bf16hi(a.x); v[2] = bf16lo(a.y); v[3] = bf16hi(a.y);
    v[4] = bf16lo(a.z); v[5] = bf16hi(a.z); v[6] = bf16lo(a.w); v[7] = bf16hi(a.w);
    v[8] = bf16lo(b.x); v[9] = bf16hi(b.x); v[10] = bf16lo(b.y); v[11] = bf16hi(b.y);
    v[12] = bf16lo(b.z); v[13] = bf16hi(b.z); v[14] = bf16lo(b.w); v[15] = bf16hi(b.w);
}

struct Range {
    int u0, u1;
};
__device__ __forceinline__ Range cta_range(int n_units, int c, int G) {
    Range r;
    r.u0 = (int)((long long)c * n_units / G);
    r.u1 = (int)((long long)(c + 1) * n_units / G);
    return r;
}

// attention items of this frame: (head, chunk) with nc chunks per head
__device__ __forceinline__ int attn_nc(int pos, int ctx) { return (min(pos + 1, ctx) + KPC - 1) / KPC; }

}  // namespace

__global__ void __launch_bounds__(NTH, 1) k_frame(const FrameProgParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSLOT * SLOT_BYTES);
    uint64_t* empty = full + NSLOT;
    float* partial = reinterpret_cast<float*>(empty + NSLOT);         // [p.partial_floats]
    float* red = partial + p.partial_floats;                           // [32]
    float* gacc = red + 32;                                            // [4 groups][4 warps][DH + 2]
    float* gm = gacc + 4 * 4 * (DH + 2);                               // [4 groups][MAXC]
    __shared__ int s_flag[8];
    __shared__ unsigned long long s_best[NCW + 1];

    const int c = blockIdx.x, G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const int pos = p.st.pos[0];
    // poll budget of the ring and phase waits (the drain after a timeout keeps the full one)
    const uint32_t budget = wait_budget(p.st);
    const unsigned long long grid_limit = (unsigned long long)budget << 4;
    uint32_t* const exit_count = &p.bar[p.n_phases];     // CTAs done with this launch
    uint32_t* const timeouts = &p.bar[p.n_phases + 1];  // CTAs whose wait ran out in this launch

    // ---------------- validation (all threads), barrier init ----------------
    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        fence_barrier_init();
        s_flag[0] = 0;  // timeout
    }
    int bad = 0;
    const bool direct = p.io->direct != 0;  // inputs already delayed (generator step)
    if (tid < p.n_streams) {
        int id = p.io->ids[tid];
        if (id == -3) id = p.st.sel[tid];
        if (id < -1 || id >= p.rows[tid]) bad = 1;
        // a delayed stream's input comes back from the delay ring: checked the same way
        const int src = pos - p.delays[tid];
        if (!direct && p.delays[tid] != 0 && src >= p.st.first_pos[0]) {
            const int in = p.st.ring[(src & 3) * PM_MAX_STREAMS_DEV + tid];
            if (in < -1 || in >= p.rows[tid]) bad = 1;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (c == 0 && tid == 0) {
            p.st.status[1] = 1u;
            set_status(p.st.status, PM_DEV_ERR_INVALID_ID);
        }
        return;  // nothing was issued and no counter touched; the frame is a no-op
    }

    if (warp == NCW) {
        // =================================== producer ===================================
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int seq = 0;
            bool ok = true;
            auto next_slot = [&](uint32_t bytes) -> int {
                const int slot = seq % NSLOT;
                if (*(volatile int*)&s_flag[0]) {
                    ok = false;
                    return -1;
                }
                if (seq >= NSLOT && !mbar_wait_n(&empty[slot], (uint32_t)((seq / NSLOT) - 1) & 1u, budget)) {
                    ok = false;
                    return -1;
                }
                mbar_arrive_expect_tx(&full[slot], bytes);
                ++seq;
                return slot;
            };
            for (int ph = 0; ph < p.n_phases && ok; ++ph) {
                const FPhase& f = p.ph[ph];
                if (f.type == PH_GEMV) {
                    const Range r = cta_range(f.n_units, c, G);
                    const uint32_t row_bytes = (uint32_t)f.K * 2u;
                    for (int ua = r.u0; ua < r.u1 && ok; ua += f.upst) {
                        const int n = min(f.upst, r.u1 - ua);
                        if (f.unit == U_PAIR_SPLIT) {
                            const uint32_t bytes = (uint32_t)n * row_bytes;
                            const int slot = next_slot(2u * bytes);
                            if (slot < 0) break;
                            uint8_t* dst = ring + (size_t)slot * SLOT_BYTES;
                            bulk_g2s(dst, f.W + (size_t)ua * f.K, bytes, &full[slot], pol);
                            bulk_g2s(dst + (size_t)f.upst * row_bytes, f.W + (size_t)(ua + f.split_rows) * f.K, bytes,
                                     &full[slot], pol);
                        } else {
                            const int rpu = (f.unit == U_ROW) ? 1 : 2;
                            const uint32_t bytes = (uint32_t)(n * rpu) * row_bytes;
                            const int slot = next_slot(bytes);
                            if (slot < 0) break;
                            bulk_g2s(ring + (size_t)slot * SLOT_BYTES, f.W + (size_t)ua * rpu * f.K, bytes, &full[slot],
                                     pol);
                        }
                    }
                } else if (f.type == PH_ATTN) {
                    const int n = min(pos + 1, p.win), lo = pos - n + 1, nc = attn_nc(pos, p.win);
                    for (int item = c; item < p.H * nc && ok; item += G) {
                        const int h = item / nc, ci = item % nc;
                        const int k0 = lo + ci * KPC;
                        const int k1 = min(k0 + KPC, pos + 1);
                        const int kend = (k1 - 1 == pos) ? pos : k1;  // the current row comes later
                        const int cnt = kend - k0;
                        const int slot = next_slot(2u * (uint32_t)cnt * DH * 2u);
                        if (slot < 0) break;
                        if (cnt > 0) {
                            uint8_t* dst = ring + (size_t)slot * SLOT_BYTES;
                            const size_t hb = (size_t)h * p.ctx * DH;
                            const int s0 = k0 % p.ctx;
                            const int first = min(cnt, p.ctx - s0);
                            for (int kv = 0; kv < 2; ++kv) {
                                const uint16_t* base = (kv == 0 ? f.kc : f.vc) + hb;
                                uint8_t* d = dst + (size_t)kv * (KPC * DH * 2);
                                bulk_g2s(d, base + (size_t)s0 * DH, (uint32_t)first * DH * 2u, &full[slot], pol);
                                if (cnt > first)
                                    bulk_g2s(d + (size_t)first * DH * 2, base, (uint32_t)(cnt - first) * DH * 2u,
                                             &full[slot], pol);
                            }
                        }
                    }
                }
            }
            if (!ok && !*(volatile int*)&s_flag[0]) {
                s_flag[0] = 1;
                timeout_abort(p.st);
                atomicAdd(timeouts, 1u);
            }
            s_flag[1] = seq;
        }
    } else {
        // =================================== consumers ===================================
        // Every wait below is bounded.  A wait that runs out sets s_flag[0]; from then on
        // the CTA keeps the same control flow (so every bar.sync stays matched) but skips
        // all waits and work, arrives on the phase counters, and exits.
        int seq = 0;
        const float eps = p.eps;
        auto timed_out = [&]() -> bool { return *(volatile int*)&s_flag[0] != 0; };
        auto note_timeout = [&]() {
            if (!timed_out()) atomicAdd(timeouts, 1u);
            s_flag[0] = 1;
            timeout_abort(p.st);
        };
        auto wait_full = [&](int slot, uint32_t parity) -> bool {
            if (timed_out()) return false;
            if (!mbar_wait_n(&full[slot], parity, budget)) {
                note_timeout();
                return false;
            }
            return true;
        };
        for (int ph = 0; ph < p.n_phases; ++ph) {
            const FPhase& f = p.ph[ph];
            // wait for every CTA to finish the previous phase
            if (ph > 0) {
                if (tid == 0 && !timed_out()) {
                    unsigned long long it = 0;
                    while (ld_acquire_u32(&p.bar[ph - 1]) < (uint32_t)G) {
                        if (++it > grid_limit) {
                            note_timeout();
                            break;
                        }
                    }
                }
                cons_bar();
            }
            const bool skip = timed_out();

            if (skip) {
                // nothing: keep arriving on the counters below
            } else if (f.type == PH_EMBED) {
                // delay assembly (every CTA computes the same inputs), 256 columns per CTA
                __shared__ int s_in[PM_MAX_STREAMS_DEV];
                if (tid < p.n_streams) {
                    const int k = tid;
                    int id = p.io->ids[k];
                    if (id == -3) id = p.st.sel[k];
                    const int src = pos - p.delays[k];
                    int in;
                    if (direct || p.delays[k] == 0)
                        in = id;
                    else if (src >= p.st.first_pos[0])
                        in = p.st.ring[(src & 3) * PM_MAX_STREAMS_DEV + k];
                    else
                        in = p.init_id[k];
                    s_in[k] = in;
                    if (c == 0 && !direct) p.st.ring[(pos & 3) * PM_MAX_STREAMS_DEV + k] = id;
                }
                if (c == 0 && tid < p.dh / 2) {
                    double sn, cs;
                    sincos((double)pos * p.rope_freq[tid], &sn, &cs);
                    p.rope_tab[tid] = make_float2((float)cs, (float)sn);
                }
                if (c == 0 && tid == 0) p.st.status[1] = 0u;
                cons_bar();
                const int col = c * 256 + 8 * tid;
                if (tid < 32 && col < p.D) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
                    for (int k = 0; k < p.n_streams; ++k) {
                        const int id = s_in[k];
                        if (id < 0) continue;
                        const uint4 w = *reinterpret_cast<const uint4*>(p.tables[k] + (size_t)id * p.D + col);
                        acc[0] += bf16lo(w.x); acc[1] += bf16hi(w.x);
                        acc[2] += bf16lo(w.y); acc[3] += bf16hi(w.y);
                        acc[4] += bf16lo(w.z); acc[5] += bf16hi(w.z);
                        acc[6] += bf16lo(w.w); acc[7] += bf16hi(w.w);
                    }
                    float4* dst = reinterpret_cast<float4*>(p.x + col);
                    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                }
            } else if (f.type == PH_GEMV) {
                const int nsl = f.K / 1024;
                const int R = NCW / nsl;  // stage rows
                const int r = warp / nsl, pp = warp % nsl;
                const bool active = r < R;
                const int RPU = (f.unit == U_ROW) ? 1 : 2;
                const uint32_t row_bytes = (uint32_t)f.K * 2u;
                // input slice: columns pp*1024 + 8*(lane + 32*ci) .. +7, ci < 4
                float xr[32];
                const float* xb = f.x + (size_t)pp * 1024;
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) {
                    const float4 a = ldcg4(xb + 8 * (lane + 32 * ci));
                    const float4 b = ldcg4(xb + 8 * (lane + 32 * ci) + 4);
                    xr[8 * ci + 0] = a.x; xr[8 * ci + 1] = a.y; xr[8 * ci + 2] = a.z; xr[8 * ci + 3] = a.w;
                    xr[8 * ci + 4] = b.x; xr[8 * ci + 5] = b.y; xr[8 * ci + 6] = b.z; xr[8 * ci + 7] = b.w;
                }
                if (f.alpha) {
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) ss = fmaf(xr[i], xr[i], ss);
                    ss = warp_sum(ss);
                    if (r == 0 && lane == 0) red[pp] = ss;
                    cons_bar();
                    float tot = 0.f;
                    for (int i = 0; i < nsl; ++i) tot += red[i];
                    const float inv = 1.0f / sqrtf(tot / (float)f.K + eps);
                    const uint16_t* al = f.alpha + (size_t)pp * 1024;
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) {
                        const uint4 av = *reinterpret_cast<const uint4*>(al + 8 * (lane + 32 * ci));
                        xr[8 * ci + 0] *= inv * bf16lo(av.x); xr[8 * ci + 1] *= inv * bf16hi(av.x);
                        xr[8 * ci + 2] *= inv * bf16lo(av.y); xr[8 * ci + 3] *= inv * bf16hi(av.y);
                        xr[8 * ci + 4] *= inv * bf16lo(av.z); xr[8 * ci + 5] *= inv * bf16hi(av.z);
                        xr[8 * ci + 6] *= inv * bf16lo(av.w); xr[8 * ci + 7] *= inv * bf16hi(av.w);
                    }
                    if (f.epi == E_HEAD && c == 0 && r == 0) {
                        float* dsts[2] = {p.h, p.io->hidden};
                        for (int t = 0; t < 2; ++t) {
                            if (!dsts[t]) continue;
                            float* hb = dsts[t] + (size_t)pp * 1024;
#pragma unroll
                            for (int ci = 0; ci < 4; ++ci) {
                                float4* d4 = reinterpret_cast<float4*>(hb + 8 * (lane + 32 * ci));
                                d4[0] = make_float4(xr[8 * ci + 0], xr[8 * ci + 1], xr[8 * ci + 2], xr[8 * ci + 3]);
                                d4[1] = make_float4(xr[8 * ci + 4], xr[8 * ci + 5], xr[8 * ci + 6], xr[8 * ci + 7]);
                            }
                        }
                    }
                }
                int i_unit, j_row;
                if (f.unit == U_PAIR_SPLIT) {
                    j_row = r / f.upst;
                    i_unit = r % f.upst;
                } else {
                    i_unit = r / RPU;
                    j_row = r % RPU;
                }
                const Range rg = cta_range(f.n_units, c, G);
                int k = 0;
                for (int ua = rg.u0; ua < rg.u1; ua += f.upst, ++k) {
                    const int slot = seq % NSLOT;
                    const bool have = wait_full(slot, (uint32_t)(seq / NSLOT) & 1u);
                    const int n = min(f.upst, rg.u1 - ua);
                    if (have && active && i_unit < n) {
                        const uint4* wrow = reinterpret_cast<const uint4*>(ring + (size_t)slot * SLOT_BYTES +
                                                                           (size_t)r * row_bytes + (size_t)pp * 2048);
                        float acc = 0.f;
#pragma unroll
                        for (int ci = 0; ci < 4; ++ci) acc += dot8(wrow[lane + 32 * ci], xr + 8 * ci);
                        acc = warp_sum(acc);
                        if (lane == 0) partial[((size_t)(k * f.upst + i_unit) * RPU + j_row) * nsl + pp] = acc;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    ++seq;
                }
                cons_bar();
                // epilogue: thread t handles local units t, t + 512, ...
                const int nu = rg.u1 - rg.u0;
                auto rowsum = [&](int lu, int j) -> float {
                    const float* pr = partial + ((size_t)lu * RPU + j) * nsl;
                    float s = 0.f;
                    for (int i = 0; i < nsl; ++i) s += pr[i];
                    return s;
                };
                if (f.epi == E_RESIDUAL) {
                    for (int lu = tid; lu < nu; lu += 512) {
                        const int row = rg.u0 + lu;
                        f.y[row] = __ldcg(f.y + row) + rowsum(lu, 0);
                    }
                } else if (f.epi == E_SWIGLU) {
                    for (int lu = tid; lu < nu; lu += 512) {
                        const float g = rowsum(lu, 0), z = rowsum(lu, 1);
                        f.y[rg.u0 + lu] = g / (1.0f + expf(-g)) * z;
                    }
                } else if (f.epi == E_QKV_ROPE) {
                    const int slot = pos % p.ctx;
                    for (int lu = tid; lu < nu; lu += 512) {
                        const int row = 2 * (rg.u0 + lu);
                        float a = rowsum(lu, 0), bb = rowsum(lu, 1);
                        const int sec = row / p.D;
                        const int idx = row - sec * p.D;
                        const int h = idx / DH, d = idx % DH;
                        if (sec < 2) {
                            const float2 t2 = p.rope_tab[d >> 1];
                            const float ra = a * t2.x - bb * t2.y;
                            const float rb = a * t2.y + bb * t2.x;
                            a = ra;
                            bb = rb;
                        }
                        if (sec == 0) {
                            *reinterpret_cast<float2*>(p.q + idx) = make_float2(a, bb);
                        } else {
                            uint16_t* cache = (sec == 1) ? f.kc : f.vc;
                            const size_t off = ((size_t)h * p.ctx + slot) * DH + d;
                            *reinterpret_cast<uint32_t*>(cache + off) =
                                (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(bb) << 16);
                        }
                    }
                } else if (f.epi == E_HEAD) {
                    float* out = p.io->logits;
                    unsigned long long best = 0ull;
                    for (int lu = tid; lu < nu; lu += 512) {
                        const int row = rg.u0 + lu;
                        const float v = rowsum(lu, 0);
                        if (out) out[row] = v;
                        best = umax64(best, pack_argmax(v, (uint32_t)row));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
                    if (lane == 0) s_best[warp] = best;
                    cons_bar();
                    if (tid == 0) {
                        unsigned long long m = 0ull;
                        for (int i = 0; i < NCW; ++i) m = umax64(m, s_best[i]);
                        atomicMax(&p.st.amax[0], m);
                    }
                }
            } else if (f.type == PH_ATTN) {
                const int n = min(pos + 1, p.win), lo = pos - n + 1, nc = attn_nc(pos, p.win);
                const int ng = warp >> 2, wq = warp & 3;  // group, warp in group
                const int g = lane >> 3, sub = lane & 7;
                float* myacc = gacc + (size_t)ng * 4 * (DH + 2);
                float* mym = gm + (size_t)ng * p.max_chunks;
                int j = 0;
                for (int item = c; item < p.H * nc; item += G, ++j) {
                    const int slot = (seq + j) % NSLOT;
                    if ((j & 3) != ng) continue;
                    const bool have = wait_full(slot, (uint32_t)((seq + j) / NSLOT) & 1u);
                    const int h = item / nc, ci = item % nc;
                    const int k0 = lo + ci * KPC;
                    const int k1 = min(k0 + KPC, pos + 1);
                    const uint8_t* sk = ring + (size_t)slot * SLOT_BYTES;
                    const uint8_t* sv = sk + KPC * DH * 2;
                    float q[16];
                    {
                        const float* qp = p.q + h * DH + 16 * sub;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float4 t4 = ldcg4(qp + 4 * v);
                            q[4 * v + 0] = t4.x * p.scale_log2;
                            q[4 * v + 1] = t4.y * p.scale_log2;
                            q[4 * v + 2] = t4.z * p.scale_log2;
                            q[4 * v + 3] = t4.w * p.scale_log2;
                        }
                    }
                    float sc[4], m = -INFINITY;
                    uint4 vr[4][2];
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int i = wq * 16 + g * 4 + it;  // key index inside the chunk
                        const int kk = k0 + i;
                        uint4 ka = make_uint4(0, 0, 0, 0), kb = ka;
                        vr[it][0] = vr[it][1] = ka;
                        if (kk < k1 && have) {
                            if (kk == pos) {
                                const size_t off = ((size_t)h * p.ctx + (pos % p.ctx)) * DH + 16 * sub;
                                const uint4* kp = reinterpret_cast<const uint4*>(f.kc + off);
                                const uint4* vp = reinterpret_cast<const uint4*>(f.vc + off);
                                ka = __ldcg(kp);
                                kb = __ldcg(kp + 1);
                                vr[it][0] = __ldcg(vp);
                                vr[it][1] = __ldcg(vp + 1);
                            } else {
                                const uint4* kp = reinterpret_cast<const uint4*>(sk + (size_t)i * DH * 2 + 32 * sub);
                                const uint4* vp = reinterpret_cast<const uint4*>(sv + (size_t)i * DH * 2 + 32 * sub);
                                ka = kp[0];
                                kb = kp[1];
                                vr[it][0] = vp[0];
                                vr[it][1] = vp[1];
                            }
                        }
                        float kv[16];
                        unpack16(ka, kb, kv);
                        float d = 0.f;
#pragma unroll
                        for (int e = 0; e < 16; ++e) d = fmaf(q[e], kv[e], d);
                        d += __shfl_xor_sync(0xffffffffu, d, 1);
                        d += __shfl_xor_sync(0xffffffffu, d, 2);
                        d += __shfl_xor_sync(0xffffffffu, d, 4);
                        sc[it] = (kk < k1) ? d : -INFINITY;
                        m = fmaxf(m, sc[it]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cnt(&empty[slot], 4u);  // the slot's 16 arrivals come from 4 warps
                    float l = 0.f, acc[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
                    if (m != -INFINITY) {
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const float w = exp2f(sc[it] - m);
                            l += w;
                            float vv[16];
                            unpack16(vr[it][0], vr[it][1], vv);
#pragma unroll
                            for (int e = 0; e < 16; ++e) acc[e] = fmaf(w, vv[e], acc[e]);
                        }
                    }
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
                    float* wa = myacc + (size_t)wq * (DH + 2);
                    if (g == 0) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) wa[16 * sub + e] = acc[e];
                        if (sub == 0) {
                            wa[DH] = m;
                            wa[DH + 1] = l;
                        }
                    }
                    group_bar(ng);
                    const int t = wq * 32 + lane;  // coordinate owned by this thread
                    float M = -INFINITY;
                    for (int w = 0; w < 4; ++w) M = fmaxf(M, myacc[w * (DH + 2) + DH]);
                    float L = 0.f, A = 0.f;
                    for (int w = 0; w < 4; ++w) {
                        const float mw = myacc[w * (DH + 2) + DH];
                        const float fw = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
                        L += myacc[w * (DH + 2) + DH + 1] * fw;
                        A += myacc[w * (DH + 2) + t] * fw;
                    }
                    group_bar(ng);
                    if (nc == 1) {
                        p.o[h * DH + t] = A / L;
                        continue;
                    }
                    float* part = p.part + ((size_t)h * p.S + ci) * (DH + 2);
                    part[t] = A;
                    if (t == 0) {
                        part[DH] = M;
                        part[DH + 1] = L;
                    }
                    __threadfence();
                    group_bar(ng);
                    if (t == 0) {
                        const uint32_t done = atomicAdd(&p.att_count[h], 1u);
                        s_flag[2 + ng] = (done == (uint32_t)nc - 1u) ? 1 : 0;
                    }
                    group_bar(ng);
                    if (!s_flag[2 + ng]) continue;
                    __threadfence();
                    const float* pb = p.part + (size_t)h * p.S * (DH + 2);
                    for (int i = t; i < nc; i += 128) mym[i] = __ldcg(pb + (size_t)i * (DH + 2) + DH);
                    group_bar(ng);
                    float Mx = -INFINITY;
                    for (int i = 0; i < nc; ++i) Mx = fmaxf(Mx, mym[i]);
                    float Lx = 0.f, Ax = 0.f;
#pragma unroll 8
                    for (int i = 0; i < nc; ++i) {
                        const float fi = (mym[i] == -INFINITY) ? 0.f : exp2f(mym[i] - Mx);
                        Lx += __ldcg(pb + (size_t)i * (DH + 2) + DH + 1) * fi;
                        Ax += __ldcg(pb + (size_t)i * (DH + 2) + t) * fi;
                    }
                    p.o[h * DH + t] = Ax / Lx;
                    if (t == 0) p.att_count[h] = 0u;
                    group_bar(ng);
                }
                seq += j;
            }
            // this CTA is done with the phase: the CTA barrier orders every consumer's writes
            // before thread 0's release-add (cumulative at gpu scope)
            cons_bar();
            if (tid == 0) red_release_add(&p.bar[ph], 1u);
        }
        // final phase: the greedy token and the frame's state advance (CTA 0), only when
        // no CTA's wait ran out in this launch (then the frame leaves no selection and the
        // position stays, like an aborted frame)
        if (!timed_out() && c == 0) {
            if (tid == 0) {
                unsigned long long it = 0;
                bool done = true;
                while (ld_acquire_u32(&p.bar[p.n_phases - 1]) < (uint32_t)G) {
                    if (++it > grid_limit) {
                        done = false;
                        note_timeout();
                        break;
                    }
                }
                if (done && ld_acquire_u32(timeouts) == 0u) {
                    __threadfence();
                    const unsigned long long key = atomicExch(&p.st.amax[0], 0ull);
                    const int32_t am = (int32_t)unpack_argmax_index(key);
                    if (p.io->token) p.io->token[0] = am;
                    p.st.sel[0] = am;
                    p.st.pos[0] = pos + 1;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (s_flag[0]) {
            // a wait ran out: let the copies already issued land before the CTA exits
            const int issued = s_flag[1];
            for (int i = issued - NSLOT < 0 ? 0 : issued - NSLOT; i < issued; ++i)
                (void)mbar_wait(&full[i % NSLOT], (uint32_t)(i / NSLOT) & 1u);
        }
        // The last CTA out clears what the launch counted with (phase counters, the exit and
        // timeout counters, the head's argmax, the attention merge counters), whether or not a
        // wait ran out: every CTA has passed its last read of them by then.
        __threadfence();
        if (atomicAdd(exit_count, 1u) == (uint32_t)G - 1u) {
            __threadfence();
            for (int i = 0; i < p.n_phases + 2; ++i) p.bar[i] = 0u;
            p.st.amax[0] = 0ull;
            for (int h = 0; h < p.H; ++h) p.att_count[h] = 0u;
        }
    }
}

bool frame_prog_supported(int D, int F, int dh) { return dh == DH && D % 1024 == 0 && F % 1024 == 0 && D <= 16384; }

size_t frame_prog_smem(int partial_floats, int max_chunks) {
    return (size_t)NSLOT * SLOT_BYTES + 16u * NSLOT + 4u * (size_t)partial_floats + 4u * 32 +
           4u * 4 * 4 * (DH + 2) + 4u * 4 * (size_t)max_chunks;
}

cudaError_t frame_prog_prepare(size_t smem) {
    return cudaFuncSetAttribute(k_frame, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_frame_prog(const FrameProgParams& p, int grid, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTH);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_frame, p);
}

int frame_prog_stage_rows(int K) { return NCW / (K / 1024); }

int frame_prog_threads() { return NTH; }

cudaError_t frame_prog_occupancy(size_t smem, int* blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_frame, NTH, smem);
}

}  // namespace pm
