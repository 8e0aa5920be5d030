// Batched projections (B >= 2) on the 5th-generation tensor cores.
//
// y[b][r] = sum_k W[r][k] x[b][k] for every projection of the temporal block and the
// text head ("PersonaPlex native LM audit", sections 3 and 5 shapes), computed swap-AB:
// the weight tile is the MMA's M = 128 operand, the batch is N = 16 / 32 / 64, the fp32
// accumulator lives in tensor memory.  Still HBM-bound (<= 64 flops per weight byte), so
// the design streams each weight byte once:
//  * work = (128-row tile, 64-element k tile) units in tile-major order, split into one
//    contiguous, balanced range per CTA (stream-K); a tile cut between CTAs is merged
//    deterministically by the last CTA to finish it (partials in slot order, completion
//    counter, no waiting);
//  * warp 4 streams A (weights, 2-D TMA, 128-byte swizzle, L2 evict-first) and B (the
//    bf16 activations, L2 evict-last: every CTA reads them) through a ring of stages;
//    the A copies of the first ring are issued before griddepcontrol.wait, and once its
//    own copies are out it prefetches the head of the next projection's weights to L2;
//  * warp 5 owns the tensor memory and issues tcgen05.mma (4 x K=16 per stage), freeing
//    each stage with tcgen05.commit; two accumulator buffers let the epilogue of one
//    tile overlap the MMAs of the next;
//  * warps 0-3 drain the accumulator (tcgen05.ld, lane = weight row) and apply the fused
//    epilogue: RMSNorm scale of the input (folded: the activations arrive as
//    bf16(alpha * x) with per-row sums of squares), residual add + the next norm's bf16
//    operand, SwiGLU, RoPE + KV-ring append, or the text head's argmax.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

#include "pm_kernels.h"
#include "tc_common.cuh"

// Tiling policy (compile-time tuning constants): CTAs per SM, fewest k-units per CTA
// (bounds how many ways a tile is split), bytes of the stage ring per CTA.
#ifndef PM_TC_CTAS_PER_SM
#define PM_TC_CTAS_PER_SM 2
#endif
#ifndef PM_TC_MIN_UNITS
#define PM_TC_MIN_UNITS 1
#endif
#ifndef PM_TC_RING_BYTES
#define PM_TC_RING_BYTES (96u * 1024u)
#endif

namespace pm {
namespace {

constexpr int KT = 64;                    // elements per k tile (128 bytes, one swizzle row)
constexpr uint32_t A_BYTES = 128u * 128u;  // 128 rows x 128 B

__host__ __device__ __forceinline__ long long unit_begin(int c, long long U, int G) { return (long long)c * U / G; }

// CTA whose unit range contains unit u
__host__ __device__ __forceinline__ int cta_of(long long u, long long U, int G) {
    int c = (int)(u * G / U);
    while (c + 1 < G && unit_begin(c + 1, U, G) <= u) ++c;
    while (c > 0 && unit_begin(c, U, G) > u) --c;
    return c;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// L2 prefetch of the first units (tile boxes) that CTA c of the next tensor-core
// projection streams, through that projection's tensor map
__device__ __forceinline__ void prefetch_next_tc(const CUtensorMap* tmN, const NextPrefetch& nx, int c) {
    const long long U = (long long)nx.n_mtiles * nx.nk;
    const long long u0 = unit_begin(c, U, nx.grid), u1 = unit_begin(c + 1, U, nx.grid);
    long long n = (long long)(nx.bytes / A_BYTES);
    if (n > u1 - u0) n = u1 - u0;
    for (long long i = 0; i < n; ++i) {
        const long long u = u0 + i;
        const int m = (int)(u / nx.nk), kt = (int)(u % nx.nk);
        if (nx.split_rows) {
            tma_prefetch_2d(tmN, kt * KT, m * 64);
            tma_prefetch_2d(tmN, kt * KT, nx.split_rows + m * 64);
        } else {
            tma_prefetch_2d(tmN, kt * KT, m * 128);
        }
    }
}

// v[i] = v[i + 16]: the next block of 16 frames moves to the front of the accumulator row
template <int NPAD>
__device__ __forceinline__ void shift_block(float (&v)[NPAD]) {
#pragma unroll
    for (int i = 0; i + 16 < NPAD; ++i) v[i] = v[i + 16];
}

// Sum over the warp of each of 16 per-lane values in 16 shuffles (instead of 16 x 5): at
// each step a lane keeps half of its values and adds its partner's copy of that half, so
// lane l ends with the total of value (l >> 1) & 15 (both lanes of a pair hold it).
__device__ __forceinline__ float warp_sum16_transposed(float (&a)[16], int lane) {
#pragma unroll
    for (int half = 8, mask = 16; half >= 1; half >>= 1, mask >>= 1) {
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? a[i] : a[i + half];
            const float keep = upper ? a[i + half] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
    return a[0] + __shfl_xor_sync(0xffffffffu, a[0], 1);
}

// RoPE over the frames of a q or k row (lane pairs hold the two coordinates of a rotation
// pair, the even coordinate first); frame b's value goes to put(b, o, aux(b)), with aux --
// a ring slot, say -- evaluated for a block of 16 frames before its first store; rolled in
// blocks of 16
template <int NPAD, class Aux, class Put>
__device__ __forceinline__ void rope_frames(float (&v)[NPAD], const TcParams& p, int d, int lane, Aux aux, Put put) {
    const bool even = (lane & 1) == 0;
    const float2* tab = p.rope_tab + (d >> 1);
#pragma unroll 1
    for (int b0 = 0; b0 < p.B; b0 += 16) {
        float2 cs[16];  // the block's rotation factors
        int ax[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const bool in = b0 + j < p.B;
            cs[j] = in ? tab[(size_t)(b0 + j) * (p.dh / 2)] : make_float2(1.f, 0.f);
            ax[j] = in ? aux(b0 + j) : 0;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (b0 + j >= p.B) break;
            const float mine = v[j];
            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
            put(b0 + j, even ? (mine * cs[j].x - other * cs[j].y) : (other * cs[j].y + mine * cs[j].x), ax[j]);
        }
        shift_block<NPAD>(v);
    }
}

// the frames of a row without rotation (v rows), as rope_frames
template <int NPAD, class Aux, class Put>
__device__ __forceinline__ void plain_frames(float (&v)[NPAD], int B, Aux aux, Put put) {
#pragma unroll 1
    for (int b0 = 0; b0 < B; b0 += 16) {
        int ax[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) ax[j] = (b0 + j < B) ? aux(b0 + j) : 0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (b0 + j < B) put(b0 + j, v[j], ax[j]);
        shift_block<NPAD>(v);
    }
}

template <int EPI, int NPAD>
__global__ void __launch_bounds__(192, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmN, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr uint32_t B_BYTES = NPAD * 128u;
    constexpr uint32_t ST_BYTES = A_BYTES + B_BYTES;
    const int nst = p.nst;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)nst * ST_BYTES);
    uint64_t* empty = full + nst;
    uint64_t* acc_full = empty + nst;  // [2]
    uint64_t* acc_empty = acc_full + 2;  // [2]
    uint64_t* fin = acc_empty + 2;       // MMA completion at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    int* flags = reinterpret_cast<int*>(tmem_slot + 4);  // [0] timeout, [1] last-of-tile, [2] issued
    float* inv = reinterpret_cast<float*>(flags + 4);    // [NPAD]
    float* xch = inv + NPAD;                              // [NPAD][64] SwiGLU exchange / reductions
    unsigned long long* red64 = reinterpret_cast<unsigned long long*>(xch + NPAD * 64);  // [4][NPAD]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.grid, c = blockIdx.x;
    const long long U = (long long)p.n_mtiles * p.nk;
    const long long w0 = unit_begin(c, U, G), w1 = unit_begin(c + 1, U, G);
    const int n = (int)(w1 - w0);
    constexpr uint32_t TMEM_COLS = (2 * NPAD < 32) ? 32 : 2 * NPAD;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        mbar_init(fin, 1);
        fence_barrier_init();
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0 && n > 0) {
            const uint64_t pol_w = l2_evict_first_policy();
            const uint64_t pol_x = l2_evict_last_policy();
            auto load_a = [&](int i) {
                const long long u = w0 + i;
                const int m = (int)(u / p.nk), kt = (int)(u % p.nk);
                uint8_t* dst = smem + (size_t)(i % nst) * ST_BYTES;
                if (p.a_tiled) {
                    tma_load_2d(dst, &tmA, 0, (int)(u * 128), &full[i % nst], pol_w);
                } else if (EPI == TE_SWIGLU) {
                    tma_load_2d(dst, &tmA, kt * KT, m * 64, &full[i % nst], pol_w);
                    tma_load_2d(dst + A_BYTES / 2, &tmA, kt * KT, p.split_rows + m * 64, &full[i % nst], pol_w);
                } else {
                    tma_load_2d(dst, &tmA, kt * KT, m * 128, &full[i % nst], pol_w);
                }
            };
            auto load_b = [&](int i) {
                const long long u = w0 + i;
                const int kt = (int)(u % p.nk);
                if (p.b_tiled)
                    tma_load_2d(smem + (size_t)(i % nst) * ST_BYTES + A_BYTES, &tmB, 0, kt * NPAD, &full[i % nst], pol_x);
                else
                    tma_load_2d(smem + (size_t)(i % nst) * ST_BYTES + A_BYTES, &tmB, kt * KT, 0, &full[i % nst], pol_x);
            };
            const int pre = n < nst ? n : nst;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], ST_BYTES);
                load_a(i);  // weights do not depend on the previous kernel
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) load_b(i);
            flags[2] = pre;
            for (int i = pre; i < n; ++i) {
                const int slot = i % nst;
                if (!mbar_wait(&empty[slot], (uint32_t)((i / nst) - 1) & 1u)) {
                    flags[0] = 1;
                    set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], ST_BYTES);
                load_a(i);
                load_b(i);
                flags[2] = i + 1;
            }
            if (p.nx.n_mtiles > 0 && c < p.nx.grid) prefetch_next_tc(&tmN, p.nx, c);
        }
    } else if (warp == 5) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0 && n > 0) {
            const uint32_t idesc = idesc_bf16_f32(128, NPAD);
            int seg = 0;
            bool ok = true;
            for (int i = 0; i < n && ok; ++i) {
                const long long u = w0 + i;
                const int kt = (int)(u % p.nk);
                const bool first = (i == 0) || (kt == 0);
                if (first && seg >= 2) {
                    if (!mbar_wait(&acc_empty[seg & 1], (uint32_t)((seg >> 1) - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const int slot = i % nst;
                if (!mbar_wait(&full[slot], (uint32_t)(i / nst) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)((seg & 1) * NPAD);
                const uint32_t a0 = smem_u32(smem + (size_t)slot * ST_BYTES);
                const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < KT / 16; ++kk)
                    tc_mma(d, sw128_desc(a0 + 32u * kk), sw128_desc(b0 + 32u * kk), idesc,
                           (first && kk == 0) ? 0u : 1u);
                tc_commit(&empty[slot]);
                if (i == n - 1 || kt == p.nk - 1) {
                    tc_commit(&acc_full[seg & 1]);
                    ++seg;
                }
            }
            if (!ok) {
                flags[0] = 1;
                set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
            }
            // every MMA this thread issued has completed before the CTA tears down
            tc_commit(fin);
            (void)mbar_wait(fin, 0u);
        }
    } else {
        // ------------------------------ epilogue (warps 0-3) ------------------------------
        pdl_wait();
        const bool aborted = *(volatile uint32_t*)&p.st.status[1] != 0u;
        const int t = threadIdx.x;  // 0..127 = accumulator lane = row within the tile
        if (t < NPAD) {
            float v = 1.0f;
            if (p.ss_in) {
                float ss = 0.f;
                for (int i = 0; i < p.ss_parts; ++i) ss += p.ss_in[(size_t)i * NPAD + t];
                v = 1.0f / sqrtf(ss / (float)p.K + p.eps);
            }
            inv[t] = v;
        }
        epi_bar();
        if (EPI == TE_HEAD) {
            // hidden state h = alpha * x * inv for this CTA's share of the columns (a
            // prefill: its last frame's, as stream seq_stream's)
            const int c0 = (int)((long long)c * p.D / G), c1 = (int)((long long)(c + 1) * p.D / G);
            for (int b = p.seq ? p.B - 1 : 0; b < p.B && !aborted; ++b) {
                const int bs = p.seq ? p.io->seq_stream : b, bo = p.seq ? 0 : b;
                for (int i = c0 + t; i < c1; i += 128) {
                    const float hv = p.x_resid[(size_t)b * p.D + i] * inv[b] *
                                     __uint_as_float((uint32_t)p.alpha[i] << 16);
                    if (p.h_internal) p.h_internal[(size_t)bs * p.D + i] = hv;
                    if (p.io->hidden) p.io->hidden[(size_t)bo * p.D + i] = hv;
                }
            }
        }
        if (n > 0) {
            const int m_first = (int)(w0 / p.nk), m_last = (int)((w1 - 1) / p.nk);
            int seg = 0;
            for (int m = m_first; m <= m_last; ++m, ++seg) {
                const int ks = (m == m_first) ? (int)(w0 % p.nk) : 0;
                const int ke = (m == m_last) ? (int)((w1 - 1) % p.nk) + 1 : p.nk;
                if (!mbar_wait(&acc_full[seg & 1], (uint32_t)(seg >> 1) & 1u)) {
                    flags[0] = 1;
                    set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                float v[NPAD];
                const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)((seg & 1) * NPAD);
#pragma unroll
                for (int q = 0; q < NPAD / 16; ++q) tmem_ld16(ta + 16u * q, v + 16 * q);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&acc_empty[seg & 1]);

                if (!(ks == 0 && ke == p.nk)) {
                    // tile cut between CTAs: deposit, and the last to arrive merges in slot order
                    const int cf = cta_of((long long)m * p.nk, U, G);
                    const int cl = cta_of((long long)m * p.nk + p.nk - 1, U, G);
                    const int nseg = cl - cf + 1;
                    float* pm_ = p.part + ((size_t)m * p.maxseg) * NPAD * 128;
                    float* mine = pm_ + (size_t)(c - cf) * NPAD * 128;
#pragma unroll
                    for (int b = 0; b < NPAD; ++b) mine[(size_t)b * 128 + t] = v[b];
                    __threadfence();
                    epi_bar();
                    if (t == 0) {
                        const uint32_t done = atomicAdd(&p.count[m], 1u);
                        flags[1] = (done == (uint32_t)nseg - 1u) ? 1 : 0;
                    }
                    epi_bar();
                    if (!flags[1]) continue;
                    __threadfence();
#pragma unroll
                    for (int b = 0; b < NPAD; ++b) v[b] = 0.f;
                    // partials summed in slot order; MSEG slots' loads are issued before any add
                    constexpr int MSEG = NPAD <= 16 ? 4 : (NPAD <= 32 ? 2 : 1);
                    for (int s0 = 0; s0 < nseg; s0 += MSEG) {
                        float tmp[MSEG][NPAD];
#pragma unroll
                        for (int j = 0; j < MSEG; ++j)
#pragma unroll
                            for (int b = 0; b < NPAD; ++b)
                                tmp[j][b] = (s0 + j < nseg) ? __ldcg(pm_ + ((size_t)(s0 + j) * NPAD + b) * 128 + t) : 0.f;
#pragma unroll
                        for (int j = 0; j < MSEG; ++j)
                            if (s0 + j < nseg)
#pragma unroll
                                for (int b = 0; b < NPAD; ++b) v[b] += tmp[j][b];
                    }
                    if (t == 0) p.count[m] = 0u;
                }
                // v[b] is the full dot product of row (tile m, lane t) with input row b
#pragma unroll
                for (int b = 0; b < NPAD; ++b) v[b] *= inv[b];

                // The per-frame epilogues run over frames in blocks of 16 in a rolled loop: a
                // straight-line body for all NPAD frames is tens of KB of code that each CTA
                // executes once, so nearly every instruction fetch missed.  Block k's values sit
                // in v[0..15] and the others move down 16 places after each block, which keeps
                // every index into v a compile-time constant (v stays in registers).
                if (EPI == TE_STORE) {
                    const int r = m * 128 + t;
                    if (!aborted && r < p.n_rows) {
#pragma unroll 1
                        for (int b0 = 0; b0 < p.B; b0 += 16) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (b0 + j < p.B) p.y[(size_t)(b0 + j) * p.y_stride + r] = v[j];
                            shift_block<NPAD>(v);
                        }
                    }
                } else if (EPI == TE_RESIDUAL) {
                    const int r = m * 128 + t;
                    const float an =
                        (!aborted && p.alpha_next) ? __uint_as_float((uint32_t)p.alpha_next[r] << 16) : 1.0f;
#pragma unroll 1
                    for (int b0 = 0; b0 < p.B; b0 += 16) {
                        float xr[16];  // 16 residual rows loaded before the first store
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            xr[j] = (!aborted && b0 + j < p.B) ? p.y[(size_t)(b0 + j) * p.y_stride + r] : 0.f;
                        float ss[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int b = b0 + j;
                            ss[j] = 0.f;
                            if (!aborted && b < p.B) {
                                const float xo = xr[j] + v[j];
                                p.y[(size_t)b * p.y_stride + r] = xo;
                                if (p.yb) p.yb[(size_t)b * p.yb_stride + r] = f32_to_bf16_rne(xo * an);
                                ss[j] = xo * xo;
                            }
                        }
                        // the warp's sums of the 16 frames' squares, lane l ending with frame (l >> 1) & 15
                        const float w = warp_sum16_transposed(ss, lane);
                        if ((lane & 1) == 0) xch[warp * NPAD + b0 + ((lane >> 1) & 15)] = w;
                        shift_block<NPAD>(v);
                    }
                    epi_bar();
                    if (t < NPAD && !aborted && p.ss_out)
                        p.ss_out[(size_t)m * NPAD + t] =
                            t < p.B ? xch[0 * NPAD + t] + xch[1 * NPAD + t] + xch[2 * NPAD + t] + xch[3 * NPAD + t]
                                    : 0.f;
                    epi_bar();
                } else if (EPI == TE_SWIGLU) {
                    // lanes 0-63: gate rows m*64 + t; lanes 64-127: value rows of the same j
                    if (t >= 64)
#pragma unroll
                        for (int b = 0; b < NPAD; ++b) xch[b * 64 + (t - 64)] = v[b];
                    epi_bar();
                    if (t < 64 && !aborted) {
                        const int jr = m * 64 + t;
#pragma unroll 1
                        for (int b0 = 0; b0 < p.B; b0 += 16) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int b = b0 + j;
                                if (b < p.B) {
                                    const float g = v[j], z = xch[b * 64 + t];
                                    p.yb[(size_t)b * p.yb_stride + jr] = f32_to_bf16_rne(g / (1.0f + expf(-g)) * z);
                                }
                            }
                            shift_block<NPAD>(v);
                        }
                    }
                    epi_bar();
                } else if (EPI == TE_QKV_ROPE) {
                    const int r = m * 128 + t;
                    const int sec = r / p.D;  // 0: q, 1: k, 2: v (a tile lies in one section)
                    const int idx = r - sec * p.D;
                    const int h = idx / p.dh, d = idx % p.dh;
                    auto none = [](int) { return 0; };
                    if (!aborted) {
                        if (sec == 0) {
                            float* dst = p.y + idx;
                            rope_frames<NPAD>(v, p, d, lane, none,
                                              [&](int b, float o, int) { dst[(size_t)b * p.y_stride] = o; });
                        } else if (p.seq) {
                            // a prefill's K/V stay out of the ring until its attention ran
                            uint16_t* dst = p.kv_new + (((size_t)(sec - 1) * p.B) * p.H + h) * p.dh + d;
                            const size_t st = (size_t)p.H * p.dh;
                            auto put = [&](int b, float o, int) { dst[(size_t)b * st] = f32_to_bf16_rne(o); };
                            if (sec == 1)
                                rope_frames<NPAD>(v, p, d, lane, none, put);
                            else
                                plain_frames<NPAD>(v, p.B, none, put);
                        } else {
                            // frame b is stream b, written to its ring slot pos[b] mod ctx
                            uint16_t* base = ((sec == 1) ? p.kc : p.vc) + (size_t)h * p.ctx * p.dh + d;
                            const size_t st = (size_t)p.H * p.ctx * p.dh;
                            auto slot = [&](int b) { return p.st.pos[b] % p.ctx; };
                            auto put = [&](int b, float o, int sl) {
                                base[(size_t)b * st + (size_t)sl * p.dh] = f32_to_bf16_rne(o);
                            };
                            if (sec == 1)
                                rope_frames<NPAD>(v, p, d, lane, slot, put);
                            else
                                plain_frames<NPAD>(v, p.B, slot, put);
                        }
                    }
                } else if (EPI == TE_HEAD) {
                    const int r = m * 128 + t;
                    float* out = p.io->logits;
                    // a prefill reports only its last frame, as stream seq_stream's
                    const int b_lo = p.seq ? p.B - 1 : 0;
                    const int s_seq = p.seq ? p.io->seq_stream : 0;
#pragma unroll 1
                    for (int b0 = 0; b0 < p.B; b0 += 16) {
                        if (b0 + 16 > b_lo) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int b = b0 + j;
                                unsigned long long key = 0ull;
                                if (b >= b_lo && b < p.B && r < p.n_rows) {
                                    const int bo = p.seq ? 0 : b, bs = p.seq ? s_seq : b;
                                    if (out && !aborted) out[(size_t)bo * p.n_rows + r] = v[j];
                                    if (p.logits_copy && !aborted) p.logits_copy[(size_t)bs * p.n_rows + r] = v[j];
                                    key = pack_argmax(v[j], (uint32_t)r);
                                }
#pragma unroll
                                for (int o = 16; o > 0; o >>= 1) key = umax64(key, __shfl_xor_sync(0xffffffffu, key, o));
                                if (lane == 0) red64[warp * NPAD + b] = key;
                            }
                        }
                        shift_block<NPAD>(v);
                    }
                    epi_bar();
                    if (t >= b_lo && t < p.B) {
                        unsigned long long k4 = umax64(umax64(red64[t], red64[NPAD + t]),
                                                       umax64(red64[2 * NPAD + t], red64[3 * NPAD + t]));
                        atomicMax(&p.st.amax[p.seq ? s_seq : t], k4);
                    }
                    __threadfence();
                    epi_bar();
                    if (t == 0) {
                        const uint32_t done = atomicAdd(&p.st.head_count[0], 1u);
                        flags[1] = (done == (uint32_t)p.n_mtiles - 1u) ? 1 : 0;
                    }
                    epi_bar();
                    if (flags[1]) {
                        __threadfence();
                        if (t >= b_lo && t < p.B) {
                            const int bs = p.seq ? s_seq : t;
                            const unsigned long long key = atomicExch(&p.st.amax[bs], 0ull);
                            const int32_t am = (int32_t)unpack_argmax_index(key);
                            if (!aborted) {
                                if (p.io->token) p.io->token[p.seq ? 0 : t] = am;
                                p.st.sel[(size_t)bs * PM_MAX_STREAMS_DEV + 0] = am;
                                p.st.pos[bs] += p.seq ? p.B : 1;
                            }
                        }
                        if (t == 0) p.st.head_count[0] = 0u;
                    }
                }
            }
        }
    }
    __syncthreads();
    if (flags[0] && threadIdx.x == 128) {
        // a wait ran out: let the copies already issued land before the CTA exits
        const int issued = flags[2];
        for (int i = issued - nst < 0 ? 0 : issued - nst; i < issued; ++i)
            (void)mbar_wait(&full[i % nst], (uint32_t)(i / nst) & 1u);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

template <int EPI, int NPAD>
cudaError_t launch_t(const CUtensorMap& A, const CUtensorMap& Bop, const CUtensorMap& N, const TcParams& p,
                     cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<EPI, NPAD>, A, Bop, N, p);
}

template <int NPAD>
cudaError_t launch_n(const CUtensorMap& A, const CUtensorMap& Bop, const CUtensorMap& N, const TcParams& p,
                     cudaStream_t s, bool pdl) {
    switch (p.epi) {
        case TE_STORE: return launch_t<TE_STORE, NPAD>(A, Bop, N, p, s, pdl);
        case TE_RESIDUAL: return launch_t<TE_RESIDUAL, NPAD>(A, Bop, N, p, s, pdl);
        case TE_SWIGLU: return launch_t<TE_SWIGLU, NPAD>(A, Bop, N, p, s, pdl);
        case TE_QKV_ROPE: return launch_t<TE_QKV_ROPE, NPAD>(A, Bop, N, p, s, pdl);
        case TE_HEAD: return launch_t<TE_HEAD, NPAD>(A, Bop, N, p, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

template <int NPAD>
cudaError_t prepare_n() {
    const int mx = 220 * 1024;
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<TE_STORE, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_tc<TE_RESIDUAL, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_tc<TE_SWIGLU, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_tc<TE_QKV_ROPE, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_tc<TE_HEAD, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
}

}  // namespace

namespace {

typedef void (*tc_kernel_t)(CUtensorMap, CUtensorMap, CUtensorMap, TcParams);

template <int NPAD>
tc_kernel_t kernel_n(int epi) {
    switch (epi) {
        case TE_STORE: return k_gemm_tc<TE_STORE, NPAD>;
        case TE_RESIDUAL: return k_gemm_tc<TE_RESIDUAL, NPAD>;
        case TE_SWIGLU: return k_gemm_tc<TE_SWIGLU, NPAD>;
        case TE_QKV_ROPE: return k_gemm_tc<TE_QKV_ROPE, NPAD>;
        case TE_HEAD: return k_gemm_tc<TE_HEAD, NPAD>;
        default: return nullptr;
    }
}

// CTAs of this kernel variant that fit on one SM at `smem` dynamic bytes (registers are
// allocated per warp in units of 256), at most PM_TC_CTAS_PER_SM
int resident_per_sm(int epi, int npad, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> memo;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, epi, npad, smem);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
    tc_kernel_t k = npad == 16 ? kernel_n<16>(epi) : npad == 32 ? kernel_n<32>(epi) : kernel_n<64>(epi);
    cudaFuncAttributes fa;
    int smem_sm = 0, reserved = 0, n = 1;
    if (k && cudaFuncGetAttributes(&fa, k) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess) {
        const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
        const int by_regs = 65536 / (6 * regs_warp);
        const int by_smem = smem_sm / (int)(smem + fa.sharedSizeBytes + reserved);
        n = by_regs < by_smem ? by_regs : by_smem;
    } else {
        cudaGetLastError();
    }
    if (n > PM_TC_CTAS_PER_SM) n = PM_TC_CTAS_PER_SM;
    if (n < 1) n = 1;
    memo[key] = n;
    return n;
}

}  // namespace

bool plan_tc(TcParams& p, int num_sms) {
    if (p.K <= 0 || p.K % KT != 0 || p.n_mtiles <= 0) return false;
    if (!(p.npad == 16 || p.npad == 32 || p.npad == 64) || p.B < 1 || p.B > p.npad) return false;
    p.nk = p.K / KT;
    const long long U = (long long)p.n_mtiles * p.nk;
    const int min_units = p.min_units > 0 ? p.min_units : PM_TC_MIN_UNITS;
    const uint32_t st_bytes = A_BYTES + (uint32_t)p.npad * 128u;
    p.nst = (int)((PM_TC_RING_BYTES) / st_bytes);
    if (p.nst < 2) p.nst = 2;
    const size_t smem = 1024 + (size_t)p.nst * st_bytes + 8u * (2 * p.nst + 5) + 16 + 16 + 4u * p.npad +
                        4u * p.npad * 64 + 8u * 4 * p.npad;
    // one wave: as many CTAs as fit on the GPU at once
    int G = resident_per_sm(p.epi, p.npad, smem) * num_sms;
    if ((long long)G * min_units > U) G = (int)((U + min_units - 1) / min_units);
    if (G < 1) G = 1;
    p.grid = G;
    int maxseg = 1;
    for (int m = 0; m < p.n_mtiles; ++m) {
        const int cf = cta_of((long long)m * p.nk, U, G), cl = cta_of((long long)m * p.nk + p.nk - 1, U, G);
        if (cl - cf + 1 > maxseg) maxseg = cl - cf + 1;
    }
    p.maxseg = maxseg;
    p.smem = smem;
    return p.smem <= 220u * 1024u;
}

cudaError_t launch_tc(const CUtensorMap& A, const CUtensorMap& Bop, const CUtensorMap& next, const TcParams& p,
                      cudaStream_t s, bool pdl) {
    switch (p.npad) {
        case 16: return launch_n<16>(A, Bop, next, p, s, pdl);
        case 32: return launch_n<32>(A, Bop, next, p, s, pdl);
        case 64: return launch_n<64>(A, Bop, next, p, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc_prepare() {
    cudaError_t e = prepare_n<16>();
    if (e == cudaSuccess) e = prepare_n<32>();
    if (e == cudaSuccess) e = prepare_n<64>();
    return e;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    typedef CUresult (*encode_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static encode_fn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f) {
            cudaGetLastError();
            return false;
        }
        fn = reinterpret_cast<encode_fn>(f);
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15u) || (inner * 2) % 16 != 0) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pm
