// Batched decode projections (2 <= B <= 16) as a weight-streaming GEMV whose inner products
// run on warp-level tensor-core MMAs (mma.sync m16n8k16: bf16 operands, fp32 accumulate).
//
// y[b][r] = sum_k W[r][k] x[b][k] for every projection of the temporal block and the text
// head ("PersonaPlex native LM audit", sections 3 and 5), for up to 16 conversations in one
// pass over the weights.  At this batch a projection is still HBM-bound (<= 32 flops per
// weight byte), so the kernel is laid out like the batch-1 GEMV, not like a GEMM:
//  * CTA c owns a contiguous, balanced range of output rows (row pairs where the epilogue
//    needs two rows together) over the whole K, so no partial sum ever leaves its CTA and
//    nothing is merged across CTAs;
//  * the CTA's rows form 16-row tiles; a stage is one tile x 512 k elements: 1 KB of each
//    row, fetched by ONE 3-D tensor copy (the weight matrix viewed as rows x (K/256) x 256,
//    box 16 x 2 x 256; SwiGLU: 8 gate rows and 8 value rows, two copies) with L2
//    evict-first.  A CTA's last tile uses a map whose box height is its remainder (two
//    remainders: the balanced split gives two row counts), so no byte outside the CTA's
//    rows is read.  Few large requests with 1 KB contiguous per row keep both the copy
//    engine and the DRAM pages efficient (one request per 1 KB row segment, or boxes only
//    128-256 B wide, each cap the stream well below the HBM rate).  Stages go through a
//    ring in k-chunk-major order, the first ring issued before griddepcontrol.wait;
//  * consumer warp w takes the 32-element k pieces w, w+4, w+8, w+12 of every chunk.  The
//    weight tile is the MMA's A operand (16 rows), the batch its B operand (8 columns; a
//    second MMA for rows 8..15).  Inside a piece the k order is permuted the same way on
//    both operands, so every fragment is one 16-byte load: thread (g, t) holds elements
//    8t..8t+7 of its rows, the first MMA takes elements {0,1 | 2,3} of each group as its
//    k pairs {2t | 2t+8}, the second MMA elements {4,5 | 6,7};
//  * after the previous kernel, one warp streams the activation chunks (one box of the bf16
//    operand per chunk, L2 evict-last: every CTA reads them) into a second ring, and another
//    sums the input's RMSNorm partials and stages the epilogue operands, both off the
//    MMA path (under a saturated memory system each of those loads takes microseconds);
//    consumers hold a chunk's activation fragments in registers across its tiles and the
//    accumulators of all the CTA's tiles across chunks;
//  * the 4 warps' partial sums meet once in shared memory, then the fused epilogue
//    (RMSNorm scale of the input, residual + the next norm's bf16 operand and the sum of
//    squares, SwiGLU, RoPE + KV-ring append, or the text head's logits and argmax) runs
//    one batch row per warp.
#include <math.h>

#include <string.h>

#include "pm_kernels.h"
#include "tc_common.cuh"

// Tiling policy: weight stages in the ring (8-column and 16-column variants), resident
// CTAs per SM.
#ifndef PM_MG_NST8
#define PM_MG_NST8 4
#endif
#ifndef PM_MG_NST16
#define PM_MG_NST16 4
#endif
#ifndef PM_MG_CTAS_PER_SM
#define PM_MG_CTAS_PER_SM 2
#endif

namespace pm {
namespace {

constexpr int CW = 4;                   // consumer warps
constexpr int KC = 512;                 // k elements per chunk (one stage row segment)
constexpr int PIECE = 32;               // k elements per warp piece (two MMAs)
constexpr int PPW = KC / PIECE / CW;    // pieces per warp per chunk
constexpr int SLOT = KC * 2;            // bytes per staged row (dense: the tensor copy's box)
constexpr int STAGE = 16 * SLOT;        // one 16-row weight tile x one chunk
constexpr int MAXT = PM_MG_MAX_TILES;   // 16-row tiles per CTA (text head)
constexpr int LO = 16;                  // row of the operand buffers where the remainder plane starts
constexpr int NPX = 16;                 // batch rows of the operand buffers
constexpr int THREADS = 32 * (CW + 3);  // consumers, weight producer, activation producer, prologue

enum RowMode { M_ROW = 0, M_ADJ = 1, M_SPLIT = 2 };

// 16-row tiles a CTA holds accumulators for, per epilogue and batch width (the full shapes'
// rows per CTA at one wave of 2 CTAs per SM: text head 7, SwiGLU 5 gate/value tile pairs,
// fused QKV 3, W_O / linear_out 1), so registers are sized for what each projection needs.
// At 16 columns the text head's 7 tiles and both operand planes would not fit the
// register budget: it takes 5 and a second half wave of CTAs.
__host__ __device__ constexpr int maxt_of(int epi, int nb) {
    return epi == TE_HEAD ? (nb == 8 ? MAXT : 5) : (epi == TE_SWIGLU ? 5 : (epi == TE_QKV_ROPE ? 3 : 2));
}

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }
// consumers + the prologue warp: the epilogue operands are in place
__device__ __forceinline__ void pbar() { asm volatile("bar.sync 2, %0;" ::"n"((CW + 1) * 32) : "memory"); }

// 3-D tensor copy of the box at (x0, x1, x2), completing on `bar`
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x0, int x1, int x2, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte shared-memory load through a 32-bit shared-window address
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NB>
struct MgLayout {
    static constexpr int NST = NB == 8 ? PM_MG_NST8 : PM_MG_NST16;
    // activation chunks in flight: two at 8 columns, so a CTA with few tiles (W_O,
    // linear_out) does not wait out each chunk's load; at 16 columns the second slot would
    // cost a weight stage the ring cannot spare at two CTAs per SM
    static constexpr int XST = NB == 8 ? 2 : 1;
    // one activation chunk: NB rows x 512 elements of the bf16 operand, then NB rows of its
    // rounding remainder
    static constexpr int XSLOT = 2 * NB * SLOT;
    static constexpr size_t FIXED = 128u + (size_t)NST * STAGE + (size_t)XST * XSLOT + 8u * (2 * NST + 2 * XST) +
                                    4u * NPX + 4u * NPX + 4u * 4;
};

template <int EPI, int NB>
__global__ void __launch_bounds__(THREADS, PM_MG_CTAS_PER_SM)
    k_gemv_mma(const __grid_constant__ CUtensorMap tmF, const __grid_constant__ CUtensorMap tmR0,
               const __grid_constant__ CUtensorMap tmR1, const __grid_constant__ CUtensorMap tmX, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    // tensor copies land on 128-byte boundaries
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
    constexpr int MODE = EPI == TE_SWIGLU ? M_SPLIT : (EPI == TE_QKV_ROPE ? M_ADJ : M_ROW);
    constexpr int RPU = MODE == M_ROW ? 1 : 2;
    constexpr int NST = MgLayout<NB>::NST;
    constexpr int XSLOT = MgLayout<NB>::XSLOT;
    constexpr int XST = MgLayout<NB>::XST;
    constexpr int MT = maxt_of(EPI, NB);
    uint8_t* ring = smem;
    uint8_t* xring = smem + (size_t)NST * STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(xring + (size_t)XST * XSLOT);
    uint64_t* empty = full + NST;
    uint64_t* xfull = empty + NST;
    uint64_t* xempty = xfull + XST;
    float* inv = reinterpret_cast<float*>(xempty + XST);  // [NPX]
    int* pslot = reinterpret_cast<int*>(inv + NPX);        // [NPX] KV-ring slot per stream
    int* flags = pslot + NPX;  // [0] timeout, [1] last CTA, [2] weight stages issued, [3] chunks issued
    float* pre = reinterpret_cast<float*>(flags + 4);      // epilogue operands (p.pre_stride per row)

    const int G = p.grid, c = blockIdx.x;
    const int n_units = MODE == M_SPLIT ? p.split_rows : p.n_rows / RPU;
    const int u0 = (int)((long long)c * n_units / G), u1 = (int)((long long)(c + 1) * n_units / G);
    const int nu = u1 - u0;
    const int nr = MODE == M_SPLIT ? nu : nu * RPU;  // outputs per batch row (SwiGLU: pairs)
    const int ntiles = MODE == M_SPLIT ? (nu + 7) / 8 : (nr + 15) / 16;
    const int K = p.K;
    const int nch = (K + KC - 1) / KC;
    const int nstages = ntiles * nch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ps = p.pre_stride;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int s = 0; s < XST; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], CW);
        }
        fence_barrier_init();
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        flags[3] = 0;
    }
    __syncthreads();
    pdl_trigger();

    if (warp == CW) {
        // ------------------------------ weight producer ------------------------------
        if (lane == 0 && nstages > 0) {
            const uint64_t pol = l2_evict_first_policy();
            // rows of the CTA's last tile, and the map whose box has that height
            const int tile_rows = MODE == M_SPLIT ? 8 : 16;
            const int last_rows = (MODE == M_SPLIT ? nu : nr) - tile_rows * (ntiles - 1);
            const CUtensorMap* tm_last = last_rows == tile_rows ? &tmF : (nu == p.h0 ? &tmR0 : &tmR1);
            for (int k = 0; k < nstages; ++k) {
                const int slot = k % NST;
                if (k >= NST && !mbar_wait(&empty[slot], (uint32_t)((k / NST) - 1) & 1u)) {
                    flags[0] = 1;
                    set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
                    break;
                }
                const int ch = k / ntiles, i = k % ntiles;
                const bool last = i == ntiles - 1;
                const CUtensorMap* tm = last ? tm_last : &tmF;
                const uint32_t rows = (uint32_t)(last ? last_rows : tile_rows);
                uint8_t* dst = ring + (size_t)slot * STAGE;
                if (MODE == M_SPLIT) {
                    mbar_arrive_expect_tx(&full[slot], 2u * rows * (uint32_t)SLOT);
                    tma_load_3d(dst, tm, 0, 2 * ch, u0 + 8 * i, &full[slot], pol);
                    tma_load_3d(dst + 8 * SLOT, tm, 0, 2 * ch, p.split_rows + u0 + 8 * i, &full[slot], pol);
                } else {
                    mbar_arrive_expect_tx(&full[slot], rows * (uint32_t)SLOT);
                    tma_load_3d(dst, tm, 0, 2 * ch, u0 * RPU + 16 * i, &full[slot], pol);
                }
                flags[2] = k + 1;
            }
        }
    } else if (warp == CW + 1) {
        // ------------------------------ activation producer ------------------------------
        if (lane == 0 && ntiles > 0) {
            pdl_wait();
            const uint64_t pol = l2_evict_last_policy();
            for (int ch = 0; ch < nch; ++ch) {
                const int slot = ch % XST;
                if (ch >= XST && !mbar_wait(&xempty[slot], (uint32_t)((ch / XST) - 1) & 1u)) {
                    flags[0] = 1;
                    set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&xfull[slot], (uint32_t)XSLOT);
                tma_load_3d(xring + (size_t)slot * XSLOT, &tmX, 0, 2 * ch, 0, &xfull[slot], pol);
                tma_load_3d(xring + (size_t)slot * XSLOT + NB * SLOT, &tmX, 0, 2 * ch, LO, &xfull[slot], pol);
                flags[3] = ch + 1;
            }
        }
    } else if (warp == CW + 2) {
        // ------------- prologue: input norm and epilogue operands, off the MMA path -------------
        pdl_wait();
        // RMSNorm of the input rows (folded: the operand is bf16(alpha * x); the sums of
        // squares arrive as per-CTA partials of the producing kernel), 16 loads in flight per lane
        {
            float ssb[NPX];
#pragma unroll
            for (int b = 0; b < NPX; ++b) ssb[b] = 0.f;
            if (p.ss_in) {
                for (int i0 = 0; i0 < p.ss_parts; i0 += 4 * 32) {
                    float4 v[4][NPX / 4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = i0 + 32 * j + lane;
#pragma unroll
                        for (int q = 0; q < NPX / 4; ++q)
                            v[j][q] = i < p.ss_parts ? __ldcg(reinterpret_cast<const float4*>(p.ss_in + (size_t)i * NPX) + q)
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < NPX / 4; ++q) {
                            ssb[4 * q + 0] += v[j][q].x;
                            ssb[4 * q + 1] += v[j][q].y;
                            ssb[4 * q + 2] += v[j][q].z;
                            ssb[4 * q + 3] += v[j][q].w;
                        }
                }
            }
#pragma unroll
            for (int b = 0; b < NPX; ++b) {
                const float tot = warp_sum(ssb[b]);
                if (lane == 0) inv[b] = p.ss_in ? 1.0f / sqrtf(tot / (float)K + p.eps) : 1.0f;
            }
            __syncwarp();
        }
        // operands: loads of 4 batch rows in flight before their stores
        if (EPI == TE_RESIDUAL) {
            for (int q = lane; q < nr; q += 32)
                pre[NPX * ps + q] = p.alpha_next ? __uint_as_float((uint32_t)p.alpha_next[u0 + q] << 16) : 1.0f;
            for (int q = lane; q < nr; q += 32) {
                for (int b0 = 0; b0 < p.B; b0 += 4) {
                    float v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[j] = b0 + j < p.B ? __ldcg(p.y + (size_t)(b0 + j) * p.y_stride + u0 + q) : 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (b0 + j < p.B) pre[(b0 + j) * ps + q] = v[j];
                }
            }
        } else if (EPI == TE_QKV_ROPE) {
            float2* cs = reinterpret_cast<float2*>(pre);
            for (int q = lane; q < nr; q += 32) {
                const int r = 2 * u0 + q;
                const int sec = r / p.D, d = (r - sec * p.D) % p.dh;
                for (int b0 = 0; b0 < p.B; b0 += 4) {
                    float2 v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[j] = (sec < 2 && b0 + j < p.B) ? p.rope_tab[(size_t)(b0 + j) * (p.dh / 2) + (d >> 1)]
                                                         : make_float2(1.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (b0 + j < p.B) cs[(b0 + j) * ps + q] = v[j];
                }
            }
            if (lane < p.B) pslot[lane] = p.st.pos[lane] % p.ctx;
        } else if (EPI == TE_HEAD) {
            // hidden state h = alpha * x * inv for this CTA's share of the columns
            const bool aborted = *(volatile uint32_t*)&p.st.status[1] != 0u;
            const int c0 = (int)((long long)c * p.D / G), c1 = (int)((long long)(c + 1) * p.D / G);
            for (int b = 0; b < p.B && !aborted; ++b) {
                for (int i = c0 + lane; i < c1; i += 32) {
                    const float hv = p.x_resid[(size_t)b * p.D + i] * inv[b] *
                                     __uint_as_float((uint32_t)p.alpha[i] << 16);
                    if (p.h_internal) p.h_internal[(size_t)b * p.D + i] = hv;
                    if (p.io->hidden) p.io->hidden[(size_t)b * p.D + i] = hv;
                }
            }
        }
        __syncwarp();
        pbar();
    } else {
        // ------------------------------ consumers ------------------------------
        const int g = lane >> 2, t = lane & 3;
        float acc[MT][NB / 8][4];
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int nb = 0; nb < NB / 8; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][nb][e] = 0.f;

        bool ok = true;
        int k = 0;
        for (int ch = 0; ch < nch && ok && ntiles > 0; ++ch) {
            const int len = min(KC, K - ch * KC);
            // this chunk's activation fragments, kept in registers across its tiles
            const int xs = ch % XST;
            if (!mbar_wait(&xfull[xs], (uint32_t)(ch / XST) & 1u)) {
                ok = false;
                break;
            }
            // bf16 operand (hi) and its rounding remainder (lo): hi + lo carries the fp32
            // activation to ~16 significant bits, so the products lose no more than fp32
            uint4 xf[PPW][NB / 8], xl[PPW][NB / 8];
            const uint32_t xa = smem_u32(xring) + (uint32_t)(xs * XSLOT + g * SLOT + (warp * PIECE + 8 * t) * 2);
#pragma unroll
            for (int j = 0; j < PPW; ++j) {
                const int pc = warp + CW * j;
#pragma unroll
                for (int nb = 0; nb < NB / 8; ++nb) {
                    const uint32_t a = xa + (uint32_t)(nb * 8 * SLOT + j * CW * PIECE * 2);
                    xf[j][nb] = pc * PIECE < len ? lds128(a) : make_uint4(0u, 0u, 0u, 0u);
                    xl[j][nb] = pc * PIECE < len ? lds128(a + NB * SLOT) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // the slot is refilled by the async proxy (bulk copy): order these generic-proxy
            // reads before that write
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&xempty[xs]);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (i < ntiles) {
                    const int slot = k % NST;
                    if (!mbar_wait(&full[slot], (uint32_t)(k / NST) & 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_u32(ring) + (uint32_t)(slot * STAGE + g * SLOT + (warp * PIECE + 8 * t) * 2);
#pragma unroll
                    for (int j = 0; j < PPW; ++j) {
                        const int pc = warp + CW * j;
                        if (pc * PIECE < len) {
                            const uint4 wa = lds128(sa + (uint32_t)(j * CW * PIECE * 2));
                            const uint4 wb = lds128(sa + (uint32_t)(8 * SLOT + j * CW * PIECE * 2));
#pragma unroll
                            for (int nb = 0; nb < NB / 8; ++nb) {
                                mma_bf16(acc[i][nb], wa.x, wb.x, wa.y, wb.y, xf[j][nb].x, xf[j][nb].y);
                                mma_bf16(acc[i][nb], wa.z, wb.z, wa.w, wb.w, xf[j][nb].z, xf[j][nb].w);
                                mma_bf16(acc[i][nb], wa.x, wb.x, wa.y, wb.y, xl[j][nb].x, xl[j][nb].y);
                                mma_bf16(acc[i][nb], wa.z, wb.z, wa.w, wb.w, xl[j][nb].z, xl[j][nb].w);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    ++k;
                }
            }
        }
        if (!ok) {
            flags[0] = 1;
            set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
        }
        pbar();  // every consumer is done with the ring; the prologue's operands are in place
        const bool aborted = *(volatile uint32_t*)&p.st.status[1] != 0u;
        float* scr = reinterpret_cast<float*>(ring);  // [CW][MT][16 slots][16 batch]
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            if (i < ntiles) {
                float* o = scr + (size_t)(warp * MT + i) * 256;
#pragma unroll
                for (int nb = 0; nb < NB / 8; ++nb) {
                    o[g * 16 + nb * 8 + 2 * t] = acc[i][nb][0];
                    o[g * 16 + nb * 8 + 2 * t + 1] = acc[i][nb][1];
                    o[(g + 8) * 16 + nb * 8 + 2 * t] = acc[i][nb][2];
                    o[(g + 8) * 16 + nb * 8 + 2 * t + 1] = acc[i][nb][3];
                }
            }
        }
        cbar();
        // y[i][slot][b] = inv[b] * (sum of the warps' partials), in warp order, in place of warp 0's
        for (int e = threadIdx.x; e < ntiles * 256; e += 32 * CW) {
            const int i = e >> 8, rem = e & 255;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < CW; ++w) v += scr[(size_t)(w * MT + i) * 256 + rem];
            scr[(size_t)i * 256 + rem] = v * inv[rem & 15];
        }
        cbar();
        const float* yt = scr;

        if (EPI == TE_RESIDUAL) {
            for (int b = warp; b < p.npad; b += CW) {
                float ss = 0.f;
                if (b < p.B && !aborted) {
                    for (int q = lane; q < nr; q += 32) {
                        const int r = u0 + q;
                        const float xo = pre[b * ps + q] + yt[(q >> 4) * 256 + (q & 15) * 16 + b];
                        p.y[(size_t)b * p.y_stride + r] = xo;
                        if (p.yb) {
                            const float v = xo * pre[NPX * ps + q];
                            const uint16_t hi = f32_to_bf16_rne(v);
                            p.yb[(size_t)b * p.yb_stride + r] = hi;
                            if (p.yb_lo_rows) p.yb[((size_t)b + p.yb_lo_rows) * p.yb_stride + r] = bf16_lo_part(v, hi);
                        }
                        ss = fmaf(xo, xo, ss);
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0 && p.ss_out && !aborted) p.ss_out[(size_t)c * p.npad + b] = ss;
            }
        } else if (EPI == TE_SWIGLU) {
            for (int b = warp; b < p.B && !aborted; b += CW) {
                for (int q = lane; q < nu; q += 32) {
                    const float gt = yt[(q >> 3) * 256 + (q & 7) * 16 + b];
                    const float z = yt[(q >> 3) * 256 + (8 + (q & 7)) * 16 + b];
                    const float v = gt / (1.0f + expf(-gt)) * z;
                    const uint16_t hi = f32_to_bf16_rne(v);
                    p.yb[(size_t)b * p.yb_stride + u0 + q] = hi;
                    if (p.yb_lo_rows) p.yb[((size_t)b + p.yb_lo_rows) * p.yb_stride + u0 + q] = bf16_lo_part(v, hi);
                }
            }
        } else if (EPI == TE_QKV_ROPE) {
            const float2* cs = reinterpret_cast<const float2*>(pre);
            for (int b = warp; b < p.B && !aborted; b += CW) {
                const int ring_slot = pslot[b];
                for (int q = lane; q < nr; q += 32) {
                    const int r = 2 * u0 + q;
                    const int sec = r / p.D, idx = r - sec * p.D;
                    const int h = idx / p.dh, d = idx % p.dh;
                    const float mine = yt[(q >> 4) * 256 + (q & 15) * 16 + b];
                    const float other = yt[((q ^ 1) >> 4) * 256 + ((q ^ 1) & 15) * 16 + b];
                    float o = mine;
                    if (sec < 2) {
                        const float2 f = cs[b * ps + q];
                        o = (d & 1) == 0 ? (mine * f.x - other * f.y) : (other * f.y + mine * f.x);
                    }
                    if (sec == 0) {
                        p.y[(size_t)b * p.y_stride + idx] = o;
                    } else {
                        uint16_t* cache = (sec == 1) ? p.kc : p.vc;
                        cache[(((size_t)b * p.H + h) * p.ctx + ring_slot) * p.dh + d] = f32_to_bf16_rne(o);
                    }
                }
            }
        } else if (EPI == TE_HEAD) {
            float* out = p.io->logits;
            for (int b = warp; b < p.B; b += CW) {
                unsigned long long key = 0ull;
                for (int q = lane; q < nr; q += 32) {
                    const int r = u0 + q;
                    const float v = yt[(q >> 4) * 256 + (q & 15) * 16 + b];
                    if (out && !aborted) out[(size_t)b * p.n_rows + r] = v;
                    if (p.logits_copy && !aborted) p.logits_copy[(size_t)b * p.n_rows + r] = v;
                    key = umax64(key, pack_argmax(v, (uint32_t)r));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) key = umax64(key, __shfl_xor_sync(0xffffffffu, key, o));
                if (lane == 0 && key != 0ull) atomicMax(&p.st.amax[b], key);
            }
            __threadfence();
            cbar();
            if (threadIdx.x == 0) {
                const uint32_t done = atomicAdd(&p.st.head_count[0], 1u);
                flags[1] = (done == (uint32_t)G - 1u) ? 1 : 0;
            }
            cbar();
            if (flags[1]) {
                __threadfence();
                if (threadIdx.x < p.B) {
                    const int b = threadIdx.x;
                    const unsigned long long key = atomicExch(&p.st.amax[b], 0ull);
                    const int32_t am = (int32_t)unpack_argmax_index(key);
                    if (!aborted) {
                        if (p.io->token) p.io->token[b] = am;
                        p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 0] = am;
                        p.st.pos[b] += 1;
                    }
                }
                if (threadIdx.x == 0) p.st.head_count[0] = 0u;
            }
        }
    }
    __syncthreads();
    if (flags[0] && threadIdx.x == 32 * CW) {
        // a wait ran out: let the copies already issued land before the CTA exits
        const int issued = flags[2];
        for (int i = issued - NST < 0 ? 0 : issued - NST; i < issued; ++i)
            (void)mbar_wait(&full[i % NST], (uint32_t)(i / NST) & 1u);
        const int xi = flags[3];
        for (int i = xi - XST < 0 ? 0 : xi - XST; i < xi; ++i)
            (void)mbar_wait(&xfull[i % XST], (uint32_t)(i / XST) & 1u);
    }
}

template <int EPI, int NB>
cudaError_t launch_e(const CUtensorMap* m, const TcParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemv_mma<EPI, NB>, m[0], m[1], m[2], m[3], p);
}

template <int NB>
cudaError_t launch_nb(const CUtensorMap* m, const TcParams& p, cudaStream_t s, bool pdl) {
    switch (p.epi) {
        case TE_RESIDUAL: return launch_e<TE_RESIDUAL, NB>(m, p, s, pdl);
        case TE_SWIGLU: return launch_e<TE_SWIGLU, NB>(m, p, s, pdl);
        case TE_QKV_ROPE: return launch_e<TE_QKV_ROPE, NB>(m, p, s, pdl);
        case TE_HEAD: return launch_e<TE_HEAD, NB>(m, p, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

template <int NB>
cudaError_t prepare_nb() {
    const int mx = 220 * 1024;
    cudaError_t e = cudaFuncSetAttribute(k_gemv_mma<TE_RESIDUAL, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemv_mma<TE_SWIGLU, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemv_mma<TE_QKV_ROPE, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemv_mma<TE_HEAD, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
}

// bf16 matrix [rows][K] viewed as rows x (K / 256) x 256, box 256 x 2 x box_rows (512
// elements of box_rows rows: 1 KB of each row), no swizzle
bool make_tmap_rows(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
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
    if ((reinterpret_cast<uintptr_t>(base) & 15u) || K % 256 != 0 || box_rows < 1 || box_rows > 256) return false;
    const cuuint64_t dims[3] = {256, K / 256, rows};
    const cuuint64_t strides[2] = {512, K * 2};
    const cuuint32_t box[3] = {256, 2, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool plan_mg(TcParams& p, int num_sms) {
    if (p.B < 1 || p.B > NPX || p.npad != NPX || p.K < 256 || p.K % 256 != 0) return false;
    if (!(p.epi == TE_RESIDUAL || p.epi == TE_SWIGLU || p.epi == TE_QKV_ROPE || p.epi == TE_HEAD)) return false;
    if (p.epi == TE_QKV_ROPE && (p.n_rows % 2 != 0 || p.dh % 2 != 0)) return false;
    const int mode = p.epi == TE_SWIGLU ? M_SPLIT : (p.epi == TE_QKV_ROPE ? M_ADJ : M_ROW);
    const long long n_units = mode == M_SPLIT ? p.split_rows : (mode == M_ADJ ? p.n_rows / 2 : p.n_rows);
    if (n_units <= 0) return false;
    // one wave of PM_MG_CTAS_PER_SM CTAs per SM, more only if a CTA's rows overflow its tiles
    long long G = (long long)PM_MG_CTAS_PER_SM * num_sms;
    if (G > n_units) G = n_units;
    long long umax = 0;
    for (;;) {
        umax = (n_units + G - 1) / G;
        const long long tiles = mode == M_SPLIT ? (umax + 7) / 8 : (umax * (mode == M_ADJ ? 2 : 1) + 15) / 16;
        if (tiles <= maxt_of(p.epi, p.B <= 8 ? 8 : 16)) break;
        G += num_sms;
    }
    p.grid = (int)G;
    p.h0 = (int)(n_units / G);  // the two unit counts of a balanced split: h0 and h0 + 1
    // epilogue operands staged by the prologue warp: rows of outputs per CTA
    const int nr_max = (int)(mode == M_ADJ ? 2 * umax : umax);
    p.pre_stride = (nr_max + 3) & ~3;
    size_t pre_floats = 0;
    if (p.epi == TE_RESIDUAL) pre_floats = (size_t)(NPX + 1) * p.pre_stride;
    if (p.epi == TE_QKV_ROPE) pre_floats = (size_t)2 * NPX * p.pre_stride;
    const bool nb8 = p.B <= 8;
    p.nst = nb8 ? MgLayout<8>::NST : MgLayout<16>::NST;
    p.smem = (nb8 ? MgLayout<8>::FIXED : MgLayout<16>::FIXED) + 4u * pre_floats;
    // the reduction scratch reuses the weight ring
    if ((size_t)CW * MAXT * 256 * 4 > (size_t)p.nst * STAGE) return false;
    return p.smem <= 110u * 1024u;
}

bool mg_tensor_maps(const TcParams& p, const uint16_t* w, uint64_t w_rows, const uint16_t* xop, CUtensorMap* m) {
    const int mode = p.epi == TE_SWIGLU ? M_SPLIT : (p.epi == TE_QKV_ROPE ? M_ADJ : M_ROW);
    const int rpu = mode == M_ADJ ? 2 : 1, tile_rows = mode == M_SPLIT ? 8 : 16;
    // remainder rows of the last tile for CTAs of h0 and h0 + 1 units (0: a full tile)
    const int r0 = (p.h0 * rpu) % tile_rows, r1 = ((p.h0 + 1) * rpu) % tile_rows;
    if (!make_tmap_rows(&m[0], w, (uint64_t)p.K, w_rows, (uint32_t)tile_rows)) return false;
    if (!make_tmap_rows(&m[1], w, (uint64_t)p.K, w_rows, (uint32_t)(r0 ? r0 : tile_rows))) return false;
    if (!make_tmap_rows(&m[2], w, (uint64_t)p.K, w_rows, (uint32_t)(r1 ? r1 : tile_rows))) return false;
    // the operand's rows and, LO rows further, its rounding remainder
    return make_tmap_rows(&m[3], xop, (uint64_t)p.K, LO + NPX, p.B <= 8 ? 8u : 16u);
}

cudaError_t launch_mg(const CUtensorMap* m, const TcParams& p, cudaStream_t s, bool pdl) {
    return p.B <= 8 ? launch_nb<8>(m, p, s, pdl) : launch_nb<16>(m, p, s, pdl);
}

cudaError_t mg_prepare() {
    cudaError_t e = prepare_nb<8>();
    if (e == cudaSuccess) e = prepare_nb<16>();
    return e;
}

}  // namespace pm
