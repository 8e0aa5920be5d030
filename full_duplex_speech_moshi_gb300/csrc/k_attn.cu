// Split-KV (flash-decoding) causal decode attention over the temporal KV ring
// ("PersonaPlex native LM audit", section 3: 32 query / key / value heads of width 128,
// keys allowed where 0 <= query_position - key_position < 3000; section 6: the cache
// holds keys after RoPE, values without).
//
// For batch row b at position p the visible keys are positions max(0, p-win+1) .. p,
// stored at ring slots position mod ctx (win = ctx for the declared mask, ctx - 1 for the
// pinned ring's labels, which hide the oldest key of a full ring).  A unit is the 64 keys
// lo + 64c .. lo + 64c + 63 of row b's window for head h.  Two ways to share them out,
// both derived on the device from the positions so a captured graph serves any cache
// length: when the batch's heads fit one wave, each head gets a cluster of CS CTAs
// (CS = 8 at B = 1, 4 at B = 2, 2 at B = 4, 1 at B = 8), each taking a contiguous share of
// the head's units, and the pieces meet in the leader CTA's shared memory through
// distributed shared memory and a cluster barrier (no global round trip); otherwise the
// units of all rows, ordered (row, head, chunk), are split into one contiguous, balanced
// range per CTA (ragged and large batches).
//
// The kernel streams K/V like the projections stream weights:
//  * a producer thread copies each unit's K rows and V rows (16 KB each, contiguous
//    ring slots; two copies where the chunk wraps) into a ring of 32 KB shared-memory
//    stages with 1-D bulk copies.  Every key but the current position was written by
//    earlier frames, so the first ring is issued before griddepcontrol.wait and overlaps
//    the fused-QKV kernel that is still writing the current K/V and the query;
//  * four consumer warps take a unit at a time: the current position's K/V row (written by
//    the kernel this one waited for) is loaded into its slot after the wait; scores with
//    128 / KPC x 2 lanes per key (reads staggered across the 16-byte columns of a row so a
//    key's lanes touch distinct banks), the base-2 exponential with the query
//    pre-scaled by log2(e)/sqrt(128) (the same softmax).  Where a CTA streams many units
//    each warp keeps its own running max / sum / weighted values over its 16 keys of every
//    unit (no barrier per unit; the warps' states merge once per piece); with few units
//    per CTA one running state spans the four warps (thread t owns coordinate t);
//  * the issuing thread walks its units incrementally (no division per unit): its work
//    between a stage coming free and the refill being issued is on every stage's cycle;
//  * a head whose units all fall in one CTA is written out directly; in the balanced split a
//    head cut between CTAs leaves one partial (weighted values, max, sum) per piece in
//    global memory and the CTA that finishes last merges them in piece order (completion
//    counter, nothing waits);
//  * stages are handed back to the copy engine after a proxy fence (generic-proxy reads
//    before the async-proxy refill).
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int DH = 128;
#ifndef PM_ATTN_KPC
#define PM_ATTN_KPC 64
#endif
constexpr int KPC = PM_ATTN_KPC;            // keys per unit (64: the per-warp softmax takes 16 keys per warp)
constexpr int LPK = 2 * 64 / KPC;           // lanes per key in the scores (4 warps x 32 lanes = KPC x LPK)
constexpr int NCOL = 128 / LPK / 8;         // 16-byte columns of a key row per lane
#ifndef PM_ATTN_NST
#define PM_ATTN_NST 2
#endif
constexpr int NST = PM_ATTN_NST;            // stages per CTA: two (64 KB) let the CTAs share an SM
                                            // with the projection kernels around them; B=1 frame
                                            // +1.6% over three, four 8% slower
constexpr int ROWB = DH * 2;                // bytes per K or V row
constexpr int STAGE = 2 * KPC * ROWB;       // K rows then V rows: 32 KB
constexpr int THREADS = 160;                // 4 consumer warps + producer warp
constexpr int MAX_PIECES = 128;             // pieces a head can be cut into (>= chunks per head)
constexpr int MAX_CLUSTER = 8;              // CTAs per head in head-per-cluster mode

__device__ __forceinline__ int n_chunks(int pos, int win) { return (min(pos + 1, win) + KPC - 1) / KPC; }

__host__ __device__ __forceinline__ long long unit_begin(int c, long long U, int G) { return (long long)c * U / G; }

// CTA whose unit range contains unit u
__device__ __forceinline__ int cta_of(long long u, long long U, int G) {
    int c = (int)(u * G / U);
    while (c + 1 < G && unit_begin(c + 1, U, G) <= u) ++c;
    while (c > 0 && unit_begin(c, U, G) > u) --c;
    return c;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// every thread of every CTA of the cluster; stores before it are visible after it
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// store to the same shared-memory variable of CTA `rank` of this cluster
__device__ __forceinline__ void dsmem_store(const void* local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

struct UnitPos {
    int b, h, ci, nc;     // row, head, chunk index, chunks of the head
    int pos, key0, key1;  // query position, first key, one past the last key of the chunk
    int lo, s0;           // the row's first visible key; ring slot of key0
};

__device__ __forceinline__ UnitPos decode_unit(long long u, const int* s_first, const int* s_nc, const int* s_pos,
                                               int B, int H, int win, int ctx) {
    UnitPos r;
    int b = 0;
    while (b + 1 < B && u >= s_first[b + 1]) ++b;
    const int nc = s_nc[b];
    const int rel = (int)(u - s_first[b]);
    r.b = b;
    r.h = rel / nc;
    r.ci = rel % nc;
    r.nc = nc;
    r.pos = s_pos[b];
    const int n = min(r.pos + 1, win);
    r.lo = r.pos - n + 1;
    r.key0 = r.lo + KPC * r.ci;
    r.key1 = min(r.key0 + KPC, r.pos + 1);
    r.s0 = r.key0 % ctx;
    return r;
}

// the unit after r in (row, head, chunk) order, without divisions: a CTA's units are
// consecutive, and the issuing thread's per-unit work sits on every stage's refill path
__device__ __forceinline__ void next_unit(UnitPos& r, const int* s_nc, const int* s_pos, int B, int H, int win,
                                          int ctx) {
    if (++r.ci == r.nc) {
        r.ci = 0;
        if (++r.h == H) {
            r.h = 0;
            if (r.b + 1 < B) ++r.b;  // (past a CTA's last unit the walk is not read)
            r.nc = s_nc[r.b];
            r.pos = s_pos[r.b];
            r.lo = r.pos - min(r.pos + 1, win) + 1;
        }
        r.key0 = r.lo;
        r.s0 = r.lo % ctx;
    } else {
        r.key0 += KPC;
        r.s0 += KPC;
        if (r.s0 >= ctx) r.s0 -= ctx;
    }
    r.key1 = min(r.key0 + KPC, r.pos + 1);
}

// Consumer variants (MODE):
//  0  one running softmax per CTA: the chunk maximum and sum meet across the four warps
//     (two consumer barriers per unit), thread t owns coordinate t of the weighted values;
//  1  as 0, with the query in registers and the weighted values over key halves x
//     coordinate pairs (one 32-bit V load per key), the halves combined once per piece;
//  2  one running softmax per warp over its 16 keys of every unit (maximum and sum by warp
//     shuffles, no barrier per unit), lane l owns coordinates 4l .. 4l+3 (one 64-bit V load
//     per key); the four warps' states are merged once per piece.  Pays when a CTA streams
//     many units.
#ifndef PM_ATTN_MANY
#define PM_ATTN_MANY 2
#endif
#ifndef PM_ATTN_FEW
#define PM_ATTN_FEW 0
#endif
template <int MODE>
__global__ void __launch_bounds__(THREADS, 2) k_attn(const AttnParams p) {
    constexpr bool QREG = MODE >= 1;  // the query held in registers (modes 1 and 2)
    static_assert(MODE != 2 || KPC == 64, "per-warp softmax takes 16 keys per warp");
    extern __shared__ __align__(128) uint8_t ring[];  // [NST][STAGE]
    __shared__ int s_first[PM_MAX_B_DEV + 1], s_nc[PM_MAX_B_DEV], s_pos[PM_MAX_B_DEV];
    __shared__ __align__(8) uint64_t full[NST], empty[NST];
    __shared__ __align__(16) float s_q[DH];
    __shared__ __align__(16) float s_p[KPC];
    __shared__ float s_wm[4], s_wl[4];
    __shared__ float s_pm[MAX_PIECES], s_pl[MAX_PIECES];
    __shared__ int s_flags[4];  // [0] timeout, [1] last piece of a head, [2] units issued
    __shared__ float s_cpart[MAX_CLUSTER][DH + 2];  // head-per-cluster: the leader's inbox
    __shared__ __align__(16) float s_comb[4][DH];    // per-half (1) or per-warp (2) pieces
    __shared__ __align__(16) float s_pw[4][16];      // mode 2: a warp's key weights

    pdl_trigger();
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    // positions change only in the frame's last kernel, so every row's window, and the
    // whole unit list, is known before the wait
    if (t < p.B) {
        const int pos = p.st.pos[t];
        s_pos[t] = pos;
        s_nc[t] = p.H * n_chunks(pos, p.win);
    }
    if (t == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        fence_barrier_init();
        s_flags[0] = 0;
        s_flags[1] = 0;
        s_flags[2] = 0;
    }
    __syncthreads();
    if (t == 0) {
        int acc = 0;
        for (int bb = 0; bb < p.B; ++bb) {
            s_first[bb] = acc;
            acc += s_nc[bb];
            s_nc[bb] /= p.H;  // chunks per head
        }
        s_first[p.B] = acc;
    }
    __syncthreads();
    const long long U = s_first[p.B];
    const int G = gridDim.x, c = blockIdx.x;
    const int CS = p.cluster;
    long long u0, u1;
    int crank = 0, chd = 0;
    if (CS > 0) {
        // head-per-cluster: head chd owns CTAs chd*CS .. chd*CS+CS-1, each a contiguous share
        chd = c / CS;
        crank = c % CS;
        const int b = chd / p.H, h = chd % p.H, nc = s_nc[b];
        const long long hs = s_first[b] + (long long)h * nc;
        u0 = hs + (long long)crank * nc / CS;
        u1 = hs + (long long)(crank + 1) * nc / CS;
    } else {
        u0 = unit_begin(c, U, G);
        u1 = unit_begin(c + 1, U, G);
    }
    const int nu = (int)(u1 - u0);
    if (nu <= 0 && CS == 0) return;  // a cluster's CTAs all reach its barrier

    if (warp == 4) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            UnitPos up = decode_unit(u0, s_first, s_nc, s_pos, p.B, p.H, p.win, p.ctx);
            for (int k = 0; k < nu; ++k) {
                const int slot = k % NST;
                if (k > 0) next_unit(up, s_nc, s_pos, p.B, p.H, p.win, p.ctx);
                if (k >= NST && !mbar_wait(&empty[slot], (uint32_t)((k / NST) - 1) & 1u)) {
                    s_flags[0] = 1;
                    set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
                    break;
                }
                // keys before the current position only: that row is written by the kernel
                // this one overlaps
                const int nk = max(0, min(up.key1, up.pos) - up.key0);
                mbar_arrive_expect_tx(&full[slot], 2u * (uint32_t)nk * ROWB);
                if (nk > 0) {
                    const size_t head = ((size_t)up.b * p.H + up.h) * (size_t)p.ctx * DH;
                    const int s0 = up.s0;
                    const int n1 = min(nk, p.ctx - s0), n2 = nk - n1;
                    uint8_t* dk = ring + (size_t)slot * STAGE;
                    uint8_t* dv = dk + KPC * ROWB;
                    bulk_g2s(dk, p.kc + head + (size_t)s0 * DH, (uint32_t)n1 * ROWB, &full[slot], pol);
                    bulk_g2s(dv, p.vc + head + (size_t)s0 * DH, (uint32_t)n1 * ROWB, &full[slot], pol);
                    if (n2 > 0) {
                        bulk_g2s(dk + n1 * ROWB, p.kc + head, (uint32_t)n2 * ROWB, &full[slot], pol);
                        bulk_g2s(dv + n1 * ROWB, p.vc + head, (uint32_t)n2 * ROWB, &full[slot], pol);
                    }
                }
                s_flags[2] = k + 1;
            }
        }
    } else {
        // ------------------------------ consumers ------------------------------
        pdl_wait();
        const bool aborted = *(volatile uint32_t*)&p.st.status[1] != 0u;
        // running softmax of the current piece of a head.  Weighted values: thread t takes
        // coordinates 2(t mod 64), 2(t mod 64)+1 over the key half t / 64 of each unit
        // (one 32-bit load of V per key); the halves meet once per piece, into `acc`
        // (coordinate t)
        float m_run = -INFINITY, l_run = 0.f, acc = 0.f, ax = 0.f, ay = 0.f;
        float mw = -INFINITY, lw = 0.f, w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;  // mode 2
        const int kh = t >> 6, dp = t & 63;
        // this lane's query columns in the order its staggered K reads visit them
        float qr[NCOL][8];
        int seg_ci0 = 0;  // first chunk of the current piece of a head
        bool ok = true;
        UnitPos up = decode_unit(u0, s_first, s_nc, s_pos, p.B, p.H, p.win, p.ctx);
        for (int k = 0; k < nu; ++k) {
            const int slot = k % NST;
            if (k > 0) next_unit(up, s_nc, s_pos, p.B, p.H, p.win, p.ctx);
            const bool first = (k == 0) || up.ci == 0;
            if (first && !aborted) {
                // this piece's query, pre-scaled for the base-2 exponential; issued before the
                // stage wait so its latency overlaps the K/V copies
                if (MODE == 2) {
                    // each lane's half of the query, in the order its staggered K reads visit it
                    const float* qg = p.q + (size_t)up.b * p.D + up.h * DH + (lane & 1) * (DH / 2);
#pragma unroll
                    for (int j = 0; j < NCOL; ++j) {
                        const int jc = (j + lane) % NCOL;
                        const float4 qa = __ldcg(reinterpret_cast<const float4*>(qg + jc * 8));
                        const float4 qb = __ldcg(reinterpret_cast<const float4*>(qg + jc * 8 + 4));
                        qr[j][0] = qa.x * p.scale_log2; qr[j][1] = qa.y * p.scale_log2;
                        qr[j][2] = qa.z * p.scale_log2; qr[j][3] = qa.w * p.scale_log2;
                        qr[j][4] = qb.x * p.scale_log2; qr[j][5] = qb.y * p.scale_log2;
                        qr[j][6] = qb.z * p.scale_log2; qr[j][7] = qb.w * p.scale_log2;
                    }
                } else {
                    s_q[t] = __ldcg(p.q + (size_t)up.b * p.D + up.h * DH + t) * p.scale_log2;
                }
                m_run = -INFINITY;
                l_run = 0.f;
                ax = 0.f;
                ay = 0.f;
                acc = 0.f;
                mw = -INFINITY;
                lw = 0.f;
                w0 = w1 = w2 = w3 = 0.f;
                seg_ci0 = up.ci;
            }
            if (!mbar_wait(&full[slot], (uint32_t)(k / NST) & 1u)) {
                ok = false;
                break;
            }
            uint8_t* st = ring + (size_t)slot * STAGE;
            const int nvalid = up.key1 - up.key0;
            if (!aborted) {
                if (MODE == 2) {
                    const int r = up.pos - up.key0;
                    if (up.key1 == up.pos + 1 && (r >> 4) == warp) {
                        // the current position's K and V rows (written by the kernel waited for),
                        // by the one warp whose keys include it
                        const size_t row = (((size_t)up.b * p.H + up.h) * p.ctx + up.pos % p.ctx) * DH;
                        reinterpret_cast<uint2*>(st + r * ROWB)[lane] =
                            __ldcg(reinterpret_cast<const uint2*>(p.kc + row) + lane);
                        reinterpret_cast<uint2*>(st + KPC * ROWB + r * ROWB)[lane] =
                            __ldcg(reinterpret_cast<const uint2*>(p.vc + row) + lane);
                        __syncwarp();
                    }
                } else if (up.key1 == up.pos + 1 || first) {
                    if (up.key1 == up.pos + 1) {
                        // the current position's K and V rows, written by the kernel waited for
                        const size_t row = (((size_t)up.b * p.H + up.h) * p.ctx + up.pos % p.ctx) * DH + t;
                        const int r = up.pos - up.key0;
                        reinterpret_cast<uint16_t*>(st + r * ROWB)[t] = __ldcg(p.kc + row);
                        reinterpret_cast<uint16_t*>(st + KPC * ROWB + r * ROWB)[t] = __ldcg(p.vc + row);
                    }
                    cons_bar();  // that row, and a new piece's query, are in place
                }
                if (MODE == 1 && first) {
                    const int part0 = (lane % LPK) * (DH / LPK);
#pragma unroll
                    for (int j = 0; j < NCOL; ++j) {
                        const int jc = (j + lane) % NCOL;
                        const float4 qa = *reinterpret_cast<const float4*>(s_q + part0 + jc * 8);
                        const float4 qb = *reinterpret_cast<const float4*>(s_q + part0 + jc * 8 + 4);
                        qr[j][0] = qa.x; qr[j][1] = qa.y; qr[j][2] = qa.z; qr[j][3] = qa.w;
                        qr[j][4] = qb.x; qr[j][5] = qb.y; qr[j][6] = qb.z; qr[j][7] = qb.w;
                    }
                }
                // scores: LPK lanes per key (128 / LPK coordinates each); warp w takes keys
                // w*KPC/4 .. w*KPC/4 + KPC/4 - 1
                const int kk = (KPC / 4) * warp + lane / LPK, part = lane % LPK;
                const int half = part;  // lanes with part 0 publish the key's weight
                float d0 = 0.f, d1 = 0.f;
                if (kk < nvalid) {
                    const uint8_t* kr = st + kk * ROWB + part * (ROWB / LPK);
                    const float* qh = s_q + part * (DH / LPK);
#pragma unroll
                    for (int j = 0; j < NCOL; ++j) {
                        const int jc = (j + lane) % NCOL;  // staggered 16-byte column
                        const uint4 kv = *reinterpret_cast<const uint4*>(kr + jc * 16);
                        float q8[8];
                        if (QREG) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) q8[e] = qr[j][e];
                        } else {
                            const float4 qa = *reinterpret_cast<const float4*>(qh + jc * 8);
                            const float4 qb = *reinterpret_cast<const float4*>(qh + jc * 8 + 4);
                            q8[0] = qa.x; q8[1] = qa.y; q8[2] = qa.z; q8[3] = qa.w;
                            q8[4] = qb.x; q8[5] = qb.y; q8[6] = qb.z; q8[7] = qb.w;
                        }
                        d0 = fmaf(q8[0], bf16lo(kv.x), d0);
                        d1 = fmaf(q8[1], bf16hi(kv.x), d1);
                        d0 = fmaf(q8[2], bf16lo(kv.y), d0);
                        d1 = fmaf(q8[3], bf16hi(kv.y), d1);
                        d0 = fmaf(q8[4], bf16lo(kv.z), d0);
                        d1 = fmaf(q8[5], bf16hi(kv.z), d1);
                        d0 = fmaf(q8[6], bf16lo(kv.w), d0);
                        d1 = fmaf(q8[7], bf16hi(kv.w), d1);
                    }
                }
                float sc = d0 + d1;
#pragma unroll
                for (int o = 1; o < LPK; o <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
                if (kk >= nvalid) sc = -INFINITY;
                if (MODE == 2) {
                    // this warp's 16 keys: maximum and sum over the warp, no barrier
                    float wm = sc;
#pragma unroll
                    for (int o = 2; o <= 16; o <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                    const float m_new = fmaxf(mw, wm);
                    const float alpha = (mw == -INFINITY) ? 0.f : exp2f(mw - m_new);
                    const float pk = (kk < nvalid) ? exp2f(sc - m_new) : 0.f;
                    float ws = pk;  // both lanes of a key hold it: the xor steps from 2 count it once
#pragma unroll
                    for (int o = 2; o <= 16; o <<= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
                    lw = lw * alpha + ws;
                    mw = m_new;
                    if (part == 0) s_pw[warp][lane >> 1] = pk;
                    __syncwarp();
                    // coordinates 4 lane .. 4 lane + 3 over the warp's valid keys (rows past
                    // nvalid hold stale data: they are skipped, never multiplied by 0)
                    const int nk = min(max(nvalid - 16 * warp, 0), 16);
                    const uint8_t* vb = st + KPC * ROWB + (16 * warp) * ROWB + lane * 8;
                    float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f, c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
                    int j = 0;
#pragma unroll 2
                    for (; j + 4 <= nk; j += 4) {
                        const float4 pj = *reinterpret_cast<const float4*>(&s_pw[warp][j]);
                        const uint2 v0 = *reinterpret_cast<const uint2*>(vb + (j + 0) * ROWB);
                        const uint2 v1 = *reinterpret_cast<const uint2*>(vb + (j + 1) * ROWB);
                        const uint2 v2 = *reinterpret_cast<const uint2*>(vb + (j + 2) * ROWB);
                        const uint2 v3 = *reinterpret_cast<const uint2*>(vb + (j + 3) * ROWB);
                        b0 = fmaf(pj.x, bf16lo(v0.x), b0);
                        b1 = fmaf(pj.x, bf16hi(v0.x), b1);
                        b2 = fmaf(pj.x, bf16lo(v0.y), b2);
                        b3 = fmaf(pj.x, bf16hi(v0.y), b3);
                        c0 = fmaf(pj.y, bf16lo(v1.x), c0);
                        c1 = fmaf(pj.y, bf16hi(v1.x), c1);
                        c2 = fmaf(pj.y, bf16lo(v1.y), c2);
                        c3 = fmaf(pj.y, bf16hi(v1.y), c3);
                        b0 = fmaf(pj.z, bf16lo(v2.x), b0);
                        b1 = fmaf(pj.z, bf16hi(v2.x), b1);
                        b2 = fmaf(pj.z, bf16lo(v2.y), b2);
                        b3 = fmaf(pj.z, bf16hi(v2.y), b3);
                        c0 = fmaf(pj.w, bf16lo(v3.x), c0);
                        c1 = fmaf(pj.w, bf16hi(v3.x), c1);
                        c2 = fmaf(pj.w, bf16lo(v3.y), c2);
                        c3 = fmaf(pj.w, bf16hi(v3.y), c3);
                    }
                    for (; j < nk; ++j) {
                        const float pj = s_pw[warp][j];
                        const uint2 v = *reinterpret_cast<const uint2*>(vb + j * ROWB);
                        b0 = fmaf(pj, bf16lo(v.x), b0);
                        b1 = fmaf(pj, bf16hi(v.x), b1);
                        b2 = fmaf(pj, bf16lo(v.y), b2);
                        b3 = fmaf(pj, bf16hi(v.y), b3);
                    }
                    w0 = w0 * alpha + (b0 + c0);
                    w1 = w1 * alpha + (b1 + c1);
                    w2 = w2 * alpha + (b2 + c2);
                    w3 = w3 * alpha + (b3 + c3);
                    __syncwarp();  // s_pw is rewritten by the next unit
                } else {
                    // chunk maximum across the 4 warps, then weights against the running maximum
                    float wm = sc;
#pragma unroll
                    for (int o = LPK; o <= 16; o <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                    if (lane == 0) s_wm[warp] = wm;
                    cons_bar();
                    const float cm = fmaxf(fmaxf(s_wm[0], s_wm[1]), fmaxf(s_wm[2], s_wm[3]));
                    const float m_new = fmaxf(m_run, cm);
                    const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
                    const float pk = (kk < nvalid) ? exp2f(sc - m_new) : 0.f;
                    if (half == 0 && kk < KPC) s_p[kk] = pk;
                    float ws = half == 0 ? pk : 0.f;
#pragma unroll
                    for (int o = 1; o <= 16; o <<= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
                    if (lane == 0) s_wl[warp] = ws;
                    cons_bar();
                    if (MODE == 1) {
                        // weighted values over this thread's key half (rows past nvalid hold stale data:
                        // they are skipped, never multiplied by 0)
                        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(st + KPC * ROWB) + dp;
                        const int j0 = kh * (KPC / 2), j1 = min(nvalid, j0 + KPC / 2);
                        float bx0 = 0.f, by0 = 0.f, bx1 = 0.f, by1 = 0.f;
                        int j = j0;
        #pragma unroll 2
                        for (; j + 4 <= j1; j += 4) {
                            const float4 pj = *reinterpret_cast<const float4*>(s_p + j);
                            const uint32_t v0 = vrow[(j + 0) * (DH / 2)], v1 = vrow[(j + 1) * (DH / 2)];
                            const uint32_t v2 = vrow[(j + 2) * (DH / 2)], v3 = vrow[(j + 3) * (DH / 2)];
                            bx0 = fmaf(pj.x, bf16lo(v0), bx0);
                            by0 = fmaf(pj.x, bf16hi(v0), by0);
                            bx1 = fmaf(pj.y, bf16lo(v1), bx1);
                            by1 = fmaf(pj.y, bf16hi(v1), by1);
                            bx0 = fmaf(pj.z, bf16lo(v2), bx0);
                            by0 = fmaf(pj.z, bf16hi(v2), by0);
                            bx1 = fmaf(pj.w, bf16lo(v3), bx1);
                            by1 = fmaf(pj.w, bf16hi(v3), by1);
                        }
                        for (; j < j1; ++j) {
                            const uint32_t v = vrow[j * (DH / 2)];
                            bx0 = fmaf(s_p[j], bf16lo(v), bx0);
                            by0 = fmaf(s_p[j], bf16hi(v), by0);
                        }
                        ax = ax * alpha + (bx0 + bx1);
                        ay = ay * alpha + (by0 + by1);
                    } else {
                        // weighted values: thread t owns coordinate t
                        // (rows past nvalid hold stale data: they are skipped, never multiplied by 0)
                        const uint16_t* vcol = reinterpret_cast<const uint16_t*>(st + KPC * ROWB) + t;
                        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                        const int n4 = nvalid & ~3;
        #pragma unroll 4
                        for (int j = 0; j < n4; j += 4) {
                            const float4 pj = *reinterpret_cast<const float4*>(s_p + j);
                            a0 = fmaf(pj.x, __uint_as_float((uint32_t)vcol[(j + 0) * DH] << 16), a0);
                            a1 = fmaf(pj.y, __uint_as_float((uint32_t)vcol[(j + 1) * DH] << 16), a1);
                            a2 = fmaf(pj.z, __uint_as_float((uint32_t)vcol[(j + 2) * DH] << 16), a2);
                            a3 = fmaf(pj.w, __uint_as_float((uint32_t)vcol[(j + 3) * DH] << 16), a3);
                        }
                        for (int j = n4; j < nvalid; ++j) a0 = fmaf(s_p[j], __uint_as_float((uint32_t)vcol[j * DH] << 16), a0);
                        acc = acc * alpha + ((a0 + a1) + (a2 + a3));
                    }
                    l_run = l_run * alpha + ((s_wl[0] + s_wl[1]) + (s_wl[2] + s_wl[3]));
                    m_run = m_new;
                }
            }
            // the stage goes back to the copy engine once every warp is done with it: order
            // these reads before its refill
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (aborted) continue;

            const bool last = (k == nu - 1) || up.ci == up.nc - 1;
            if (!last) continue;
            if (MODE == 2) {
                // the four warps' running states of the piece, into coordinate t
                if (lane == 0) {
                    s_wm[warp] = mw;
                    s_wl[warp] = lw;
                }
                *reinterpret_cast<float4*>(&s_comb[warp][4 * lane]) = make_float4(w0, w1, w2, w3);
                cons_bar();
                const float M = fmaxf(fmaxf(s_wm[0], s_wm[1]), fmaxf(s_wm[2], s_wm[3]));
                float A = 0.f, L = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float f = (s_wm[w] == -INFINITY) ? 0.f : exp2f(s_wm[w] - M);
                    A = fmaf(f, s_comb[w][t], A);
                    L = fmaf(f, s_wl[w], L);
                }
                acc = A;
                l_run = L;
                m_run = M;
                cons_bar();
            } else if (MODE == 1) {
                // the two key halves of the piece, into coordinate t
                s_comb[kh][2 * dp] = ax;
                s_comb[kh][2 * dp + 1] = ay;
                cons_bar();
                acc = s_comb[0][t] + s_comb[1][t];
                cons_bar();
            }
            if (CS > 1) continue;  // pieces of a cluster's head meet in its leader
            float* ob = p.o + (size_t)up.b * p.D + up.h * DH;
            uint16_t* obb = p.ob ? p.ob + (size_t)up.b * p.D + up.h * DH : nullptr;
            const size_t lo_off = (size_t)p.ob_lo_rows * p.D;
            if (seg_ci0 == 0 && up.ci == up.nc - 1) {
                // the whole head was this CTA's
                const float v = acc / l_run;
                ob[t] = v;
                if (obb) {
                    const uint16_t hi = f32_to_bf16_rne(v);
                    obb[t] = hi;
                    if (lo_off) obb[lo_off + t] = bf16_lo_part(v, hi);
                }
                continue;
            }
            // a piece of a head cut between CTAs: deposit, the last piece to arrive merges
            const size_t hb = ((size_t)up.b * p.H + up.h) * p.S;
            float* part = p.part + (hb + seg_ci0) * (DH + 2);
            part[t] = acc;
            if (t == 0) {
                part[DH] = m_run;
                part[DH + 1] = l_run;
            }
            __threadfence();
            cons_bar();
            const long long hs = (u0 + k) - up.ci;  // the head's first unit
            const int cf = cta_of(hs, U, G), cl = cta_of(hs + up.nc - 1, U, G);
            if (t == 0) {
                const uint32_t done = atomicAdd(&p.count[(size_t)up.b * p.H + up.h], 1u);
                s_flags[1] = (done == (uint32_t)(cl - cf)) ? 1 : 0;
            }
            cons_bar();
            if (!s_flags[1]) continue;
            __threadfence();
            // pieces in order: piece i starts at the head's first unit in CTA cf + i
            const int np = cl - cf + 1;
            for (int i = t; i < np; i += 128) {
                const long long st_u = unit_begin(cf + i, U, G);
                const int ci = (int)((st_u > hs ? st_u : hs) - hs);
                s_pm[i] = __ldcg(p.part + (hb + ci) * (DH + 2) + DH);
                s_pl[i] = __ldcg(p.part + (hb + ci) * (DH + 2) + DH + 1);
            }
            cons_bar();
            float M = -INFINITY;
            for (int i = 0; i < np; ++i) M = fmaxf(M, s_pm[i]);
            float L = 0.f, A = 0.f;
            for (int i0 = 0; i0 < np; i0 += 8) {
                // eight pieces' values loaded before any is combined (one round trip, not eight)
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[j] = 0.f;
                    if (i0 + j < np) {
                        const long long st_u = unit_begin(cf + i0 + j, U, G);
                        const int ci = (int)((st_u > hs ? st_u : hs) - hs);
                        v[j] = __ldcg(p.part + (hb + ci) * (DH + 2) + t);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (i0 + j < np) {
                        const float f = (s_pm[i0 + j] == -INFINITY) ? 0.f : exp2f(s_pm[i0 + j] - M);
                        L += s_pl[i0 + j] * f;
                        A += v[j] * f;
                    }
                }
            }
            const float v = A / L;
            ob[t] = v;
            if (obb) {
                const uint16_t hi = f32_to_bf16_rne(v);
                obb[t] = hi;
                if (lo_off) obb[lo_off + t] = bf16_lo_part(v, hi);
            }
            if (t == 0) p.count[(size_t)up.b * p.H + up.h] = 0u;
            cons_bar();
        }
        if (!ok) {
            s_flags[0] = 1;
            set_status(p.st.status, PM_DEV_ERR_TIMEOUT);
        }
        if (CS > 1 && !aborted) {
            // this CTA's piece of the head (empty pieces: max -inf, sum 0) into the leader
            dsmem_store(&s_cpart[crank][t], 0, acc);
            if (t == 0) {
                dsmem_store(&s_cpart[crank][DH], 0, m_run);
                dsmem_store(&s_cpart[crank][DH + 1], 0, l_run);
            }
        }
    }
    if (CS > 1) {
        cluster_sync_all();
        if (crank == 0 && t < DH && *(volatile uint32_t*)&p.st.status[1] == 0u) {
            float M = -INFINITY;
            for (int i = 0; i < CS; ++i) M = fmaxf(M, s_cpart[i][DH]);
            float L = 0.f, A = 0.f;
            for (int i = 0; i < CS; ++i) {
                const float f = (s_cpart[i][DH] == -INFINITY) ? 0.f : exp2f(s_cpart[i][DH] - M);
                L += s_cpart[i][DH + 1] * f;
                A += s_cpart[i][t] * f;
            }
            const int b = chd / p.H, h = chd % p.H;
            const float v = A / L;
            p.o[(size_t)b * p.D + h * DH + t] = v;
            if (p.ob) {
                const uint16_t hi = f32_to_bf16_rne(v);
                p.ob[(size_t)b * p.D + h * DH + t] = hi;
                if (p.ob_lo_rows) p.ob[((size_t)b + p.ob_lo_rows) * p.D + h * DH + t] = bf16_lo_part(v, hi);
            }
        }
    }
    __syncthreads();
    if (s_flags[0] && t == 128) {
        // a wait ran out: let the copies already issued land before the CTA exits
        const int issued = s_flags[2];
        for (int i = issued - NST < 0 ? 0 : issued - NST; i < issued; ++i)
            (void)mbar_wait(&full[i % NST], (uint32_t)(i / NST) & 1u);
    }
}

}  // namespace

int attn_max_splits(int ctx) { return (ctx + KPC - 1) / KPC; }

void attn_plan(AttnParams& p, int num_sms) {
    const int slots = 2 * num_sms;  // resident CTAs
    if (p.B * p.H <= slots) {
        int cs = 1;
        while (cs < MAX_CLUSTER && p.B * p.H * cs * 2 <= slots) cs *= 2;
        p.cluster = cs;
        p.grid = p.B * p.H * cs;
    } else {
        p.cluster = 0;
        p.grid = slots;
    }
}

cudaError_t attn_prepare() {
    cudaError_t e = cudaFuncSetAttribute(k_attn<PM_ATTN_MANY>, cudaFuncAttributeMaxDynamicSharedMemorySize, NST * STAGE);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn<PM_ATTN_FEW>, cudaFuncAttributeMaxDynamicSharedMemorySize, NST * STAGE);
    return e;
}

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.S < attn_max_splits(p.ctx) || p.S > MAX_PIECES || p.B > PM_MAX_B_DEV || p.grid < 1 || p.win < 1 ||
        p.win > p.ctx || p.D != p.H * DH)
        return cudaErrorInvalidValue;
    if (p.cluster < 0 || p.cluster > MAX_CLUSTER || (p.cluster > 0 && p.grid != p.B * p.H * p.cluster))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = NST * STAGE;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (p.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    // many units per CTA (one or two CTAs per head, or the balanced split) vs one or two
    return (p.cluster == 0 || p.cluster <= 2) ? cudaLaunchKernelEx(&cfg, k_attn<PM_ATTN_MANY>, p)
                                              : cudaLaunchKernelEx(&cfg, k_attn<PM_ATTN_FEW>, p);
}

}  // namespace pm
