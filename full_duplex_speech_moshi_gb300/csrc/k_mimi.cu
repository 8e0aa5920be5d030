// Streaming Mimi decoder: code frames -> 24 kHz PCM, one 80 ms frame per stream and call
// ("PersonaPlex native LM audit", chapter "Exact Mimi codec construction": the DECODE
// order of "Complete encode/decode order", the split quantizer, the depthwise latent
// upsampler, the decoder transformer of "Both codec transformer stacks", "SEANet decoder,
// every stage", and the streaming rules of "Stateful streaming, padding and dependency
// boundaries").
//
// One CUDA graph per batch size B, every launch after the first with programmatic
// dependent launch (each kernel lets its successor start at once, stages its weights -- which
// no earlier kernel writes -- and only then waits for its predecessor's results):
//   k_mimi_front      codes -> split-RVQ lookup -> the two output projections -> latent;
//                     the depthwise ConvTranspose (kernel 4, stride 2) makes the frame's two
//                     25 Hz positions from this latent and the previous one
//   per block         LayerNorm-prologue GEMV (in_proj) -> k_mimi_attn (RoPE, ring append,
//                     causal window) -> GEMV (out_proj) + LayerScale + residual ->
//                     LayerNorm GEMV (lin1) + GELU -> GEMV (lin2) + LayerScale + residual
//   SEANet decoder    every convolution as a "phased" product: output row (phase p, channel
//                     co), column u, = bias + sum over input channels ci and taps m of
//                     Wt[p, co][m][ci] x[ci][u - (NT - 1) + m], with the activated input x
//                     (ELU where the decoder applies one).  A Conv1d is one phase with NT = k
//                     taps; a ConvTranspose1d of kernel 2s and stride s is s phases with two
//                     taps each (output n = u s + p takes tap p of input u and tap p + s of
//                     input u - 1).  Weights are re-laid tap-major once, in pm_mimi_create.
//                     A convolution keeps its last k - 1 activated inputs; a transposed
//                     convolution its column u = T (the s outputs the next frame completes).
//   k_mimi_finish     advances each stream's frame counter and position
// Streaming state is double-buffered by frame parity: a kernel reads the state of parity
// (frame & 1) and writes parity (frame + 1) & 1, so no kernel waits for another's reads,
// and a call with an invalid code (checked on the device for device codes) advances
// nothing.
//
// Activations fp32, weights bf16 (widened exactly), fp32 accumulation; RoPE angles in
// double from the integer position.  The result is the non-streaming causal decoder's,
// frame by frame.
#include <math.h>
#include <string.h>

#include <string>
#include <vector>

#include "../../include/pm_mimi.h"
#include "pm_common.cuh"

namespace pm {
namespace {

constexpr int MDH = 64;    // transformer head width
constexpr int GW = 4;      // rows (warps) per CTA of the transformer GEMVs

struct MimiIO {
    const int32_t* codes;  // decoder: [B][n_q] input codes
    float* pcm;            // decoder: [B][frame_samples] output PCM
    const float* pcm_in;   // encoder: [B][frame_samples] input PCM
    int32_t* codes_out;    // encoder: [B][n_q] output codes
    float* latent_out;     // encoder: [B][dim] unquantised latent, or NULL
};

struct MimiState {
    int32_t* frame;     // [B_max] frames decoded since reset (state parity = frame & 1)
    int32_t* pos;       // [B_max] 25 Hz position of the frame's first position
    uint32_t* abort;    // [1] nonzero: this call's codes were invalid (nothing advances)
    uint32_t* status;   // [1] sticky: bit 0 an invalid device code, bit 1 a wait ran out
    const uint32_t* wait_budget;  // [1] polls of the quantiser's copy waits
};

__device__ __forceinline__ float bf(const uint16_t* p, size_t i) { return __uint_as_float((uint32_t)p[i] << 16); }

__device__ __forceinline__ float elu_f(float x) { return x > 0.f ? x : expm1f(x); }

__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

__device__ __forceinline__ bool aborted(const MimiState& st) { return *(volatile const uint32_t*)st.abort != 0u; }

__device__ __forceinline__ uint2 ldg_u2(const uint16_t* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// copy n elements with NB loads in flight per thread: ld(i) reads element i, st(i, v) stores it
template <int NB, typename LoadF, typename StoreF>
__device__ __forceinline__ void batched_copy(int n, LoadF ld, StoreF st) {
    for (int i0 = threadIdx.x; i0 < n; i0 += NB * (int)blockDim.x) {
        decltype(ld(0)) v[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int i = i0 + j * (int)blockDim.x;
            if (i < n) v[j] = ld(i);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int i = i0 + j * (int)blockDim.x;
            if (i < n) st(i, v[j]);
        }
    }
}

// ------------------------------------------------------------------------------------
// codes -> latent -> the frame's two upsampled positions
// ------------------------------------------------------------------------------------
struct FrontParams {
    const MimiIO* io;
    MimiState st;
    const uint16_t* cb[16];     // codebooks [card][cb_dim]
    const uint16_t* sem_out;    // [dim][cb_dim]
    const uint16_t* ac_out;     // [dim][cb_dim]
    const uint16_t* up;         // [dim][1][4]
    float* prev;                // [2][B_max][dim] the previous frame's latent, by parity
    float* X;                   // [B][2][dim] residual stream of the transformer
    int B_max, dim, cb_dim, card, n_q;
};

// grid (dim / 16, B), 256 threads: warp w makes channels 16 x + 2 w, 16 x + 2 w + 1
__global__ void __launch_bounds__(256) k_mimi_front(const FrontParams p) {
    extern __shared__ float sm[];
    float* sem = sm;              // semantic vector  [cb_dim]
    float* ac = sm + p.cb_dim;    // acoustic sum     [cb_dim]
    __shared__ int s_codes[16];
    __shared__ int s_bad;
    const int b = blockIdx.y, t = threadIdx.x, warp = t >> 5, lane = t & 31;
    pdl_trigger();
    if (t == 0) s_bad = 0;
    if (t < p.n_q) {
        const int c = p.io->codes[(size_t)b * p.n_q + t];
        s_codes[t] = c;
        if (c < 0 || c >= p.card) atomicOr(&s_bad, 1);
    }
    __syncthreads();
    if (s_bad) {
        // an invalid code anywhere makes the whole call a no-op
        if (t == 0) {
            atomicExch(p.st.abort, 1u);
            atomicOr(p.st.status, 1u);
        }
        return;
    }
    for (int k = t; k < p.cb_dim; k += blockDim.x) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < p.n_q) v[j] = bf(p.cb[j], (size_t)s_codes[j] * p.cb_dim + k);
        float a = 0.f;
#pragma unroll
        for (int j = 1; j < 16; ++j)
            if (j < p.n_q) a += v[j];
        sem[k] = v[0];
        ac[k] = a;
    }
    __syncthreads();
    const int par = p.st.frame[b] & 1;
    for (int r = 0; r < 2; ++r) {
        const int c = blockIdx.x * 16 + warp * 2 + r;
        if (c >= p.dim) break;
        const uint16_t* ws = p.sem_out + (size_t)c * p.cb_dim;
        const uint16_t* wa = p.ac_out + (size_t)c * p.cb_dim;
        float v = 0.f;
#pragma unroll 4
        for (int k = 4 * lane; k < p.cb_dim; k += 128) {
            const uint2 a = ldg_u2(ws + k), e = ldg_u2(wa + k);
            const float4 x = *reinterpret_cast<const float4*>(sem + k);
            const float4 y = *reinterpret_cast<const float4*>(ac + k);
            v = fmaf(bf16lo(a.x), x.x, v);
            v = fmaf(bf16hi(a.x), x.y, v);
            v = fmaf(bf16lo(a.y), x.z, v);
            v = fmaf(bf16hi(a.y), x.w, v);
            v = fmaf(bf16lo(e.x), y.x, v);
            v = fmaf(bf16hi(e.x), y.y, v);
            v = fmaf(bf16lo(e.y), y.z, v);
            v = fmaf(bf16hi(e.y), y.w, v);
        }
        const float lat = warp_sum(v);
        if (lane == 0) {
            const float pr = p.prev[((size_t)par * p.B_max + b) * p.dim + c];
            // transposed depthwise convolution, kernel 4, stride 2, trimmed by 2 on the
            // right: output 2t + i = tap i of input t + tap i + 2 of input t - 1
            const float w0 = bf(p.up, (size_t)c * 4 + 0), w1 = bf(p.up, (size_t)c * 4 + 1);
            const float w2 = bf(p.up, (size_t)c * 4 + 2), w3 = bf(p.up, (size_t)c * 4 + 3);
            p.X[((size_t)b * 2 + 0) * p.dim + c] = fmaf(w0, lat, w2 * pr);
            p.X[((size_t)b * 2 + 1) * p.dim + c] = fmaf(w1, lat, w3 * pr);
            p.prev[((size_t)(par ^ 1) * p.B_max + b) * p.dim + c] = lat;
        }
    }
}

// ------------------------------------------------------------------------------------
// transformer projections: y[q][r] = sum_k W[r][k] x[q][k] over the call's 2B positions
// ------------------------------------------------------------------------------------
enum MPro { MP_NONE = 0, MP_LN = 1 };
enum MEpi { ME_STORE = 0, ME_GELU = 1, ME_SCALE_RES = 2 };

struct MGemvParams {
    const uint16_t* W;      // [R][K]
    const float* x;         // [nq][K]
    const uint16_t* ln_w;   // MP_LN: LayerNorm weight and bias [K]
    const uint16_t* ln_b;
    float eps;
    float* y;               // [nq][R]; ME_SCALE_RES: the residual stream, added to
    const uint16_t* scale;  // ME_SCALE_RES: LayerScale [R]
    MimiState st;
    int R, K, nq;
};

// grid ceil(R / 4), 128 threads, a warp per output row.  The CTA's 4 weight rows (and the
// LayerNorm parameters, the LayerScale) are staged in shared memory before the wait; lane l
// then takes elements 4 l + 128 i .. + 3 of its row for every position.  NQ bounds the
// call's positions 2B (nq <= NQ <= 16); K a multiple of 128.
template <int PRO, int EPI, int NQ>
__global__ void __launch_bounds__(128) k_mimi_gemv(const MGemvParams p) {
    extern __shared__ __align__(16) float xs[];  // [nq][K] | LN weight [K] | LN bias [K] | W [4][K] bf16
    __shared__ float s_m[16], s_r[16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int r0 = blockIdx.x * GW, r = r0 + warp, K = p.K;
    float* lnw = xs + p.nq * K;
    float* lnb = lnw + K;
    uint16_t* ws = reinterpret_cast<uint16_t*>(lnb + K);
    pdl_trigger();
    {
        const int nrow = min(GW, p.R - r0), n8 = nrow * K / 8;
        const uint4* src = reinterpret_cast<const uint4*>(p.W + (size_t)r0 * K);
        batched_copy<4>(n8, [&](int i) { return __ldg(src + i); },
                        [&](int i, uint4 v) { reinterpret_cast<uint4*>(ws)[i] = v; });
    }
    float scale = 0.f;
    if (EPI == ME_SCALE_RES && r < p.R) scale = bf(p.scale, r);
    if (PRO == MP_LN)
        batched_copy<4>(K, [&](int k) { return make_float2(bf(p.ln_w, k), bf(p.ln_b, k)); },
                        [&](int k, float2 v) {
                            lnw[k] = v.x;
                            lnb[k] = v.y;
                        });
    pdl_wait();
    if (aborted(p.st)) return;
    batched_copy<4>(p.nq * K / 4, [&](int i) { return reinterpret_cast<const float4*>(p.x)[i]; },
                    [&](int i, float4 v) { reinterpret_cast<float4*>(xs)[i] = v; });
    __syncthreads();
    if (PRO == MP_LN) {
        // mean and biased variance per position, then (x - m) / sqrt(v + eps) * w + b
        for (int q = warp; q < p.nq; q += GW) {
            const float4* xq = reinterpret_cast<const float4*>(xs + q * K);
            float s0 = 0.f, s1 = 0.f;
            for (int k = lane; k < K / 4; k += 32) {
                const float4 v = xq[k];
                s0 += v.x + v.y;
                s1 += v.z + v.w;
            }
            const float m = warp_sum(s0 + s1) / (float)K;
            float v0 = 0.f, v1 = 0.f;
            for (int k = lane; k < K / 4; k += 32) {
                const float4 v = xq[k];
                const float a = v.x - m, b2 = v.y - m, c = v.z - m, d = v.w - m;
                v0 = fmaf(a, a, fmaf(b2, b2, v0));
                v1 = fmaf(c, c, fmaf(d, d, v1));
            }
            const float var = warp_sum(v0 + v1);
            if (lane == 0) {
                s_m[q] = m;
                s_r[q] = 1.0f / sqrtf(var / (float)K + p.eps);
            }
        }
        __syncthreads();
        for (int q = 0; q < p.nq; ++q)
            for (int k = t; k < K; k += blockDim.x) xs[q * K + k] = fmaf((xs[q * K + k] - s_m[q]) * s_r[q], lnw[k], lnb[k]);
        __syncthreads();
    }
    if (r >= p.R) return;
    float acc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[q] = 0.f;
    const uint16_t* wrow = ws + (size_t)warp * K;
    for (int k = 4 * lane; k < K; k += 128) {
        const uint2 w = *reinterpret_cast<const uint2*>(wrow + k);
        const float w0 = bf16lo(w.x), w1 = bf16hi(w.x), w2 = bf16lo(w.y), w3 = bf16hi(w.y);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (q < p.nq) {
                const float4 x = *reinterpret_cast<const float4*>(xs + q * K + k);
                acc[q] = fmaf(w3, x.w, fmaf(w2, x.z, fmaf(w1, x.y, fmaf(w0, x.x, acc[q]))));
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        if (q < p.nq) {
            const float v = warp_sum(acc[q]);
            if (lane == q) {
                float* o = p.y + (size_t)q * p.R + r;
                if (EPI == ME_STORE) *o = v;
                if (EPI == ME_GELU) *o = gelu_f(v);
                if (EPI == ME_SCALE_RES) *o = fmaf(v, scale, *o);
            }
        }
    }
}

// ------------------------------------------------------------------------------------
// attention: RoPE, ring append, causal window (a CTA per stream and head)
// ------------------------------------------------------------------------------------
struct MAttnParams {
    const float* qkv;     // [B][2][3 dim]: q, k, v
    float* o;             // [B][2][dim]
    float* kc;            // this block's keys   [B_max][H][RS][64], after RoPE
    float* vc;            // this block's values [B_max][H][RS][64]
    const double* freq;   // [32] RoPE frequencies of the coordinate pairs
    MimiState st;
    int dim, H, ctx, RS;  // RS = ctx + 1 ring slots: the frame's second key must not evict
                          // the oldest key its first query still sees
    float scale_log2;     // log2(e) / sqrt(64)
};

// The window holds keys base .. pos0 + 1, base = pos0 - ctx + 1: NW = ctx + 1 rows.  The
// rows of earlier frames are final when the call starts, so they are staged into shared
// memory before the wait; the frame's two keys and values are made after it (RoPE) and go
// both to the ring and to the staged window.  Then a thread per key computes both queries'
// scores, the CTA takes the softmax, and pairs of threads sum the values.
__global__ void __launch_bounds__(256) k_mimi_attn(const MAttnParams p) {
    extern __shared__ __align__(16) float asm_[];
    const int NW = p.ctx + 1;
    float* Ks = asm_;                                  // [NW][65]
    float* Vs = Ks + (((size_t)NW * 65 + 3) & ~(size_t)3);  // [NW][64], 16-byte aligned
    float* sc = Vs + (size_t)NW * 64;    // [2][NW] scores, then probabilities
    __shared__ float qr[2][MDH];
    __shared__ float red[2][8];
    __shared__ float s_max[2], s_sum[2];
    __shared__ float part[2][2][MDH];
    const int b = blockIdx.x, h = blockIdx.y;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const size_t hb = ((size_t)b * p.H + h) * p.RS;
    pdl_trigger();
    const int pos0 = p.st.pos[b];        // set by the previous call's last kernel
    const int base = pos0 - p.ctx + 1;
    {
        // old rows: positions max(0, base) .. pos0 - 1, 16 float4 per row and tensor
        const int first = max(0, base), n_old = pos0 - first;
        const int n4 = n_old * 16;
        for (int i0 = t; i0 < 2 * n4; i0 += 4 * blockDim.x) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < 2 * n4) {
                    const int tensor = i >= n4, ii = i - tensor * n4, row = ii >> 4, c4 = ii & 15;
                    const int kp = first + row;
                    v[j] = reinterpret_cast<const float4*>((tensor ? p.vc : p.kc) + (hb + (size_t)(kp % p.RS)) * MDH)[c4];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < 2 * n4) {
                    const int tensor = i >= n4, ii = i - tensor * n4, row = ii >> 4, c4 = ii & 15;
                    const int sr = first + row - base;
                    if (tensor) {
                        reinterpret_cast<float4*>(Vs + (size_t)sr * 64)[c4] = v[j];
                    } else {
                        float* d = Ks + (size_t)sr * 65 + 4 * c4;
                        d[0] = v[j].x;
                        d[1] = v[j].y;
                        d[2] = v[j].z;
                        d[3] = v[j].w;
                    }
                }
            }
        }
    }
    pdl_wait();
    if (aborted(p.st)) return;
    // RoPE on adjacent pairs (2j, 2j + 1) of q and k at the frame's two positions; the
    // angle is reduced modulo 2 pi in double before the single-precision sine and cosine
    if (t < MDH) {
        const int i = t / (MDH / 2), j = t % (MDH / 2);
        const int pos = pos0 + i;
        const double a = (double)pos * p.freq[j];
        const double two_pi = 6.283185307179586476925;
        const float ang = (float)(a - two_pi * rint(a * (1.0 / two_pi)));
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float* row = p.qkv + ((size_t)b * 2 + i) * 3 * p.dim + h * MDH;
        const float q0 = row[2 * j], q1 = row[2 * j + 1];
        const float k0 = row[p.dim + 2 * j], k1 = row[p.dim + 2 * j + 1];
        const float v0 = row[2 * p.dim + 2 * j], v1 = row[2 * p.dim + 2 * j + 1];
        const float kr0 = k0 * cs - k1 * sn, kr1 = k0 * sn + k1 * cs;
        qr[i][2 * j] = q0 * cs - q1 * sn;
        qr[i][2 * j + 1] = q0 * sn + q1 * cs;
        float* kd = p.kc + (hb + (size_t)(pos % p.RS)) * MDH;
        float* vd = p.vc + (hb + (size_t)(pos % p.RS)) * MDH;
        kd[2 * j] = kr0;
        kd[2 * j + 1] = kr1;
        vd[2 * j] = v0;
        vd[2 * j + 1] = v1;
        const int sr = pos - base;  // ctx - 1 + i
        Ks[(size_t)sr * 65 + 2 * j] = kr0;
        Ks[(size_t)sr * 65 + 2 * j + 1] = kr1;
        Vs[(size_t)sr * 64 + 2 * j] = v0;
        Vs[(size_t)sr * 64 + 2 * j + 1] = v1;
    }
    __syncthreads();
    // scores: query i (position pos0 + i) sees keys max(0, pos0 + i - ctx + 1) .. pos0 + i,
    // i.e. rows i .. ctx - 1 + i of the window, without negative positions
    float mx[2] = {-INFINITY, -INFINITY};
    for (int r = t; r < NW; r += blockDim.x) {
        const float* kr = Ks + (size_t)r * 65;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll 16
        for (int d = 0; d < MDH; ++d) {
            const float k = kr[d];
            a0 = fmaf(qr[0][d], k, a0);
            a1 = fmaf(qr[1][d], k, a1);
        }
        const bool live = base + r >= 0;
        const float s0 = (live && r <= p.ctx - 1) ? a0 * p.scale_log2 : -INFINITY;
        const float s1 = (live && r >= 1) ? a1 * p.scale_log2 : -INFINITY;
        sc[r] = s0;
        sc[NW + r] = s1;
        mx[0] = fmaxf(mx[0], s0);
        mx[1] = fmaxf(mx[1], s1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float m = mx[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red[i][warp] = m;
    }
    __syncthreads();
    if (t < 2) {
        float m = red[t][0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[t][w]);
        s_max[t] = m;
    }
    __syncthreads();
    float sm[2] = {0.f, 0.f};
    for (int r = t; r < NW; r += blockDim.x) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float e = exp2f(sc[i * NW + r] - s_max[i]);
            sc[i * NW + r] = e;
            sm[i] += e;
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float v = warp_sum(sm[i]);
        if (lane == 0) red[i][warp] = v;
    }
    __syncthreads();
    if (t < 2) {
        float v = 0.f;
        for (int w = 0; w < 8; ++w) v += red[t][w];
        s_sum[t] = v;
    }
    // values: thread (half, i, d) sums rows r_lo + half, r_lo + half + 2, ... of query i;
    // rows of negative positions (before the stream's first frame) were never staged
    const int d = t & 63, i = (t >> 6) & 1, half = t >> 7, r_lo = max(0, -base);
    float a = 0.f;
    for (int r = r_lo + half; r < NW; r += 2) a = fmaf(sc[i * NW + r], Vs[(size_t)r * 64 + d], a);
    part[half][i][d] = a;
    __syncthreads();
    if (t < 2 * MDH) {
        const int ii = t >> 6, dd = t & 63;
        p.o[((size_t)b * 2 + ii) * p.dim + h * MDH + dd] = (part[0][ii][dd] + part[1][ii][dd]) / s_sum[ii];
    }
}

size_t attn_smem(int ctx) {
    const size_t NW = (size_t)ctx + 1;
    return 4u * (((NW * 65 + 3) & ~(size_t)3) + NW * 64 + 2 * NW);
}

// ------------------------------------------------------------------------------------
// SEANet convolutions as phased products (see the file header)
// ------------------------------------------------------------------------------------
struct MConvParams {
    const float* in;        // [B][Cin][T S] (or [B][T S][Cin] when in_pm), already activated;
                            // input channel ci' = ci S + p at position t is element t S + p of
                            // channel ci (S = 1: plain channels)
    const MimiIO* io_in;    // when set, the input is the caller's PCM (io_in->pcm_in)
    float* out;             // the output as computed, or NULL: Conv1d [B][Cout][T],
                            // ConvTranspose1d [B][Cout][T s]
    float* out_act;         // ELU of the output (what the next convolution reads), or NULL
    const float* res_in;    // residual added to the output (same layout), or NULL
    const MimiIO* io_out;   // when set, the output is the caller's PCM (io_out->pcm)
    const uint16_t* Wt;     // tap-major [R = P Cout][NT][Cin]
    const uint16_t* bias;   // [Cout]
    float* state;           // Conv1d: [2][B_max][Cin][NT-1] activated inputs;
                            // ConvTranspose1d: [2][B_max][Cout][P] column T of the last call
    MimiState st;
    int B_max, Cin, Cout, NT, P, T, U;  // P phases (1: Conv1d); U = T (Conv1d) or T + 1; Cin
                                        // counts input channels ci' (S per original channel)
    int S;                  // input positions folded into a channel (a stride-S convolution)
    int rep;                // at a stream's first frame, positions before 0 repeat position 0
    int no_bias, out_pm;    // no bias; output position-major [B][T][Cout]
    int in_pm, rows_per_cta;
};

// (activated) input of channel ci at position src of this call: a Conv1d takes src < 0 from
// its state, a ConvTranspose1d reads zeros outside 0..T-1 (its carried column stands in)
__device__ __forceinline__ float conv_load(const MConvParams& p, int b, int ci, int src, const float* st_old) {
    const int c0 = ci / p.S, ph = ci - c0 * p.S, Cs = p.Cin / p.S, TS = p.T * p.S;
    const float* in = p.io_in ? p.io_in->pcm_in : p.in;
    if (src < 0) {
        if (p.rep && p.st.frame[b] == 0)  // replicated left padding: the stream's first position
            return p.in_pm ? in[(size_t)b * TS * Cs + c0] : in[((size_t)b * Cs + c0) * TS];
        return (p.P == 1 && p.NT > 1) ? st_old[((size_t)b * p.Cin + ci) * (p.NT - 1) + (p.NT - 1 + src)] : 0.f;
    }
    if (src >= p.T) return 0.f;
    const int t = src * p.S + ph;
    return p.in_pm ? in[((size_t)b * TS + t) * Cs + c0] : in[((size_t)b * Cs + c0) * TS + t];
}

// output of row (phase, co), column u: bias (+ carried column, + residual) -> the raw
// output, its ELU, or the PCM
__device__ __forceinline__ void conv_put(const MConvParams& p, int b, int row, int u, float acc, int par) {
    int co = row, n = u, len = p.T;
    float v = acc;
    if (p.P > 1) {
        const int ph = row / p.Cout;
        co = row - ph * p.Cout;
        const size_t tl = ((size_t)b * p.Cout + co) * p.P + ph;
        if (u == p.T) {  // the column the next call completes: kept without the bias
            p.state[(size_t)(par ^ 1) * p.B_max * p.Cout * p.P + tl] = acc;
            return;
        }
        if (u == 0) v += p.state[(size_t)par * p.B_max * p.Cout * p.P + tl];
        n = u * p.P + ph;
        len = p.T * p.P;
    }
    if (!p.no_bias) v += bf(p.bias, co);
    const size_t o = p.out_pm ? ((size_t)b * len + n) * p.Cout + co : ((size_t)b * p.Cout + co) * len + n;
    if (p.res_in) v += p.res_in[o];
    if (p.io_out) {
        p.io_out->pcm[o] = v;
        return;
    }
    if (p.out) p.out[o] = v;
    if (p.out_act) p.out_act[o] = elu_f(v);
}

// the next call's Conv1d state: the last NT - 1 activated inputs, from a window that holds
// positions u0 - (NT - 1) ..
__device__ __forceinline__ void conv_save_state(const MConvParams& p, int b, int par, const float* win, int WL,
                                                int u0) {
    const int km = p.NT - 1;
    float* st_new = p.state + (size_t)(par ^ 1) * p.B_max * p.Cin * km;
    for (int i = threadIdx.x; i < p.Cin * km; i += blockDim.x) {
        const int ci = i / km, m = i - ci * km;
        st_new[((size_t)b * p.Cin + ci) * km + m] = win[ci * WL + (p.T - u0) + m];
    }
}

// U <= UMAX: grid (ceil(R / RC), B) with RC = rows_per_cta (8 or 16), a warp per row (warp w
// takes rows w, w + 8), lanes over input channels.  The CTA stages its RC rows of weights
// ([RC][NT][Cin], contiguous) before the wait and the window [Cin][U + NT - 1] (odd row
// stride) after it.
template <int UMAX>
__global__ void __launch_bounds__(256) k_mimi_conv_rows(const MConvParams p) {
    extern __shared__ __align__(16) uint8_t smraw[];
    const int R = p.P * p.Cout, KR = p.NT * p.Cin, RC = p.rows_per_cta;
    const int r0 = blockIdx.x * RC, nrow = min(RC, R - r0);
    uint16_t* ws = reinterpret_cast<uint16_t*>(smraw);
    float* win = reinterpret_cast<float*>(smraw + (((size_t)RC * KR * 2 + 15) & ~(size_t)15));
    const int WL = (p.U + p.NT - 1) | 1;
    const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    const uint16_t* src = p.Wt + (size_t)r0 * KR;
    if ((KR & 7) == 0) {
        batched_copy<4>(nrow * KR / 8, [&](int i) { return __ldg(reinterpret_cast<const uint4*>(src) + i); },
                        [&](int i, uint4 v) { reinterpret_cast<uint4*>(ws)[i] = v; });
    } else {
        batched_copy<8>(nrow * KR, [&](int i) { return src[i]; }, [&](int i, uint16_t v) { ws[i] = v; });
    }
    pdl_wait();
    if (aborted(p.st)) return;
    const int par = p.st.frame[b] & 1;
    const float* st_old = p.state + (size_t)par * p.B_max * p.Cin * (p.NT - 1);
    const int WW = p.U + p.NT - 1;
    batched_copy<8>(
        p.Cin * WW,
        [&](int i) {
            const int ci = i / WW;
            return conv_load(p, b, ci, i - ci * WW - (p.NT - 1), st_old);
        },
        [&](int i, float v) {
            const int ci = i / WW;
            win[ci * WL + (i - ci * WW)] = v;
        });
    __syncthreads();
    if (p.P == 1 && p.NT > 1 && blockIdx.x == 0) conv_save_state(p, b, par, win, WL, 0);
    for (int rr = warp; rr < nrow; rr += 8) {
        float acc[UMAX];
#pragma unroll
        for (int u = 0; u < UMAX; ++u) acc[u] = 0.f;
        const uint16_t* wrow = ws + (size_t)rr * KR;
        for (int ci = lane; ci < p.Cin; ci += 32) {
            const float* x = win + ci * WL;
            for (int m = 0; m < p.NT; ++m) {
                const float w = __uint_as_float((uint32_t)wrow[m * p.Cin + ci] << 16);
#pragma unroll
                for (int u = 0; u < UMAX; ++u)
                    if (u < p.U) acc[u] = fmaf(w, x[u + m], acc[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < UMAX; ++u) {
            if (u < p.U) {
                const float v = warp_sum(acc[u]);
                if (lane == u) conv_put(p, b, r0 + rr, u, v, par);
            }
        }
    }
}

// grid (ceil(U / 32), ceil(R / CO), B): lane = column u0 + lane; the 8 warps split the input
// channels (warp w takes ci = w, w + 8, ...), each accumulating the CTA's CO rows, and the
// partial sums meet in shared memory in a fixed order.  Weights are staged before the wait
// as [NT Cin][CO] (a channel's CO rows adjacent), the activated window [Cin][32 + NT - 1]
// after it.
size_t tiled_smem(int Cin, int NT, int CO) {
    return (((size_t)NT * Cin * CO * 2 + 15) & ~(size_t)15) + ((4u * (size_t)Cin * (32 + NT - 1) + 15) & ~(size_t)15) +
           4u * 8 * CO * 32;
}

template <int CO>
__global__ void __launch_bounds__(256) k_mimi_conv_tiled(const MConvParams p) {
    extern __shared__ __align__(16) uint8_t smraw[];
    const int R = p.P * p.Cout, KR = p.NT * p.Cin, WL = 32 + p.NT - 1;
    uint16_t* ws = reinterpret_cast<uint16_t*>(smraw);
    float* win = reinterpret_cast<float*>(smraw + (((size_t)KR * CO * 2 + 15) & ~(size_t)15));
    float* red = win + ((((size_t)p.Cin * WL) + 3) & ~(size_t)3);
    const int b = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.y * CO, u0 = blockIdx.x * 32;
    pdl_trigger();
    batched_copy<8>(
        CO * KR,
        [&](int i) { return row0 + i / KR < R ? p.Wt[(size_t)row0 * KR + i] : (uint16_t)0; },
        [&](int i, uint16_t v) {
            const int r = i / KR;
            ws[(i - r * KR) * CO + r] = v;
        });
    pdl_wait();
    if (aborted(p.st)) return;
    const int par = p.st.frame[b] & 1;
    const float* st_old = p.state + (size_t)par * p.B_max * p.Cin * (p.NT - 1);
    batched_copy<8>(
        p.Cin * WL,
        [&](int i) {
            const int ci = i / WL;
            return conv_load(p, b, ci, u0 - (p.NT - 1) + (i - ci * WL), st_old);
        },
        [&](int i, float v) { win[i] = v; });
    __syncthreads();
    if (p.P == 1 && p.NT > 1 && blockIdx.y == 0 && u0 + 32 >= p.T) conv_save_state(p, b, par, win, WL, u0);
    float acc[CO];
#pragma unroll
    for (int r = 0; r < CO; ++r) acc[r] = 0.f;
    for (int ci = warp; ci < p.Cin; ci += 8) {
        const float* x = win + ci * WL + lane;
        for (int m = 0; m < p.NT; ++m) {
            const float xv = x[m];
            const uint2* wv = reinterpret_cast<const uint2*>(ws + (size_t)(m * p.Cin + ci) * CO);
#pragma unroll
            for (int g = 0; g < CO / 4; ++g) {
                const uint2 w = wv[g];
                acc[4 * g + 0] = fmaf(bf16lo(w.x), xv, acc[4 * g + 0]);
                acc[4 * g + 1] = fmaf(bf16hi(w.x), xv, acc[4 * g + 1]);
                acc[4 * g + 2] = fmaf(bf16lo(w.y), xv, acc[4 * g + 2]);
                acc[4 * g + 3] = fmaf(bf16hi(w.y), xv, acc[4 * g + 3]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < CO; ++r) red[(warp * CO + r) * 32 + lane] = acc[r];
    __syncthreads();
    for (int i = threadIdx.x; i < CO * 32; i += blockDim.x) {
        const int r = i >> 5, l = i & 31;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += red[(w * CO + r) * 32 + l];
        const int row = row0 + r, u = u0 + l;
        if (row < R && u < p.U) conv_put(p, b, row, u, v, par);
    }
}

struct FinishParams {
    MimiState st;
    const MimiIO* io;
    int B, frame_samples;
};

__global__ void __launch_bounds__(256) k_mimi_finish(const FinishParams p) {
    pdl_wait();
    const bool ab = aborted(p.st);
    if (ab) {
        for (int i = threadIdx.x; i < p.B * p.frame_samples; i += blockDim.x) p.io->pcm[i] = 0.f;
    } else if (threadIdx.x < p.B) {
        p.st.frame[threadIdx.x] += 1;
        p.st.pos[threadIdx.x] += 2;
    }
    __syncthreads();
    if (threadIdx.x == 0) *p.st.abort = 0u;
}

// ------------------------------------------------------------------------------------
// split residual vector quantisation of the latent: one cluster of RQ CTAs per stream
// ------------------------------------------------------------------------------------
constexpr int RQ = 8;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// store to the same shared-memory variable of CTA `rank` of the cluster
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(r), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(unsigned long long* local, uint32_t rank, unsigned long long v) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(r), "l"(v) : "memory");
}

struct RvqParams {
    const float* e;            // [B][dim] the latent after the downsampler
    const uint16_t* w_sem;     // semantic input projection [cb_dim][dim]
    const uint16_t* w_ac;      // acoustic input projection [cb_dim][dim]
    const uint16_t* cb[16];    // codebooks [card][cb_dim]
    const MimiIO* io;          // codes_out, latent_out
    MimiState st;              // status word (bit 1: a bounded wait ran out) and wait budget
    int dim, cb_dim, card, n_q;
};

// grid (RQ, B), clusters of RQ along x, 256 threads.  CTA k of a stream's cluster makes
// projection rows k R2 .. (R2 = 2 cb_dim / RQ; the semantic rows first) and sends them to
// every CTA of the cluster.  Its slice of every codebook (entries k card/RQ .. + card/RQ)
// streams through shared memory in halves, two buffers, by bulk copies on the copy engine
// -- the slices do not depend on the latent, so they run a level ahead of the scan; per
// level the CTA scans its slice (squared distance, a warp per entry, four at a time) and
// the cluster agrees on the smallest (distance, index) key through shared-memory slots
// and a cluster barrier.  The semantic search runs beside the first acoustic level; each
// acoustic level subtracts the chosen entry from the residual all CTAs hold.
__global__ void __launch_bounds__(256) k_mimi_rvq(const RvqParams p) {
    extern __shared__ __align__(16) uint8_t smraw[];
    __shared__ unsigned long long keys[2][2][RQ];  // [phase parity][search][rank]
    __shared__ unsigned long long wkey[8];
    __shared__ __align__(8) uint64_t full[2];      // one mbarrier per codebook buffer
    const int R2 = 2 * p.cb_dim / RQ, per = p.card / RQ, half = per / 2;
    const uint32_t chunk = (uint32_t)half * p.cb_dim * 2;
    uint16_t* cbuf = reinterpret_cast<uint16_t*>(smraw);                                  // [2][half][cb_dim]
    uint16_t* wsm = reinterpret_cast<uint16_t*>(smraw + 2 * (size_t)chunk);              // [R2][dim]
    float* es = reinterpret_cast<float*>(smraw + 2 * (size_t)chunk + (size_t)R2 * p.dim * 2);  // [dim]
    float* z = es + p.dim;                                                               // [2][cb_dim]
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.y, t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int e0 = (int)rank * per, n_chunks = 2 * p.n_q;
    const uint32_t budget = *(volatile const uint32_t*)p.st.wait_budget;
    int n_issued[2] = {0, 0};  // thread 0: copies issued into each buffer
    // chunk c: codebook c / 2, half c % 2 of this CTA's slice, into buffer c % 2
    auto issue = [&](int c) {
        uint64_t* bar = &full[c & 1];
        ++n_issued[c & 1];
        mbar_arrive_expect_tx(bar, chunk);
        bulk_g2s(cbuf + (size_t)(c & 1) * half * p.cb_dim, p.cb[c >> 1] + (size_t)(e0 + (c & 1) * half) * p.cb_dim,
                 chunk, bar, l2_evict_first_policy());
    };
    pdl_trigger();
    // every CTA of the cluster must be running before any stores into it: arrive now, wait
    // before the first remote store
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (t == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (t == 0) {
        issue(0);
        issue(1);
    }
    {
        const int r0 = (int)rank * R2;  // projection rows of this CTA
        const int n8 = R2 * p.dim / 8;
        batched_copy<4>(
            n8,
            [&](int i) {
                const int row = r0 + (i * 8) / p.dim, k = (i * 8) % p.dim;
                const uint16_t* w = row < p.cb_dim ? p.w_sem + (size_t)row * p.dim : p.w_ac + (size_t)(row - p.cb_dim) * p.dim;
                return __ldg(reinterpret_cast<const uint4*>(w + k));
            },
            [&](int i, uint4 v) { reinterpret_cast<uint4*>(wsm)[i] = v; });
    }
    pdl_wait();
    for (int k = t; k < p.dim; k += blockDim.x) es[k] = p.e[(size_t)b * p.dim + k];
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    // input projections: warp w makes rows w, w + 8, ... of this CTA's R2 and stores each
    // into every CTA of the cluster
    for (int rr = warp; rr < R2; rr += 8) {
        const uint16_t* w = wsm + (size_t)rr * p.dim;
        float a = 0.f;
        for (int k = 4 * lane; k < p.dim; k += 128) {
            const uint2 wv = *reinterpret_cast<const uint2*>(w + k);
            const float4 x = *reinterpret_cast<const float4*>(es + k);
            a = fmaf(bf16lo(wv.x), x.x, fmaf(bf16hi(wv.x), x.y, fmaf(bf16lo(wv.y), x.z, fmaf(bf16hi(wv.y), x.w, a))));
        }
        a = warp_sum(a);
        const int row = (int)rank * R2 + rr;
        if (lane < RQ) st_cluster_f32(z + row, (uint32_t)lane, a);  // row < cb_dim: semantic
    }
    cluster_sync();
    bool ok = true;
    int c = 0;  // next chunk to consume
    for (int ph = 0; ph + 1 < p.n_q; ++ph) {
        const int ns = ph == 0 ? 2 : 1;
        for (int sidx = 0; sidx < ns; ++sidx) {
            // ph 0: search 0 = semantic codebook 0 on z[0], search 1 = acoustic codebook 1
            const int j = ph == 0 ? sidx : ph + 1;
            const float* v = z + (j == 0 ? 0 : p.cb_dim);
            unsigned long long best = ~0ull;
            for (int h = 0; h < 2; ++h, ++c) {
                if (!mbar_wait_n(&full[c & 1], (uint32_t)(c >> 1) & 1u, budget)) ok = false;
                const uint16_t* cb = cbuf + (size_t)(c & 1) * half * p.cb_dim;
                // four entries in flight per warp: warp w takes entries 4 w .. 4 w + 3, + 32, ...
                for (int en0 = 4 * warp; en0 < half; en0 += 32) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int k = 8 * lane; k < p.cb_dim; k += 256) {
                        const float4 x0 = *reinterpret_cast<const float4*>(v + k);
                        const float4 x1 = *reinterpret_cast<const float4*>(v + k + 4);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (en0 + u >= half) break;
                            const uint4 cv = *reinterpret_cast<const uint4*>(cb + (size_t)(en0 + u) * p.cb_dim + k);
                            const float d0 = x0.x - bf16lo(cv.x), d1 = x0.y - bf16hi(cv.x), d2 = x0.z - bf16lo(cv.y),
                                        d3 = x0.w - bf16hi(cv.y), d4 = x1.x - bf16lo(cv.z), d5 = x1.y - bf16hi(cv.z),
                                        d6 = x1.z - bf16lo(cv.w), d7 = x1.w - bf16hi(cv.w);
                            const float a = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, d[u]))));
                            d[u] = fmaf(d4, d4, fmaf(d5, d5, fmaf(d6, d6, fmaf(d7, d7, a))));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float du = warp_sum(d[u]);
                        const uint32_t idx = (uint32_t)(e0 + h * half + en0 + u);
                        const unsigned long long key = ((unsigned long long)float_order_key(du) << 32) | idx;
                        if (en0 + u < half && key < best) best = key;
                    }
                }
                __syncthreads();  // every warp is done with this buffer
                // after a wait ran out no copy is issued into a buffer whose last copy may
                // still be landing
                if (t == 0 && ok && c + 2 < n_chunks) issue(c + 2);
            }
            if (lane == 0) wkey[warp] = best;
            __syncthreads();
            if (t == 0) {
                unsigned long long m = wkey[0];
                for (int w = 1; w < 8; ++w) m = wkey[w] < m ? wkey[w] : m;
                for (uint32_t r = 0; r < RQ; ++r) st_cluster_u64(&keys[ph & 1][sidx][rank], r, m);
            }
            __syncthreads();
        }
        cluster_sync();
        for (int sidx = 0; sidx < ns; ++sidx) {
            unsigned long long m = keys[ph & 1][sidx][0];
            for (int r = 1; r < RQ; ++r) m = keys[ph & 1][sidx][r] < m ? keys[ph & 1][sidx][r] : m;
            const int code = (int)(uint32_t)(m & 0xFFFFFFFFull) % p.card;
            const int j = ph == 0 ? sidx : ph + 1;
            if (rank == 0 && t == 0) p.io->codes_out[(size_t)b * p.n_q + j] = code;
            if (j > 0)  // the acoustic residual moves on
                for (int k = t; k < p.cb_dim; k += blockDim.x) z[p.cb_dim + k] -= bf(p.cb[j], (size_t)code * p.cb_dim + k);
        }
        __syncthreads();
    }
    if (!ok && t == 0) atomicOr(p.st.status, 2u);
    if (t == 0)  // every copy issued has landed before the CTA exits (the full poll budget)
        for (int bf_ = 0; bf_ < 2; ++bf_)
            if (n_issued[bf_] > 0) (void)mbar_wait_n(&full[bf_], (uint32_t)(n_issued[bf_] - 1) & 1u, PM_SPIN_LIMIT);
    if (rank == 0 && p.io->latent_out)
        for (int k = t; k < p.dim; k += blockDim.x) p.io->latent_out[(size_t)b * p.dim + k] = es[k];
}

size_t rvq_smem(int dim, int cb_dim, int card) {
    return 2 * (size_t)(card / RQ / 2) * cb_dim * 2 + (size_t)(2 * cb_dim / RQ) * dim * 2 + 4u * (size_t)(dim + 2 * cb_dim);
}

// tap-major relayout, once at creation: Conv1d W [Cout][Cin/S][NT S] -> Wt [Cout][NT][Cin]
// with input channel ci' = ci S + p taking kernel index m S + p (S = 1: Wt[co][m][ci] =
// W[co][ci][m]); ConvTranspose1d W [Cin][Cout][2s] -> Wt [s][Cout][2][Cin], tap m = 1 being
// kernel index p (input u) and m = 0 kernel index p + s (input u - 1)
__global__ void k_mimi_relayout(const uint16_t* W, uint16_t* Wt, int Cin, int Cout, int NT, int P, int S) {
    const size_t n = (size_t)P * Cout * NT * Cin;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int ci = (int)(i % Cin);
        const size_t rest = i / Cin;
        const int m = (int)(rest % NT);
        const size_t row = rest / NT;
        if (P == 1) {
            const int c0 = ci / S, ph = ci - c0 * S;
            Wt[i] = W[(row * (Cin / S) + c0) * ((size_t)NT * S) + (size_t)m * S + ph];
        } else {
            const int ph = (int)(row / Cout), co = (int)(row % Cout), k = 2 * P;
            Wt[i] = W[((size_t)ci * Cout + co) * k + ph + (1 - m) * P];
        }
    }
}

}  // namespace
}  // namespace pm

// =====================================================================================
// C ABI
// =====================================================================================
using namespace pm;

// buffer codes of a convolution's input / outputs: >= 0 an activation buffer, or
constexpr int BUF_NONE = -100;  // no such output
constexpr int BUF_X = -1;       // the transformer residual stream [B][2][dim] (position-major)
constexpr int BUF_IO = -2;      // the caller's PCM (decoder output, encoder input)
constexpr int BUF_LAT = -3;     // the encoder's latent [B][dim]

struct MimiLayer {         // one SEANet (or resampling) convolution, as recorded
    const uint16_t* Wt;    // tap-major weights
    const uint16_t* bias;
    float* state;
    int Cin, Cout, NT, P, T, S;  // Cin counts folded input channels (S per original channel)
    int rep, no_bias;
    int in_buf;            // input buffer (activated)
    int out_raw, out_act;  // buffers for the output and for its ELU
    int res_buf;           // buffer added to the output
    int wi;                // canonical index of the weight (the bias follows it)
    int kind;              // PM_MIMI_K_* of the launch
};

struct pm_mimi_ctx {
    pm_mimi_config cfg{};
    int encoder = 0;                     // 0: decoder context, 1: encoder context
    int device = 0;
    int frame_samples = 0;
    cudaStream_t stream = nullptr, cap = nullptr;
    std::vector<const uint16_t*> w;      // canonical tensors
    void* block = nullptr;
    uint16_t* wt_block = nullptr;        // tap-major convolution weights
    MimiState st{};
    MimiIO* io = nullptr;                // device I/O block
    int32_t* codes_dev = nullptr;        // decoder: host codes staged here
    float* pcm_dev = nullptr;            // encoder: host PCM staged here
    uint8_t* host_io = nullptr;          // pinned: I/O block image + host codes / PCM
    size_t host_io_bytes = 0;
    cudaEvent_t io_done = nullptr;
    float *prev = nullptr, *X = nullptr, *qkv = nullptr, *o = nullptr, *hf = nullptr, *kv = nullptr, *lat = nullptr;
    double* freq = nullptr;
    std::vector<float*> acts;            // SEANet activations
    std::vector<float*> states;          // streaming state per layer [2][B_max][per_stream]
    std::vector<size_t> state_per_stream;
    std::vector<MimiLayer> layers;       // convolutions in order
    std::vector<cudaGraphExec_t> graphs; // per B
    std::string err;
};

namespace {

thread_local std::string g_mimi_create_error;

int mimi_channels(const pm_mimi_config& c) { return c.n_filters << c.n_ratios; }

pm_status mfail(pm_mimi_ctx* c, pm_status s, const std::string& m) {
    if (c) c->err = m;
    return s;
}

// positions of each group in the decoder's canonical tensor order
struct MimiIdx {
    int cb0, sem_out, ac_out, up, layer0, dec0w, stage0, outw, total;
};
MimiIdx mimi_index(const pm_mimi_config& c) {
    MimiIdx x;
    x.cb0 = 0;
    x.sem_out = c.n_q;
    x.ac_out = c.n_q + 1;
    x.up = c.n_q + 2;
    x.layer0 = c.n_q + 3;
    x.dec0w = x.layer0 + 10 * c.n_layers;
    x.stage0 = x.dec0w + 2;
    x.outw = x.stage0 + 6 * c.n_ratios;
    x.total = x.outw + 2;
    return x;
}

// positions in the encoder's canonical order
struct MimiEncIdx {
    int enc0w, stage0, outw, layer0, ds, sem_in, ac_in, cb0, total;
};
MimiEncIdx mimi_enc_index(const pm_mimi_config& c) {
    MimiEncIdx x;
    x.enc0w = 0;
    x.stage0 = 2;
    x.outw = 2 + 6 * c.n_ratios;
    x.layer0 = x.outw + 2;
    x.ds = x.layer0 + 10 * c.n_layers;
    x.sem_in = x.ds + 1;
    x.ac_in = x.ds + 2;
    x.cb0 = x.ds + 3;
    x.total = x.cb0 + c.n_q;
    return x;
}

const char* mimi_check(const pm_mimi_config* c) {
    if (c->B_max < 1 || c->B_max > PM_MIMI_MAX_B) return "B_max outside 1..8";
    if (c->heads < 1 || c->dim != c->heads * MDH) return "dim must be 64 x heads";
    if (c->dim % 256 != 0 || c->ffn % 256 != 0 || c->dim > 2048 || c->ffn > 4096)
        return "dim and ffn must be multiples of 256 (dim <= 2048, ffn <= 4096)";
    if (c->cb_dim < 8 || c->cb_dim % 8 != 0 || c->cb_dim > 4096) return "cb_dim must be a multiple of 8 (<= 4096)";
    if (c->card < 1 || c->n_q < 2 || c->n_q > 16) return "codebooks: card >= 1, 2 <= n_q <= 16";
    if (c->n_layers < 0 || c->ctx < 2) return "transformer: n_layers >= 0, ctx >= 2";
    if (c->up_kernel != 4 || c->up_stride != 2) return "the latent resamplers must be kernel 4, stride 2";
    if (c->n_ratios < 1 || c->n_ratios > PM_MIMI_MAX_RATIOS || c->n_filters < 1) return "SEANet stages";
    for (int i = 0; i < c->n_ratios; ++i)
        if (c->ratios[i] < 1 || c->ratios[i] > 16) return "SEANet ratios must be 1..16";
    if (c->kernel < 1 || c->last_kernel < 1 || c->res_kernel < 1 || c->compress < 1) return "SEANet kernels";
    if (c->kernel > 16 || c->last_kernel > 16 || c->res_kernel > 16) return "SEANet kernels above 16";
    if (c->n_filters % c->compress != 0) return "n_filters must be a multiple of compress";
    if (!(c->ln_eps > 0.f) || !(c->rope_theta > 0.f)) return "ln_eps and rope_theta must be positive";
    return nullptr;
}

// the encoder's extra constraints (the cluster search and its projection slices)
const char* mimi_encoder_check(const pm_mimi_config* c) {
    if (c->card % (2 * RQ) != 0) return "the encoder needs card to be a multiple of 16";
    if ((2 * c->cb_dim) % RQ != 0 || c->cb_dim % 8 != 0) return "the encoder needs cb_dim a multiple of 8";
    if (c->dim % 128 != 0) return "the encoder needs dim a multiple of 128";
    return nullptr;
}

MimiLayer make_layer(int Cin, int Cout, int NT, int P, int T, int S, int in, int raw, int act, int res, int wi, int kind) {
    MimiLayer L;
    memset(&L, 0, sizeof L);
    L.Cin = Cin;
    L.Cout = Cout;
    L.NT = NT;
    L.P = P;
    L.T = T;
    L.S = S;
    L.in_buf = in;
    L.out_raw = raw;
    L.out_act = act;
    L.res_buf = res;
    L.wi = wi;
    L.kind = kind;
    return L;
}

// the decoder's SEANet convolutions in order.  Every convolution after the first reads an
// ELU, so each producer writes its output activated (the ELU computed once per element);
// the transposed convolution also keeps its raw output, which the residual unit's second
// convolution adds.  Buffers: 0 = first convolution (activated); stage i: 1 + 3i raw y,
// 2 + 3i ELU(y) -- reused for ELU of the residual sum, the next stage's input, once the
// unit's first convolution has read it --, 3 + 3i the unit's activated middle.
std::vector<MimiLayer> seanet_layers(const pm_mimi_config& f) {
    const MimiIdx ix = mimi_index(f);
    std::vector<MimiLayer> v;
    int C = mimi_channels(f), T = 2;
    v.push_back(make_layer(f.dim, C, f.kernel, 1, T, 1, BUF_X, BUF_NONE, 0, BUF_NONE, ix.dec0w, PM_MIMI_K_CONV_FIRST));
    int cur = 0;
    for (int i = 0; i < f.n_ratios; ++i) {
        const int r = f.ratios[i], co = C / 2, h = co / f.compress, w = ix.stage0 + 6 * i;
        const int yraw = 1 + 3 * i, yact = 2 + 3 * i, mid = 3 + 3 * i;
        v.push_back(make_layer(C, co, 2, r, T, 1, cur, yraw, yact, BUF_NONE, w, PM_MIMI_K_CONVTR));
        T *= r;
        v.push_back(make_layer(co, h, f.res_kernel, 1, T, 1, yact, BUF_NONE, mid, BUF_NONE, w + 2, PM_MIMI_K_RES1));
        v.push_back(make_layer(h, co, 1, 1, T, 1, mid, BUF_NONE, yact, yraw, w + 4, PM_MIMI_K_RES2));
        cur = yact;
        C = co;
    }
    v.push_back(make_layer(C, 1, f.last_kernel, 1, T, 1, cur, BUF_IO, BUF_NONE, BUF_NONE, ix.outw, PM_MIMI_K_CONV_LAST));
    return v;
}

// the encoder's convolutions in order: the SEANet encoder (stages in the reversed ratio
// order, each a residual unit then a stride-r convolution of kernel 2r folded as S = r input
// positions per channel and two taps), the last convolution into the transformer stream,
// and, recorded after the transformer, the latent downsampler.  Buffers per stage i: 3i raw
// x, 3i + 1 ELU(x) (reused for ELU of the residual sum), 3i + 2 the unit's activated middle;
// the stage's strided convolution writes stage i + 1's raw and ELU.
std::vector<MimiLayer> seanet_encoder_layers(const pm_mimi_config& f) {
    const MimiEncIdx ix = mimi_enc_index(f);
    std::vector<MimiLayer> v;
    int C = f.n_filters, T = 2;
    for (int i = 0; i < f.n_ratios; ++i) T *= f.ratios[i];
    v.push_back(make_layer(1, C, f.kernel, 1, T, 1, BUF_IO, 0, 1, BUF_NONE, ix.enc0w, PM_MIMI_K_CONV_FIRST));
    for (int i = 0; i < f.n_ratios; ++i) {
        const int r = f.ratios[f.n_ratios - 1 - i], h = C / f.compress, w = ix.stage0 + 6 * i;
        const int xraw = 3 * i, xact = 3 * i + 1, mid = 3 * i + 2;
        v.push_back(make_layer(C, h, f.res_kernel, 1, T, 1, xact, BUF_NONE, mid, BUF_NONE, w, PM_MIMI_K_RES1));
        v.push_back(make_layer(h, C, 1, 1, T, 1, mid, BUF_NONE, xact, xraw, w + 2, PM_MIMI_K_RES2));
        v.push_back(make_layer(C * r, 2 * C, 2, 1, T / r, r, xact, 3 * (i + 1), 3 * (i + 1) + 1, BUF_NONE, w + 4,
                               PM_MIMI_K_DOWN));
        C *= 2;
        T /= r;
    }
    v.push_back(make_layer(C, f.dim, f.last_kernel, 1, T, 1, 3 * f.n_ratios + 1, BUF_X, BUF_NONE, BUF_NONE, ix.outw,
                           PM_MIMI_K_CONV_LAST));
    MimiLayer ds = make_layer(2 * f.dim, f.dim, 2, 1, 1, 2, BUF_X, BUF_LAT, BUF_NONE, BUF_NONE, ix.ds, PM_MIMI_K_RESAMPLE);
    ds.rep = 1;
    ds.no_bias = 1;
    v.push_back(ds);
    return v;
}

// per-stream element counts of each layer's state (0: none)
size_t layer_state(const MimiLayer& L) {
    if (L.P > 1) return (size_t)L.Cout * L.P;
    return (size_t)L.Cin * (L.NT - 1);
}

// the launch shape of a layer: row kernel (U <= 32) or tiled, with its shared memory
struct ConvLaunch {
    int rows;          // 1: k_mimi_conv_rows
    int umax;          // rows: 4, 16 or 32
    int rpc;           // rows: rows per CTA (8 or 16)
    int CO;            // tiled: rows per CTA (4, 8 or 16)
    dim3 grid;
    size_t smem;
};
size_t rows_smem(const MimiLayer& L, int rpc, int U) {
    return (((size_t)rpc * L.NT * L.Cin * 2 + 15) & ~(size_t)15) + 4u * (size_t)L.Cin * ((U + L.NT - 1) | 1);
}
ConvLaunch conv_launch(const MimiLayer& L, int B) {
    ConvLaunch c;
    memset(&c, 0, sizeof c);
    const int R = L.P * L.Cout, U = L.P > 1 ? L.T + 1 : L.T;
    if (U <= 32) {
        // a warp per row; two rows per warp where one would give more than two CTAs per SM
        // (fewer CTAs stage the same window) and the weights still fit
        c.rows = 1;
        c.umax = U <= 4 ? 4 : U <= 16 ? 16 : 32;
        c.rpc = ((R + 7) / 8) * B > 2 * 152 && rows_smem(L, 16, U) <= 200u * 1024u ? 16 : 8;
        c.grid = dim3((unsigned)((R + c.rpc - 1) / c.rpc), (unsigned)B);
        c.smem = rows_smem(L, c.rpc, U);
        return c;
    }
    // the most rows per CTA (fewest CTAs staging the same window) that still fills the SMs
    const int tiles = (U + 31) / 32;
    c.CO = 4;
    for (int co = 16; co > 4; co /= 2)
        if (tiles * ((R + co - 1) / co) * B >= 152) {
            c.CO = co;
            break;
        }
    c.grid = dim3((unsigned)tiles, (unsigned)((R + c.CO - 1) / c.CO), (unsigned)B);
    c.smem = tiled_smem(L.Cin, L.NT, c.CO);
    return c;
}

template <typename K, typename P>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const P& params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, params);
}

size_t gemv_smem(int nq, int K) { return 4u * (size_t)(nq + 2) * K + 2u * GW * (size_t)K; }

template <int PRO, int EPI>
cudaError_t mgemv(const MGemvParams& p, cudaStream_t s) {
    const dim3 g((unsigned)((p.R + GW - 1) / GW)), b(32 * GW);
    const size_t sm = gemv_smem(p.nq, p.K);
    if (p.nq <= 2) return launch_pdl(k_mimi_gemv<PRO, EPI, 2>, g, b, sm, s, p);
    if (p.nq <= 4) return launch_pdl(k_mimi_gemv<PRO, EPI, 4>, g, b, sm, s, p);
    if (p.nq <= 8) return launch_pdl(k_mimi_gemv<PRO, EPI, 8>, g, b, sm, s, p);
    return launch_pdl(k_mimi_gemv<PRO, EPI, 16>, g, b, sm, s, p);
}

// per-launch events of the profiling calls (NULL when recording into a graph)
struct MimiMarks {
    std::vector<cudaEvent_t> ev;
    std::vector<int32_t> kind;
    void mark(cudaStream_t s, int32_t k) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return;
        cudaEventRecord(e, s);
        ev.push_back(e);
        kind.push_back(k);
    }
};

// a transformer stack over the context's X: layer0 = canonical index of block 0's norm1.w
pm_status record_transformer(pm_mimi_ctx* c, int B, cudaStream_t s, int layer0, MimiMarks* mk) {
    const pm_mimi_config& f = c->cfg;
    const int D = f.dim, nq = 2 * B, RS = f.ctx + 1;
    const size_t kv_block = (size_t)f.B_max * f.heads * RS * MDH;
    for (int l = 0; l < f.n_layers; ++l) {
        // canonical per-block order: norm1.w, norm1.b, in_proj, out_proj, scale1, norm2.w,
        // norm2.b, lin1, lin2, scale2
        const int w0 = layer0 + 10 * l;
        MGemvParams g;
        memset(&g, 0, sizeof g);
        g.st = c->st;
        g.eps = f.ln_eps;
        g.nq = nq;
        g.W = c->w[w0 + 2];
        g.x = c->X;
        g.ln_w = c->w[w0 + 0];
        g.ln_b = c->w[w0 + 1];
        g.y = c->qkv;
        g.R = 3 * D;
        g.K = D;
        if (mgemv<MP_LN, ME_STORE>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi in_proj launch");
        if (mk) mk->mark(s, PM_MIMI_K_IN_PROJ);
        MAttnParams a;
        memset(&a, 0, sizeof a);
        a.qkv = c->qkv;
        a.o = c->o;
        a.kc = c->kv + (size_t)(2 * l) * kv_block;
        a.vc = c->kv + (size_t)(2 * l + 1) * kv_block;
        a.freq = c->freq;
        a.st = c->st;
        a.dim = D;
        a.H = f.heads;
        a.ctx = f.ctx;
        a.RS = RS;
        a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)MDH));
        if (launch_pdl(k_mimi_attn, dim3((unsigned)B, (unsigned)f.heads), dim3(256), attn_smem(f.ctx), s, a) !=
            cudaSuccess)
            return mfail(c, PM_ERR_CUDA, "mimi attention launch");
        if (mk) mk->mark(s, PM_MIMI_K_ATTN);
        g.W = c->w[w0 + 3];
        g.x = c->o;
        g.y = c->X;
        g.scale = c->w[w0 + 4];
        g.R = D;
        g.K = D;
        if (mgemv<MP_NONE, ME_SCALE_RES>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi out_proj launch");
        if (mk) mk->mark(s, PM_MIMI_K_OUT_PROJ);
        g.W = c->w[w0 + 7];
        g.x = c->X;
        g.ln_w = c->w[w0 + 5];
        g.ln_b = c->w[w0 + 6];
        g.y = c->hf;
        g.R = f.ffn;
        g.K = D;
        if (mgemv<MP_LN, ME_GELU>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi lin1 launch");
        if (mk) mk->mark(s, PM_MIMI_K_LIN1);
        g.W = c->w[w0 + 8];
        g.x = c->hf;
        g.y = c->X;
        g.scale = c->w[w0 + 9];
        g.R = D;
        g.K = f.ffn;
        if (mgemv<MP_NONE, ME_SCALE_RES>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi lin2 launch");
        if (mk) mk->mark(s, PM_MIMI_K_LIN2);
    }
    return PM_OK;
}

float* buf_ptr(pm_mimi_ctx* c, int code) {
    if (code >= 0) return c->acts[code];
    if (code == BUF_X) return c->X;
    if (code == BUF_LAT) return c->lat;
    return nullptr;
}

// convolutions first .. last - 1 of the context's plan
pm_status record_convs(pm_mimi_ctx* c, int B, cudaStream_t s, size_t first, size_t last, MimiMarks* mk) {
    const pm_mimi_config& f = c->cfg;
    for (size_t i = first; i < last; ++i) {
        const MimiLayer& L = c->layers[i];
        MConvParams q;
        memset(&q, 0, sizeof q);
        q.in = buf_ptr(c, L.in_buf);
        q.io_in = L.in_buf == BUF_IO ? c->io : nullptr;  // the encoder's first convolution reads the caller's PCM
        q.in_pm = L.in_buf == BUF_X;
        q.out = buf_ptr(c, L.out_raw);
        q.out_pm = L.out_raw == BUF_X;
        q.io_out = L.out_raw == BUF_IO ? c->io : nullptr;  // the decoder's last convolution writes the caller's PCM
        q.out_act = L.out_act == BUF_NONE ? nullptr : buf_ptr(c, L.out_act);
        q.res_in = L.res_buf == BUF_NONE ? nullptr : buf_ptr(c, L.res_buf);
        q.Wt = L.Wt;
        q.bias = L.bias;
        q.state = L.state;
        q.st = c->st;
        q.B_max = f.B_max;
        q.Cin = L.Cin;
        q.Cout = L.Cout;
        q.NT = L.NT;
        q.P = L.P;
        q.T = L.T;
        q.U = L.P > 1 ? L.T + 1 : L.T;
        q.S = L.S;
        q.rep = L.rep;
        q.no_bias = L.no_bias;
        const ConvLaunch cl = conv_launch(L, B);
        q.rows_per_cta = cl.rpc;
        cudaError_t e;
        if (cl.rows)
            e = cl.umax == 4    ? launch_pdl(k_mimi_conv_rows<4>, cl.grid, dim3(256), cl.smem, s, q)
                : cl.umax == 16 ? launch_pdl(k_mimi_conv_rows<16>, cl.grid, dim3(256), cl.smem, s, q)
                                : launch_pdl(k_mimi_conv_rows<32>, cl.grid, dim3(256), cl.smem, s, q);
        else
            e = cl.CO == 16  ? launch_pdl(k_mimi_conv_tiled<16>, cl.grid, dim3(256), cl.smem, s, q)
                : cl.CO == 8 ? launch_pdl(k_mimi_conv_tiled<8>, cl.grid, dim3(256), cl.smem, s, q)
                             : launch_pdl(k_mimi_conv_tiled<4>, cl.grid, dim3(256), cl.smem, s, q);
        if (e != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi convolution launch");
        if (mk) mk->mark(s, L.kind);
    }
    return PM_OK;
}

pm_status record_finish(pm_mimi_ctx* c, int B, cudaStream_t s, MimiMarks* mk) {
    FinishParams fin;
    fin.st = c->st;
    fin.io = c->io;
    fin.B = B;
    fin.frame_samples = c->encoder ? 0 : c->frame_samples;
    if (launch_pdl(k_mimi_finish, dim3(1), dim3(256), 0, s, fin) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "mimi finish launch");
    if (mk) mk->mark(s, PM_MIMI_K_FINISH);
    return PM_OK;
}

pm_status record_decoder(pm_mimi_ctx* c, int B, cudaStream_t s, MimiMarks* mk) {
    const pm_mimi_config& f = c->cfg;
    const MimiIdx ix = mimi_index(f);
    FrontParams fp;
    memset(&fp, 0, sizeof fp);
    fp.io = c->io;
    fp.st = c->st;
    for (int j = 0; j < f.n_q; ++j) fp.cb[j] = c->w[ix.cb0 + j];
    fp.sem_out = c->w[ix.sem_out];
    fp.ac_out = c->w[ix.ac_out];
    fp.up = c->w[ix.up];
    fp.prev = c->prev;
    fp.X = c->X;
    fp.B_max = f.B_max;
    fp.dim = f.dim;
    fp.cb_dim = f.cb_dim;
    fp.card = f.card;
    fp.n_q = f.n_q;
    // the first launch follows the I/O copies, not a kernel: no programmatic dependency
    k_mimi_front<<<dim3((unsigned)((f.dim + 15) / 16), (unsigned)B), 256, 8u * f.cb_dim, s>>>(fp);
    if (cudaGetLastError() != cudaSuccess) return mfail(c, PM_ERR_CUDA, "k_mimi_front launch");
    if (mk) mk->mark(s, PM_MIMI_K_FRONT);
    pm_status st = record_transformer(c, B, s, ix.layer0, mk);
    if (st == PM_OK) st = record_convs(c, B, s, 0, c->layers.size(), mk);
    if (st == PM_OK) st = record_finish(c, B, s, mk);
    return st;
}

pm_status record_encoder(pm_mimi_ctx* c, int B, cudaStream_t s, MimiMarks* mk) {
    const pm_mimi_config& f = c->cfg;
    const MimiEncIdx ix = mimi_enc_index(f);
    const size_t n = c->layers.size();  // the last one is the downsampler, after the transformer
    pm_status st = record_convs(c, B, s, 0, n - 1, mk);
    if (st == PM_OK) st = record_transformer(c, B, s, ix.layer0, mk);
    if (st == PM_OK) st = record_convs(c, B, s, n - 1, n, mk);
    if (st != PM_OK) return st;
    RvqParams rp;
    memset(&rp, 0, sizeof rp);
    rp.e = c->lat;
    rp.w_sem = c->w[ix.sem_in];
    rp.w_ac = c->w[ix.ac_in];
    for (int j = 0; j < f.n_q; ++j) rp.cb[j] = c->w[ix.cb0 + j];
    rp.io = c->io;
    rp.st = c->st;
    rp.dim = f.dim;
    rp.cb_dim = f.cb_dim;
    rp.card = f.card;
    rp.n_q = f.n_q;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(RQ, (unsigned)B);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = rvq_smem(f.dim, f.cb_dim, f.card);
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = RQ;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, k_mimi_rvq, rp) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi rvq launch");
        if (mk) mk->mark(s, PM_MIMI_K_RVQ);
    }
    return record_finish(c, B, s, mk);
}

// largest dynamic shared memory any launch of this context asks for
size_t mimi_smem_need(const pm_mimi_config& f, const std::vector<MimiLayer>& layers, int encoder) {
    size_t m = gemv_smem(2 * f.B_max, f.dim > f.ffn ? f.dim : f.ffn);
    if (attn_smem(f.ctx) > m) m = attn_smem(f.ctx);
    if (encoder && rvq_smem(f.dim, f.cb_dim, f.card) > m) m = rvq_smem(f.dim, f.cb_dim, f.card);
    for (const MimiLayer& L : layers)
        for (int B : {1, f.B_max}) {
            const ConvLaunch cl = conv_launch(L, B);
            if (cl.smem > m) m = cl.smem;
        }
    return m;
}

cudaError_t mimi_func_attributes(size_t smem) {
    const int v = (int)smem;
    cudaError_t e = cudaSuccess;
    auto set = [&](const void* fn) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
    };
#define PM_MIMI_SET_GEMV(NQ)                                   \
    set((const void*)k_mimi_gemv<MP_LN, ME_STORE, NQ>);        \
    set((const void*)k_mimi_gemv<MP_LN, ME_GELU, NQ>);         \
    set((const void*)k_mimi_gemv<MP_NONE, ME_SCALE_RES, NQ>);
    PM_MIMI_SET_GEMV(2)
    PM_MIMI_SET_GEMV(4)
    PM_MIMI_SET_GEMV(8)
    PM_MIMI_SET_GEMV(16)
#undef PM_MIMI_SET_GEMV
    set((const void*)k_mimi_conv_rows<4>);
    set((const void*)k_mimi_conv_rows<16>);
    set((const void*)k_mimi_conv_rows<32>);
    set((const void*)k_mimi_conv_tiled<4>);
    set((const void*)k_mimi_conv_tiled<8>);
    set((const void*)k_mimi_conv_tiled<16>);
    set((const void*)k_mimi_front);
    set((const void*)k_mimi_attn);
    set((const void*)k_mimi_rvq);
    return e;
}

pm_status mimi_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors, void* cuda_stream,
                      pm_mimi_ctx** out, int encoder) {
    g_mimi_create_error.clear();
    const char* fn = encoder ? "pm_mimi_encoder_create: " : "pm_mimi_create: ";
    auto refuse = [&](pm_status s, const std::string& m) {
        g_mimi_create_error = fn + m;
        return s;
    };
    if (!cfg || !tensors || !out) return refuse(PM_ERR_ARG, "NULL argument");
    *out = nullptr;
    if (const char* why = mimi_check(cfg)) return refuse(PM_ERR_ARG, why);
    if (encoder)
        if (const char* why = mimi_encoder_check(cfg)) return refuse(PM_ERR_ARG, why);
    const int total = encoder ? mimi_enc_index(*cfg).total : mimi_index(*cfg).total;
    if (n_tensors != total) return refuse(PM_ERR_ARG, "expected " + std::to_string(total) + " tensors");
    for (int i = 0; i < n_tensors; ++i) {
        if (!tensors[i] || (reinterpret_cast<uintptr_t>(tensors[i]) & 15u))
            return refuse(PM_ERR_ARG, "tensor " + std::to_string(i) + " NULL or not 16-byte aligned");
        cudaPointerAttributes a;
        const bool dev = cudaPointerGetAttributes(&a, tensors[i]) == cudaSuccess &&
                         (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged);
        cudaGetLastError();
        if (!dev) return refuse(PM_ERR_ARG, "tensor " + std::to_string(i) + " is not device memory");
    }
    const std::vector<MimiLayer> layers = encoder ? seanet_encoder_layers(*cfg) : seanet_layers(*cfg);
    const size_t smem = mimi_smem_need(*cfg, layers, encoder);
    if (smem > 227u * 1024u) return refuse(PM_ERR_UNSUPPORTED, "shared memory above 227 KB");
    pm_mimi_ctx* c = new pm_mimi_ctx();
    c->cfg = *cfg;
    c->encoder = encoder;
    const pm_mimi_config& f = c->cfg;
    c->frame_samples = 2;
    for (int i = 0; i < f.n_ratios; ++i) c->frame_samples *= f.ratios[i];
    cudaGetDevice(&c->device);
    c->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    for (int i = 0; i < n_tensors; ++i) c->w.push_back(static_cast<const uint16_t*>(tensors[i]));
    c->layers = layers;
    auto bail = [&](pm_status s, const char* m) {
        pm_mimi_destroy(c);
        g_mimi_create_error = std::string(fn) + m;
        return s;
    };
    if (mimi_func_attributes(smem) != cudaSuccess) {
        cudaGetLastError();
        return bail(PM_ERR_CUDA, "cudaFuncSetAttribute");
    }
    // one allocation for state, activations and I/O
    const int BM = f.B_max, D = f.dim;
    void *p_frame, *p_pos, *p_abort, *p_status, *p_budget, *p_io, *p_codes, *p_pcm, *p_prev, *p_X, *p_qkv, *p_o,
        *p_hf, *p_kv, *p_lat, *p_freq;
    std::vector<std::pair<void**, size_t>> items = {
        {&p_frame, 4u * BM},
        {&p_pos, 4u * BM},
        {&p_abort, 4u},
        {&p_status, 4u},
        {&p_budget, 4u},
        {&p_io, sizeof(MimiIO)},
        {&p_codes, 4u * BM * f.n_q},
        {&p_pcm, encoder ? 4u * BM * c->frame_samples : 16u},
        {&p_prev, 4u * 2 * BM * D},
        {&p_X, 4u * BM * 2 * D},
        {&p_qkv, 4u * BM * 2 * 3 * D},
        {&p_o, 4u * BM * 2 * D},
        {&p_hf, 4u * BM * 2 * f.ffn},
        {&p_kv, 4u * (size_t)f.n_layers * 2 * BM * f.heads * (f.ctx + 1) * MDH},
        {&p_lat, 4u * BM * D},
        {&p_freq, 8u * (MDH / 2)},
    };
    int n_act = 0;
    for (const MimiLayer& L : c->layers)
        for (int k : {L.in_buf, L.out_raw, L.out_act, L.res_buf}) n_act = k + 1 > n_act ? k + 1 : n_act;
    std::vector<size_t> act_sizes(n_act, 0);
    for (const MimiLayer& L : c->layers) {
        const size_t n = (size_t)BM * L.Cout * (L.P > 1 ? L.T * L.P : L.T);
        for (int k : {L.out_raw, L.out_act})
            if (k >= 0 && n > act_sizes[k]) act_sizes[k] = n;
    }
    c->acts.assign(act_sizes.size(), nullptr);
    for (size_t i = 0; i < act_sizes.size(); ++i) items.push_back({reinterpret_cast<void**>(&c->acts[i]), 4u * act_sizes[i]});
    c->states.assign(c->layers.size(), nullptr);
    c->state_per_stream.assign(c->layers.size(), 0);
    for (size_t i = 0; i < c->layers.size(); ++i) {
        c->state_per_stream[i] = layer_state(c->layers[i]);
        items.push_back({reinterpret_cast<void**>(&c->states[i]), 4u * 2 * BM * c->state_per_stream[i]});
    }
    size_t total_bytes = 0;
    for (auto& it : items) total_bytes = (total_bytes + 255) / 256 * 256 + (it.second + 15) / 16 * 16;
    if (cudaMalloc(&c->block, total_bytes) != cudaSuccess) {
        cudaGetLastError();
        return bail(PM_ERR_OOM, "device allocation");
    }
    if (cudaMemset(c->block, 0, total_bytes) != cudaSuccess) return bail(PM_ERR_CUDA, "cudaMemset");
    size_t off = 0;
    for (auto& it : items) {
        off = (off + 255) / 256 * 256;
        *it.first = static_cast<uint8_t*>(c->block) + off;
        off += (it.second + 15) / 16 * 16;
    }
    c->st.frame = (int32_t*)p_frame;
    c->st.pos = (int32_t*)p_pos;
    c->st.abort = (uint32_t*)p_abort;
    c->st.status = (uint32_t*)p_status;
    c->st.wait_budget = (const uint32_t*)p_budget;
    {
        const uint32_t b0 = PM_SPIN_LIMIT;
        if (cudaMemcpy(p_budget, &b0, 4, cudaMemcpyHostToDevice) != cudaSuccess) return bail(PM_ERR_CUDA, "cudaMemcpy");
    }
    c->io = (MimiIO*)p_io;
    c->codes_dev = (int32_t*)p_codes;
    c->pcm_dev = (float*)p_pcm;
    c->prev = (float*)p_prev;
    c->X = (float*)p_X;
    c->qkv = (float*)p_qkv;
    c->o = (float*)p_o;
    c->hf = (float*)p_hf;
    c->kv = (float*)p_kv;
    c->lat = (float*)p_lat;
    c->freq = (double*)p_freq;
    // tap-major convolution weights, re-laid from the caller's tensors once
    std::vector<size_t> wt_off;
    size_t wt_total = 0;
    for (const MimiLayer& L : c->layers) {
        wt_off.push_back(wt_total);
        wt_total += ((size_t)L.P * L.Cout * L.NT * L.Cin + 7) / 8 * 8;
    }
    if (cudaMalloc((void**)&c->wt_block, 2 * wt_total) != cudaSuccess) {
        cudaGetLastError();
        return bail(PM_ERR_OOM, "device allocation (re-laid weights)");
    }
    for (size_t i = 0; i < c->layers.size(); ++i) {
        MimiLayer& L = c->layers[i];
        L.Wt = c->wt_block + wt_off[i];
        L.bias = L.no_bias ? nullptr : c->w[L.wi + 1];
        L.state = c->states[i];
        k_mimi_relayout<<<256, 256>>>(c->w[L.wi], c->wt_block + wt_off[i], L.Cin, L.Cout, L.NT, L.P, L.S);
        if (cudaGetLastError() != cudaSuccess) return bail(PM_ERR_CUDA, "relayout launch");
    }
    // RoPE frequency of pair j: theta^(-2j / 64)
    std::vector<double> fq(MDH / 2);
    for (int j = 0; j < MDH / 2; ++j) fq[j] = exp(-log((double)f.rope_theta) * (2.0 * j) / (double)MDH);
    if (cudaMemcpy(c->freq, fq.data(), 8u * fq.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(PM_ERR_CUDA, "cudaMemcpy");
    c->host_io_bytes = 64u + (encoder ? 4u * BM * c->frame_samples : 4u * BM * f.n_q);
    if (cudaHostAlloc((void**)&c->host_io, c->host_io_bytes, cudaHostAllocDefault) != cudaSuccess)
        return bail(PM_ERR_OOM, "pinned host allocation");
    if (cudaEventCreateWithFlags(&c->io_done, cudaEventDisableTiming) != cudaSuccess)
        return bail(PM_ERR_CUDA, "cudaEventCreate");
    if (cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess)
        return bail(PM_ERR_CUDA, "cudaStreamCreate");
    c->graphs.assign(BM + 1, nullptr);
    if (cudaDeviceSynchronize() != cudaSuccess) return bail(PM_ERR_CUDA, "cudaDeviceSynchronize");
    *out = c;
    return PM_OK;
}

// device, managed or host-mapped memory: the pointer the kernels use, or NULL
template <typename T>
T* device_view(T* p) {
    cudaPointerAttributes a;
    T* d = nullptr;
    if (p && cudaPointerGetAttributes(&a, p) == cudaSuccess) {
        if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) d = p;
        if (a.type == cudaMemoryTypeHost && a.devicePointer) d = static_cast<T*>(a.devicePointer);
    }
    cudaGetLastError();
    return d;
}

bool is_device(const void* p) {
    cudaPointerAttributes a;
    const bool d = p && cudaPointerGetAttributes(&a, p) == cudaSuccess &&
                   (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged);
    cudaGetLastError();
    return d;
}

// decoder: validate the call's pointers and codes, then copy the I/O block (and host codes)
// on the context's stream; graph or eager launches follow
pm_status mimi_stage(pm_mimi_ctx* c, int B, const int32_t* codes, float* pcm) {
    const pm_mimi_config& f = c->cfg;
    if (c->encoder) return mfail(c, PM_ERR_STATE, "pm_mimi_decode on an encoder context");
    if (B < 1 || B > f.B_max || !codes || !pcm) return mfail(c, PM_ERR_ARG, "pm_mimi_decode: bad B or NULL pointer");
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    float* pcm_dev = device_view(pcm);
    if (!pcm_dev || (reinterpret_cast<uintptr_t>(pcm) & 3u))
        return mfail(c, PM_ERR_ARG, "pm_mimi_decode: pcm must be 4-byte aligned device, managed or host-mapped memory");
    const bool dev_codes = is_device(codes);
    if (!dev_codes)
        for (int i = 0; i < B * f.n_q; ++i)
            if (codes[i] < 0 || codes[i] >= f.card)
                return mfail(c, PM_ERR_INVALID_ID,
                             "pm_mimi_decode: code " + std::to_string(codes[i]) + " at " + std::to_string(i) + " out of range");
    // the previous call's copies out of the pinned staging must be done before it is reused
    if (cudaEventSynchronize(c->io_done) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaEventSynchronize");
    MimiIO io;
    memset(&io, 0, sizeof io);
    io.codes = dev_codes ? codes : c->codes_dev;
    io.pcm = pcm_dev;
    memcpy(c->host_io, &io, sizeof io);
    if (!dev_codes) {
        memcpy(c->host_io + 64, codes, 4u * B * f.n_q);
        if (cudaMemcpyAsync(c->codes_dev, c->host_io + 64, 4u * B * f.n_q, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
            return mfail(c, PM_ERR_CUDA, "codes copy");
    }
    if (cudaMemcpyAsync(c->io, c->host_io, sizeof io, cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
        cudaEventRecord(c->io_done, c->stream) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "I/O block copy");
    return PM_OK;
}

// encoder: the same for PCM in, codes (and the latent) out
pm_status mimi_stage_enc(pm_mimi_ctx* c, int B, const float* pcm, int32_t* codes, float* latent) {
    const pm_mimi_config& f = c->cfg;
    if (!c->encoder) return mfail(c, PM_ERR_STATE, "pm_mimi_encode on a decoder context");
    if (B < 1 || B > f.B_max || !pcm || !codes) return mfail(c, PM_ERR_ARG, "pm_mimi_encode: bad B or NULL pointer");
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    int32_t* codes_dev = device_view(codes);
    if (!codes_dev || (reinterpret_cast<uintptr_t>(codes) & 3u))
        return mfail(c, PM_ERR_ARG, "pm_mimi_encode: codes must be 4-byte aligned device, managed or host-mapped memory");
    float* lat_dev = nullptr;
    if (latent) {
        lat_dev = device_view(latent);
        if (!lat_dev || (reinterpret_cast<uintptr_t>(latent) & 3u))
            return mfail(c, PM_ERR_ARG, "pm_mimi_encode: latent must be device, managed or host-mapped memory");
    }
    const bool dev_pcm = is_device(pcm);
    if (dev_pcm && (reinterpret_cast<uintptr_t>(pcm) & 3u)) return mfail(c, PM_ERR_ARG, "pm_mimi_encode: pcm not aligned");
    if (cudaEventSynchronize(c->io_done) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaEventSynchronize");
    MimiIO io;
    memset(&io, 0, sizeof io);
    io.pcm_in = dev_pcm ? pcm : c->pcm_dev;
    io.codes_out = codes_dev;
    io.latent_out = lat_dev;
    memcpy(c->host_io, &io, sizeof io);
    if (!dev_pcm) {
        const size_t n = 4u * (size_t)B * c->frame_samples;
        memcpy(c->host_io + 64, pcm, n);
        if (cudaMemcpyAsync(c->pcm_dev, c->host_io + 64, n, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
            return mfail(c, PM_ERR_CUDA, "pcm copy");
    }
    if (cudaMemcpyAsync(c->io, c->host_io, sizeof io, cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
        cudaEventRecord(c->io_done, c->stream) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "I/O block copy");
    return PM_OK;
}

pm_status mimi_record(pm_mimi_ctx* c, int B, cudaStream_t s, MimiMarks* mk) {
    return c->encoder ? record_encoder(c, B, s, mk) : record_decoder(c, B, s, mk);
}

pm_status mimi_graph(pm_mimi_ctx* c, int B) {
    if (B < 1 || B > c->cfg.B_max || c->graphs[B]) return PM_OK;
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    if (cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "cudaStreamBeginCapture");
    pm_status st = mimi_record(c, B, c->cap, nullptr);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(c->cap, &g);
    if (st != PM_OK || e != cudaSuccess || cudaGraphInstantiate(&c->graphs[B], g, 0) != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        c->graphs[B] = nullptr;
        cudaGetLastError();
        return st != PM_OK ? st : mfail(c, PM_ERR_CUDA, "mimi graph capture");
    }
    cudaGraphDestroy(g);
    return PM_OK;
}

pm_status mimi_profile_run(pm_mimi_ctx* c, int B, float* ms, int32_t* kind, int n_max, int* n) {
    MimiMarks mk;
    cudaEvent_t start;
    if (cudaEventCreate(&start) != cudaSuccess || cudaEventRecord(start, c->stream) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "profile: event");
    pm_status st = mimi_record(c, B, c->stream, &mk);
    const bool synced = cudaStreamSynchronize(c->stream) == cudaSuccess;
    int k = 0;
    cudaEvent_t prev = start;
    for (size_t i = 0; i < mk.ev.size(); ++i) {
        float t = 0.f;
        if (synced && k < n_max && cudaEventElapsedTime(&t, prev, mk.ev[i]) == cudaSuccess) {
            ms[k] = t;
            kind[k] = mk.kind[i];
            ++k;
        }
        prev = mk.ev[i];
    }
    for (auto e : mk.ev) cudaEventDestroy(e);
    cudaEventDestroy(start);
    *n = k;
    if (st != PM_OK) return st;
    return synced ? PM_OK : mfail(c, PM_ERR_CUDA, "profile: synchronize");
}

}  // namespace

extern "C" int pm_mimi_tensor_count(const pm_mimi_config* cfg) {
    if (!cfg || mimi_check(cfg)) return -1;
    return mimi_index(*cfg).total;
}

extern "C" int pm_mimi_encoder_tensor_count(const pm_mimi_config* cfg) {
    if (!cfg || mimi_check(cfg) || mimi_encoder_check(cfg)) return -1;
    return mimi_enc_index(*cfg).total;
}

extern "C" pm_status pm_mimi_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors,
                                    void* cuda_stream, pm_mimi_ctx** out) {
    return mimi_create(cfg, tensors, n_tensors, cuda_stream, out, 0);
}

extern "C" pm_status pm_mimi_encoder_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors,
                                            void* cuda_stream, pm_mimi_ctx** out) {
    return mimi_create(cfg, tensors, n_tensors, cuda_stream, out, 1);
}

extern "C" void pm_mimi_destroy(pm_mimi_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    if (c->block) cudaStreamSynchronize(c->stream);
    for (auto g : c->graphs)
        if (g) cudaGraphExecDestroy(g);
    if (c->io_done) cudaEventDestroy(c->io_done);
    if (c->host_io) cudaFreeHost(c->host_io);
    if (c->cap) cudaStreamDestroy(c->cap);
    if (c->wt_block) cudaFree(c->wt_block);
    if (c->block) cudaFree(c->block);
    delete c;
}

extern "C" pm_status pm_mimi_decode(pm_mimi_ctx* c, int B, const int32_t* codes, float* pcm) {
    if (!c) return PM_ERR_ARG;
    if (c->encoder) return mfail(c, PM_ERR_STATE, "pm_mimi_decode on an encoder context");
    pm_status st = mimi_graph(c, B);
    if (st == PM_OK) st = mimi_stage(c, B, codes, pcm);
    if (st != PM_OK) return st;
    if (cudaGraphLaunch(c->graphs[B], c->stream) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi launch");
    return PM_OK;
}

extern "C" pm_status pm_mimi_encode(pm_mimi_ctx* c, int B, const float* pcm, int32_t* codes, float* latent) {
    if (!c) return PM_ERR_ARG;
    if (!c->encoder) return mfail(c, PM_ERR_STATE, "pm_mimi_encode on a decoder context");
    pm_status st = mimi_graph(c, B);
    if (st == PM_OK) st = mimi_stage_enc(c, B, pcm, codes, latent);
    if (st != PM_OK) return st;
    if (cudaGraphLaunch(c->graphs[B], c->stream) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi launch");
    return PM_OK;
}

extern "C" pm_status pm_mimi_profile(pm_mimi_ctx* c, int B, const int32_t* codes, float* pcm, float* ms,
                                     int32_t* kind, int n_max, int* n) {
    if (!c) return PM_ERR_ARG;
    if (!ms || !kind || !n || n_max < 1) return mfail(c, PM_ERR_ARG, "pm_mimi_profile: NULL output or n_max < 1");
    pm_status st = mimi_stage(c, B, codes, pcm);
    return st != PM_OK ? st : mimi_profile_run(c, B, ms, kind, n_max, n);
}

extern "C" pm_status pm_mimi_encode_profile(pm_mimi_ctx* c, int B, const float* pcm, int32_t* codes, float* latent,
                                            float* ms, int32_t* kind, int n_max, int* n) {
    if (!c) return PM_ERR_ARG;
    if (!ms || !kind || !n || n_max < 1) return mfail(c, PM_ERR_ARG, "pm_mimi_encode_profile: NULL output or n_max < 1");
    pm_status st = mimi_stage_enc(c, B, pcm, codes, latent);
    return st != PM_OK ? st : mimi_profile_run(c, B, ms, kind, n_max, n);
}

extern "C" pm_status pm_mimi_reset(pm_mimi_ctx* c, const int32_t* mask) {
    if (!c) return PM_ERR_ARG;
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    const pm_mimi_config& f = c->cfg;
    const int BM = f.B_max;
    // a fresh stream: frame 0 at position 0, no previous latent, zero convolution history
    // and zero carried columns (the ring needs no clearing: the window only reaches
    // positions written since the reset)
    for (int b = 0; b < BM; ++b) {
        if (mask && !mask[b]) continue;
        bool ok = cudaMemsetAsync(c->st.frame + b, 0, 4, c->stream) == cudaSuccess &&
                  cudaMemsetAsync(c->st.pos + b, 0, 4, c->stream) == cudaSuccess;
        for (int par = 0; par < 2 && ok; ++par) {
            ok = cudaMemsetAsync(c->prev + ((size_t)par * BM + b) * f.dim, 0, 4u * f.dim, c->stream) == cudaSuccess;
            for (size_t i = 0; i < c->states.size() && ok; ++i) {
                const size_t n = c->state_per_stream[i];
                if (n) ok = cudaMemsetAsync(c->states[i] + ((size_t)par * BM + b) * n, 0, 4u * n, c->stream) == cudaSuccess;
            }
        }
        if (!ok) return mfail(c, PM_ERR_CUDA, "pm_mimi_reset: cudaMemsetAsync");
    }
    return PM_OK;
}

extern "C" pm_status pm_mimi_status(pm_mimi_ctx* c) {
    if (!c) return PM_ERR_ARG;
    if (cudaSetDevice(c->device) != cudaSuccess || cudaStreamSynchronize(c->stream) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "pm_mimi_status: synchronize");
    uint32_t s = 0;
    if (cudaMemcpy(&s, c->st.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess || cudaMemset(c->st.status, 0, 4) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "pm_mimi_status: read");
    if (s & 2u) return mfail(c, PM_ERR_TIMEOUT, "a bounded wait of the quantiser ran out (that call's codes are undefined)");
    if (s & ~1u) return mfail(c, PM_ERR_CUDA, "unknown device status");
    return s ? mfail(c, PM_ERR_INVALID_ID, "a code given in device memory was out of range (that call was a no-op)") : PM_OK;
}

extern "C" pm_status pm_mimi_set_wait_budget(pm_mimi_ctx* c, uint32_t polls) {
    if (!c) return PM_ERR_ARG;
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    const uint32_t v = polls == PM_WAIT_BUDGET_DEFAULT ? (uint32_t)PM_SPIN_LIMIT : polls;
    // ordered on the context's stream: calls before it keep the old budget
    if (cudaStreamSynchronize(c->stream) != cudaSuccess ||
        cudaMemcpy((void*)c->st.wait_budget, &v, 4, cudaMemcpyHostToDevice) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "pm_mimi_set_wait_budget");
    return PM_OK;
}

extern "C" pm_status pm_mimi_get_frames(pm_mimi_ctx* c, int32_t* frames) {
    if (!c || !frames) return PM_ERR_ARG;
    if (cudaSetDevice(c->device) != cudaSuccess || cudaStreamSynchronize(c->stream) != cudaSuccess ||
        cudaMemcpy(frames, c->st.frame, 4u * c->cfg.B_max, cudaMemcpyDeviceToHost) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "pm_mimi_get_frames");
    return PM_OK;
}

extern "C" const char* pm_mimi_last_error(const pm_mimi_ctx* c) {
    return c ? c->err.c_str() : g_mimi_create_error.c_str();
}
