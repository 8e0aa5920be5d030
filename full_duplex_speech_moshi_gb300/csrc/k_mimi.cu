// Streaming Mimi decoder: code frames -> 24 kHz PCM, one 80 ms frame per stream and call
// ("PersonaPlex native LM audit", chapter "Exact Mimi codec construction": the DECODE
// order of "Complete encode/decode order", the split quantizer, the depthwise latent
// upsampler, the decoder transformer of "Both codec transformer stacks", "SEANet decoder,
// every stage", and the streaming rules of "Stateful streaming, padding and dependency
// boundaries").
//
// One CUDA graph per batch size B:
//   k_mimi_front      codes -> split-RVQ lookup -> the two output projections -> latent;
//                     the depthwise ConvTranspose (kernel 4, stride 2) makes the frame's two
//                     25 Hz positions from this latent and the previous one
//   per block         LayerNorm-prologue GEMV (in_proj) -> k_mimi_attn (RoPE, ring append,
//                     causal window) -> GEMV (out_proj) + LayerScale + residual ->
//                     LayerNorm GEMV (lin1) + GELU -> GEMV (lin2) + LayerScale + residual
//   SEANet decoder    causal Conv1d / ConvTranspose1d with ELU on their inputs and the
//                     residual units; a convolution keeps its last k-1 (activated) inputs,
//                     a transposed convolution its k-s unfinished outputs
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

constexpr int MDH = 64;  // transformer head width
constexpr int TILE = 32; // positions per CTA of the tiled convolutions

struct MimiIO {
    const int32_t* codes;  // [B][n_q]
    float* pcm;            // [B][frame_samples]
};

struct MimiState {
    int32_t* frame;     // [B_max] frames decoded since reset (state parity = frame & 1)
    int32_t* pos;       // [B_max] 25 Hz position of the frame's first position
    uint32_t* abort;    // [1] nonzero: this call's codes were invalid (nothing advances)
    uint32_t* status;   // [1] sticky: an invalid device code was seen
};

__device__ __forceinline__ float bf(const uint16_t* p, size_t i) { return __uint_as_float((uint32_t)p[i] << 16); }

__device__ __forceinline__ float elu_f(float x) { return x > 0.f ? x : expm1f(x); }

__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

__device__ __forceinline__ bool aborted(const MimiState& st) { return *(volatile const uint32_t*)st.abort != 0u; }

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

// grid (dim / 64, B), 256 threads: warp w makes channels 64 x + 8 w .. + 7
__global__ void __launch_bounds__(256) k_mimi_front(const FrontParams p) {
    extern __shared__ float sm[];
    float* sem = sm;              // semantic vector  [cb_dim]
    float* ac = sm + p.cb_dim;    // acoustic sum     [cb_dim]
    __shared__ int s_codes[16];
    __shared__ int s_bad;
    const int b = blockIdx.y, t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t == 0) s_bad = 0;
    __syncthreads();
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
        sem[k] = bf(p.cb[0], (size_t)s_codes[0] * p.cb_dim + k);
        float a = 0.f;
        for (int j = 1; j < p.n_q; ++j) a += bf(p.cb[j], (size_t)s_codes[j] * p.cb_dim + k);
        ac[k] = a;
    }
    __syncthreads();
    const int par = p.st.frame[b] & 1;
    for (int r = 0; r < 8; ++r) {
        const int c = blockIdx.x * 64 + warp * 8 + r;
        if (c >= p.dim) break;
        const uint16_t* ws = p.sem_out + (size_t)c * p.cb_dim;
        const uint16_t* wa = p.ac_out + (size_t)c * p.cb_dim;
        float v = 0.f;
        for (int k = 8 * lane; k < p.cb_dim; k += 256) {
            const uint4 a = *reinterpret_cast<const uint4*>(ws + k);
            const uint4 e = *reinterpret_cast<const uint4*>(wa + k);
            const float* x = sem + k;
            const float* y = ac + k;
            v = fmaf(bf16lo(a.x), x[0], v);
            v = fmaf(bf16hi(a.x), x[1], v);
            v = fmaf(bf16lo(a.y), x[2], v);
            v = fmaf(bf16hi(a.y), x[3], v);
            v = fmaf(bf16lo(a.z), x[4], v);
            v = fmaf(bf16hi(a.z), x[5], v);
            v = fmaf(bf16lo(a.w), x[6], v);
            v = fmaf(bf16hi(a.w), x[7], v);
            v = fmaf(bf16lo(e.x), y[0], v);
            v = fmaf(bf16hi(e.x), y[1], v);
            v = fmaf(bf16lo(e.y), y[2], v);
            v = fmaf(bf16hi(e.y), y[3], v);
            v = fmaf(bf16lo(e.z), y[4], v);
            v = fmaf(bf16hi(e.z), y[5], v);
            v = fmaf(bf16lo(e.w), y[6], v);
            v = fmaf(bf16hi(e.w), y[7], v);
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

// grid ceil(R / 8), 256 threads, a warp per output row; nq <= 16, K a multiple of 128
template <int PRO, int EPI>
__global__ void __launch_bounds__(256) k_mimi_gemv(const MGemvParams p) {
    extern __shared__ float xs[];  // [nq][K]
    __shared__ float s_m[16], s_r[16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    if (aborted(p.st)) return;
    for (int i = 4 * t; i < p.nq * p.K; i += 4 * blockDim.x)
        *reinterpret_cast<float4*>(xs + i) = *reinterpret_cast<const float4*>(p.x + i);
    __syncthreads();
    if (PRO == MP_LN) {
        // mean and biased variance per position, then (x - m) / sqrt(v + eps) * w + b
        for (int q = warp; q < p.nq; q += 8) {
            float s = 0.f;
            for (int k = lane; k < p.K; k += 32) s += xs[q * p.K + k];
            const float m = warp_sum(s) / (float)p.K;
            float v = 0.f;
            for (int k = lane; k < p.K; k += 32) {
                const float d = xs[q * p.K + k] - m;
                v = fmaf(d, d, v);
            }
            v = warp_sum(v);
            if (lane == 0) {
                s_m[q] = m;
                s_r[q] = 1.0f / sqrtf(v / (float)p.K + p.eps);
            }
        }
        __syncthreads();
        for (int i = t; i < p.nq * p.K; i += blockDim.x) {
            const int q = i / p.K, k = i - q * p.K;
            xs[i] = fmaf((xs[i] - s_m[q]) * s_r[q], bf(p.ln_w, k), bf(p.ln_b, k));
        }
        __syncthreads();
    }
    const int r = blockIdx.x * 8 + warp;
    if (r >= p.R) return;
    float acc[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
    const uint16_t* wr = p.W + (size_t)r * p.K;
    for (int k = 4 * lane; k < p.K; k += 128) {
        const uint2 w = *reinterpret_cast<const uint2*>(wr + k);
        const float w0 = bf16lo(w.x), w1 = bf16hi(w.x), w2 = bf16lo(w.y), w3 = bf16hi(w.y);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            if (q < p.nq) {
                const float4 x = *reinterpret_cast<const float4*>(xs + q * p.K + k);
                float a = acc[q];
                a = fmaf(w0, x.x, a);
                a = fmaf(w1, x.y, a);
                a = fmaf(w2, x.z, a);
                a = fmaf(w3, x.w, a);
                acc[q] = a;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        if (q < p.nq) {
            const float v = warp_sum(acc[q]);
            if (lane == 0) {
                float* o = p.y + (size_t)q * p.R + r;
                if (EPI == ME_STORE) *o = v;
                if (EPI == ME_GELU) *o = gelu_f(v);
                if (EPI == ME_SCALE_RES) *o = fmaf(v, bf(p.scale, r), *o);
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

__global__ void __launch_bounds__(256) k_mimi_attn(const MAttnParams p) {
    __shared__ float qr[2][MDH];
    __shared__ float s_m[8][2], s_l[8][2];
    __shared__ float s_o[8][2][MDH];
    const int b = blockIdx.x, h = blockIdx.y;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (aborted(p.st)) return;
    const int pos0 = p.st.pos[b];
    const size_t hb = ((size_t)b * p.H + h) * p.RS;
    // RoPE on adjacent pairs (2j, 2j + 1) of q and k at the frame's two positions
    if (t < MDH) {
        const int i = t / (MDH / 2), j = t % (MDH / 2);
        const int pos = pos0 + i;
        double sn, cs;
        sincos((double)pos * p.freq[j], &sn, &cs);
        const float c = (float)cs, s = (float)sn;
        const float* row = p.qkv + ((size_t)b * 2 + i) * 3 * p.dim + h * MDH;
        const float q0 = row[2 * j], q1 = row[2 * j + 1];
        const float k0 = row[p.dim + 2 * j], k1 = row[p.dim + 2 * j + 1];
        qr[i][2 * j] = q0 * c - q1 * s;
        qr[i][2 * j + 1] = q0 * s + q1 * c;
        float* kd = p.kc + (hb + (size_t)(pos % p.RS)) * MDH;
        float* vd = p.vc + (hb + (size_t)(pos % p.RS)) * MDH;
        kd[2 * j] = k0 * c - k1 * s;
        kd[2 * j + 1] = k0 * s + k1 * c;
        vd[2 * j] = row[2 * p.dim + 2 * j];
        vd[2 * j + 1] = row[2 * p.dim + 2 * j + 1];
    }
    __syncthreads();
    // the query at position pos sees keys max(0, pos - ctx + 1) .. pos; warp w takes keys
    // lo + w, lo + w + 8, ... with a running maximum and sum; lane l holds coordinates 2l, 2l+1
    for (int i = 0; i < 2; ++i) {
        const int pos = pos0 + i, lo = max(0, pos - p.ctx + 1);
        const float qa = qr[i][2 * lane], qb = qr[i][2 * lane + 1];
        float m = -INFINITY, l = 0.f, a0 = 0.f, a1 = 0.f;
        for (int kp = lo + warp; kp <= pos; kp += 8) {
            const float2 kv = *reinterpret_cast<const float2*>(p.kc + (hb + (size_t)(kp % p.RS)) * MDH + 2 * lane);
            const float2 vv = *reinterpret_cast<const float2*>(p.vc + (hb + (size_t)(kp % p.RS)) * MDH + 2 * lane);
            const float sc = warp_sum(fmaf(qa, kv.x, qb * kv.y)) * p.scale_log2;
            const float mn = fmaxf(m, sc);
            const float f = exp2f(m - mn), e = exp2f(sc - mn);
            l = fmaf(l, f, e);
            a0 = fmaf(a0, f, e * vv.x);
            a1 = fmaf(a1, f, e * vv.y);
            m = mn;
        }
        if (lane == 0) {
            s_m[warp][i] = m;
            s_l[warp][i] = l;
        }
        s_o[warp][i][2 * lane] = a0;
        s_o[warp][i][2 * lane + 1] = a1;
    }
    __syncthreads();
    if (t < 2 * MDH) {
        const int i = t / MDH, d = t % MDH;
        float M = -INFINITY;
        for (int w = 0; w < 8; ++w) M = fmaxf(M, s_m[w][i]);
        float L = 0.f, A = 0.f;
        for (int w = 0; w < 8; ++w) {
            const float f = (s_m[w][i] == -INFINITY) ? 0.f : exp2f(s_m[w][i] - M);
            L = fmaf(s_l[w][i], f, L);
            A = fmaf(s_o[w][i][d], f, A);
        }
        p.o[((size_t)b * 2 + i) * p.dim + h * MDH + d] = A / L;
    }
}

// ------------------------------------------------------------------------------------
// SEANet: causal Conv1d (stride 1) and ConvTranspose1d (kernel 2s, stride s)
// ------------------------------------------------------------------------------------
struct MConvParams {
    const float* in;        // [B][Cin][T] (or [B][T][Cin] when in_pm)
    float* out;             // [B][Cout][T out]: written, or added to (res)
    const MimiIO* io_out;   // when set, the output is the caller's PCM (io_out->pcm)
    const uint16_t* W;      // Conv1d [Cout][Cin][k]; ConvTranspose1d [Cin][Cout][k]
    const uint16_t* bias;   // [Cout]
    float* state;           // Conv1d: [2][B_max][Cin][k-1] activated inputs;
                            // ConvTranspose1d: [2][B_max][Cout][k-s] unfinished outputs
    MimiState st;
    int B_max, Cin, Cout, k, s, T;  // T: input positions of this call
    int elu_in, in_pm, res;
};

// input column tau of channel ci after the optional ELU; tau < 0 is the streaming state
__device__ __forceinline__ float conv_in(const MConvParams& p, int b, int ci, int tau, const float* st_old) {
    if (tau < 0) return st_old[((size_t)b * p.Cin + ci) * (p.k - 1) + (p.k - 1 + tau)];
    const float v = p.in_pm ? p.in[((size_t)b * p.T + tau) * p.Cin + ci] : p.in[((size_t)b * p.Cin + ci) * p.T + tau];
    return p.elu_in ? elu_f(v) : v;
}

__device__ __forceinline__ float* conv_out(const MConvParams& p) { return p.io_out ? p.io_out->pcm : p.out; }

// T <= 16: grid (ceil(Cout / 8), B), a warp per output channel, lanes split the Cin x k
// reduction; the CTA stages the activated window [Cin][k - 1 + T] in shared memory
__global__ void __launch_bounds__(256) k_mimi_conv_w(const MConvParams p) {
    extern __shared__ float win[];
    if (aborted(p.st)) return;
    const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int par = p.st.frame[b] & 1, km = p.k - 1, WL = km + p.T;
    const float* st_old = km ? p.state + (size_t)par * p.B_max * p.Cin * km : nullptr;
    for (int i = threadIdx.x; i < p.Cin * WL; i += blockDim.x) {
        const int ci = i / WL, m = i - ci * WL;
        win[i] = conv_in(p, b, ci, m - km, st_old);
    }
    __syncthreads();
    if (km && blockIdx.x == 0) {
        float* st_new = p.state + (size_t)(par ^ 1) * p.B_max * p.Cin * km;
        for (int i = threadIdx.x; i < p.Cin * km; i += blockDim.x) {
            const int ci = i / km, m = i - ci * km;
            st_new[((size_t)b * p.Cin + ci) * km + m] = win[ci * WL + p.T + m];
        }
    }
    const int co = blockIdx.x * 8 + warp;
    if (co >= p.Cout) return;
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.f;
    const uint16_t* wr = p.W + (size_t)co * p.Cin * p.k;
    for (int idx = lane; idx < p.Cin * p.k; idx += 32) {
        const int ci = idx / p.k, j = idx - ci * p.k;
        const float w = bf(wr, idx);
        const float* x = win + ci * WL + j;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t < p.T) acc[t] = fmaf(w, x[t], acc[t]);
    }
    float* out = conv_out(p);
    const float bias = bf(p.bias, co);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        if (t < p.T) {
            const float v = warp_sum(acc[t]) + bias;
            if (lane == 0) {
                float* o = out + ((size_t)b * p.Cout + co) * p.T + t;
                *o = p.res ? *o + v : v;
            }
        }
    }
}

// grid (ceil(T / 32), ceil(Cout / 8), B): lane = position in the tile, warp = channel; the
// CTA stages the activated inputs [Cin][32 + k - 1] once
__global__ void __launch_bounds__(256) k_mimi_conv_t(const MConvParams p) {
    extern __shared__ float win[];
    if (aborted(p.st)) return;
    const int b = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int par = p.st.frame[b] & 1, km = p.k - 1, WL = TILE + km;
    const int t0 = blockIdx.x * TILE;
    const float* st_old = km ? p.state + (size_t)par * p.B_max * p.Cin * km : nullptr;
    for (int i = threadIdx.x; i < p.Cin * WL; i += blockDim.x) {
        const int ci = i / WL, m = i - ci * WL, tau = t0 - km + m;
        win[i] = tau < p.T ? conv_in(p, b, ci, tau, st_old) : 0.f;
    }
    __syncthreads();
    if (km && blockIdx.y == 0 && t0 + TILE >= p.T) {
        // the last tile's window holds the call's last k - 1 inputs
        float* st_new = p.state + (size_t)(par ^ 1) * p.B_max * p.Cin * km;
        for (int i = threadIdx.x; i < p.Cin * km; i += blockDim.x) {
            const int ci = i / km, m = i - ci * km;
            st_new[((size_t)b * p.Cin + ci) * km + m] = win[ci * WL + (p.T - t0) + m];
        }
    }
    const int co = blockIdx.y * 8 + warp, t = t0 + lane;
    if (co >= p.Cout || t >= p.T) return;
    float acc = bf(p.bias, co);
    const uint16_t* wr = p.W + (size_t)co * p.Cin * p.k;
    for (int ci = 0; ci < p.Cin; ++ci) {
        const float* x = win + ci * WL + lane;
        for (int j = 0; j < p.k; ++j) acc = fmaf(bf(wr, ci * p.k + j), x[j], acc);
    }
    float* o = conv_out(p) + ((size_t)b * p.Cout + co) * p.T + t;
    *o = p.res ? *o + acc : acc;
}

// ConvTranspose1d, k = 2s: output n takes tap n mod s of input n / s and tap n mod s + s of
// input n / s - 1.  grid (ceil((T + 1) s / 32), ceil(Cout / 8), B): the call emits outputs
// 0 .. T s - 1 (the first s completed by the previous call's tail) and keeps T s .. T s + s - 1
__global__ void __launch_bounds__(256) k_mimi_convtr(const MConvParams p) {
    extern __shared__ float xs[];  // [Cin][NT] activated inputs t_lo .. t_lo + NT - 1
    if (aborted(p.st)) return;
    const int b = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int par = p.st.frame[b] & 1, s = p.s, keep = p.k - p.s, len = p.T * s;
    const int n0 = blockIdx.x * TILE;
    const int t_lo = max(0, n0 / s - 1), t_hi = min(p.T - 1, (n0 + TILE - 1) / s);
    const int NT = t_hi - t_lo + 1;
    for (int i = threadIdx.x; i < p.Cin * NT; i += blockDim.x) {
        const int ci = i / NT, m = i - ci * NT;
        const float v = p.in[((size_t)b * p.Cin + ci) * p.T + t_lo + m];
        xs[i] = p.elu_in ? elu_f(v) : v;
    }
    __syncthreads();
    const int co = blockIdx.y * 8 + warp, n = n0 + lane;
    if (co >= p.Cout || n >= len + keep) return;
    const int t1 = n / s, j1 = n - t1 * s;
    const bool v1 = t1 < p.T, v0 = t1 >= 1;
    const int i1 = v1 ? t1 - t_lo : 0, i0 = v0 ? t1 - 1 - t_lo : 0;
    float acc = 0.f;
    for (int ci = 0; ci < p.Cin; ++ci) {
        const uint16_t* w = p.W + ((size_t)ci * p.Cout + co) * p.k;
        const float* x = xs + ci * NT;
        if (v1) acc = fmaf(bf(w, j1), x[i1], acc);
        if (v0) acc = fmaf(bf(w, j1 + s), x[i0], acc);
    }
    const float* tl_old = p.state + (size_t)par * p.B_max * p.Cout * keep;
    float* tl_new = p.state + (size_t)(par ^ 1) * p.B_max * p.Cout * keep;
    if (n < len) {
        if (n < keep) acc += tl_old[((size_t)b * p.Cout + co) * keep + n];
        p.out[((size_t)b * p.Cout + co) * len + n] = acc + bf(p.bias, co);
    } else {
        tl_new[((size_t)b * p.Cout + co) * keep + (n - len)] = acc;
    }
}

struct FinishParams {
    MimiState st;
    const MimiIO* io;
    int B, frame_samples;
};

__global__ void __launch_bounds__(256) k_mimi_finish(const FinishParams p) {
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

}  // namespace
}  // namespace pm

// =====================================================================================
// C ABI
// =====================================================================================
using namespace pm;

struct pm_mimi_ctx {
    pm_mimi_config cfg{};
    int device = 0;
    int frame_samples = 0;
    cudaStream_t stream = nullptr, cap = nullptr;
    std::vector<const uint16_t*> w;      // canonical tensors
    void* block = nullptr;
    MimiState st{};
    MimiIO* io = nullptr;                // device I/O block
    int32_t* codes_dev = nullptr;        // host codes staged here
    uint8_t* host_io = nullptr;          // pinned: I/O block image + host codes
    cudaEvent_t io_done = nullptr;
    float *prev = nullptr, *X = nullptr, *qkv = nullptr, *o = nullptr, *hf = nullptr, *kv = nullptr;
    double* freq = nullptr;
    std::vector<float*> acts;            // SEANet activations
    std::vector<float*> states;          // SEANet streaming state [2][B_max][per_stream]
    std::vector<size_t> state_per_stream;
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

// positions of each group in the canonical tensor order
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

const char* mimi_check(const pm_mimi_config* c) {
    if (c->B_max < 1 || c->B_max > PM_MIMI_MAX_B) return "B_max outside 1..8";
    if (c->heads < 1 || c->dim != c->heads * MDH) return "dim must be 64 x heads";
    if (c->dim % 256 != 0 || c->ffn % 256 != 0 || c->dim > 2048 || c->ffn > 4096)
        return "dim and ffn must be multiples of 256 (dim <= 2048, ffn <= 4096)";
    if (c->cb_dim < 8 || c->cb_dim % 8 != 0 || c->cb_dim > 4096) return "cb_dim must be a multiple of 8 (<= 4096)";
    if (c->card < 1 || c->n_q < 2 || c->n_q > 16) return "codebooks: card >= 1, 2 <= n_q <= 16";
    if (c->n_layers < 0 || c->ctx < 2) return "transformer: n_layers >= 0, ctx >= 2";
    if (c->up_kernel != 4 || c->up_stride != 2) return "the latent upsampler must be kernel 4, stride 2";
    if (c->n_ratios < 1 || c->n_ratios > PM_MIMI_MAX_RATIOS || c->n_filters < 1) return "SEANet stages";
    for (int i = 0; i < c->n_ratios; ++i)
        if (c->ratios[i] < 1 || c->ratios[i] > 16) return "SEANet ratios must be 1..16";
    if (c->kernel < 1 || c->last_kernel < 1 || c->res_kernel < 1 || c->compress < 1) return "SEANet kernels";
    if (c->kernel > 16 || c->last_kernel > 16 || c->res_kernel > 16) return "SEANet kernels above 16";
    if (c->n_filters % c->compress != 0) return "n_filters must be a multiple of compress";
    if (!(c->ln_eps > 0.f) || !(c->rope_theta > 0.f)) return "ln_eps and rope_theta must be positive";
    return nullptr;
}

// per-stream element counts of the state buffers, in recording order
std::vector<size_t> state_sizes(const pm_mimi_config& f) {
    std::vector<size_t> v;
    int C = mimi_channels(f);
    v.push_back((size_t)f.dim * (f.kernel - 1));
    for (int i = 0; i < f.n_ratios; ++i) {
        const int co = C / 2;
        v.push_back((size_t)co * f.ratios[i]);             // transposed-convolution tail (k - s = r)
        v.push_back((size_t)co * (f.res_kernel - 1));      // residual unit's first convolution
        C = co;
    }
    v.push_back((size_t)C * (f.last_kernel - 1));
    return v;
}

template <int PRO, int EPI>
cudaError_t mgemv(const MGemvParams& p, cudaStream_t s) {
    const size_t smem = 4u * (size_t)p.nq * p.K;
    k_mimi_gemv<PRO, EPI><<<(p.R + 7) / 8, 256, smem, s>>>(p);
    return cudaGetLastError();
}

size_t conv_w_smem(int Cin, int k, int T) { return 4u * (size_t)Cin * (k - 1 + T); }
size_t conv_t_smem(int Cin, int k) { return 4u * (size_t)Cin * (TILE + k - 1); }
size_t convtr_smem(int Cin, int s) { return 4u * (size_t)Cin * (TILE / s + 3); }

pm_status launch_conv(pm_mimi_ctx* c, const MConvParams& q, int B, cudaStream_t s) {
    if (q.T <= 16) {
        k_mimi_conv_w<<<dim3((unsigned)((q.Cout + 7) / 8), (unsigned)B), 256, conv_w_smem(q.Cin, q.k, q.T), s>>>(q);
    } else {
        k_mimi_conv_t<<<dim3((unsigned)((q.T + TILE - 1) / TILE), (unsigned)((q.Cout + 7) / 8), (unsigned)B), 256,
                        conv_t_smem(q.Cin, q.k), s>>>(q);
    }
    return cudaGetLastError() == cudaSuccess ? PM_OK : mfail(c, PM_ERR_CUDA, "mimi convolution launch");
}

pm_status record_mimi(pm_mimi_ctx* c, int B, cudaStream_t s) {
    const pm_mimi_config& f = c->cfg;
    const MimiIdx ix = mimi_index(f);
    const int D = f.dim;
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
    fp.dim = D;
    fp.cb_dim = f.cb_dim;
    fp.card = f.card;
    fp.n_q = f.n_q;
    k_mimi_front<<<dim3((unsigned)((D + 63) / 64), (unsigned)B), 256, 8u * f.cb_dim, s>>>(fp);
    if (cudaGetLastError() != cudaSuccess) return mfail(c, PM_ERR_CUDA, "k_mimi_front launch");
    const int nq = 2 * B, RS = f.ctx + 1;
    const size_t kv_block = (size_t)f.B_max * f.heads * RS * MDH;
    for (int l = 0; l < f.n_layers; ++l) {
        // canonical per-block order: norm1.w, norm1.b, in_proj, out_proj, scale1, norm2.w,
        // norm2.b, lin1, lin2, scale2
        const int w0 = ix.layer0 + 10 * l;
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
        k_mimi_attn<<<dim3((unsigned)B, (unsigned)f.heads), 256, 0, s>>>(a);
        if (cudaGetLastError() != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi attention launch");
        g.W = c->w[w0 + 3];
        g.x = c->o;
        g.y = c->X;
        g.scale = c->w[w0 + 4];
        g.R = D;
        g.K = D;
        if (mgemv<MP_NONE, ME_SCALE_RES>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi out_proj launch");
        g.W = c->w[w0 + 7];
        g.x = c->X;
        g.ln_w = c->w[w0 + 5];
        g.ln_b = c->w[w0 + 6];
        g.y = c->hf;
        g.R = f.ffn;
        g.K = D;
        if (mgemv<MP_LN, ME_GELU>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi lin1 launch");
        g.W = c->w[w0 + 8];
        g.x = c->hf;
        g.y = c->X;
        g.scale = c->w[w0 + 9];
        g.R = D;
        g.K = f.ffn;
        if (mgemv<MP_NONE, ME_SCALE_RES>(g, s) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi lin2 launch");
    }
    // SEANet decoder
    auto conv_params = [&](const float* in, float* out, int wi, float* state, int Cin, int Cout, int k, int T) {
        MConvParams q;
        memset(&q, 0, sizeof q);
        q.in = in;
        q.out = out;
        q.W = c->w[wi];
        q.bias = c->w[wi + 1];
        q.state = state;
        q.st = c->st;
        q.B_max = f.B_max;
        q.Cin = Cin;
        q.Cout = Cout;
        q.k = k;
        q.s = 1;
        q.T = T;
        q.elu_in = 1;
        return q;
    };
    int T = 2, C = mimi_channels(f), si = 0;
    MConvParams q = conv_params(c->X, c->acts[0], ix.dec0w, c->states[si++], D, C, f.kernel, T);
    q.elu_in = 0;  // the first convolution takes the transformer output as it is
    q.in_pm = 1;
    pm_status ps = launch_conv(c, q, B, s);
    if (ps) return ps;
    const float* cur = c->acts[0];
    for (int i = 0; i < f.n_ratios; ++i) {
        const int r = f.ratios[i], co = C / 2, hd = co / f.compress, w = ix.stage0 + 6 * i;
        float* y = c->acts[1 + 2 * i];
        float* hmid = c->acts[2 + 2 * i];
        q = conv_params(cur, y, w, c->states[si++], C, co, 2 * r, T);
        q.s = r;
        const int n_out = T * r + r;
        k_mimi_convtr<<<dim3((unsigned)((n_out + TILE - 1) / TILE), (unsigned)((co + 7) / 8), (unsigned)B), 256,
                        convtr_smem(C, r), s>>>(q);
        if (cudaGetLastError() != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi transposed convolution launch");
        T *= r;
        // residual unit: y += conv_k1(ELU(conv_k(ELU(y))))
        if ((ps = launch_conv(c, conv_params(y, hmid, w + 2, c->states[si++], co, hd, f.res_kernel, T), B, s))) return ps;
        q = conv_params(hmid, y, w + 4, nullptr, hd, co, 1, T);
        q.res = 1;
        if ((ps = launch_conv(c, q, B, s))) return ps;
        cur = y;
        C = co;
    }
    q = conv_params(cur, nullptr, ix.outw, c->states[si++], C, 1, f.last_kernel, T);
    q.io_out = c->io;  // straight into the caller's PCM
    if ((ps = launch_conv(c, q, B, s))) return ps;
    FinishParams fin;
    fin.st = c->st;
    fin.io = c->io;
    fin.B = B;
    fin.frame_samples = c->frame_samples;
    k_mimi_finish<<<1, 256, 0, s>>>(fin);
    if (cudaGetLastError() != cudaSuccess) return mfail(c, PM_ERR_CUDA, "mimi finish launch");
    return PM_OK;
}

// largest dynamic shared memory any launch of this configuration asks for
size_t mimi_smem_need(const pm_mimi_config& f) {
    size_t m = 4u * 2 * f.B_max * (size_t)(f.dim > f.ffn ? f.dim : f.ffn);
    int T = 2, C = mimi_channels(f);
    auto conv = [&](int Cin, int k, int TT) {
        const size_t v = TT <= 16 ? conv_w_smem(Cin, k, TT) : conv_t_smem(Cin, k);
        if (v > m) m = v;
    };
    conv(f.dim, f.kernel, T);
    for (int i = 0; i < f.n_ratios; ++i) {
        const int r = f.ratios[i], co = C / 2;
        if (convtr_smem(C, r) > m) m = convtr_smem(C, r);
        T *= r;
        conv(co, f.res_kernel, T);
        conv(co / f.compress, 1, T);
        C = co;
    }
    conv(C, f.last_kernel, T);
    return m;
}

cudaError_t mimi_func_attributes(size_t smem) {
    const int v = (int)smem;
    cudaError_t e = cudaSuccess;
    auto set = [&](const void* fn) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
    };
    set((const void*)k_mimi_gemv<MP_LN, ME_STORE>);
    set((const void*)k_mimi_gemv<MP_LN, ME_GELU>);
    set((const void*)k_mimi_gemv<MP_NONE, ME_SCALE_RES>);
    set((const void*)k_mimi_conv_w);
    set((const void*)k_mimi_conv_t);
    set((const void*)k_mimi_convtr);
    set((const void*)k_mimi_front);
    return e;
}

}  // namespace

extern "C" int pm_mimi_tensor_count(const pm_mimi_config* cfg) {
    if (!cfg || mimi_check(cfg)) return -1;
    return mimi_index(*cfg).total;
}

extern "C" pm_status pm_mimi_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors,
                                    void* cuda_stream, pm_mimi_ctx** out) {
    g_mimi_create_error.clear();
    auto refuse = [](pm_status s, const std::string& m) {
        g_mimi_create_error = m;
        return s;
    };
    if (!cfg || !tensors || !out) return refuse(PM_ERR_ARG, "pm_mimi_create: NULL argument");
    *out = nullptr;
    if (const char* why = mimi_check(cfg)) return refuse(PM_ERR_ARG, std::string("pm_mimi_create: ") + why);
    const MimiIdx ix = mimi_index(*cfg);
    if (n_tensors != ix.total)
        return refuse(PM_ERR_ARG, "pm_mimi_create: expected " + std::to_string(ix.total) + " tensors");
    for (int i = 0; i < n_tensors; ++i) {
        if (!tensors[i] || (reinterpret_cast<uintptr_t>(tensors[i]) & 15u))
            return refuse(PM_ERR_ARG, "pm_mimi_create: tensor " + std::to_string(i) + " NULL or not 16-byte aligned");
        cudaPointerAttributes a;
        const bool dev = cudaPointerGetAttributes(&a, tensors[i]) == cudaSuccess &&
                         (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged);
        cudaGetLastError();
        if (!dev) return refuse(PM_ERR_ARG, "pm_mimi_create: tensor " + std::to_string(i) + " is not device memory");
    }
    const size_t smem = mimi_smem_need(*cfg);
    if (smem > 227u * 1024u) return refuse(PM_ERR_UNSUPPORTED, "pm_mimi_create: shared memory above 227 KB");
    pm_mimi_ctx* c = new pm_mimi_ctx();
    c->cfg = *cfg;
    const pm_mimi_config& f = c->cfg;
    c->frame_samples = 2;
    for (int i = 0; i < f.n_ratios; ++i) c->frame_samples *= f.ratios[i];
    cudaGetDevice(&c->device);
    c->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    for (int i = 0; i < n_tensors; ++i) c->w.push_back(static_cast<const uint16_t*>(tensors[i]));
    auto bail = [&](pm_status s, const char* m) {
        pm_mimi_destroy(c);
        g_mimi_create_error = std::string("pm_mimi_create: ") + m;
        return s;
    };
    if (mimi_func_attributes(smem) != cudaSuccess) {
        cudaGetLastError();
        return bail(PM_ERR_CUDA, "cudaFuncSetAttribute");
    }
    // one allocation for state, activations and I/O
    const int BM = f.B_max, D = f.dim;
    void *p_frame, *p_pos, *p_abort, *p_status, *p_io, *p_codes, *p_prev, *p_X, *p_qkv, *p_o, *p_hf, *p_kv, *p_freq;
    std::vector<std::pair<void**, size_t>> items = {
        {&p_frame, 4u * BM},
        {&p_pos, 4u * BM},
        {&p_abort, 4u},
        {&p_status, 4u},
        {&p_io, sizeof(MimiIO)},
        {&p_codes, 4u * BM * f.n_q},
        {&p_prev, 4u * 2 * BM * D},
        {&p_X, 4u * BM * 2 * D},
        {&p_qkv, 4u * BM * 2 * 3 * D},
        {&p_o, 4u * BM * 2 * D},
        {&p_hf, 4u * BM * 2 * f.ffn},
        {&p_kv, 4u * (size_t)f.n_layers * 2 * BM * f.heads * (f.ctx + 1) * MDH},
        {&p_freq, 8u * (MDH / 2)},
    };
    // activations: the first convolution's output, per stage the transposed convolution's
    // output (the residual stream) and the residual unit's middle
    int T = 2, C = mimi_channels(f);
    std::vector<size_t> act_sizes = {(size_t)BM * C * T};
    for (int i = 0; i < f.n_ratios; ++i) {
        const int co = C / 2;
        T *= f.ratios[i];
        act_sizes.push_back((size_t)BM * co * T);
        act_sizes.push_back((size_t)BM * (co / f.compress) * T);
        C = co;
    }
    c->state_per_stream = state_sizes(f);
    c->acts.assign(act_sizes.size(), nullptr);
    c->states.assign(c->state_per_stream.size(), nullptr);
    for (size_t i = 0; i < act_sizes.size(); ++i) items.push_back({reinterpret_cast<void**>(&c->acts[i]), 4u * act_sizes[i]});
    for (size_t i = 0; i < c->states.size(); ++i)
        items.push_back({reinterpret_cast<void**>(&c->states[i]), 4u * 2 * BM * c->state_per_stream[i]});
    size_t total = 0;
    for (auto& it : items) total = (total + 255) / 256 * 256 + (it.second + 15) / 16 * 16;
    if (cudaMalloc(&c->block, total) != cudaSuccess) {
        cudaGetLastError();
        return bail(PM_ERR_OOM, "device allocation");
    }
    if (cudaMemset(c->block, 0, total) != cudaSuccess) return bail(PM_ERR_CUDA, "cudaMemset");
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
    c->io = (MimiIO*)p_io;
    c->codes_dev = (int32_t*)p_codes;
    c->prev = (float*)p_prev;
    c->X = (float*)p_X;
    c->qkv = (float*)p_qkv;
    c->o = (float*)p_o;
    c->hf = (float*)p_hf;
    c->kv = (float*)p_kv;
    c->freq = (double*)p_freq;
    // RoPE frequency of pair j: theta^(-2j / 64)
    std::vector<double> fq(MDH / 2);
    for (int j = 0; j < MDH / 2; ++j) fq[j] = exp(-log((double)f.rope_theta) * (2.0 * j) / (double)MDH);
    if (cudaMemcpy(c->freq, fq.data(), 8u * fq.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(PM_ERR_CUDA, "cudaMemcpy");
    if (cudaHostAlloc((void**)&c->host_io, 64u + 4u * BM * f.n_q, cudaHostAllocDefault) != cudaSuccess)
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

extern "C" void pm_mimi_destroy(pm_mimi_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    if (c->block) cudaStreamSynchronize(c->stream);
    for (auto g : c->graphs)
        if (g) cudaGraphExecDestroy(g);
    if (c->io_done) cudaEventDestroy(c->io_done);
    if (c->host_io) cudaFreeHost(c->host_io);
    if (c->cap) cudaStreamDestroy(c->cap);
    if (c->block) cudaFree(c->block);
    delete c;
}

extern "C" pm_status pm_mimi_decode(pm_mimi_ctx* c, int B, const int32_t* codes, float* pcm) {
    if (!c) return PM_ERR_ARG;
    const pm_mimi_config& f = c->cfg;
    if (B < 1 || B > f.B_max || !codes || !pcm) return mfail(c, PM_ERR_ARG, "pm_mimi_decode: bad B or NULL pointer");
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    cudaPointerAttributes a;
    float* pcm_dev = nullptr;
    if (cudaPointerGetAttributes(&a, pcm) == cudaSuccess) {
        if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) pcm_dev = pcm;
        if (a.type == cudaMemoryTypeHost && a.devicePointer) pcm_dev = static_cast<float*>(a.devicePointer);
    }
    cudaGetLastError();
    if (!pcm_dev || (reinterpret_cast<uintptr_t>(pcm) & 3u))
        return mfail(c, PM_ERR_ARG, "pm_mimi_decode: pcm must be 4-byte aligned device, managed or host-mapped memory");
    const bool dev_codes = cudaPointerGetAttributes(&a, codes) == cudaSuccess &&
                           (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged);
    cudaGetLastError();
    if (!dev_codes)
        for (int i = 0; i < B * f.n_q; ++i)
            if (codes[i] < 0 || codes[i] >= f.card)
                return mfail(c, PM_ERR_INVALID_ID,
                             "pm_mimi_decode: code " + std::to_string(codes[i]) + " at " + std::to_string(i) + " out of range");
    if (!c->graphs[B]) {
        if (cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
            return mfail(c, PM_ERR_CUDA, "cudaStreamBeginCapture");
        pm_status st = record_mimi(c, B, c->cap);
        cudaGraph_t g = nullptr;
        const cudaError_t e = cudaStreamEndCapture(c->cap, &g);
        if (st != PM_OK || e != cudaSuccess || cudaGraphInstantiate(&c->graphs[B], g, 0) != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            c->graphs[B] = nullptr;
            cudaGetLastError();
            return st != PM_OK ? st : mfail(c, PM_ERR_CUDA, "mimi graph capture");
        }
        cudaGraphDestroy(g);
    }
    // the previous call's copies out of the pinned staging must be done before it is reused
    if (cudaEventSynchronize(c->io_done) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaEventSynchronize");
    MimiIO io;
    io.codes = dev_codes ? codes : c->codes_dev;
    io.pcm = pcm_dev;
    memcpy(c->host_io, &io, sizeof io);
    if (!dev_codes) {
        memcpy(c->host_io + 64, codes, 4u * B * f.n_q);
        if (cudaMemcpyAsync(c->codes_dev, c->host_io + 64, 4u * B * f.n_q, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
            return mfail(c, PM_ERR_CUDA, "codes copy");
    }
    if (cudaMemcpyAsync(c->io, c->host_io, sizeof io, cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
        cudaEventRecord(c->io_done, c->stream) != cudaSuccess || cudaGraphLaunch(c->graphs[B], c->stream) != cudaSuccess)
        return mfail(c, PM_ERR_CUDA, "mimi launch");
    return PM_OK;
}

extern "C" pm_status pm_mimi_reset(pm_mimi_ctx* c, const int32_t* mask) {
    if (!c) return PM_ERR_ARG;
    if (cudaSetDevice(c->device) != cudaSuccess) return mfail(c, PM_ERR_CUDA, "cudaSetDevice");
    const pm_mimi_config& f = c->cfg;
    const int BM = f.B_max;
    // a fresh stream: frame 0 at position 0, no previous latent, zero convolution history
    // and zero transposed-convolution tails (the ring needs no clearing: the window only
    // reaches positions written since the reset)
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
    return s ? mfail(c, PM_ERR_INVALID_ID, "a code given in device memory was out of range (that call was a no-op)") : PM_OK;
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
