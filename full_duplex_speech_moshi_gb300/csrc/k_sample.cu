// Temperature / top-k sampling of the text token and of the depth codes
// ("PersonaPlex native LM audit", section 7 "One exact generator step": the generator
// samples the text token and each depth position's code; released defaults text
// temperature 0.7 / top-k 25, audio temperature 0.8 / top-k 250).
//
// One CTA per batch row, 1024 threads:
//  * every logit gets the unique 64-bit key (order-preserving bits of the fp32 value,
//    then the complement of its index), so "larger logit, then lower index" is plain key
//    order and the top-k set has no ties;
//  * the k-th largest key is found exactly by an 8-pass radix select (8 bits per pass,
//    one shared histogram, warp-aggregated increments); the row is staged in shared
//    memory when it fits (text head: 32000 logits = 125 KB);
//  * the k survivors are sorted (bitonic, descending), weighted exp((l - l_max) / T) and
//    prefix-summed; u = (first word of Philox4x64-10 >> 40) * 2^-24 with key (seed, 0)
//    and counter (frame position, row, substep, 0) -- Salmon, Moraes, Dror, Shaw,
//    "Parallel random numbers: as easy as 1, 2, 3" (SC'11); the pick is the first
//    survivor whose running sum exceeds u * total;
//  * T <= 0 or k <= 1 is greedy: the argmax, lowest index on ties.
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int NT = 1024;  // threads per CTA (also the largest top-k)

__device__ __forceinline__ unsigned long long logit_key(float v, int i) { return pack_argmax(v, (uint32_t)i); }

// Philox4x64-10 block; returns the first output word
__device__ __forceinline__ unsigned long long philox4x64_w0(unsigned long long c0, unsigned long long c1,
                                                            unsigned long long c2, unsigned long long c3,
                                                            unsigned long long k0, unsigned long long k1) {
    const unsigned long long M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const unsigned long long W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const unsigned long long hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const unsigned long long hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const unsigned long long n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

__global__ void __launch_bounds__(NT) k_sample(const SampleParams p) {
    extern __shared__ float s_row[];  // staged logits (when p.stage)
    __shared__ unsigned int s_hist[256];
    __shared__ unsigned long long s_cand[NT];
    __shared__ float s_scan[NT / 32];
    __shared__ unsigned long long s_red[NT / 32];
    __shared__ int s_bin, s_above, s_cnt, s_pick, s_skip;
    __shared__ float s_u, s_total;

    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();

    // ---- configuration and the counter of this row ----
    float T;
    int k;
    unsigned long long seed, c0;
    const unsigned long long c1 = (unsigned long long)b;
    unsigned long long c2;
    if (p.mode == SM_PLAIN) {
        T = p.temperature;
        k = p.top_k;
        seed = p.seed;
        c0 = (unsigned long long)p.position;
        c2 = (unsigned long long)p.substep;
    } else {
        const bool text = p.mode == SM_TEXT;
        T = text ? p.cfg->text_temperature : p.cfg->audio_temperature;
        k = text ? p.cfg->text_top_k : p.cfg->audio_top_k;
        seed = p.cfg->seed;
        // the frame being decoded: the text head has already advanced the position
        c0 = (unsigned long long)(long long)(p.st.pos[b] - 1);
        c2 = text ? 0ull : (unsigned long long)(1 + p.q);
    }
    if (tid == 0) {
        int skip = 0;
        if (p.mode != SM_PLAIN && *(volatile uint32_t*)&p.st.status[1] != 0u) skip = 1;  // frame aborted
        if (p.mode == SM_DEPTH && p.st.dep_sup[(size_t)b * p.Q + p.q] >= 0) skip = 1;      // code supplied
        s_skip = skip;
    }
    __syncthreads();
    if (s_skip) return;
    const int V = p.V;
    if (k > V) k = V;
    const float* g_row = p.logits + (size_t)b * p.ld;
    const float* row = g_row;
    if (p.stage) {
        for (int i = tid; i < V; i += NT) s_row[i] = g_row[i];
        row = s_row;
    }
    __syncthreads();

    int32_t tok;
    if (T <= 0.0f || k <= 1) {
        // ---- greedy: the largest key ----
        unsigned long long best = 0ull;
        for (int i = tid; i < V; i += NT) best = umax64(best, logit_key(row[i], i));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (lane == 0) s_red[warp] = best;
        __syncthreads();
        if (tid == 0) {
            unsigned long long m = 0ull;
            for (int w = 0; w < NT / 32; ++w) m = umax64(m, s_red[w]);
            s_pick = (int)unpack_argmax_index(m);
        }
        __syncthreads();
        tok = s_pick;
    } else {
        // ---- exact k-th largest key: 8-pass radix select ----
        unsigned long long prefix = 0ull, mask = 0ull;
        int kk = k;  // rank still to find among the keys matching the prefix
        for (int pass = 0; pass < 8; ++pass) {
            const int shift = 56 - 8 * pass;
            for (int i = tid; i < 256; i += NT) s_hist[i] = 0u;
            __syncthreads();
            for (int i0 = 0; i0 < V; i0 += NT) {
                const int i = i0 + tid;
                bool in = false;
                unsigned int bin = 0u;
                if (i < V) {
                    const unsigned long long key = logit_key(row[i], i);
                    in = (key & mask) == prefix;
                    bin = (unsigned int)(key >> shift) & 255u;
                }
                const unsigned int act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const unsigned int same = __match_any_sync(act, bin);
                    if ((__ffs(same) - 1) == lane) atomicAdd(&s_hist[bin], (unsigned int)__popc(same));
                }
            }
            __syncthreads();
            if (warp == 0) {
                // bins from the top: lane l holds bins 255 - 8l .. 248 - 8l
                unsigned int c[8], sum = 0u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = s_hist[255 - (lane * 8 + j)];
                    sum += c[j];
                }
                unsigned int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const unsigned int excl = incl - sum;
                if (excl < (unsigned int)kk && (unsigned int)kk <= incl) {
                    unsigned int run = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (run + c[j] >= (unsigned int)kk) {
                            s_bin = 255 - (lane * 8 + j);
                            s_above = (int)run;
                            break;
                        }
                        run += c[j];
                    }
                }
            }
            __syncthreads();
            prefix |= (unsigned long long)s_bin << shift;
            mask |= 0xFFull << shift;
            kk -= s_above;
            __syncthreads();
        }
        // ---- the k survivors (keys >= the k-th largest), sorted descending ----
        if (tid == 0) s_cnt = 0;
        __syncthreads();
        for (int i = tid; i < V; i += NT) {
            const unsigned long long key = logit_key(row[i], i);
            if (key >= prefix) {
                const int slot = atomicAdd(&s_cnt, 1);
                if (slot < NT) s_cand[slot] = key;
            }
        }
        __syncthreads();
        int P = 1;
        while (P < k) P <<= 1;
        for (int i = k + tid; i < P; i += NT) s_cand[i] = 0ull;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P; i += NT) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const bool desc = (i & size) == 0;
                        const unsigned long long a = s_cand[i], c = s_cand[j];
                        if (desc ? (a < c) : (a > c)) {
                            s_cand[i] = c;
                            s_cand[j] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
        // ---- weights, running sums, the draw ----
        const int top_idx = (int)unpack_argmax_index(s_cand[0]);
        const float lmax = row[top_idx];
        const float inv_t = 1.0f / T;
        float w = 0.0f;
        int idx = 0;
        if (tid < k) {
            idx = (int)unpack_argmax_index(s_cand[tid]);
            w = expf((row[idx] - lmax) * inv_t);
        }
        // inclusive block scan of w over threads 0..k-1 (warp scans, then a scan of the
        // warp totals)
        float incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_scan[warp] = incl;
        if (tid == 0) {
            const unsigned long long x = philox4x64_w0(c0, c1, c2, 0ull, seed, 0ull);
            s_u = (float)(unsigned int)(x >> 40) * (1.0f / 16777216.0f);
            s_pick = k - 1;
        }
        __syncthreads();
        if (warp == 0) {
            float v = s_scan[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            s_scan[lane] = v;  // inclusive over warps
        }
        __syncthreads();
        const float cum = (warp > 0 ? s_scan[warp - 1] : 0.0f) + incl;
        if (tid == k - 1) s_total = cum;
        __syncthreads();
        // the first survivor whose running sum exceeds u * total (the last one if rounding
        // leaves none above)
        const float target = s_u * s_total;
        if (tid < k && cum > target) atomicMin(&s_pick, tid);
        __syncthreads();
        tok = (int)unpack_argmax_index(s_cand[s_pick]);
    }

    if (tid != 0) return;
    if (p.mode == SM_PLAIN) {
        p.tokens[b] = tok;
    } else if (p.mode == SM_TEXT) {
        if (p.io->token) p.io->token[b] = tok;
        p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 0] = tok;
    } else {
        p.st.dep_codes[(size_t)b * p.Q + p.q] = tok;
        if (p.dio->codes) p.dio->codes[(size_t)b * p.Q + p.q] = tok;
        if (1 + p.q < p.n_streams) p.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + 1 + p.q] = tok;
    }
}

}  // namespace

static size_t sample_smem(int V) { return (V <= PM_SAMPLE_STAGE_MAX) ? (size_t)V * 4u : 0u; }

cudaError_t sample_prepare() {
    return cudaFuncSetAttribute(k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(PM_SAMPLE_STAGE_MAX * 4));
}

cudaError_t launch_sample(const SampleParams& p, cudaStream_t s, bool pdl) {
    if (p.V < 1 || p.B < 1) return cudaErrorInvalidValue;
    SampleParams q = p;
    q.stage = p.V <= PM_SAMPLE_STAGE_MAX ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sample_smem(p.V);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_sample, q);
}

}  // namespace pm
