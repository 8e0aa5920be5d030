// Temperature / top-k sampling of the text token and of the depth codes
// ("PersonaPlex native LM audit", section 7 "One exact generator step": the generator
// samples the text token and each depth position's code; released defaults text
// temperature 0.7 / top-k 25, audio temperature 0.8 / top-k 250).
//
// One CTA per batch row, 1024 threads:
//  * every logit gets the unique 64-bit key (order-preserving bits of the fp32 value,
//    then the complement of its index), so "larger logit, then lower index" is plain key
//    order and the top-k set has no ties;
//  * a short list surely holding the top k: with M the largest logit, the keys within
//    DELTA of M outrank all others, so the smallest DELTA of a geometric ladder
//    (0.25 * 2^j) admitting at least k (and at most 4096) keys gives it, in three
//    cheap passes over the row (max, ladder counts, gather); a list of at most 1024 keys
//    is ranked directly (each key counts the larger ones);
//  * otherwise (many near-equal logits) the k-th largest key is found exactly by an
//    8-pass radix select (8 bits per pass, per-warp histograms) over the list or the
//    row, and the k survivors are ranked;
//  * the row is staged in shared memory when it fits (text head: 32000 logits = 125 KB);
//  * the k survivors, in descending order, are weighted exp((l - l_max) / T) and
//    prefix-summed; u = (first word of Philox4x64-10 >> 40) * 2^-24 with key (seed, 0)
//    and counter (frame position, row, substep, 0) -- Salmon, Moraes, Dror, Shaw,
//    "Parallel random numbers: as easy as 1, 2, 3" (SC'11); the pick is the first
//    survivor whose running sum exceeds u * total;
//  * T <= 0 or k <= 1 is greedy: the argmax, lowest index on ties.
#include <math.h>

#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int NT = 1024;        // threads per CTA (also the largest top-k)
constexpr int KEY_LIST = 4096;  // keys the selection gathers into its shared list
constexpr int NLAD = 13;        // ladder of logit distances below the maximum

// rung j of the distance ladder: 0.25 * 2^j, the last rung unbounded
__device__ __forceinline__ float ladder(int j) { return j == NLAD - 1 ? INFINITY : ldexpf(0.25f, j); }

__device__ __forceinline__ unsigned long long logit_key(float v, int i) { return pack_argmax(v, (uint32_t)i); }

// slot for this lane in a shared list when `take`: one atomic per warp on the list count
__device__ __forceinline__ int warp_append_slot(bool take, int* count) {
    const unsigned int m = __ballot_sync(0xffffffffu, take);
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (m && lane == __ffs(m) - 1) base = atomicAdd(count, __popc(m));
    base = __shfl_sync(0xffffffffu, base, m ? __ffs(m) - 1 : 0);
    return base + __popc(m & ((1u << lane) - 1u));
}

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
    __shared__ unsigned int s_whist[NT / 32][256];  // one histogram per warp (no cross-warp contention)
    __shared__ unsigned int s_hist[256];
    __shared__ unsigned long long s_cand[NT];
    __shared__ float s_scan[NT / 32];
    __shared__ unsigned long long s_red[NT / 32];
    __shared__ unsigned long long s_keys[KEY_LIST];
    __shared__ int s_bin, s_above, s_inbin, s_cnt, s_pick, s_skip;
    __shared__ float s_u, s_total, s_maxv;
    __shared__ float s_redf[NT / 32];
    __shared__ unsigned int s_lad[NLAD];
    __shared__ int s_rung;

    // a prefill's text token is stream seq_stream's (one row)
    const int b = p.seq ? p.io->seq_stream : (int)blockIdx.x;
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
        // ---- a short list that surely holds the top k ----
        // With M the largest logit, every key whose logit is within DELTA of M outranks
        // every key outside, so the smallest DELTA of a geometric ladder that admits at
        // least k keys (and at most the list capacity) gives a list containing the top k.
        float mx = -INFINITY;
        for (int i = tid; i < V; i += NT) mx = fmaxf(mx, row[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_redf[warp] = mx;
        __syncthreads();
        if (tid < 32) {
            float v = s_redf[tid];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (tid == 0) s_maxv = v;
        }
        for (int j = tid; j < NLAD; j += NT) s_lad[j] = 0u;
        __syncthreads();
        const float M = s_maxv;
        unsigned int cnt[NLAD];
#pragma unroll
        for (int j = 0; j < NLAD; ++j) cnt[j] = 0u;
        for (int i = tid; i < V; i += NT) {
            const float d = M - row[i];
#pragma unroll
            for (int j = 0; j < NLAD; ++j) cnt[j] += (d <= ladder(j)) ? 1u : 0u;
        }
#pragma unroll
        for (int j = 0; j < NLAD; ++j) {
            unsigned int c = cnt[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (lane == 0) atomicAdd(&s_lad[j], c);
        }
        __syncthreads();
        if (tid == 0) {
            int pick = -1;
            for (int j = 0; j < NLAD; ++j)
                if (s_lad[j] >= (unsigned int)k) {
                    if (s_lad[j] <= (unsigned int)KEY_LIST) pick = j;
                    break;
                }
            s_rung = pick;
            s_cnt = 0;
        }
        __syncthreads();
        int listed = -1;  // keys in s_keys (-1: the radix select scans the row)
        if (s_rung >= 0) {
            const float delta = ladder(s_rung);
            for (int i0 = 0; i0 < V; i0 += NT) {
                const int i = i0 + tid;
                const float v = i < V ? row[i] : 0.0f;
                const bool take = i < V && (M - v) <= delta;
                const int slot = warp_append_slot(take, &s_cnt);
                if (take) s_keys[slot] = logit_key(v, i);
            }
            __syncthreads();
            listed = s_cnt;
        }
        if (listed >= 0 && listed <= NT) {
            // ---- rank the list directly: key ranks are unique ----
            if (tid < listed) {
                const unsigned long long key = s_keys[tid];
                int rank = 0;
                for (int i = 0; i < listed; ++i) rank += (s_keys[i] > key) ? 1 : 0;
                if (rank < k) s_cand[rank] = key;
            }
            __syncthreads();
        } else {
            // ---- exact k-th largest key: 8-pass radix select (over the list, or over the
            // row until few enough keys match the prefix to gather them) ----
            unsigned long long prefix = 0ull, mask = 0ull;
            int kk = k;  // rank still to find among the keys matching the prefix
            for (int pass = 0; pass < 8; ++pass) {
                const int shift = 56 - 8 * pass;
                for (int i = lane; i < 256; i += 32) s_whist[warp][i] = 0u;
                __syncthreads();
                const int n_scan = listed < 0 ? V : listed;
                for (int i0 = 0; i0 < n_scan; i0 += NT) {
                    const int i = i0 + tid;
                    bool in = false;
                    unsigned int bin = 0u;
                    if (i < n_scan) {
                        const unsigned long long key = listed < 0 ? logit_key(row[i], i) : s_keys[i];
                        in = (key & mask) == prefix;
                        bin = (unsigned int)(key >> shift) & 255u;
                    }
                    const unsigned int act = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        // one add when the warp's keys share the bin, else one per key
                        const unsigned int b0 = __shfl_sync(act, bin, __ffs(act) - 1);
                        if (__all_sync(act, bin == b0)) {
                            if ((__ffs(act) - 1) == lane) s_whist[warp][b0] += (unsigned int)__popc(act);
                        } else {
                            atomicAdd(&s_whist[warp][bin], 1u);
                        }
                    }
                }
                __syncthreads();
                for (int i = tid; i < 256; i += NT) {
                    unsigned int t = 0u;
                    for (int w = 0; w < NT / 32; ++w) t += s_whist[w][i];
                    s_hist[i] = t;
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
                                s_inbin = (int)c[j];
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
                if (listed < 0 && pass < 7 && s_inbin <= KEY_LIST) {
                    // gather the keys matching the new prefix (their order is irrelevant)
                    if (tid == 0) s_cnt = 0;
                    __syncthreads();
                    for (int i0 = 0; i0 < V; i0 += NT) {
                        const int i = i0 + tid;
                        const unsigned long long key = i < V ? logit_key(row[i], i) : 0ull;
                        const bool take = i < V && (key & mask) == prefix;
                        const int slot = warp_append_slot(take, &s_cnt);
                        if (take) s_keys[slot] = key;
                    }
                    __syncthreads();
                    listed = s_cnt;
                }
                __syncthreads();
            }
            // ---- the k survivors (keys >= the k-th largest), ranked into order: every key
            // above the prefix's bins is one, wherever it was scanned from ----
            if (tid == 0) s_cnt = 0;
            __syncthreads();
            for (int i0 = 0; i0 < V; i0 += NT) {
                const int i = i0 + tid;
                const unsigned long long key = i < V ? logit_key(row[i], i) : 0ull;
                const bool take = i < V && key >= prefix;
                const int slot = warp_append_slot(take, &s_cnt);
                if (take && slot < NT) s_keys[slot] = key;
            }
            __syncthreads();
            if (tid < k) {
                const unsigned long long key = s_keys[tid];
                int rank = 0;
                for (int i = 0; i < k; ++i) rank += (s_keys[i] > key) ? 1 : 0;
                s_cand[rank] = key;
            }
            __syncthreads();
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
        if (p.io->token) p.io->token[p.seq ? 0 : b] = tok;
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
