/*
 * Float64 CPU oracle of the Moshi/PersonaPlex per-frame decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow statement of what the decode
 * step computes, used to check the CUDA path.  Only the test suite, the smoke check
 * and the bench's CPU-baseline leg may load it; the library never does.  It shares no
 * code with the CUDA path.
 *
 * Authority: "PersonaPlex native LM audit" (clockless-atlas personaplex-research page):
 *   section 3 "Native temporal computation"  -- embedding sum, block equations, RMSNorm32,
 *            RoPE (adjacent pairs, theta 1e4), causal window mask, final norm + text head;
 *   section 4 "Native depth computation"      -- sixteen positions, six per-position blocks,
 *            shared norm scales, no RoPE, no final depth norm;
 *   section 6 "Three distinct caches"         -- K stored after RoPE, V not;
 *   section 7 "One exact generator step"      -- stream order and delays.
 * RMSNorm closed form: the same page, connector chapter section 2 ("RMSNorm(x; g, e)").
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   - attention scale 1/sqrt(d_h) (the SDPA default);
 *   - RoPE pair (2j, 2j+1), angle pos * exp(-ln(theta) * 2j / d_h),
 *     (a, b) -> (a cos - b sin, a sin + b cos);
 *   - fused QKV rows: Q = rows 0..D-1, K = D..2D-1, V = 2D..3D-1; head h = rows h*dh..;
 *   - SwiGLU: rows 0..F-1 are the gate g (SiLU applied), rows F..2F-1 are z;
 *   - depth step q uses rows q*3*Dd .. of the packed QKV and rows q*Dd .. of the packed
 *     output projection; its Q/K/V split inside the slice follows the temporal order;
 *   - argmax ties go to the lowest index;
 *   - a stream's frame at position p reads, for a stream of delay d, the IDs given at
 *     position p-d; positions before the first frame since reset or position set read
 *     the initial ID of that stream.
 *
 * Sampling (same page, section 7: the generator samples the text token and each depth
 * position's code, released defaults text temperature 0.7 / top-k 25, audio 0.8 / 250):
 *   - the page names temperature and top-k and nothing finer; the reading taken: keep the
 *     k largest logits (ties at the cut to the lower index), weights exp((l - l_max) / T)
 *     over those, and the first candidate, in descending-logit order, whose running sum
 *     of weights exceeds u * total; T <= 0 or k <= 1 is greedy (the argmax);
 *   - u comes from Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 *     as easy as 1, 2, 3", SC'11) with key (seed, 0) and counter (frame position, batch
 *     row, substep, 0), substep 0 for the text token and 1 + q for depth position q:
 *     u = (first output word >> 40) * 2^-24.
 *
 * Pinned ring mode (same page, section 6, "Observed source-level boundary"): the ring
 * labels slot i, with end_index = end_offset mod capacity and delta = i - end_index, as
 * position end_offset + delta when delta <= 0 and end_offset + delta - capacity otherwise;
 * a key is attended to when its label lies in 0..query position.  After the current
 * key's write (end_offset = position + 1) a full ring therefore hides its oldest key.  The
 * depth cache uses the same mapping with capacity dep_ctx (the pages show it for 16).
 *
 * Arithmetic is float64 throughout.  Weights are bf16 bit patterns, widened exactly.
 * Nothing is blocked, fused or reordered beyond the definitions above.  Loops over
 * output rows run under OpenMP; each row's sum is a plain serial loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "pm_oracle.h"

/* ------------------------------------------------------------------------- */
/* scalar helpers                                                             */
/* ------------------------------------------------------------------------- */

double orc_bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* y[r] = sum_c W[r][c] * x[c]; W is bf16 [rows][cols], row-major ([out, in]). */
void orc_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t* w = W + (size_t)r * (size_t)cols;
        double acc = 0.0;
        for (int c = 0; c < cols; ++c) acc += orc_bf16_to_double(w[c]) * x[c];
        y[r] = acc;
    }
}

/* RMSNorm(x; alpha, eps) = alpha * x / sqrt(mean_j x_j^2 + eps); no mean subtraction. */
void orc_rmsnorm(const double* x, const uint16_t* alpha, int n, double eps, double* out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) out[i] = orc_bf16_to_double(alpha[i]) * x[i] * inv;
}

/* Rotate one head vector v[dh] in place for absolute position pos: coordinate pairs
 * (2j, 2j+1), frequency f_j = exp(-ln(theta) * 2j / dh), angle pos * f_j. */
void orc_rope(double* v, int dh, long pos, double theta) {
    for (int j = 0; j < dh / 2; ++j) {
        double f = exp(-log(theta) * (2.0 * j) / (double)dh);
        double ang = (double)pos * f;
        double c = cos(ang), s = sin(ang);
        double a = v[2 * j], b = v[2 * j + 1];
        v[2 * j] = a * c - b * s;
        v[2 * j + 1] = a * s + b * c;
    }
}

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* One head of softmax attention for a single query:
 * o = sum_i softmax_i(q . k_i / sqrt(dh)) v_i over n keys.
 * keys[i] / vals[i] point at dh-vectors. */
void orc_attend(const double* q, const double* const* keys, const double* const* vals, int n, int dh,
                double* o) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    double scale = 1.0 / sqrt((double)dh);
    for (int i = 0; i < n; ++i) {
        double d = 0.0;
        for (int c = 0; c < dh; ++c) d += q[c] * keys[i][c];
        s[i] = d * scale;
        if (s[i] > m) m = s[i];
    }
    double den = 0.0;
    for (int i = 0; i < n; ++i) {
        s[i] = exp(s[i] - m);
        den += s[i];
    }
    for (int c = 0; c < dh; ++c) o[c] = 0.0;
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < dh; ++c) o[c] += (s[i] / den) * vals[i][c];
    free(s);
}

void orc_ring_labels(long capacity, long end_offset, long* labels) {
    const long end_index = end_offset % capacity;
    for (long i = 0; i < capacity; ++i) {
        const long delta = i - end_index;
        labels[i] = (delta <= 0) ? end_offset + delta : end_offset + delta - capacity;
    }
}

static int cmp_long(const void* a, const void* b) {
    const long x = *(const long*)a, y = *(const long*)b;
    return (x > y) - (x < y);
}

int orc_visible_positions(long pos, long capacity, int pinned, long* vis) {
    int n = 0;
    if (!pinned) {
        long lo = pos - capacity + 1;
        if (lo < 0) lo = 0;
        for (long p = lo; p <= pos; ++p) vis[n++] = p;
        return n;
    }
    long* labels = (long*)malloc(sizeof(long) * (size_t)capacity);
    orc_ring_labels(capacity, pos + 1, labels);
    for (long i = 0; i < capacity; ++i)
        if (labels[i] >= 0 && labels[i] <= pos) vis[n++] = labels[i];
    free(labels);
    qsort(vis, (size_t)n, sizeof(long), cmp_long);
    return n;
}

/* lowest index among the maxima */
int orc_argmax(const double* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ------------------------------------------------------------------------- */
/* sampling                                                                   */
/* ------------------------------------------------------------------------- */

/* Philox4x64-10: ten rounds of the 4x64 S-box (two 64x64 -> 128-bit multiplies per
 * round with the multipliers published for Philox by Salmon et al., 2011), the key
 * bumped by the two Weyl constants between rounds. */
void orc_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const unsigned __int128 p0 = (unsigned __int128)M0 * c0;
        const unsigned __int128 p1 = (unsigned __int128)M1 * c2;
        const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

double orc_uniform24(uint64_t seed, uint64_t c0, uint64_t c1, uint64_t c2) {
    const uint64_t ctr[4] = {c0, c1, c2, 0}, key[2] = {seed, 0};
    uint64_t out[4];
    orc_philox4x64(ctr, key, out);
    return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

/* order for the top-k cut: larger logit first, then lower index */
static const double* g_sort_logits;
static int by_logit_desc(const void* a, const void* b) {
    const int i = *(const int*)a, j = *(const int*)b;
    const double li = g_sort_logits[i], lj = g_sort_logits[j];
    if (li > lj) return -1;
    if (li < lj) return 1;
    return (i < j) ? -1 : (i > j) ? 1 : 0;
}

int orc_sample_topk(const double* logits, int V, double temperature, int top_k, uint64_t seed, uint64_t c0,
                    uint64_t c1, uint64_t c2, double* margin, double* cut_gap) {
    if (margin) *margin = INFINITY;
    if (cut_gap) *cut_gap = INFINITY;
    if (temperature <= 0.0 || top_k <= 1) return orc_argmax(logits, V);
    const int k = top_k < V ? top_k : V;
    int* idx = (int*)malloc(sizeof(int) * (size_t)V);
    for (int i = 0; i < V; ++i) idx[i] = i;
    g_sort_logits = logits;
    qsort(idx, (size_t)V, sizeof(int), by_logit_desc);
    if (cut_gap && k < V) *cut_gap = logits[idx[k - 1]] - logits[idx[k]];
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    const double lmax = logits[idx[0]];
    double total = 0.0;
    for (int j = 0; j < k; ++j) {
        w[j] = exp((logits[idx[j]] - lmax) / temperature);
        total += w[j];
    }
    const double target = orc_uniform24(seed, c0, c1, c2) * total;
    int pick = k - 1;
    double run = 0.0, below = 0.0;
    for (int j = 0; j < k; ++j) {
        below = run;
        run += w[j];
        if (run > target) {
            pick = j;
            break;
        }
    }
    if (margin) {
        const double d0 = target - below, d1 = run - target;
        *margin = (d0 < d1 ? d0 : d1) / total;
    }
    const int token = idx[pick];
    free(w);
    free(idx);
    return token;
}

/* ------------------------------------------------------------------------- */
/* model                                                                      */
/* ------------------------------------------------------------------------- */

struct orc_model {
    orc_config c;
    const uint16_t* text_emb;
    const uint16_t** audio_emb; /* n_streams - 1 */
    const uint16_t** norm1;     /* per layer */
    const uint16_t** w_qkv;
    const uint16_t** w_o;
    const uint16_t** norm2;
    const uint16_t** w_in;
    const uint16_t** w_out;
    const uint16_t* out_norm;
    const uint16_t* text_head;
    /* depformer (NULL when dep_layers == 0) */
    const uint16_t** dep_in;        /* dep_steps */
    const uint16_t* dep_text_emb;
    const uint16_t** dep_audio_emb; /* dep_steps - 1 */
    const uint16_t** dep_norm1;     /* dep_layers */
    const uint16_t** dep_qkv;
    const uint16_t** dep_o;
    const uint16_t** dep_norm2;
    const uint16_t** dep_w_in;      /* dep_layers * dep_steps, index j*steps+q */
    const uint16_t** dep_w_out;
    const uint16_t** dep_head;      /* dep_steps */
};

static const uint16_t** take(const uint16_t* const* t, int* at, int n) {
    const uint16_t** a = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; ++i) a[i] = t[(*at)++];
    return a;
}

int orc_tensor_count(const orc_config* c) {
    int n = 1 + (c->n_streams - 1) + 6 * c->n_layers + 2;
    if (c->dep_layers > 0) {
        int Q = c->dep_steps;
        n += Q + 1 + (Q - 1) + c->dep_layers * (4 + 2 * Q) + Q;
    }
    return n;
}

orc_model* orc_create(const orc_config* c, const uint16_t* const* t, int n_tensors) {
    if (n_tensors != orc_tensor_count(c)) return NULL;
    orc_model* m = (orc_model*)calloc(1, sizeof *m);
    m->c = *c;
    int at = 0;
    m->text_emb = t[at++];
    m->audio_emb = take(t, &at, c->n_streams - 1);
    m->norm1 = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    m->w_qkv = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    m->w_o = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    m->norm2 = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    m->w_in = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    m->w_out = (const uint16_t**)malloc(sizeof(void*) * (size_t)c->n_layers);
    for (int l = 0; l < c->n_layers; ++l) {
        m->norm1[l] = t[at++];
        m->w_qkv[l] = t[at++];
        m->w_o[l] = t[at++];
        m->norm2[l] = t[at++];
        m->w_in[l] = t[at++];
        m->w_out[l] = t[at++];
    }
    m->out_norm = t[at++];
    m->text_head = t[at++];
    if (c->dep_layers > 0) {
        int Q = c->dep_steps, J = c->dep_layers;
        m->dep_in = take(t, &at, Q);
        m->dep_text_emb = t[at++];
        m->dep_audio_emb = take(t, &at, Q - 1);
        m->dep_norm1 = (const uint16_t**)malloc(sizeof(void*) * (size_t)J);
        m->dep_qkv = (const uint16_t**)malloc(sizeof(void*) * (size_t)J);
        m->dep_o = (const uint16_t**)malloc(sizeof(void*) * (size_t)J);
        m->dep_norm2 = (const uint16_t**)malloc(sizeof(void*) * (size_t)J);
        m->dep_w_in = (const uint16_t**)malloc(sizeof(void*) * (size_t)(J * Q));
        m->dep_w_out = (const uint16_t**)malloc(sizeof(void*) * (size_t)(J * Q));
        for (int j = 0; j < J; ++j) {
            m->dep_norm1[j] = t[at++];
            m->dep_qkv[j] = t[at++];
            m->dep_o[j] = t[at++];
            m->dep_norm2[j] = t[at++];
            for (int q = 0; q < Q; ++q) m->dep_w_in[j * Q + q] = t[at++];
            for (int q = 0; q < Q; ++q) m->dep_w_out[j * Q + q] = t[at++];
        }
        m->dep_head = take(t, &at, Q);
    }
    return m;
}

void orc_destroy(orc_model* m) {
    if (!m) return;
    free(m->audio_emb);
    free(m->norm1); free(m->w_qkv); free(m->w_o); free(m->norm2); free(m->w_in); free(m->w_out);
    if (m->c.dep_layers > 0) {
        free(m->dep_in); free(m->dep_audio_emb); free(m->dep_norm1); free(m->dep_qkv);
        free(m->dep_o); free(m->dep_norm2); free(m->dep_w_in); free(m->dep_w_out); free(m->dep_head);
    }
    free(m);
}

/* rows of embedding table k (stream 0 = text) */
static int stream_rows(const orc_config* c, int k) { return k == 0 ? c->text_in : c->audio_in; }

static int stream_init(const orc_config* c, int k) { return k == 0 ? c->init_text : c->init_audio; }

int orc_validate_ids(const orc_config* c, const int32_t* ids) {
    for (int k = 0; k < c->n_streams; ++k)
        if (ids[k] < -1 || ids[k] >= stream_rows(c, k)) return ORC_ERR_INVALID_ID;
    return ORC_OK;
}

/* x = sum over streams of E_k[in[k]], with ID -1 contributing an exact zero vector. */
void orc_embed(const orc_model* m, const int32_t* in, double* x) {
    const orc_config* c = &m->c;
    for (int i = 0; i < c->D; ++i) x[i] = 0.0;
    for (int k = 0; k < c->n_streams; ++k) {
        if (in[k] == -1) continue;
        const uint16_t* table = (k == 0) ? m->text_emb : m->audio_emb[k - 1];
        const uint16_t* row = table + (size_t)in[k] * (size_t)c->D;
        for (int i = 0; i < c->D; ++i) x[i] += orc_bf16_to_double(row[i]);
    }
}

/* ------------------------------------------------------------------------- */
/* stream state (incremental decode)                                          */
/* ------------------------------------------------------------------------- */

struct orc_stream {
    long pos;        /* absolute position of the next frame */
    long first_pos;  /* position of the first frame since reset / position set */
    int32_t* id_hist;   /* [hist_cap][n_streams], indexed by pos - first_pos */
    long hist_cap;
    /* K/V per layer, indexed by absolute position: [layer][pos][D] */
    double** K;
    double** V;
    long kv_cap;
    int n_layers;    /* so that freeing needs no model (it may be gone at teardown) */
};

orc_stream* orc_stream_new(const orc_model* m) {
    orc_stream* s = (orc_stream*)calloc(1, sizeof *s);
    s->n_layers = m->c.n_layers;
    s->K = (double**)calloc((size_t)m->c.n_layers, sizeof(double*));
    s->V = (double**)calloc((size_t)m->c.n_layers, sizeof(double*));
    return s;
}

void orc_stream_free(const orc_model* m, orc_stream* s) {
    (void)m;
    if (!s) return;
    for (int l = 0; l < s->n_layers; ++l) { free(s->K[l]); free(s->V[l]); }
    free(s->K); free(s->V); free(s->id_hist);
    free(s);
}

static void ensure_kv(const orc_model* m, orc_stream* s, long npos) {
    if (npos <= s->kv_cap) return;
    long cap = s->kv_cap ? s->kv_cap : 64;
    while (cap < npos) cap *= 2;
    size_t D = (size_t)m->c.D;
    for (int l = 0; l < m->c.n_layers; ++l) {
        s->K[l] = (double*)realloc(s->K[l], sizeof(double) * D * (size_t)cap);
        s->V[l] = (double*)realloc(s->V[l], sizeof(double) * D * (size_t)cap);
    }
    s->kv_cap = cap;
}

void orc_stream_set_position(const orc_model* m, orc_stream* s, long pos) {
    (void)m;
    s->pos = pos;
    s->first_pos = pos;
}

/* Load K and V for absolute positions first..first+n-1 of one layer.  k, v are bf16 bit
 * patterns laid out [H][n][dh] (the head-major layout of the GPU cache), widened exactly. */
void orc_stream_load_kv(const orc_model* m, orc_stream* s, int layer, long first, long n, const uint16_t* k,
                        const uint16_t* v) {
    const orc_config* c = &m->c;
    ensure_kv(m, s, first + n);
    for (long p = 0; p < n; ++p)
        for (int h = 0; h < c->H; ++h)
            for (int d = 0; d < c->dh; ++d) {
                size_t src = ((size_t)h * (size_t)n + (size_t)p) * (size_t)c->dh + (size_t)d;
                size_t dst = (size_t)(first + p) * (size_t)c->D + (size_t)h * (size_t)c->dh + (size_t)d;
                s->K[layer][dst] = orc_bf16_to_double(k[src]);
                s->V[layer][dst] = orc_bf16_to_double(v[src]);
            }
}

long orc_stream_position(const orc_stream* s) { return s->pos; }

/* Delay assembly: stream k at position p reads the IDs given at p - delay[k]; before the
 * first frame since reset/position set it reads the stream's initial ID. */
static void assemble(const orc_model* m, const orc_stream* s, int32_t* in) {
    const orc_config* c = &m->c;
    for (int k = 0; k < c->n_streams; ++k) {
        long src = s->pos - c->delays[k];
        if (src < s->first_pos)
            in[k] = stream_init(c, k);
        else
            in[k] = s->id_hist[(size_t)(src - s->first_pos) * (size_t)c->n_streams + (size_t)k];
    }
}

int orc_delay_assemble(const orc_model* m, orc_stream* s, const int32_t* ids, int32_t* in_out) {
    const orc_config* c = &m->c;
    if (orc_validate_ids(c, ids) != ORC_OK) return ORC_ERR_INVALID_ID;
    long idx = s->pos - s->first_pos;
    if (idx + 1 > s->hist_cap) {
        long cap = s->hist_cap ? s->hist_cap * 2 : 64;
        while (cap < idx + 1) cap *= 2;
        s->id_hist = (int32_t*)realloc(s->id_hist, sizeof(int32_t) * (size_t)c->n_streams * (size_t)cap);
        s->hist_cap = cap;
    }
    memcpy(s->id_hist + (size_t)idx * (size_t)c->n_streams, ids, sizeof(int32_t) * (size_t)c->n_streams);
    assemble(m, s, in_out);
    return ORC_OK;
}

/* One temporal block at position pos, in place on x[D]; appends K/V at pos. */
static void temporal_block(const orc_model* m, orc_stream* s, int l, double* x) {
    const orc_config* c = &m->c;
    const int D = c->D, H = c->H, dh = c->dh, F = c->ffn;
    const long pos = s->pos;
    double* u = (double*)malloc(sizeof(double) * (size_t)D);
    double* qkv = (double*)malloc(sizeof(double) * 3 * (size_t)D);
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    double* a = (double*)malloc(sizeof(double) * (size_t)D);
    double* gz = (double*)malloc(sizeof(double) * 2 * (size_t)F);
    double* sg = (double*)malloc(sizeof(double) * (size_t)F);
    double* f = (double*)malloc(sizeof(double) * (size_t)D);

    orc_rmsnorm(x, m->norm1[l], D, c->eps, u);
    orc_matvec(m->w_qkv[l], 3 * D, D, u, qkv);
    double* q = qkv;
    double* k = qkv + D;
    double* v = qkv + 2 * D;
    for (int h = 0; h < H; ++h) {
        orc_rope(q + h * dh, dh, pos, c->rope_theta);
        orc_rope(k + h * dh, dh, pos, c->rope_theta);
    }
    ensure_kv(m, s, pos + 1);
    memcpy(s->K[l] + (size_t)pos * (size_t)D, k, sizeof(double) * (size_t)D);
    memcpy(s->V[l] + (size_t)pos * (size_t)D, v, sizeof(double) * (size_t)D);

    /* keys allowed where 0 <= pos - key_pos < ctx (or the pinned ring's labels) */
    long* vis = (long*)malloc(sizeof(long) * (size_t)c->ctx);
    const int n = orc_visible_positions(pos, c->ctx, c->pinned_ring, vis);
    const double** kp = (const double**)malloc(sizeof(void*) * (size_t)n);
    const double** vp = (const double**)malloc(sizeof(void*) * (size_t)n);
    for (int h = 0; h < H; ++h) {
        for (int i = 0; i < n; ++i) {
            kp[i] = s->K[l] + (size_t)vis[i] * (size_t)D + (size_t)h * (size_t)dh;
            vp[i] = s->V[l] + (size_t)vis[i] * (size_t)D + (size_t)h * (size_t)dh;
        }
        orc_attend(q + h * dh, kp, vp, n, dh, o + h * dh);
    }
    free(kp); free(vp); free(vis);

    orc_matvec(m->w_o[l], D, D, o, a);
    for (int i = 0; i < D; ++i) x[i] += a[i]; /* y = x + a */

    orc_rmsnorm(x, m->norm2[l], D, c->eps, u);
    orc_matvec(m->w_in[l], 2 * F, D, u, gz);
    for (int j = 0; j < F; ++j) sg[j] = orc_silu(gz[j]) * gz[F + j];
    orc_matvec(m->w_out[l], D, F, sg, f);
    for (int i = 0; i < D; ++i) x[i] += f[i]; /* block output = y + f */

    free(u); free(qkv); free(o); free(a); free(gz); free(sg); free(f);
}

int orc_frame_step(const orc_model* m, orc_stream* s, const int32_t* ids, double* hidden, double* residual,
                   double* logits, int32_t* argmax) {
    int32_t in[64];
    int rc = orc_delay_assemble(m, s, ids, in);
    if (rc != ORC_OK) return rc;
    return orc_frame_forward(m, s, in, hidden, residual, logits, argmax);
}

/* The temporal forward of one frame from its already-delayed inputs in[n_streams] (what
 * the generator's token ring hands the model): embedding sum, the blocks at the stream's
 * position, final norm, text head.  The stream's ID history is not touched. */
int orc_frame_forward(const orc_model* m, orc_stream* s, const int32_t* in, double* hidden, double* residual,
                      double* logits, int32_t* argmax) {
    const orc_config* c = &m->c;
    if (orc_validate_ids(c, in) != ORC_OK) return ORC_ERR_INVALID_ID;
    double* x = (double*)malloc(sizeof(double) * (size_t)c->D);
    double* h = (double*)malloc(sizeof(double) * (size_t)c->D);
    orc_embed(m, in, x);
    for (int l = 0; l < c->n_layers; ++l) temporal_block(m, s, l, x);
    if (residual) memcpy(residual, x, sizeof(double) * (size_t)c->D);
    orc_rmsnorm(x, m->out_norm, c->D, c->eps, h);
    if (hidden) memcpy(hidden, h, sizeof(double) * (size_t)c->D);
    double* lg = logits ? logits : (double*)malloc(sizeof(double) * (size_t)c->text_out);
    orc_matvec(m->text_head, c->text_out, c->D, h, lg);
    if (argmax) *argmax = orc_argmax(lg, c->text_out);
    if (!logits) free(lg);
    free(x); free(h);
    s->pos += 1;
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* full-sequence form (explicit mask matrix), frames 0..T-1 from reset          */
/* ------------------------------------------------------------------------- */

int orc_full_sequence(const orc_model* m, int T, const int32_t* ids, double* hidden, double* logits,
                      int32_t* argmax) {
    const orc_config* c = &m->c;
    const int D = c->D, H = c->H, dh = c->dh, F = c->ffn, S = c->n_streams;
    for (int t = 0; t < T; ++t)
        if (orc_validate_ids(c, ids + (size_t)t * S) != ORC_OK) return ORC_ERR_INVALID_ID;

    double* X = (double*)malloc(sizeof(double) * (size_t)T * D);
    double* U = (double*)malloc(sizeof(double) * (size_t)T * D);
    double* QKV = (double*)malloc(sizeof(double) * (size_t)T * 3 * D);
    double* O = (double*)malloc(sizeof(double) * (size_t)T * D);
    double* A = (double*)malloc(sizeof(double) * (size_t)T * D);
    double* GZ = (double*)malloc(sizeof(double) * (size_t)T * 2 * F);
    double* SG = (double*)malloc(sizeof(double) * (size_t)T * F);
    double* P = (double*)malloc(sizeof(double) * (size_t)T * T);

    /* delayed inputs for every frame, then the embedding sum */
    for (int t = 0; t < T; ++t) {
        int32_t in[64];
        for (int k = 0; k < S; ++k) {
            int src = t - c->delays[k];
            in[k] = src < 0 ? stream_init(c, k) : ids[(size_t)src * S + k];
        }
        orc_embed(m, in, X + (size_t)t * D);
    }
    for (int l = 0; l < c->n_layers; ++l) {
        for (int t = 0; t < T; ++t) {
            orc_rmsnorm(X + (size_t)t * D, m->norm1[l], D, c->eps, U + (size_t)t * D);
            orc_matvec(m->w_qkv[l], 3 * D, D, U + (size_t)t * D, QKV + (size_t)t * 3 * D);
            for (int h = 0; h < H; ++h) {
                orc_rope(QKV + (size_t)t * 3 * D + h * dh, dh, t, c->rope_theta);
                orc_rope(QKV + (size_t)t * 3 * D + D + h * dh, dh, t, c->rope_theta);
            }
        }
        /* mask matrix M[t][s] = 0 if key s is visible to query t (0 <= t - s < ctx, or the
         * pinned ring's labels with end_offset t + 1), else -inf */
        char* allow = (char*)calloc((size_t)T * T, 1);
        long* vis = (long*)malloc(sizeof(long) * (size_t)c->ctx);
        for (int t = 0; t < T; ++t) {
            const int nv = orc_visible_positions(t, c->ctx, c->pinned_ring, vis);
            for (int i = 0; i < nv; ++i) allow[(size_t)t * T + vis[i]] = 1;
        }
        free(vis);
        for (int h = 0; h < H; ++h) {
            for (int t = 0; t < T; ++t) {
                double mx = -INFINITY;
                for (int s2 = 0; s2 < T; ++s2) {
                    int allowed = allow[(size_t)t * T + s2];
                    double d = 0.0;
                    for (int e = 0; e < dh; ++e)
                        d += QKV[(size_t)t * 3 * D + h * dh + e] * QKV[(size_t)s2 * 3 * D + D + h * dh + e];
                    P[(size_t)t * T + s2] = allowed ? d / sqrt((double)dh) : -INFINITY;
                    if (P[(size_t)t * T + s2] > mx) mx = P[(size_t)t * T + s2];
                }
                double den = 0.0;
                for (int s2 = 0; s2 < T; ++s2) {
                    double e = P[(size_t)t * T + s2] == -INFINITY ? 0.0 : exp(P[(size_t)t * T + s2] - mx);
                    P[(size_t)t * T + s2] = e;
                    den += e;
                }
                for (int e = 0; e < dh; ++e) {
                    double acc = 0.0;
                    for (int s2 = 0; s2 < T; ++s2)
                        acc += P[(size_t)t * T + s2] / den * QKV[(size_t)s2 * 3 * D + 2 * D + h * dh + e];
                    O[(size_t)t * D + h * dh + e] = acc;
                }
            }
        }
        free(allow);
        for (int t = 0; t < T; ++t) {
            double* x = X + (size_t)t * D;
            orc_matvec(m->w_o[l], D, D, O + (size_t)t * D, A + (size_t)t * D);
            for (int i = 0; i < D; ++i) x[i] += A[(size_t)t * D + i];
            orc_rmsnorm(x, m->norm2[l], D, c->eps, U + (size_t)t * D);
            orc_matvec(m->w_in[l], 2 * F, D, U + (size_t)t * D, GZ + (size_t)t * 2 * F);
            for (int j = 0; j < F; ++j)
                SG[(size_t)t * F + j] = orc_silu(GZ[(size_t)t * 2 * F + j]) * GZ[(size_t)t * 2 * F + F + j];
            orc_matvec(m->w_out[l], D, F, SG + (size_t)t * F, A + (size_t)t * D);
            for (int i = 0; i < D; ++i) x[i] += A[(size_t)t * D + i];
        }
    }
    for (int t = 0; t < T; ++t) {
        double* h = U + (size_t)t * D;
        orc_rmsnorm(X + (size_t)t * D, m->out_norm, D, c->eps, h);
        if (hidden) memcpy(hidden + (size_t)t * D, h, sizeof(double) * (size_t)D);
        double* lg = (double*)malloc(sizeof(double) * (size_t)c->text_out);
        orc_matvec(m->text_head, c->text_out, D, h, lg);
        if (logits) memcpy(logits + (size_t)t * c->text_out, lg, sizeof(double) * (size_t)c->text_out);
        if (argmax) argmax[t] = orc_argmax(lg, c->text_out);
        free(lg);
    }
    free(X); free(U); free(QKV); free(O); free(A); free(GZ); free(SG); free(P);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* depformer: sixteen sequential positions, fresh depth context each call       */
/* ------------------------------------------------------------------------- */

int orc_depformer_step(const orc_model* m, const double* hidden, int32_t text_tok, const int32_t* supplied,
                       double* logits, int32_t* codes) {
    return orc_depformer_step_sampled(m, hidden, text_tok, supplied, NULL, 0, 0, logits, codes, NULL);
}

int orc_depformer_step_sampled(const orc_model* m, const double* hidden, int32_t text_tok, const int32_t* supplied,
                               const orc_sampling* smp, uint64_t pos, uint64_t row, double* logits, int32_t* codes,
                               double* margins) {
    const orc_config* c = &m->c;
    if (c->dep_layers <= 0) return ORC_ERR_ARG;
    const int Dd = c->dep_D, Hd = c->dep_H, dd = c->dep_dh, Fd = c->dep_ffn, Q = c->dep_steps;
    const int J = c->dep_layers, V = c->dep_card;
    if (text_tok < 0 || text_tok >= c->dep_text_in) return ORC_ERR_INVALID_ID;
    for (int q = 0; q < Q; ++q)
        /* a supplied code is a depth input row: 0..dep_audio_in-1, which includes the initial
         * audio ID that the generator's first model step supplies at delayed positions */
        if (supplied[q] < -1 || supplied[q] >= c->dep_audio_in) return ORC_ERR_INVALID_ID;

    double* z = (double*)malloc(sizeof(double) * (size_t)Dd);
    double* u = (double*)malloc(sizeof(double) * (size_t)Dd);
    double* qkv = (double*)malloc(sizeof(double) * 3 * (size_t)Dd);
    double* o = (double*)malloc(sizeof(double) * (size_t)Dd);
    double* a = (double*)malloc(sizeof(double) * (size_t)Dd);
    double* gz = (double*)malloc(sizeof(double) * 2 * (size_t)Fd);
    double* sg = (double*)malloc(sizeof(double) * (size_t)Fd);
    /* depth K/V per layer: [Q positions][Dd]; opened fresh for this call */
    double* Kd = (double*)calloc((size_t)J * Q * Dd, sizeof(double));
    double* Vd = (double*)calloc((size_t)J * Q * Dd, sizeof(double));
    const double** kp = (const double**)malloc(sizeof(void*) * (size_t)Q);
    const double** vp = (const double**)malloc(sizeof(void*) * (size_t)Q);
    long* dvis = (long*)malloc(sizeof(long) * (size_t)(c->dep_ctx > Q ? c->dep_ctx : Q));

    int32_t prev = text_tok;
    for (int q = 0; q < Q; ++q) {
        /* z = W_in,q h + (q = 0 ? E_text[text] : E_audio,q-1[previous code]) */
        orc_matvec(m->dep_in[q], Dd, c->D, hidden, z);
        const uint16_t* emb = (q == 0) ? m->dep_text_emb : m->dep_audio_emb[q - 1];
        for (int i = 0; i < Dd; ++i) z[i] += orc_bf16_to_double(emb[(size_t)prev * Dd + i]);

        for (int j = 0; j < J; ++j) {
            orc_rmsnorm(z, m->dep_norm1[j], Dd, c->eps, u);
            orc_matvec(m->dep_qkv[j] + (size_t)q * 3 * Dd * Dd, 3 * Dd, Dd, u, qkv);
            memcpy(Kd + ((size_t)j * Q + q) * Dd, qkv + Dd, sizeof(double) * (size_t)Dd);
            memcpy(Vd + ((size_t)j * Q + q) * Dd, qkv + 2 * Dd, sizeof(double) * (size_t)Dd);
            const int n = orc_visible_positions(q, c->dep_ctx, c->pinned_ring, dvis);
            for (int h = 0; h < Hd; ++h) {
                for (int i = 0; i < n; ++i) {
                    kp[i] = Kd + ((size_t)j * Q + dvis[i]) * Dd + (size_t)h * dd;
                    vp[i] = Vd + ((size_t)j * Q + dvis[i]) * Dd + (size_t)h * dd;
                }
                orc_attend(qkv + h * dd, kp, vp, n, dd, o + h * dd);
            }
            orc_matvec(m->dep_o[j] + (size_t)q * Dd * Dd, Dd, Dd, o, a);
            for (int i = 0; i < Dd; ++i) z[i] += a[i];
            orc_rmsnorm(z, m->dep_norm2[j], Dd, c->eps, u);
            orc_matvec(m->dep_w_in[j * Q + q], 2 * Fd, Dd, u, gz);
            for (int i = 0; i < Fd; ++i) sg[i] = orc_silu(gz[i]) * gz[Fd + i];
            orc_matvec(m->dep_w_out[j * Q + q], Dd, Fd, sg, a);
            for (int i = 0; i < Dd; ++i) z[i] += a[i];
        }
        double* lg = logits + (size_t)q * V;
        orc_matvec(m->dep_head[q], V, Dd, z, lg); /* no final depth norm */
        int32_t code;
        double mg = INFINITY;
        if (supplied[q] >= 0)
            code = supplied[q];
        else if (smp)
            code = orc_sample_topk(lg, V, smp->temperature, smp->top_k, smp->seed, pos, row, 1u + (uint64_t)q, &mg,
                                   NULL);
        else
            code = orc_argmax(lg, V);
        if (margins) margins[q] = mg;
        codes[q] = code;
        prev = code;
    }
    free(z); free(u); free(qkv); free(o); free(a); free(gz); free(sg); free(Kd); free(Vd);
    free(kp); free(vp); free(dvis);
    return ORC_OK;
}

/* Threads of the OpenMP row loops from now on (n >= 1); returns the previous count.  Used to
 * time the oracle on one core beside all of them; no arithmetic depends on it. */
int orc_set_threads(int n) {
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}

