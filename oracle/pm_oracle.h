/*
 * Float64 CPU oracle of the Moshi/PersonaPlex per-frame decode step.
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the bench's
 * CPU-baseline leg, never by the library.  See pm_oracle.c for the passages followed.
 *
 * Weights are bf16 bit patterns (uint16_t) in PyTorch [out, in] orientation, passed as an
 * array of pointers in the canonical order:
 *   text_emb [text_in][D]; emb.i [audio_in][D] for i < n_streams-1;
 *   per layer l: norm1 [D], in_proj [3D][D], out_proj [D][D], norm2 [D],
 *                linear_in [2F][D], linear_out [D][F];
 *   out_norm [D]; text_linear [text_out][D];
 *   if dep_layers > 0: depformer_in.q [Dd][D] (q < Q); depformer_text_emb [dep_text_in][Dd];
 *     depformer_emb.q [dep_audio_in][Dd] (q < Q-1);
 *     per depth layer j: norm1 [Dd], in_proj [Q*3*Dd][Dd], out_proj [Q*Dd][Dd], norm2 [Dd],
 *       gating.q.linear_in [2Fd][Dd] (q < Q), gating.q.linear_out [Dd][Fd] (q < Q);
 *     linears.q [dep_card][Dd] (q < Q).
 * The oracle borrows the pointers; they must outlive the model.
 */
#ifndef PM_ORACLE_H
#define PM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_INVALID_ID = 2 };

typedef struct {
    int D, H, dh, ffn, n_layers, ctx;
    int text_in, text_out, audio_in, n_streams;
    int delays[64];
    int init_text, init_audio;
    double eps, rope_theta;
    int dep_D, dep_H, dep_dh, dep_ffn, dep_layers, dep_steps, dep_ctx, dep_card, dep_text_in, dep_audio_in;
    int pinned_ring; /* 0: the declared mask; 1: the pinned ring's position labels (both caches) */
} orc_config;

typedef struct orc_model orc_model;
typedef struct orc_stream orc_stream;

/* scalar steps, exposed so that each can be pinned on its own */
double orc_bf16_to_double(uint16_t h);
void orc_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y);
void orc_rmsnorm(const double* x, const uint16_t* alpha, int n, double eps, double* out);
void orc_rope(double* v, int dh, long pos, double theta);
double orc_silu(double g);
void orc_attend(const double* q, const double* const* keys, const double* const* vals, int n, int dh, double* o);
int orc_argmax(const double* v, int n);
/* position labels of a ring of `capacity` slots after `end_offset` writes, as the pinned
 * implementation reports them; and the positions a query at `pos` may attend to (its own
 * key written, so end_offset = pos + 1), ascending, into vis[] (capacity entries); returns
 * their count.  pinned = 0 gives the declared mask 0 <= pos - p < capacity. */
void orc_ring_labels(long capacity, long end_offset, long* labels);
int orc_visible_positions(long pos, long capacity, int pinned, long* vis);

int orc_tensor_count(const orc_config* c);
orc_model* orc_create(const orc_config* c, const uint16_t* const* tensors, int n_tensors);
void orc_destroy(orc_model* m);
int orc_validate_ids(const orc_config* c, const int32_t* ids);
void orc_embed(const orc_model* m, const int32_t* in, double* x);

orc_stream* orc_stream_new(const orc_model* m);
void orc_stream_free(const orc_model* m, orc_stream* s);
void orc_stream_set_position(const orc_model* m, orc_stream* s, long pos);
void orc_stream_load_kv(const orc_model* m, orc_stream* s, int layer, long first, long n, const uint16_t* k,
                        const uint16_t* v);
long orc_stream_position(const orc_stream* s);
/* records ids[n_streams] for the stream's current position and returns the delayed inputs */
int orc_delay_assemble(const orc_model* m, orc_stream* s, const int32_t* ids, int32_t* in_out);

/* One frame: ids[n_streams] undelayed; outputs hidden = h after the final norm [D],
 * residual = x before it [D] (may be NULL), logits [text_out] (may be NULL), argmax. */
int orc_frame_step(const orc_model* m, orc_stream* s, const int32_t* ids, double* hidden, double* residual,
                   double* logits, int32_t* argmax);
/* One frame from already-delayed inputs in[n_streams] (no delay assembly, ID history
 * untouched); same outputs as orc_frame_step, position advanced by one. */
int orc_frame_forward(const orc_model* m, orc_stream* s, const int32_t* in, double* hidden, double* residual,
                      double* logits, int32_t* argmax);
/* Frames 0..T-1 from reset, every layer evaluated over all T positions with an explicit
 * mask matrix.  ids [T][n_streams]; hidden [T][D]; logits [T][text_out]; argmax [T]. */
int orc_full_sequence(const orc_model* m, int T, const int32_t* ids, double* hidden, double* logits,
                      int32_t* argmax);
/* Depformer: hidden [D] (h after the final norm), text token, supplied [Q] (-1 = greedy);
 * outputs logits [Q][dep_card] and codes [Q]. */
int orc_depformer_step(const orc_model* m, const double* hidden, int32_t text_tok, const int32_t* supplied,
                       double* logits, int32_t* codes);

/* sampling: Philox4x64-10 block (counter ctr, key), the 24-bit uniform of the counter
 * (c0, c1, c2, 0) under key (seed, 0), and temperature / top-k sampling of one row of
 * logits with that uniform.  margin (may be NULL): distance of u * total from the nearest
 * cumulative boundary of the pick, relative to the total; cut_gap (may be NULL): logit
 * gap between the k-th and (k+1)-th largest (INFINITY when k >= V or greedy). */
typedef struct {
    double temperature;
    int top_k;
    uint64_t seed;
} orc_sampling;
void orc_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
double orc_uniform24(uint64_t seed, uint64_t c0, uint64_t c1, uint64_t c2);
int orc_sample_topk(const double* logits, int V, double temperature, int top_k, uint64_t seed, uint64_t c0,
                    uint64_t c1, uint64_t c2, double* margin, double* cut_gap);
/* Depformer with sampled codes where none is supplied (smp NULL = greedy): position q's
 * counter is (pos, row, 1 + q).  margins [Q] (may be NULL): the pick margins (INFINITY
 * where supplied or greedy). */
int orc_depformer_step_sampled(const orc_model* m, const double* hidden, int32_t text_tok, const int32_t* supplied,
                               const orc_sampling* smp, uint64_t pos, uint64_t row, double* logits, int32_t* codes,
                               double* margins);

/* threads of the OpenMP row loops from now on (n >= 1); returns the previous count */
int orc_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
