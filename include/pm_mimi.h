/*
 * pm_mimi.h -- C ABI of the GB300 (sm_103a) streaming Mimi codec: the decoder takes one
 * 80 ms frame of codes per stream and call to 1,920 samples of 24 kHz PCM; the encoder
 * takes 1,920 samples to one frame of codes.
 *
 * What the calls compute is defined on the page "PersonaPlex native LM audit"
 * (clockless-atlas personaplex-research), chapter "Exact Mimi codec construction":
 *   - "Complete encode/decode order", DECODE: semantic code lookup and the semantic
 *     output projection, plus the sum of the acoustic lookups and the acoustic output
 *     projection; the learned depthwise ConvTranspose1d (kernel 4, stride 2, no bias) from
 *     12.5 Hz to 25 Hz; the decoder transformer; the SEANet decoder;
 *   - "Split quantizer: exact paths and active capacity" (codebook 0 semantic, 1..n_q-1
 *     acoustic, bias-free output projections [dim, cb_dim]);
 *   - "Both codec transformer stacks" (per block LayerNorm -> self-attention with RoPE,
 *     causal window 0 <= q - k < ctx -> LayerScale -> residual -> LayerNorm -> Linear ->
 *     GELU -> Linear -> LayerScale -> residual; 64-wide heads);
 *   - "SEANet decoder, every stage" (Conv1d dim -> n_filters 2^n_ratios, kernel `kernel`;
 *     per stage ELU -> ConvTranspose1d C -> C/2, kernel 2r, stride r, then the residual
 *     unit x + Conv(k1)(ELU(Conv(k res_kernel, C/2 -> C/2/compress)(ELU(x)))); ELU ->
 *     Conv1d -> 1 channel, kernel last_kernel; every convolution with a bias);
 *   - "Stateful streaming, padding and dependency boundaries": causal convolutions pad
 *     kernel - stride on the left, causal transposed convolutions trim kernel - stride on
 *     the right; a streaming codec emits exactly the non-streaming result frame by frame;
 *   - ENCODE: "SEANet encoder, every stage" (Conv1d 1 -> n_filters, kernel `kernel`; per
 *     stage, in the reversed ratio order, the residual unit then ELU -> Conv1d C -> 2C,
 *     kernel 2r, stride r; ELU -> Conv1d -> dim, kernel last_kernel), the encoder
 *     transformer (a separate stack), "Learned resampling around the quantizer" (Conv1d
 *     dim -> dim, kernel 4, stride 2, no bias, the first position replicated as left
 *     padding), and the split quantizer (semantic projection -> nearest entry of codebook
 *     0; acoustic projection -> residual chain over codebooks 1..n_q-1).
 * Readings where the chapter is silent: RoPE turns adjacent pairs (2j, 2j+1) of each head
 * by position * rope_theta^(-2j/64); the attention scale is 1/sqrt(64); GELU is the erf
 * form; ELU has alpha 1; transformer positions count the 25 Hz grid from 0 at reset;
 * "nearest" is the smallest squared Euclidean distance (fp32), the lowest index on ties.
 *
 * Conventions (as in pm.h).
 *  - Calls are asynchronous on the CUDA stream given to pm_mimi_create; outputs are valid
 *    once it has synchronised.  Calls on one context must not overlap.
 *  - Weights are caller-owned device memory, bf16, 16-byte aligned, valid until
 *    pm_mimi_destroy, given as an array of pointers in this canonical order (PyTorch
 *    layouts: Linear [out][in], Conv1d [out][in][k], ConvTranspose1d [in][out][k]):
 *      q.codebook.0 .. q.codebook.{n_q-1}  [card][cb_dim]
 *      q.sem.out [dim][cb_dim], q.ac.out [dim][cb_dim], up.weight [dim][1][4]
 *      per block l < n_layers: norm1.w [dim], norm1.b [dim], in_proj [3 dim][dim] (q, k,
 *        v rows), out_proj [dim][dim], scale1 [dim], norm2.w, norm2.b, lin1 [ffn][dim],
 *        lin2 [dim][ffn], scale2 [dim]
 *      dec.0.w [C0][dim][kernel], dec.0.b [C0]          (C0 = n_filters << n_ratios)
 *      per stage i (C -> C/2, r = ratios[i], h = C/2/compress): up.w [C][C/2][2r],
 *        up.b [C/2], res.w1 [h][C/2][res_kernel], res.b1 [h], res.w2 [C/2][h][1],
 *        res.b2 [C/2]
 *      dec.out.w [1][n_filters][last_kernel], dec.out.b [1]
 *    pm_mimi_tensor_count() gives the count.
 *  - Everything else (streaming state, the transformer's key/value ring of ctx + 1
 *    positions per block, activations, one CUDA graph per batch size) is allocated by
 *    pm_mimi_create; no later call allocates device memory.
 *  - Errors: host-visible arguments are validated before anything launches (pm_status,
 *    pm_mimi_last_error).  Codes given in device memory are validated on the device: an
 *    invalid one turns the whole call into a no-op (no state advances, the PCM output is
 *    zeros) reported by the next pm_mimi_status().
 *  - Arithmetic: fp32 activations and accumulation, bf16 weights widened exactly.
 */
#ifndef PM_MIMI_H
#define PM_MIMI_H

#include "pm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pm_mimi_ctx pm_mimi_ctx;

#define PM_MIMI_MAX_B 8
#define PM_MIMI_MAX_RATIOS 8

typedef struct {
    int B_max;            /* streams the context serves, 1..PM_MIMI_MAX_B */
    int dim;              /* latent / transformer width: 64 x heads, a multiple of 256 (512) */
    int cb_dim;           /* codebook vector width, a multiple of 8 (256) */
    int card;             /* entries per codebook (2048) */
    int n_q;              /* codebooks used: 1 semantic + n_q - 1 acoustic, 2..16 (8) */
    int n_layers;         /* decoder transformer blocks (8) */
    int heads;            /* attention heads of width 64 (8) */
    int ffn;              /* feed-forward width, a multiple of 256 (2048) */
    int ctx;              /* attention window in 25 Hz positions (250) */
    int n_filters;        /* SEANet base width (64) */
    int n_ratios;         /* SEANet stages (4) */
    int ratios[PM_MIMI_MAX_RATIOS]; /* upsampling ratio per stage, 1..16 (8, 6, 5, 4) */
    int kernel;           /* first convolution's kernel (7) */
    int last_kernel;      /* last convolution's kernel (3) */
    int res_kernel;       /* residual unit's first kernel (3) */
    int compress;         /* residual unit's width divisor (2) */
    int up_kernel;        /* latent upsampler kernel: must be 4 */
    int up_stride;        /* latent upsampler stride: must be 2 */
    float ln_eps;         /* LayerNorm epsilon (1e-5) */
    float rope_theta;     /* RoPE base (10000) */
} pm_mimi_config;

/* Number of tensors pm_mimi_create expects for this configuration, or -1 if the
 * configuration is not supported. */
int pm_mimi_tensor_count(const pm_mimi_config* cfg);

/* The encoder's canonical tensor order (same layout conventions):
 *      enc.0.w [n_filters][1][kernel], enc.0.b
 *      per stage i (C = n_filters << i, r = ratios[n_ratios - 1 - i], h = C / compress):
 *        res.w1 [h][C][res_kernel], res.b1 [h], res.w2 [C][h][1], res.b2 [C],
 *        down.w [2C][C][2r], down.b [2C]
 *      enc.out.w [dim][n_filters << n_ratios][last_kernel], enc.out.b [dim]
 *      per block l < n_layers: the ten tensors of a decoder block (the encoder's own stack)
 *      ds.weight [dim][dim][4] (the downsampler, no bias)
 *      q.sem.in [cb_dim][dim], q.ac.in [cb_dim][dim] (input projections)
 *      q.codebook.0 .. q.codebook.{n_q-1} [card][cb_dim] (the tables the decoder reads)
 * Count, or -1 if the encoder does not support the configuration (it also needs card a
 * multiple of 8 and dim a multiple of 128). */
int pm_mimi_encoder_tensor_count(const pm_mimi_config* cfg);

/* Create a decoder for up to cfg->B_max streams, all at frame 0.  tensors: n_tensors
 * device pointers in the canonical order above.  cuda_stream: the stream every call runs
 * on (NULL = legacy default stream).  PM_ERR_ARG for a bad configuration, pointer or
 * count; PM_ERR_UNSUPPORTED if a kernel would need more than 227 KB of shared memory;
 * PM_ERR_OOM if the device allocation fails.  On failure *out is NULL and
 * pm_mimi_last_error(NULL) says why. */
pm_status pm_mimi_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors, void* cuda_stream,
                         pm_mimi_ctx** out);

/* Create an encoder context (same conventions as pm_mimi_create; the tensors in the
 * encoder's order).  pm_mimi_reset, pm_mimi_status, pm_mimi_get_frames, pm_mimi_last_error
 * and pm_mimi_destroy serve both kinds; pm_mimi_decode on an encoder context, or
 * pm_mimi_encode on a decoder context, is PM_ERR_STATE. */
pm_status pm_mimi_encoder_create(const pm_mimi_config* cfg, const void* const* tensors, int n_tensors,
                                 void* cuda_stream, pm_mimi_ctx** out);

/* Encode the next frame of streams 0..B-1.
 *  pcm     [B][frame_samples] fp32, host or device memory (host PCM is copied in through
 *          pinned staging).
 *  codes   [B][n_q] int32 out: semantic code then the acoustic codes; device, managed or
 *          host-mapped memory, 4-byte aligned.
 *  latent  [B][dim] fp32 out, or NULL: the unquantised latent after the downsampler.
 * Each stream advances by one frame.  Every float input gives in-range codes (no device
 * validation is needed); non-finite PCM gives unspecified codes. */
pm_status pm_mimi_encode(pm_mimi_ctx* ctx, int B, const float* pcm, int32_t* codes, float* latent);

/* Decode the next frame of streams 0..B-1.
 *  codes  [B][n_q] int32 code indices 0..card-1, host or device memory.  Host codes are
 *         checked before anything launches (PM_ERR_INVALID_ID, nothing runs); device codes
 *         on the device (see Errors).
 *  pcm    [B][frame_samples] fp32 (frame_samples = up_stride x prod(ratios) = 1920),
 *         device, managed or host-mapped memory, 4-byte aligned: the frame's samples,
 *         which continue the stream's previous frames exactly.
 * Each stream advances by one frame (two 25 Hz positions).  The first call with a given B
 * captures that batch size's graph (synchronous; later calls only launch it). */
pm_status pm_mimi_decode(pm_mimi_ctx* ctx, int B, const int32_t* codes, float* pcm);

/* Kinds of the launches pm_mimi_profile times, in launch order: the front; per block
 * in_proj, attention, out_proj, lin1, lin2; the first convolution; per stage the
 * transposed convolution and the residual unit's two convolutions; the last convolution;
 * the finishing kernel. */
#define PM_MIMI_K_FRONT 0
#define PM_MIMI_K_IN_PROJ 1
#define PM_MIMI_K_ATTN 2
#define PM_MIMI_K_OUT_PROJ 3
#define PM_MIMI_K_LIN1 4
#define PM_MIMI_K_LIN2 5
#define PM_MIMI_K_CONV_FIRST 6
#define PM_MIMI_K_CONVTR 7
#define PM_MIMI_K_RES1 8
#define PM_MIMI_K_RES2 9
#define PM_MIMI_K_CONV_LAST 10
#define PM_MIMI_K_FINISH 11
#define PM_MIMI_K_DOWN 12      /* encoder: a SEANet stride-r convolution */
#define PM_MIMI_K_RESAMPLE 13  /* encoder: the latent downsampler */
#define PM_MIMI_K_RVQ 14       /* encoder: input projections + residual quantisation */

/* pm_mimi_decode launched kernel by kernel (not from the graph) with a CUDA event after
 * each launch, then synchronised: ms[i] is the device time between launch i's event and
 * the previous one, kind[i] its PM_MIMI_K_* kind; *n receives the count (at most n_max;
 * 2 + 5 n_layers + 3 n_ratios + 2 launches).  Same arguments, results and state advance
 * as pm_mimi_decode.  For measurement, not for serving: it creates and destroys events. */
pm_status pm_mimi_profile(pm_mimi_ctx* ctx, int B, const int32_t* codes, float* pcm, float* ms, int32_t* kind,
                          int n_max, int* n);

/* pm_mimi_encode launched kernel by kernel, timed the same way (the encoder's launches: the
 * first convolution; per stage the residual unit's two convolutions and the strided
 * convolution; the last convolution; the transformer; the downsampler; the quantiser; the
 * finishing kernel). */
pm_status pm_mimi_encode_profile(pm_mimi_ctx* ctx, int B, const float* pcm, int32_t* codes, float* latent,
                                 float* ms, int32_t* kind, int n_max, int* n);

/* Return the streams whose mask entry is nonzero (all streams if mask is NULL; a host
 * array of B_max entries) to frame 0 with empty history, ordered on the context's stream. */
pm_status pm_mimi_reset(pm_mimi_ctx* ctx, const int32_t* mask);

/* Synchronise the context's stream; PM_ERR_INVALID_ID if a call since the last
 * pm_mimi_status met an invalid device code (that call was a no-op), PM_ERR_TIMEOUT if a
 * bounded wait ran out (pm_mimi_set_wait_budget), else PM_OK.  Reading clears both. */
pm_status pm_mimi_status(pm_mimi_ctx* ctx);

/* Poll budget of the encoder's bounded waits (the quantiser's waits for its codebook
 * copies; PM_WAIT_BUDGET_DEFAULT restores the normal budget).  A wait that runs out makes
 * that call's codes undefined and the next pm_mimi_status returns PM_ERR_TIMEOUT; the
 * streaming state advances as usual (the quantiser holds none), and copies already issued
 * are waited for with the normal budget before the kernel exits.  Synchronises the
 * context's stream; for tests of that path. */
pm_status pm_mimi_set_wait_budget(pm_mimi_ctx* ctx, uint32_t polls);

/* Synchronise and copy the frames decoded since reset per stream ([B_max] int32, host). */
pm_status pm_mimi_get_frames(pm_mimi_ctx* ctx, int32_t* frames);

/* Message of the last failed call on this context; with NULL, why the last
 * pm_mimi_create on this thread failed. */
const char* pm_mimi_last_error(const pm_mimi_ctx* ctx);

/* Free everything the context owns (not the weights); either kind. */
void pm_mimi_destroy(pm_mimi_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* PM_MIMI_H */
