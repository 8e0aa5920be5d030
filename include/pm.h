/*
 * pm.h -- C ABI of the GB300 (sm_103a) per-frame streaming decode step of the
 * Moshi/PersonaPlex temporal transformer and its depformer.
 *
 * What the calls compute is defined on the page "PersonaPlex native LM audit"
 * (clockless-atlas personaplex-research):
 *   pm_frame_step      section 3 "Native temporal computation" (embedding sum, 32 blocks
 *                      of RMSNorm32 -> fused QKV -> RoPE -> causal windowed attention ->
 *                      W_O + residual -> RMSNorm32 -> SwiGLU FFN + residual, final
 *                      RMSNorm32, untied text head) with the stream delays of section 7
 *                      "One exact generator step" and the KV cache of section 6;
 *   pm_depformer_step  section 4 "Native depth computation" (sixteen sequential
 *                      positions, six blocks with per-position weights and shared norm
 *                      scales, fresh depth context per frame, supplied codes replace the
 *                      sampled ones).
 * Selection is greedy (argmax, lowest index on ties).
 *
 * Conventions.
 *  - Every call is asynchronous on the CUDA stream given to pm_create; outputs are valid
 *    once that stream has synchronised.  Calls on one context must not overlap.
 *  - Weights are caller-owned device memory, bf16, PyTorch [out, in] row-major.
 *    Norm scales are bf16 vectors.  They must stay valid until pm_destroy.
 *  - The temporal KV cache is caller-owned device memory, bf16, laid out
 *    [n_layers][2 (K, V)][B_max][H][ctx][dh]; keys are stored after RoPE.  Position p of
 *    stream b lives in slot p mod ctx.  Size: pm_kv_cache_bytes().
 *  - Everything else (positions, delay ring, activations, depth cache, CUDA graphs) is
 *    owned by the context and allocated in pm_create; no call after pm_create allocates
 *    device memory.
 *  - Errors: every call validates its host-visible arguments before launching anything
 *    and returns a pm_status; on error no state changes and pm_last_error() says why.
 *    IDs given in device memory are validated on the device: an invalid one makes the
 *    whole frame a no-op (no KV write, no position advance) and is reported by the next
 *    pm_device_status().
 */
#ifndef PM_H
#define PM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pm_ctx pm_ctx;

typedef enum {
    PM_OK = 0,
    PM_ERR_ARG = 1,          /* bad pointer, size or configuration */
    PM_ERR_INVALID_ID = 2,   /* a token ID outside -1..rows-1 (or -2), or a feedback ID with no prior selection */
    PM_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    PM_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out (reported by pm_device_status) */
    PM_ERR_STATE = 5,        /* call not valid in the context's current state */
    PM_ERR_OOM = 6,          /* device allocation in pm_create failed */
    PM_ERR_UNSUPPORTED = 7   /* shape not supported by this build's kernels */
} pm_status;

/* Special token IDs (section 3 of the audit: -1 embeds to an exact zero vector; -2 is the
 * ungenerated-cache sentinel and is never a valid input). */
#define PM_ID_NONE (-1)
#define PM_ID_UNGENERATED (-2)
/* Library extension: the token this context selected for the same stream on the stream's
 * previous frame (text: the greedy text token of the previous pm_frame_step; audio stream
 * k = 1..16: depformer code q = k-1 of the previous pm_depformer_step).  Lets greedy
 * feedback stay on the device. */
#define PM_ID_FEEDBACK (-3)

#define PM_MAX_STREAMS 32

typedef struct {
    int B_max;            /* largest batch the context serves (1..64) */
    /* temporal transformer */
    int D, H, dh, ffn;    /* 4096, 32, 128, 11264 (gated hidden width) */
    int n_layers, ctx;    /* 32, 3000 */
    int text_in;          /* text embedding rows, 32001 (32000 = initial text ID) */
    int text_out;         /* text head rows, 32000 */
    int audio_in;         /* audio embedding rows, 2049 (2048 = initial audio ID) */
    int n_streams;        /* 17: text, 8 agent audio, 8 user audio */
    int delays[PM_MAX_STREAMS];  /* per stream, 0..3: {0,0,1,1,1,1,1,1,1,0,1,1,1,1,1,1,1} */
    int init_text, init_audio;   /* 32000, 2048 */
    float eps;            /* 1e-8 */
    float rope_theta;     /* 1e4 */
    /* depformer (dep_layers = 0: none) */
    int dep_D, dep_H, dep_dh, dep_ffn;  /* 1024, 16, 64, 2816 */
    int dep_layers, dep_steps, dep_ctx; /* 6, 16, 8 (or 16) */
    int dep_card;                       /* depth head rows, 2048 */
    int dep_text_in, dep_audio_in;      /* 32001, 2049 */
    unsigned flags;                     /* PM_FLAG_* */
} pm_config;

/* pm_config.flags: run batch-1 frames as one persistent cooperative launch (a phase
 * program with grid-wide barriers) instead of the default chain of one kernel per step.
 * Needs D and ffn multiples of 1024 and cooperative launch; otherwise the chain runs.
 * Measured on GB300 at 2.707 ms per 32-block frame against 2.374 ms for the chain. */
#define PM_FLAG_FRAME_PROGRAM 1u

/* pm_config.flags: attention windows of the pinned ring cache ("PersonaPlex native LM
 * audit", section 6, "Observed source-level boundary"): its position labels hide the
 * oldest key of a full ring, so a query sees min(pos + 1, ctx - 1) temporal keys and
 * min(q + 1, dep_ctx - 1) depth keys instead of the declared mask's ctx / dep_ctx.
 * Off by default (the declared mask).  Needs ctx >= 2 and dep_ctx >= 2. */
#define PM_FLAG_PINNED_RING 2u

/* pm_config.flags: run batch-1 depformer calls as a chain of one kernel per projection
 * instead of the default persistent launch (clusters of 4 CTAs per depth head, grid-wide
 * barriers between its phases).  The persistent launch keeps re-laid copies of the
 * depformer's W_o (per-head blocks) and linear_out (transposed), made in pm_create from
 * the weights as they are then (2 * J * Q * (dep_D^2 + dep_ffn * dep_D) bytes: 754 MB at
 * the full shape); it needs dep_dh = 64, dep_D = 64 * dep_H <= 1024, cooperative launch and
 * room for dep_H clusters, and is not used while depth codes are sampled or for B > 1. */
#define PM_FLAG_DEPFORMER_CHAIN 4u

/* pm_config.flags: run batches of 2..16 streams on the tcgen05 GEMM (32 batch columns)
 * instead of the warp-level MMA GEMV.  For comparison only: the GEMM takes bf16 activation
 * operands without the rounding-remainder plane, which at B = 16 moved a greedy token at a
 * top-2 gap of 1.3e-2 (the default path carries the remainder). */
#define PM_FLAG_BATCHED_TCGEN05 8u

/* Temporal weights: device pointers.  Per-layer members point to host arrays of
 * n_layers device pointers (copied by pm_create). */
typedef struct {
    const void* text_emb;                      /* [text_in][D] */
    const void* audio_emb[PM_MAX_STREAMS - 1]; /* n_streams-1 tables [audio_in][D] */
    const void* const* norm1;                  /* [D] attention-norm scale per layer */
    const void* const* in_proj;                /* [3D][D] fused Q,K,V (rows Q 0..D-1, K D..2D-1, V 2D..3D-1) */
    const void* const* out_proj;               /* [D][D] */
    const void* const* norm2;                  /* [D] FFN-norm scale per layer */
    const void* const* linear_in;              /* [2F][D]: rows 0..F-1 gate (SiLU), F..2F-1 value */
    const void* const* linear_out;             /* [D][F] */
    const void* out_norm;                      /* [D] */
    const void* text_linear;                   /* [text_out][D] */
} pm_temporal_weights;

/* Depformer weights (section 4 of the audit, parameter names of section 5). */
typedef struct {
    const void* const* dep_in;      /* dep_steps pointers, [dep_D][D] */
    const void* text_emb;           /* [dep_text_in][dep_D] */
    const void* const* audio_emb;   /* dep_steps-1 pointers, [dep_audio_in][dep_D] */
    const void* const* norm1;       /* dep_layers pointers, [dep_D], shared by all positions */
    const void* const* in_proj;     /* dep_layers pointers, [dep_steps*3*dep_D][dep_D]; position q uses rows q*3*dep_D.. */
    const void* const* out_proj;    /* dep_layers pointers, [dep_steps*dep_D][dep_D]; position q uses rows q*dep_D.. */
    const void* const* norm2;       /* dep_layers pointers, [dep_D] */
    const void* const* linear_in;   /* dep_layers*dep_steps pointers (index j*dep_steps+q), [2*dep_ffn][dep_D] */
    const void* const* linear_out;  /* same indexing, [dep_D][dep_ffn] */
    const void* const* heads;       /* dep_steps pointers, [dep_card][dep_D] */
} pm_depformer_weights;

/* Bytes of the caller-owned temporal KV cache for this configuration. */
size_t pm_kv_cache_bytes(const pm_config* cfg);

/* Create a context on the current CUDA device.  `dw` may be NULL (no depformer).
 * `kv_cache`: device pointer, pm_kv_cache_bytes(cfg) bytes, 256-byte aligned.
 * `cuda_stream`: a cudaStream_t (NULL = legacy default stream).  All positions start
 * at 0 (reset).  Returns PM_ERR_UNSUPPORTED for shapes the kernels do not cover. */
pm_status pm_create(const pm_config* cfg, const pm_temporal_weights* tw, const pm_depformer_weights* dw,
                    void* kv_cache, void* cuda_stream, pm_ctx** out);

/* Reset streams (host mask [B_max], nonzero = reset; NULL = all): position 0, empty
 * delay history, no prior selection, generator offset 0 with empty token and provided
 * rings.  Cache bytes are not cleared (the mask hides them). */
pm_status pm_reset(pm_ctx* ctx, const int32_t* stream_mask);

/* Set the positions of streams 0..B-1 (host array [B], each >= 0).  Used when the caller
 * has written the KV history of positions < pos itself.  Delayed streams read their
 * initial IDs on the first frame after a position set. */
pm_status pm_set_positions(pm_ctx* ctx, int B, const int32_t* pos);

/* Read back the positions of streams 0..B_max-1 (synchronises the stream). */
pm_status pm_get_positions(pm_ctx* ctx, int32_t* pos_out);

/* One temporal frame for streams 0..B-1.
 *  ids         [B][n_streams] int32, host or device memory: the undelayed token of each
 *              stream at this frame (-1 none, PM_ID_FEEDBACK allowed).  Host memory is
 *              copied before the call returns.
 *  text_logits [B][text_out] fp32 device memory, or NULL.
 *  hidden      [B][D] fp32 device memory, 16-byte aligned: h after the final RMSNorm,
 *              or NULL.
 *  text_token  [B] int32, device or host-mapped memory: the selected text token (greedy,
 *              or drawn after pm_set_sampling), or NULL.
 * An output that is neither device, managed nor host-mapped memory, or a hidden pointer
 * that is not 16-byte aligned, is PM_ERR_ARG (nothing is launched).
 * Advances each stream's position by one. */
pm_status pm_frame_step(pm_ctx* ctx, int B, const int32_t* ids, float* text_logits, float* hidden,
                        int32_t* text_token);

/* Prefill: T frames of stream `stream` from its current position, as if pm_frame_step
 * ran T times with these IDs for that stream alone ("PersonaPlex native LM audit",
 * section 9: the startup voice prompt, silence frames and system text prompt each advance
 * one model step), computed as passes of up to 64 frames whose projections are 64-row
 * tensor-core GEMMs and whose attention is causal within the pass.
 *  ids         [T][n_streams] int32, host or device memory: each frame's undelayed tokens
 *              (-1 none; no PM_ID_FEEDBACK).  Host memory is copied before the call returns.
 *  text_logits [1][text_out] fp32 device memory, hidden [1][D], text_token [1]: the last
 *              frame's outputs (greedy or drawn token), or NULL.
 * Advances the stream's position by T; its selection slot holds the last frame's text
 * token (so PM_ID_FEEDBACK and the depformer's default token continue from it).  Results
 * equal T single frames up to the tensor-core path's rounding (bf16 activation operands). */
pm_status pm_prefill(pm_ctx* ctx, int stream, int T, const int32_t* ids, float* text_logits, float* hidden,
                     int32_t* text_token);

/* One depformer frame (sixteen positions) for streams 0..B-1.
 *  hidden    [B][D] fp32 device memory, or NULL = the h of this context's last frame.
 *  text_tok  [B] int32 host or device memory, or NULL = the text token this context
 *            selected on its last frame.
 *  supplied  [B][dep_steps] int32 host or device memory, or NULL = all greedy:
 *            -1 = select (argmax, or drawn after pm_set_sampling), otherwise the code
 *            to use (0..dep_audio_in-1: a row of the next position's depth embedding,
 *            which includes the initial audio ID the generator supplies on its first
 *            model step).
 *  logits    [B][dep_steps][dep_card] fp32 device memory, or NULL.
 *  codes     [B][dep_steps] int32 device or host-mapped memory, or NULL. */
pm_status pm_depformer_step(pm_ctx* ctx, int B, const float* hidden, const int32_t* text_tok,
                            const int32_t* supplied, float* logits, int32_t* codes);

/* One generator step for streams 0..B-1 ("PersonaPlex native LM audit", section 7 "One
 * exact generator step"; its token ring [B,17,4] and provided ring of section 6).  Each
 * stream has a generator offset s (0 after pm_reset), separate from its position.
 *  provided     [B][n_streams] int32 host memory, or NULL: per stream the code handed in
 *               at this call (-1 = none): the user's codebooks (streams 9..16), or forced
 *               text / agent codes.  It is placed at ring column (s + delay[k]) mod 4 and
 *               marked provided; a provided target replaces the selection (text: also as
 *               the depformer's conditioning token).  Codes are 0..rows-1 of both the
 *               temporal and the depth tables of that stream; anything else is
 *               PM_ERR_INVALID_ID (nothing runs).
 *  out          [B][n_streams] int32 device or host-mapped memory, or NULL: the aligned
 *               output frame, stream k from column (s - max_delay + delay[k]) mod 4 (text
 *               and codebook 0 selected on the previous call, delayed codebooks on this
 *               one); -1 where out_valid is 0.
 *  out_valid    [B] int32 or NULL: 1 once the initial delay padding is over (s > max_delay).
 *  text_logits  [B][text_out] fp32, hidden [B][D] fp32 (16-byte aligned), depth_logits
 *               [B][dep_steps][dep_card] fp32: this call's model outputs, or NULL.
 * Steps per call: place the provided codes; while s <= delay[k] insert stream k's initial
 * ID at column s mod 4 (provided); at s = 0 nothing else (a batch whose rows are all at
 * s = 0 runs no model; rows at s = 0 in a batch that runs are restored to their position
 * and selections afterwards); otherwise run the temporal frame on column (s - 1) mod 4 as
 * given (no delay assembly: the ring has applied the delays) and the depformer with the
 * provided targets, write the selections into the unprovided slots of column s mod 4,
 * clear the provided flags of column (s - 1) mod 4, emit the aligned output, advance s.
 * Selection follows pm_set_sampling (greedy by default).  A stream driven by this call
 * should not also be stepped with pm_frame_step (PM_ID_FEEDBACK and the delay history
 * are that call's mechanism).  Needs a depformer with dep_steps = n_streams - 1. */
pm_status pm_generator_step(pm_ctx* ctx, int B, const int32_t* provided, int32_t* out, int32_t* out_valid,
                            float* text_logits, float* hidden, float* depth_logits);

/* Kernel families of a temporal frame, as reported by pm_profile_frame. */
typedef enum {
    PM_KERNEL_EMBED = 0,       /* delay assembly + embedding gather-sum */
    PM_KERNEL_QKV = 1,         /* RMSNorm + fused QKV + RoPE + KV append */
    PM_KERNEL_ATTENTION = 2,   /* split-KV decode attention */
    PM_KERNEL_OUT_PROJ = 3,    /* W_O + residual */
    PM_KERNEL_LINEAR_IN = 4,   /* RMSNorm + linear_in + SwiGLU */
    PM_KERNEL_LINEAR_OUT = 5,  /* linear_out + residual */
    PM_KERNEL_HEAD = 6,        /* final RMSNorm + text head + greedy token */
    PM_KERNEL_FRAME = 7,       /* the whole batch-1 frame as one persistent launch */
    PM_KERNEL_SAMPLE = 8       /* temperature / top-k sampling of the text token */
} pm_kernel_kind;

/* Same computation and state change as pm_frame_step, but the frame's kernels are
 * launched one at a time (no graph, no overlap between kernels) with a CUDA event after
 * each on the context's stream.  Writes each launch's device time in milliseconds to
 * kernel_ms[i] and its pm_kernel_kind to kernel_kind[i] (host arrays of max_launches
 * entries; a frame has 2 + 5 * n_layers launches, one more with text sampling), the
 * count to *n_launches, and
 * synchronises the stream.  For measurement only. */
pm_status pm_profile_frame(pm_ctx* ctx, int B, const int32_t* ids, float* text_logits, float* hidden,
                           int32_t* text_token, float* kernel_ms, int32_t* kernel_kind, int max_launches,
                           int* n_launches);

/* Sampling ("PersonaPlex native LM audit", section 7: the generator samples the text
 * token and every depth code; released defaults text temperature 0.7 / top-k 25, audio
 * 0.8 / top-k 250).  Greedy (the argmax, lowest index on ties) until this is called.
 * With temperature > 0 and top_k > 1 a token is drawn from the top_k largest logits
 * (ties at the cut kept by lower index) with weights exp((l - l_max) / temperature),
 * scanning them in descending order for the first running weight above u * total, where
 * u = (first word of Philox4x64-10 >> 40) * 2^-24 under key (seed, 0) and counter
 * (frame position, batch row, substep, 0): substep 0 for the text token, 1 + q for depth
 * position q; the frame position is the stream's position before the frame.  The drawn
 * text token replaces the greedy one everywhere (text_token output, PM_ID_FEEDBACK, the
 * depformer's default conditioning token); drawn depth codes replace the greedy ones
 * where no code is supplied.  temperature <= 0 or top_k <= 1 selects greedy for that
 * stream kind; top_k above 1024 is PM_ERR_ARG (it is clamped to the vocabulary size).
 * Ordered with the context's other calls on its stream; the next frame after a switch
 * between greedy and sampled captures new graphs. */
pm_status pm_set_sampling(pm_ctx* ctx, float text_temperature, int text_top_k, float audio_temperature,
                          int audio_top_k, unsigned long long seed);

/* Standalone sampling of B rows of logits with the rule of pm_set_sampling (counter
 * (position, row, substep, 0) for row b).
 *  logits  fp32 device memory, row b at logits + b * ld (ld >= V), V >= 1.
 *  tokens  [B] int32 device or host-mapped memory.
 * temperature <= 0 or top_k <= 1: the argmax.  top_k above 1024 is PM_ERR_ARG.  One
 * launch on the context's stream; touches no context state. */
pm_status pm_sample(pm_ctx* ctx, int B, const float* logits, int V, int ld, float temperature, int top_k,
                    unsigned long long seed, long long position, int substep, int32_t* tokens);

/* Stream snapshots (the startup voice prompt is replayed once and its state reused:
 * "PersonaPlex native LM audit", section 9, cached voice prompts restore temporal history
 * and the token ring).  A snapshot holds one stream's position, first position since
 * reset, delay history, last selections, the generator's offset, token ring and provided
 * ring, and the KV rows of every ring slot that holds a position (min(position, ctx)
 * slots).  pm_snapshot_bytes: the buffer a snapshot of this
 * configuration needs at most (header + all ctx slots). */
size_t pm_snapshot_bytes(const pm_config* cfg);

/* Copy stream `stream`'s decode state into `dst` (device memory, pm_snapshot_bytes bytes,
 * 16-byte aligned).  Synchronises the context's stream (the position decides how many
 * slots are copied). */
pm_status pm_snapshot(pm_ctx* ctx, int stream, void* dst);

/* Make stream `stream` continue exactly as the snapshotted stream would: state and KV rows
 * from `src` (device memory written by pm_snapshot of a context with the same n_layers,
 * H, dh, ctx and n_streams; PM_ERR_ARG otherwise).  The snapshot's delay-ring entries that
 * later frames read and its selections are checked on the host first: an ID outside
 * -1..rows-1 (a selection outside -2..rows-1, a generator ring code outside -2..rows-1 or
 * a provided flag other than 0 / 1) is PM_ERR_ARG and nothing is restored.  The
 * next frame is bit-identical to the snapshotted stream's next frame on the same path.
 * Synchronises the context's stream. */
pm_status pm_restore(pm_ctx* ctx, int stream, const void* src);

/* Synchronise the stream and return (and clear) any device-side error: an invalid ID
 * given in device memory (PM_ERR_INVALID_ID) or a bounded wait that ran out
 * (PM_ERR_TIMEOUT).  A frame in which a wait ran out is abandoned like a frame with an
 * invalid ID: its later kernels skip their writes, the position does not advance and no
 * selection is recorded, so the next frame repeats that position. */
pm_status pm_device_status(pm_ctx* ctx);

/* Fault injection for tests of the timeout path.  Sets the poll budget of the bounded
 * waits of the batch-1 kernel chain's projections and of the persistent frame program
 * (their shared-memory ring waits and grid-wide phase barriers), in stream order.
 * polls = 0 makes every such wait give up at once, so the next frame times out:
 * pm_device_status then returns PM_ERR_TIMEOUT.  PM_WAIT_BUDGET_DEFAULT restores the
 * normal budget.  Copies already issued by a CTA whose wait ran out are still waited for
 * with the normal budget before it exits. */
#define PM_WAIT_BUDGET_DEFAULT 0xFFFFFFFFu
pm_status pm_set_wait_budget(pm_ctx* ctx, uint32_t polls);

/* Final RMSNorm + text head + greedy token with no context and no device allocation.
 * The model describes no such call: this is a library entry point for callers that cannot
 * allocate device memory (code running during CUDA stream capture, real-time threads
 * that must not block on the allocator, hosts that own all device memory).
 *  residual  [B][D] fp32 device memory, 16-byte aligned: the residual stream after the
 *            last block.
 *  out_norm  bf16 [D]; text_linear bf16 [V][D] (device, 16-byte aligned).
 *  hidden    [B][D] fp32, 16-byte aligned (normalised state h) or NULL;
 *  logits    [B][V] fp32 or NULL;
 *  token     [B] int32 greedy token (lowest index on ties) or NULL;
 *  status    [1] int32 or NULL: once the stream reaches the end of the call, PM_OK, or
 *            PM_ERR_TIMEOUT if a bounded wait of the head ran out (outputs incomplete).
 * Outputs are device, managed or host-mapped memory; anything else is PM_ERR_ARG.
 * Same arithmetic as the head of pm_frame_step.  Scratch is a 10,240-byte static device
 * array in the library, so B may be at most 64 (PM_ERR_UNSUPPORTED beyond, or if D is
 * not a multiple of 256).  The first call on each device resolves that array's address
 * and clears it (synchronous); make it before any stream capture.  Later calls only
 * launch kernels on `cuda_stream` (NULL = legacy default stream).  All calls share the
 * array: calls that overlap on the GPU race. */
pm_status pm_text_head_noalloc(int B, int D, int V, const float* residual, const void* out_norm,
                               const void* text_linear, float eps, float* hidden, float* logits, int32_t* token,
                               int32_t* status, void* cuda_stream);

/* Message of the last failed call on this context (empty string if none); with a NULL
 * context, the reason the last pm_create on this thread failed. */
const char* pm_last_error(const pm_ctx* ctx);

/* Free everything the context owns (not the weights or the KV cache). */
void pm_destroy(pm_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* PM_H */
