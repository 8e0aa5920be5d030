// Host-side interface between the C-ABI layer (pm_api.cu) and the kernel translation
// units.  Plain structs of device pointers and sizes; every launch goes on `stream` and,
// when `pdl` is set, may begin before the previous kernel in the stream has finished
// (programmatic dependent launch: the kernel waits with griddepcontrol.wait before it
// reads anything the previous kernel wrote).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

#include "pm_common.cuh"

namespace pm {

// ----------------------------------------------------------------------------------
// weight-streaming GEMV  y = W x  (bf16 W [rows][K], fp32 x), B = 1 row of x per CTA
// ----------------------------------------------------------------------------------
enum Unit { U_ROW = 0, U_PAIR_ADJ = 1, U_PAIR_SPLIT = 2 };
enum Prologue {
    PRO_PLAIN = 0,    // x as given
    PRO_RMSNORM = 1,  // x normalised (fp32 RMSNorm, learned scale)
    PRO_DEPATTN = 2,  // x = depth attention output, computed by every CTA from q and the depth cache
    PRO_RMSNORM_EMB = 3  // depformer layer 0: x = input projection + E[previous code], written to
                         // x_out (the residual stream) by CTA 0, then normalised
};
enum Epilogue {
    E_STORE = 0,      // y[row] = dot
    E_RESIDUAL = 1,   // y[row] += dot
    E_SWIGLU = 2,     // y[u] = SiLU(dot(row u)) * dot(row u + F)
    E_QKV_ROPE = 3,   // temporal fused QKV: RoPE on Q, K; K, V into the KV ring
    E_HEAD = 4,       // text head: logits + argmax, frame finalisation
    E_DEP_QKV = 6,    // depth QKV: q to y, k, v into the depth cache at position q
    E_DEP_HEAD = 7    // depth head: logits + argmax or supplied code
};

// matrices one GEMV launch can take as consecutive segments of its rows
#define PM_GEMV_MAX_SEG 32

struct GemvParams {
    const uint16_t* W;     // [rows][K]
    int nseg, seg_units;   // > 1: units s*seg_units .. are rows of Wseg[s] (W unused)
    const uint16_t* Wseg[PM_GEMV_MAX_SEG];
    int K;
    int n_units;           // units (rows or row pairs) of the whole matrix
    int split_rows;        // U_PAIR_SPLIT: unit u = rows u and u + split_rows
    // plan (filled by plan_gemv)
    int CH, P, upst, warps, nst, grid_per_b, units_cta_max;
    uint32_t stage_bytes;
    size_t smem;
    int B;
    // input vector
    const float* x;        // [B][x_stride]
    int x_stride;
    const uint16_t* alpha; // norm scale [K] (PRO_RMSNORM)
    float eps;
    // main output
    float* y;              // [B][y_stride]
    int y_stride;
    // shared state
    DevState st;
    // E_QKV_ROPE
    int D, H, dh, ctx, B_max;
    uint16_t* kc;          // K cache of this layer: [B_max][H][ctx][dh]
    uint16_t* vc;          // V cache of this layer
    const float2* rope_tab;   // [B][dh/2] (cos, sin) of this frame's positions
    // E_HEAD
    const FrameIO* io;
    float* h_internal;     // [B][K] normalised input copy (the hidden state), written by CTA 0
    // depformer
    const DepIO* dio;
    int q;                 // depth position
    int Q;                 // depth positions per frame
    const uint16_t* emb;   // PRO_RMSNORM_EMB table [rows][K]
    float* x_out;          // PRO_RMSNORM_EMB: the assembled (pre-norm) input [B][K], by CTA 0
    uint16_t* dkc;         // E_DEP_QKV / PRO_DEPATTN: depth K cache of this layer [B_max][Hd][Q][dhd]
    uint16_t* dvc;
    int dep_ctx;           // PRO_DEPATTN: attention window (x = q of depth position q)
    int x_in_smem;         // plan input: the prologue builds x in shared memory (PRO_DEPATTN)
    float dep_scale_log2;
    int n_streams;
    float* logits_copy;    // E_HEAD / E_DEP_HEAD: also write the logits here ([B][y_stride]), or null
};

// Choose the tiling for a GEMV of row length K over n_units units of rows_per_unit rows.
// Returns false if the shape is not supported (K % 256 != 0 or K too large).
bool plan_gemv(GemvParams& p, int rows_per_unit, int num_sms);

cudaError_t launch_gemv(int pro, int epi, int unit, const GemvParams& p, cudaStream_t s, bool pdl);

// Raise the dynamic shared-memory limit of every GEMV variant (once per process/device).
cudaError_t gemv_prepare();

// ----------------------------------------------------------------------------------
// embedding gather-sum with delay assembly and ID validation
// ----------------------------------------------------------------------------------
struct EmbedParams {
    const uint16_t* tables[PM_MAX_STREAMS_DEV];  // stream k -> table (0 = text)
    const FrameIO* io;
    DevState st;
    float* x;        // [B][D]
    int D, B, n_streams;
    int rows[PM_MAX_STREAMS_DEV];
    int init_id[PM_MAX_STREAMS_DEV];
    int delays[PM_MAX_STREAMS_DEV];
    // RoPE table of this frame: rope_tab[b][j] = (cos, sin)(pos_b * freq[j]), j < dh/2
    float2* rope_tab;
    const double* rope_freq;
    int dh;
    // prefill: rows are frames pos .. pos+B-1 of stream io->seq_stream with these inputs
    // (delays already applied and IDs validated by k_seq_prepare), or null
    const int32_t* resolved;  // [B][n_streams]
    // tensor-core path (B >= 2): bf16(alpha * x) operand [npad][D] and per-CTA sums of x^2
    uint16_t* xb;
    int xb_lo_rows;  // > 0: also the rounding remainder of the operand at row b + xb_lo_rows
    const uint16_t* alpha;
    float* ss;       // [D/1024][npad]
    int npad;
};
cudaError_t launch_embed(const EmbedParams& p, cudaStream_t s, bool pdl);

// ----------------------------------------------------------------------------------
// split-KV decode attention over the temporal ring (dh = 128)
// ----------------------------------------------------------------------------------
struct AttnParams {
    uint16_t* ob;          // [npad][D] bf16 copy of o for the tensor-core W_O, or null
    int ob_lo_rows;        // > 0: also the rounding remainder bf16(o - ob) at row b + ob_lo_rows
    const float* q;        // [B][D] rotated queries
    const uint16_t* kc;    // [B_max][H][ctx][dh]
    const uint16_t* vc;
    float* o;              // [B][D]
    float* part;           // [B][H][S][dh + 2] chunk partials
    uint32_t* count;       // [B][H], zero between launches
    DevState st;
    int B, H, ctx, S, D;
    int win;               // most keys a query sees (ctx, or ctx - 1 for the pinned ring)
    int grid;              // CTAs (attn_plan)
    int cluster;           // CTAs per head in head-per-cluster mode (1..8), 0 = balanced split
    float scale_log2;      // log2(e) / sqrt(dh)
};
cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl);
cudaError_t attn_prepare();  // opt-in shared memory of the attention kernel
// grid and mode for B rows of H heads (sets p.grid, p.cluster)
void attn_plan(AttnParams& p, int num_sms);
// chunks (CTAs per head) the attention grid needs for a window of ctx keys; AttnParams.S
// must be at least this and `part` must hold S chunks per head
int attn_max_splits(int ctx);

// ----------------------------------------------------------------------------------
// prefill (T frames of one stream as one batched pass)
// ----------------------------------------------------------------------------------
#define PM_SEQ_MAX_ROWS 64       // frames per prefill pass
#define PM_SEQ_KPC 256           // keys per attention work item
#define PM_SEQ_MAX_CHUNKS 16     // work items per head (window + rows up to 4096 keys)
#define PM_SEQ_PART_STRIDE 132   // floats per attention partial (128 values, max, sum, pad)
struct SeqPrepParams {
    const FrameIO* io;
    DevState st;
    int32_t* resolved;       // [T][n_streams] out
    int T, n_streams;
    int rows[PM_MAX_STREAMS_DEV];
    int init_id[PM_MAX_STREAMS_DEV];
    int delays[PM_MAX_STREAMS_DEV];
};
cudaError_t launch_seq_prepare(const SeqPrepParams& p, cudaStream_t s, bool pdl);
struct AttnSeqParams {
    const float* q;          // [T][D] rotated queries
    const uint16_t* kc;      // this layer's K cache [B_max][H][ctx][dh] (positions < pos)
    const uint16_t* vc;
    const uint16_t* kv_new;  // [2][T][H][dh] this pass's K and V (positions pos .. pos+T-1)
    float* o;                // [T][D]
    uint16_t* ob;            // [npad][D] bf16 copy of o, or null
    float* part;             // [T][H][PM_SEQ_MAX_CHUNKS][PM_SEQ_PART_STRIDE]
    DevState st;
    const FrameIO* io;
    int T, H, ctx, win, D, grid;
    float scale_log2;
};
cudaError_t launch_attn_seq(const AttnSeqParams& p, cudaStream_t s, bool pdl);
// after the pass attention: merges each row's chunk partials (windows of several chunks)
// and copies the pass's K/V rows into the ring (the last row of each slot)
cudaError_t launch_seq_commit(const AttnSeqParams& p, cudaStream_t s, bool pdl);
cudaError_t attn_seq_prepare();
int attn_seq_max_chunks(int win);

// ----------------------------------------------------------------------------------
// depformer helpers
// ----------------------------------------------------------------------------------
struct DepBeginParams {
    const DepIO* dio;
    DevState st;
    float* h_internal;     // [B][D] hidden the chain reads
    int32_t* dep_sup;      // [B][Q] validated supplied codes
    int B, D, Q, sup_rows, text_rows;  // sup_rows: depth audio embedding rows (supplied codes < it)
};
cudaError_t launch_dep_begin(const DepBeginParams& p, cudaStream_t s, bool pdl);

// ----------------------------------------------------------------------------------
// generator step (token ring + provided ring, section 7 of the audit)
// ----------------------------------------------------------------------------------
struct GenParams {
    DevState st;
    int32_t* ring;            // [B_max][PM_MAX_STREAMS_DEV][4] codes (-2: never written)
    int32_t* prov;            // [B_max][PM_MAX_STREAMS_DEV][4] provided flags
    int32_t* off;             // [B_max] generator offsets
    const int32_t* provided;  // [B][S] codes handed in (-1: none), or null
    int32_t* in;              // [B][S] the frame's inputs
    int32_t* dep_tok;         // [B] depth conditioning token
    int32_t* dep_sup;         // [B][Q] provided depth targets (-1: select)
    int32_t* pos_save;        // [B_max] position before the call's frame
    int32_t* sel_save;        // [B_max][PM_MAX_STREAMS_DEV] selections before the call's frame
    int32_t* out;             // [B][S] aligned output codes, or null
    int32_t* valid;           // [B] 1 where out holds a frame, or null
    int B, S, Q, max_delay;
    int ran;                  // the frame and the depformer ran in this call
    int delays[PM_MAX_STREAMS_DEV];
    int init[PM_MAX_STREAMS_DEV];
};
// phase 0: steps 1-3 (before the frame), 1: depth inputs (before the depformer), 2: steps 6-7
cudaError_t launch_gen(int phase, const GenParams& p, cudaStream_t s);

// ----------------------------------------------------------------------------------
// depformer call for batch 1 as one persistent launch (clusters of 4 CTAs per depth head)
// ----------------------------------------------------------------------------------
#define PM_DF_MAX_Q 16
#define PM_DF_MAX_J 8
struct DepFusedParams {
    DevState st;
    const DepIO* dio;
    const uint16_t* dep_in[PM_DF_MAX_Q];           // [Dd][D] per position
    const uint16_t* temb;                           // [dep_text_in][Dd]
    const uint16_t* aemb[PM_DF_MAX_Q];              // [dep_audio_in][Dd] per position 1..Q-1
    const uint16_t* norm1[PM_DF_MAX_J];
    const uint16_t* norm2[PM_DF_MAX_J];
    const uint16_t* qkv[PM_DF_MAX_J];               // [Q * 3 * Dd][Dd]
    const uint16_t* lin_in[PM_DF_MAX_J * PM_DF_MAX_Q];  // [2 * Fd][Dd], index j * Q + q
    const uint16_t* heads[PM_DF_MAX_Q];             // [card][Dd]
    const uint16_t* wo_packed;                      // [J][Q][H][4][Dd / 4][64]
    const uint16_t* wout_t;                         // [J][Q][Fd][Dd]
    uint16_t* dk[PM_DF_MAX_J];                      // depth cache of block j, batch row 0: [H][Q][64]
    uint16_t* dv[PM_DF_MAX_J];
    float* dzin;                                    // [Q][Dd] input projections
    float* part_att;                                // [H][Dd]
    float* part_ffn;                                // [H][Dd]
    unsigned long long* amax;                       // [Q]
    uint32_t* bar;                                  // [3]: arrivals, exits, timeouts
    int G, D, Dd, H, Fd, Q, J, card, n_streams, text_rows, sup_rows, dep_win;
    float eps, scale_log2;
};
size_t depth_fused_smem();
bool depth_fused_supported(int D, int Dd, int H, int dh, int Fd, int Q, int card, int G_sms);
cudaError_t depth_fused_prepare(size_t smem);
cudaError_t depth_fused_max_clusters(size_t smem, int G, int* n);
cudaError_t launch_depth_fused(const DepFusedParams& p, size_t smem, cudaStream_t s);
// one (block, position): W_o slice [Dd][Dd] into the packed head blocks, linear_out [Dd][Fd]
// into its transpose
cudaError_t depth_relayout(const uint16_t* wo_q, uint16_t* wo_dst, const uint16_t* wout_q, uint16_t* woutT_dst, int Dd,
                           int Fd, int H, cudaStream_t s);



// ----------------------------------------------------------------------------------
// temperature / top-k sampling (one CTA per row)
// ----------------------------------------------------------------------------------
enum SampleMode {
    SM_PLAIN = 0,  // given rows, settings and counter; tokens to `tokens`
    SM_TEXT = 1,   // the frame's text token from the head's logits (context settings)
    SM_DEPTH = 2   // depth position q's code where none is supplied (context settings)
};
// rows of up to this many logits are staged in shared memory (128 KB; the kernel's
// static shared memory takes another 75 KB)
#define PM_SAMPLE_STAGE_MAX 32768
// largest top-k the sampler serves (one survivor per thread)
#define PM_SAMPLE_MAX_TOP_K 1024
struct SampleParams {
    int mode;
    const float* logits;   // row b at logits + b * ld
    int ld, V, B;
    int stage;             // set by launch_sample
    // SM_PLAIN settings; counter (position, row, substep, 0)
    float temperature;
    int top_k;
    unsigned long long seed;
    long long position;
    int substep;
    int32_t* tokens;       // SM_PLAIN output [B]
    // SM_TEXT / SM_DEPTH: settings, state, outputs; counter (pos - 1, row, 0 or 1 + q, 0)
    const SampleCfg* cfg;
    DevState st;
    const FrameIO* io;
    const DepIO* dio;
    int q, Q, n_streams;
    int seq;
};
cudaError_t launch_sample(const SampleParams& p, cudaStream_t s, bool pdl);
// (SampleParams.seq: SM_TEXT for a prefill -- one row, stream io->seq_stream)
cudaError_t sample_prepare();

// ----------------------------------------------------------------------------------
// batched projections on the tensor cores (tcgen05, accumulators in TMEM), B >= 2
// ----------------------------------------------------------------------------------
enum TcEpilogue {
    TE_STORE = 0,     // y[b][row] = acc
    TE_RESIDUAL = 1,  // y[b][row] += acc; yb = bf16(alpha_next * y); per-tile sum of y^2
    TE_SWIGLU = 2,    // tile = 64 gate rows + 64 value rows: yb[b][j] = bf16(SiLU(g) * z)
    TE_QKV_ROPE = 3,  // RoPE on q, k rows; q to y (fp32), k, v to the KV ring (bf16)
    TE_HEAD = 4       // text head logits + greedy token, frame finalisation, hidden state
};

// The head of the next projection's weights, fetched into L2 by this kernel's producer
// once its own copies are issued: while this kernel drains (last stages, split-K merges,
// epilogue), HBM already serves the first tiles that the next projection's CTA with the
// same index will stream, so that kernel's first loads hit L2.
struct NextPrefetch {
    int n_mtiles;          // next projection's 128-row tiles (0 = nothing to prefetch)
    int nk;                // its 64-element k tiles per row
    int grid;              // its CTAs
    int split_rows;        // TE_SWIGLU: value rows start here (two 64-row boxes per unit), else 0
    uint32_t bytes;        // bytes per CTA to prefetch
};

struct TcParams {
    int epi;
    int K, nk;               // row length, 64-element k tiles
    int n_rows;              // rows that are real outputs (guards the last tile)
    int n_mtiles;            // 128-row tiles (TE_SWIGLU: 64 gate/value row pairs per tile)
    int split_rows;          // TE_SWIGLU: value rows start here
    int B, npad;             // batch rows, MMA N (16, 32 or 64)
    int grid, nst, maxseg;   // plan (plan_tc)
    int min_units;           // plan input: fewest (tile, k-tile) units per CTA (0 = default)
    int a_tiled;             // A is pre-tiled: unit u is rows u*128 .. +127 of a [units*128][64] tensor
    int b_tiled;             // B is pre-tiled: k tile kt is rows kt*npad .. of a [nk*npad][64] tensor
    size_t smem;
    // RMSNorm of the input: inv[b] = 1 / sqrt(sum(ss_in[part][b]) / K + eps)
    const float* ss_in;      // [ss_parts][npad] or null (no norm)
    int ss_parts;
    float eps;
    // outputs
    float* y;                // fp32 [B][y_stride]
    int y_stride;
    uint16_t* yb;            // bf16 [npad][yb_stride] operand of the next projection, or null
    int yb_stride;
    int yb_lo_rows;          // > 0: also its rounding remainder at row b + yb_lo_rows (batched GEMV)
    const uint16_t* alpha_next;  // TE_RESIDUAL: scale folded into yb (next RMSNorm's alpha)
    float* ss_out;           // TE_RESIDUAL: [n_mtiles][npad] per-tile sum of squares of y
    // stream-K partials and per-tile completion counters (zero between launches)
    float* part;             // [n_mtiles][maxseg][npad][128]
    uint32_t* count;         // [n_mtiles]
    DevState st;
    // TE_QKV_ROPE
    int D, H, dh, ctx;
    uint16_t* kc;
    uint16_t* vc;
    const float2* rope_tab;  // [B][dh/2] (cos, sin) of this frame's positions
    // TE_HEAD
    const FrameIO* io;
    float* h_internal;       // [B][D] hidden state
    const float* x_resid;    // [B][D] residual before the final norm
    const uint16_t* alpha;   // final norm scale [D]
    float* logits_copy;      // also write the logits here ([B][n_rows]), or null
    NextPrefetch nx;         // read through the `next` tensor map
    // prefill: rows are frames pos .. pos+B-1 of stream io->seq_stream (TE_QKV_ROPE: their
    // K/V go to kv_new, committed to the ring after the attention; TE_HEAD: only the last
    // row's outputs, positions advance by B)
    int seq;
    uint16_t* kv_new;        // [2][B][H][dh] bf16 (K rows, then V rows)
    // batched GEMV path (k_gemv_mma, 2 <= B <= 16): plain pointers instead of tensor maps
    const uint16_t* w;       // weights [rows][K] bf16
    const uint16_t* xop;     // activation operand [16][K] bf16 (rows >= B are ignored)
    int pre_stride;          // plan: floats per batch row of the staged epilogue operands
    int h0;                  // plan: units of the smaller CTAs (the others own h0 + 1)
};

bool plan_tc(TcParams& p, int num_sms);

// Batched decode projections, 2 <= B <= 16, as a weight-streaming GEMV on warp-level MMAs
// (k_gemv_mma): same epilogues as the tensor-core path except TE_STORE; the sums of
// squares it writes (TE_RESIDUAL) are per CTA: ss_out[c][npad] for c < grid.
#define PM_MG_MAX_TILES 8    // 16-row tiles per CTA
bool plan_mg(TcParams& p, int num_sms);
// tensor maps of a planned projection: the weights [w_rows][K] with boxes of a full tile
// and of the two last-tile remainders, and the activation operand [16][K]
bool mg_tensor_maps(const TcParams& p, const uint16_t* w, uint64_t w_rows, const uint16_t* xop, CUtensorMap* m);
cudaError_t launch_mg(const CUtensorMap* m, const TcParams& p, cudaStream_t s, bool pdl);
cudaError_t mg_prepare();
// `next`: tensor map of the next projection's weights (read when p.nx.n_mtiles > 0)
cudaError_t launch_tc(const CUtensorMap& A, const CUtensorMap& Bop, const CUtensorMap& next, const TcParams& p,
                      cudaStream_t s, bool pdl);
cudaError_t tc_prepare();
// 2-D bf16 tensor map, 128-byte swizzle, box {64, box_rows}; false if the driver refuses it
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);

// ----------------------------------------------------------------------------------
// persistent frame program (B = 1): one cooperative launch runs the whole frame
// ----------------------------------------------------------------------------------
enum PhaseType { PH_EMBED = 0, PH_GEMV = 1, PH_ATTN = 2 };

struct FPhase {
    int type;
    int epi;            // PH_GEMV: E_QKV_ROPE, E_RESIDUAL, E_SWIGLU, E_HEAD
    int unit;           // U_ROW, U_PAIR_ADJ, U_PAIR_SPLIT
    int K;              // row length (multiple of 1024)
    int n_units;
    int split_rows;     // U_PAIR_SPLIT
    int upst;           // units per shared-memory stage
    const uint16_t* W;  // [rows][K] bf16
    const float* x;     // input vector [K]
    const uint16_t* alpha;  // RMSNorm scale of the input, or null
    float* y;           // output vector
    uint16_t* kc;       // QKV / attention: this layer's K cache [H][ctx][dh] (batch row 0)
    uint16_t* vc;
};

struct FrameProgParams {
    const FPhase* ph;
    int n_phases;
    DevState st;
    const FrameIO* io;
    const uint16_t* tables[PM_MAX_STREAMS_DEV];
    int rows[PM_MAX_STREAMS_DEV];
    int init_id[PM_MAX_STREAMS_DEV];
    int delays[PM_MAX_STREAMS_DEV];
    int n_streams;
    const double* rope_freq;
    float2* rope_tab;
    float* x;
    float* q;
    float* o;
    float* h;
    int D, H, dh, ctx;
    int win;                 // most keys a query sees (ctx, or ctx - 1 for the pinned ring)
    float eps, scale_log2;
    float* part;        // [H][S][dh + 2] attention chunk partials
    uint32_t* att_count;  // [H]
    int S, max_chunks;
    int partial_floats; // shared-memory row partials (max over GEMV phases)
    uint32_t* bar;      // [n_phases] grid-barrier arrival counters, zero between frames
};

bool frame_prog_supported(int D, int F, int dh);
int frame_prog_stage_rows(int K);
size_t frame_prog_smem(int partial_floats, int max_chunks);
cudaError_t frame_prog_prepare(size_t smem);
cudaError_t launch_frame_prog(const FrameProgParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t frame_prog_occupancy(size_t smem, int* blocks_per_sm);

}  // namespace pm
