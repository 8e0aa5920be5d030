// Host-side interface between the C-ABI layer (pm_api.cu) and the kernel translation
// units.  Plain structs of device pointers and sizes; every launch goes on `stream` and,
// when `pdl` is set, may begin before the previous kernel in the stream has finished
// (programmatic dependent launch: the kernel waits with griddepcontrol.wait before it
// reads anything the previous kernel wrote).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pm_common.cuh"

namespace pm {

// ----------------------------------------------------------------------------------
// weight-streaming GEMV  y = W x  (bf16 W [rows][K], fp32 x), B = 1 row of x per CTA
// ----------------------------------------------------------------------------------
enum Unit { U_ROW = 0, U_PAIR_ADJ = 1, U_PAIR_SPLIT = 2 };
enum Prologue { PRO_PLAIN = 0, PRO_RMSNORM = 1 };
enum Epilogue {
    E_STORE = 0,      // y[row] = dot
    E_RESIDUAL = 1,   // y[row] += dot
    E_SWIGLU = 2,     // y[u] = SiLU(dot(row u)) * dot(row u + F)
    E_QKV_ROPE = 3,   // temporal fused QKV: RoPE on Q, K; K, V into the KV ring
    E_HEAD = 4,       // text head: logits + argmax, frame finalisation
    E_EMB_ADD = 5,    // depformer input: y[row] = dot + E[token][row]
    E_DEP_QKV = 6,    // depth QKV: q to y, k, v into the depth cache at position q
    E_DEP_HEAD = 7    // depth head: logits + argmax or supplied code
};

struct GemvParams {
    const uint16_t* W;     // [rows][K]
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
    const double* rope_freq;  // [dh/2]
    // E_HEAD
    const FrameIO* io;
    float* h_internal;     // [B][K] normalised input copy (the hidden state), written by CTA 0
    // depformer
    const DepIO* dio;
    int q;                 // depth position
    int Q;                 // depth positions per frame
    const uint16_t* emb;   // E_EMB_ADD table [rows_emb][y dim]
    int emb_rows;
    uint16_t* dkc;         // E_DEP_QKV: depth K cache of this layer [B_max][Hd][Q][dhd]
    uint16_t* dvc;
    int n_streams;
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
};
cudaError_t launch_embed(const EmbedParams& p, cudaStream_t s, bool pdl);

// ----------------------------------------------------------------------------------
// split-KV decode attention over the temporal ring (dh = 128)
// ----------------------------------------------------------------------------------
struct AttnParams {
    const float* q;        // [B][D] rotated queries
    const uint16_t* kc;    // [B_max][H][ctx][dh]
    const uint16_t* vc;
    float* o;              // [B][D]
    float* part;           // [B][H][S][dh + 2] chunk partials
    uint32_t* count;       // [B][H], zero between launches
    DevState st;
    int B, H, ctx, S, D;
    float scale_log2;      // log2(e) / sqrt(dh)
};
cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl);
// chunks (CTAs per head) the attention grid needs for a window of ctx keys; AttnParams.S
// must be at least this and `part` must hold S chunks per head
int attn_max_splits(int ctx);

// ----------------------------------------------------------------------------------
// depformer helpers
// ----------------------------------------------------------------------------------
struct DepBeginParams {
    const DepIO* dio;
    DevState st;
    float* h_internal;     // [B][D] hidden the chain reads
    int32_t* dep_sup;      // [B][Q] validated supplied codes
    int B, D, Q, card, text_rows;
};
cudaError_t launch_dep_begin(const DepBeginParams& p, cudaStream_t s, bool pdl);

struct DepAttnParams {
    const float* q;        // [B][Dd]
    const uint16_t* kc;    // depth K cache of this layer [B_max][Hd][Q][dhd]
    const uint16_t* vc;
    float* o;              // [B][Dd]
    DevState st;
    int B, Hd, dhd, Q, q_pos, dep_ctx, Dd;
    float scale_log2;
};
cudaError_t launch_dep_attn(const DepAttnParams& p, cudaStream_t s, bool pdl);

}  // namespace pm
