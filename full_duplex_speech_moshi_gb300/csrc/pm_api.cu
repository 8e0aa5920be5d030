// C ABI of the decode step (declared in include/pm.h): context set-up, argument
// validation, and one CUDA graph per (call kind, batch size) in which every kernel after
// the first is a programmatic dependent launch.
//
// Per-call inputs and output pointers travel through small device-side structs (FrameIO,
// DepIO) refreshed by one host-to-device copy before each graph launch, so a graph is
// captured once per batch size and replayed for every frame.  Positions, the delay ring
// and the last selected tokens live in device memory and are advanced by the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/pm.h"
#include "pm_kernels.h"

using namespace pm;

namespace {

constexpr int kMaxB = 64;
constexpr int kStagingSlots = 8;

struct Staging {
    uint8_t* host = nullptr;  // pinned
    cudaEvent_t done = nullptr;
};

}  // namespace

struct pm_ctx {
    pm_config cfg{};
    int device = 0;
    int num_sms = 0;
    cudaStream_t stream = nullptr;   // caller's stream: every launch goes here
    cudaStream_t cap = nullptr;      // private stream used only for graph capture
    bool has_dep = false;
    // weights (device)
    const uint16_t* tables[PM_MAX_STREAMS_DEV] = {};
    std::vector<const uint16_t*> norm1, in_proj, out_proj, norm2, lin_in, lin_out;
    const uint16_t* out_norm = nullptr;
    const uint16_t* text_linear = nullptr;
    std::vector<const uint16_t*> d_in, d_aemb, d_norm1, d_qkv, d_o, d_norm2, d_lin_in, d_lin_out, d_heads;
    const uint16_t* d_temb = nullptr;
    uint16_t* kv = nullptr;
    // owned device memory
    void* block = nullptr;
    size_t block_bytes = 0;
    DevState st{};
    uint8_t* io_region = nullptr;      // FrameIO + ids
    uint8_t* dio_region = nullptr;     // DepIO + text_tok + supplied
    float *x = nullptr, *q = nullptr, *o = nullptr, *s = nullptr, *h = nullptr;
    float* att_part = nullptr;
    uint32_t* att_count = nullptr;
    double* rope_freq = nullptr;
    float2* rope_tab = nullptr;        // [B_max][dh/2]
    // tensor-core path (B >= 2): bf16 operands, sums of squares, stream-K scratch
    int npad_max = 0;
    uint16_t *xb = nullptr, *ob = nullptr, *sb = nullptr;
    float* ss = nullptr;               // [D/128][npad_max]
    float* tc_part = nullptr;
    uint32_t* tc_count = nullptr;
    float *dz = nullptr, *dq = nullptr, *ds = nullptr;
    float* dzin = nullptr;  // [B_max][dep_steps][dep_D]: the depformer input projections of a call
    uint16_t* dkv = nullptr;
    // sampling: device-resident settings, the logits the samplers read, which kinds sample
    SampleCfg* scfg = nullptr;
    SampleCfg scfg_host{};
    float* slog = nullptr;    // [B_max][text_out]
    float* dslog = nullptr;   // [B_max][dep_card]
    bool text_smp = false, audio_smp = false;
    // prefill: resolved inputs of a pass, attention partials and counters, graphs per T
    int32_t* seq_resolved = nullptr;
    float* seq_part = nullptr;
    uint16_t* seq_kv = nullptr;        // [2][PM_SEQ_MAX_ROWS][H][dh] a pass's K/V before commit
    std::map<int, cudaGraphExec_t> prefill_graphs;
    // staging
    Staging slots[kStagingSlots];
    int next_slot = 0;
    // graphs
    std::map<int, cudaGraphExec_t> frame_graphs, dep_graphs;
    std::string err;
    size_t tc_part_floats = 0;
    int tc_count_max = 0;
    int ss_parts_max = 0;              // sum-of-squares partials the ss buffer holds (batched GEMV)
    // persistent batch-1 frame program (null when the shape or device does not allow it)
    bool prog = false;
    FPhase* d_phases = nullptr;
    uint32_t* prog_bar = nullptr;      // [n_phases + 2]: phase counters, exit and timeout counters
    uint32_t* wait_budget = nullptr;   // device word: poll budget of the GEMV and frame-program waits
    // generator (token ring + provided ring per stream, offsets; device-resident) and the host's
    // copy of the offsets (they change only through pm_generator_step, pm_reset, pm_restore)
    int32_t *gen_ring = nullptr, *gen_prov = nullptr, *gen_off = nullptr, *gen_in = nullptr;
    int32_t *gen_tok = nullptr, *gen_sup = nullptr, *gen_pos_save = nullptr, *gen_sel_save = nullptr;
    std::vector<int> gen_s;
    // persistent batch-1 depformer (null when the shape, the device or the flags exclude it)
    bool dep_fused = false;
    void* df_block = nullptr;          // re-laid W_o / linear_out copies and the call's scratch
    DepFusedParams df{};
    size_t df_smem = 0;
    size_t prog_smem = 0;
    FrameProgParams prog_params{};
    // set while pm_profile_frame records a frame eagerly
    std::vector<cudaEvent_t>* prof_ev = nullptr;
    std::vector<int>* prof_kind = nullptr;
};

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// message of the last pm_create failure on this thread (pm_last_error(NULL) returns it)
static thread_local std::string g_create_err;

static pm_status fail(pm_ctx* c, pm_status st, const std::string& msg) {
    if (c) c->err = msg;
    return st;
}

static pm_status cuda_fail(pm_ctx* c, cudaError_t e, const char* where) {
    return fail(c, PM_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define PM_CUDA(call)                                          \
    do {                                                       \
        cudaError_t e_ = (call);                               \
        if (e_ != cudaSuccess) return cuda_fail(c, e_, #call); \
    } while (0)

extern "C" size_t pm_kv_cache_bytes(const pm_config* cfg) {
    if (!cfg) return 0;
    return (size_t)cfg->n_layers * 2u * (size_t)cfg->B_max * (size_t)cfg->H * (size_t)cfg->ctx * (size_t)cfg->dh *
           2u;
}

static const char* check_config(const pm_config* c) {
    if (c->B_max < 1 || c->B_max > kMaxB) return "B_max must be 1..64";
    if (c->dh != 128) return "temporal head width dh must be 128";
    if (c->H < 1 || c->D != c->H * c->dh) return "D must equal H * dh";
    if (c->D % 256 != 0 || c->ffn % 256 != 0) return "D and ffn must be multiples of 256";
    if (c->n_layers < 1 || c->ctx < 1) return "n_layers and ctx must be positive";
    if (c->n_streams < 1 || c->n_streams > PM_MAX_STREAMS) return "n_streams must be 1..32";
    if (c->text_in < 1 || c->audio_in < 1 || c->text_out < 1) return "table sizes must be positive";
    for (int k = 0; k < c->n_streams; ++k)
        if (c->delays[k] < 0 || c->delays[k] > 3) return "delays must be 0..3";
    if (c->init_text < 0 || c->init_text >= c->text_in) return "init_text outside the text table";
    if (c->init_audio < 0 || c->init_audio >= c->audio_in) return "init_audio outside the audio tables";
    if (!(c->eps > 0.f) || !(c->rope_theta > 0.f)) return "eps and rope_theta must be positive";
    if ((c->flags & PM_FLAG_PINNED_RING) && c->ctx < 2) return "the pinned ring needs ctx >= 2";
    if (c->dep_layers > 0) {
        if (c->dep_dh != 64 || c->dep_D != c->dep_H * c->dep_dh) return "depformer needs dep_dh 64 and dep_D = dep_H * 64";
        if (c->dep_D % 256 != 0 || c->dep_ffn % 256 != 0) return "dep_D and dep_ffn must be multiples of 256";
        if (c->dep_steps < 1 || c->dep_steps > 32) return "dep_steps must be 1..32";
        if (c->dep_ctx < 1 || c->dep_ctx > 16) return "dep_ctx must be 1..16";
        if ((c->flags & PM_FLAG_PINNED_RING) && c->dep_ctx < 2) return "the pinned ring needs dep_ctx >= 2";
        if (c->dep_card < 1 || c->dep_text_in < 1 || c->dep_audio_in < c->dep_card) return "bad depformer table sizes";
    }
    return nullptr;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// ------------------------------------------------------------------------------------
// small state kernel (reset / position set)
// ------------------------------------------------------------------------------------
struct SetStateArgs {
    DevState st;
    int32_t* gen_ring;  // non-null: also reset the generator (ring unwritten, no flags, offset 0)
    int32_t* gen_prov;
    int32_t* gen_off;
    int n;
    int32_t pos[kMaxB];
    int32_t apply[kMaxB];
};

__global__ void k_set_state(const SetStateArgs a) {
    const int b = blockIdx.x;
    if (b >= a.n || !a.apply[b]) return;
    if (threadIdx.x == 0) {
        a.st.pos[b] = a.pos[b];
        a.st.first_pos[b] = a.pos[b];
        a.st.amax[b] = 0ull;
        a.st.head_count[b] = 0u;
        a.st.dep_amax[b] = 0ull;
        a.st.dep_count[b] = 0u;
    }
    if (threadIdx.x < PM_MAX_STREAMS_DEV) a.st.sel[(size_t)b * PM_MAX_STREAMS_DEV + threadIdx.x] = -2;
    if (a.gen_ring) {
        for (int i = threadIdx.x; i < 4 * PM_MAX_STREAMS_DEV; i += blockDim.x) {
            a.gen_ring[(size_t)b * 4 * PM_MAX_STREAMS_DEV + i] = -2;
            a.gen_prov[(size_t)b * 4 * PM_MAX_STREAMS_DEV + i] = 0;
        }
        if (threadIdx.x == 0) a.gen_off[b] = 0;
    }
}

// ------------------------------------------------------------------------------------
// graph construction
// ------------------------------------------------------------------------------------
static GemvParams base_params(pm_ctx* c) {
    GemvParams p;
    memset(&p, 0, sizeof p);
    p.st = c->st;
    p.eps = c->cfg.eps;
    p.io = reinterpret_cast<const FrameIO*>(c->io_region);
    p.dio = reinterpret_cast<const DepIO*>(c->dio_region);
    p.n_streams = c->cfg.n_streams;
    return p;
}

static pm_status plan(pm_ctx* c, GemvParams& p, int rpu, const char* what) {
    if (!plan_gemv(p, rpu, c->num_sms)) return fail(c, PM_ERR_UNSUPPORTED, std::string("no GEMV plan for ") + what);
    return PM_OK;
}

// Bytes per CTA of the next projection's weights that a tensor-core projection prefetches
// into L2 after issuing its own copies (tuning constant; 0 disables).  Off: with the
// epilogues rolled, 256 KB per CTA made the 64-row prefill pass and B = 40 about 2% slower
// (the prefetch competes with the projection's own weight stream).
#ifndef PM_PF_TC_BYTES
#define PM_PF_TC_BYTES 0u
#endif

static NextPrefetch next_tc(pm_ctx* c, int epi, int K, int n_mtiles, int split_rows, int npad) {
    NextPrefetch nx;
    memset(&nx, 0, sizeof nx);
    TcParams t;
    memset(&t, 0, sizeof t);
    t.epi = epi;
    t.K = K;
    t.n_mtiles = n_mtiles;
    t.npad = npad;
    t.B = 1;
    if (PM_PF_TC_BYTES == 0u || !plan_tc(t, c->num_sms)) return nx;
    nx.n_mtiles = n_mtiles;
    nx.nk = t.nk;
    nx.grid = t.grid;
    nx.split_rows = split_rows;
    nx.bytes = PM_PF_TC_BYTES;
    return nx;
}

typedef pm_status (*record_fn)(pm_ctx*, int, cudaStream_t);

// profiling mark: an event after the launch just issued (only inside pm_profile_frame)
static pm_status mark(pm_ctx* c, cudaStream_t s, int kind) {
    if (!c->prof_ev) return PM_OK;
    cudaEvent_t e;
    PM_CUDA(cudaEventCreate(&e));
    c->prof_ev->push_back(e);
    c->prof_kind->push_back(kind);
    PM_CUDA(cudaEventRecord(e, s));
    return PM_OK;
}

// the drawn text token replaces the head's greedy one (when text sampling is on)
static pm_status record_text_sample(pm_ctx* c, int B, cudaStream_t s, bool pdl, bool seq = false) {
    if (!c->text_smp) return PM_OK;
    SampleParams sp;
    memset(&sp, 0, sizeof sp);
    sp.mode = SM_TEXT;
    sp.seq = seq ? 1 : 0;  // a prefill draws only its last frame's token
    sp.logits = c->slog;
    sp.ld = c->cfg.text_out;
    sp.V = c->cfg.text_out;
    sp.B = seq ? 1 : B;
    sp.cfg = c->scfg;
    sp.st = c->st;
    sp.io = reinterpret_cast<const FrameIO*>(c->io_region);
    sp.dio = reinterpret_cast<const DepIO*>(c->dio_region);
    sp.n_streams = c->cfg.n_streams;
    PM_CUDA(launch_sample(sp, s, pdl));
    return mark(c, s, PM_KERNEL_SAMPLE);
}

static pm_status record_frame(pm_ctx* c, int B, cudaStream_t s) {
    const pm_config& f = c->cfg;
    const int D = f.D, F = f.ffn;
    if (B == 1 && c->prog && !c->text_smp) {
        pm_status ms = mark(c, s, -1);
        if (ms) return ms;
        PM_CUDA(launch_frame_prog(c->prog_params, c->num_sms, c->prog_smem, s));
        return mark(c, s, PM_KERNEL_FRAME);
    }
    EmbedParams ep;
    memset(&ep, 0, sizeof ep);
    for (int k = 0; k < f.n_streams; ++k) {
        ep.tables[k] = c->tables[k];
        ep.rows[k] = (k == 0) ? f.text_in : f.audio_in;
        ep.init_id[k] = (k == 0) ? f.init_text : f.init_audio;
        ep.delays[k] = f.delays[k];
    }
    ep.io = reinterpret_cast<const FrameIO*>(c->io_region);
    ep.st = c->st;
    ep.x = c->x;
    ep.D = D;
    ep.B = B;
    ep.n_streams = f.n_streams;
    ep.rope_tab = c->rope_tab;
    ep.rope_freq = c->rope_freq;
    ep.dh = f.dh;
    const bool pdl = c->prof_ev == nullptr;  // eager profiling runs each kernel alone
    pm_status ms = mark(c, s, -1);
    if (ms) return ms;
    PM_CUDA(launch_embed(ep, s, false));
    if ((ms = mark(c, s, PM_KERNEL_EMBED))) return ms;

    const size_t layer_elems = (size_t)f.B_max * f.H * f.ctx * f.dh;
    for (int l = 0; l < f.n_layers; ++l) {
        uint16_t* kc = c->kv + (size_t)(2 * l + 0) * layer_elems;
        uint16_t* vc = c->kv + (size_t)(2 * l + 1) * layer_elems;
        // RMSNorm1 + fused QKV + RoPE + KV append
        GemvParams p = base_params(c);
        p.W = c->in_proj[l];
        p.K = D;
        p.n_units = 3 * D / 2;
        p.B = B;
        p.x = c->x;
        p.x_stride = D;
        p.alpha = c->norm1[l];
        p.y = c->q;
        p.y_stride = D;
        p.D = D;
        p.H = f.H;
        p.dh = f.dh;
        p.ctx = f.ctx;
        p.B_max = f.B_max;
        p.kc = kc;
        p.vc = vc;
        p.rope_tab = c->rope_tab;
        pm_status ps = plan(c, p, 2, "in_proj");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_RMSNORM, E_QKV_ROPE, U_PAIR_ADJ, p, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_QKV))) return ms;
        // attention
        AttnParams ap;
        memset(&ap, 0, sizeof ap);
        ap.q = c->q;
        ap.kc = kc;
        ap.vc = vc;
        ap.o = c->o;
        ap.part = c->att_part;
        ap.count = c->att_count;
        ap.st = c->st;
        ap.B = B;
        ap.H = f.H;
        ap.ctx = f.ctx;
        ap.S = attn_max_splits(f.ctx);
        ap.win = f.ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);
        attn_plan(ap, c->num_sms);
        ap.D = D;
        ap.scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dh));
        PM_CUDA(launch_attn(ap, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_ATTENTION))) return ms;
        // W_O + residual
        p = base_params(c);
        p.W = c->out_proj[l];
        p.K = D;
        p.n_units = D;
        p.B = B;
        p.x = c->o;
        p.x_stride = D;
        p.y = c->x;
        p.y_stride = D;
        ps = plan(c, p, 1, "out_proj");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_PLAIN, E_RESIDUAL, U_ROW, p, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_OUT_PROJ))) return ms;
        // RMSNorm2 + linear_in + SwiGLU
        p = base_params(c);
        p.W = c->lin_in[l];
        p.K = D;
        p.n_units = F;
        p.split_rows = F;
        p.B = B;
        p.x = c->x;
        p.x_stride = D;
        p.alpha = c->norm2[l];
        p.y = c->s;
        p.y_stride = F;
        ps = plan(c, p, 2, "linear_in");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_RMSNORM, E_SWIGLU, U_PAIR_SPLIT, p, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_LINEAR_IN))) return ms;
        // linear_out + residual
        p = base_params(c);
        p.W = c->lin_out[l];
        p.K = F;
        p.n_units = D;
        p.B = B;
        p.x = c->s;
        p.x_stride = F;
        p.y = c->x;
        p.y_stride = D;
        ps = plan(c, p, 1, "linear_out");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_PLAIN, E_RESIDUAL, U_ROW, p, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_LINEAR_OUT))) return ms;
    }
    // final RMSNorm + text head + argmax + frame finalisation
    GemvParams p = base_params(c);
    p.W = c->text_linear;
    p.K = D;
    p.n_units = f.text_out;
    p.B = B;
    p.x = c->x;
    p.x_stride = D;
    p.alpha = c->out_norm;
    p.y_stride = f.text_out;
    p.h_internal = c->h;
    if (c->text_smp) p.logits_copy = c->slog;
    pm_status ps = plan(c, p, 1, "text_linear");
    if (ps) return ps;
    PM_CUDA(launch_gemv(PRO_RMSNORM, E_HEAD, U_ROW, p, s, pdl));
    if ((ms = mark(c, s, PM_KERNEL_HEAD))) return ms;
    return record_text_sample(c, B, s, pdl);
}


// batch columns of the batched paths: 16 = the warp-MMA GEMV (2 <= B <= 16), 32 / 64 = the
// tcgen05 GEMM; PM_FLAG_BATCHED_TCGEN05 sends B <= 16 to the GEMM as well
static int npad_for(const pm_ctx* c, int B) {
    if (c->cfg.flags & PM_FLAG_BATCHED_TCGEN05) return B <= 32 ? 32 : 64;
    return B <= 16 ? 16 : (B <= 32 ? 32 : 64);
}

// B >= 2: every projection on the tensor cores (k_gemm_tc), same kernel families and order
// `seq`: a prefill pass -- the B rows are frames pos .. pos+B-1 of stream io->seq_stream
static pm_status record_frame_tc_impl(pm_ctx* c, int B, cudaStream_t s, bool seq) {
    const pm_config& f = c->cfg;
    const int D = f.D, F = f.ffn, npad = npad_for(c, B);
    if (npad > c->npad_max) return fail(c, PM_ERR_UNSUPPORTED, "batch larger than the tensor-core buffers");
    const bool pdl = c->prof_ev == nullptr;
    if (seq) {
        SeqPrepParams sp;
        memset(&sp, 0, sizeof sp);
        sp.io = reinterpret_cast<const FrameIO*>(c->io_region);
        sp.st = c->st;
        sp.resolved = c->seq_resolved;
        sp.T = B;
        sp.n_streams = f.n_streams;
        for (int k = 0; k < f.n_streams; ++k) {
            sp.rows[k] = (k == 0) ? f.text_in : f.audio_in;
            sp.init_id[k] = (k == 0) ? f.init_text : f.init_audio;
            sp.delays[k] = f.delays[k];
        }
        PM_CUDA(launch_seq_prepare(sp, s, false));
    }
    EmbedParams ep;
    memset(&ep, 0, sizeof ep);
    for (int k = 0; k < f.n_streams; ++k) {
        ep.tables[k] = c->tables[k];
        ep.rows[k] = (k == 0) ? f.text_in : f.audio_in;
        ep.init_id[k] = (k == 0) ? f.init_text : f.init_audio;
        ep.delays[k] = f.delays[k];
    }
    ep.io = reinterpret_cast<const FrameIO*>(c->io_region);
    ep.st = c->st;
    ep.x = c->x;
    ep.D = D;
    ep.B = B;
    ep.n_streams = f.n_streams;
    ep.rope_tab = c->rope_tab;
    ep.rope_freq = c->rope_freq;
    ep.dh = f.dh;
    ep.xb = c->xb;
    // 2 <= B <= 16 decode runs the batched GEMV on warp-level MMAs (k_gemv_mma), which
    // also reads each bf16 operand's rounding remainder (rows 16..31 of the operand buffers)
    const bool mg = !seq && npad == 16;
    const int lo_rows = mg ? 16 : 0;
    ep.xb_lo_rows = lo_rows;
    ep.alpha = c->norm1[0];
    ep.ss = c->ss;
    ep.npad = npad;
    ep.resolved = seq ? c->seq_resolved : nullptr;
    pm_status ms = mark(c, s, -1);
    if (ms) return ms;
    PM_CUDA(launch_embed(ep, s, seq && pdl));
    if ((ms = mark(c, s, PM_KERNEL_EMBED))) return ms;

    CUtensorMap mx, mo, msb;
    if (!make_tmap_bf16(&mx, c->xb, D, npad, npad) || !make_tmap_bf16(&mo, c->ob, D, npad, npad) ||
        !make_tmap_bf16(&msb, c->sb, F, npad, npad))
        return fail(c, PM_ERR_CUDA, "tensor map encoding failed (activations)");
    auto base = [&](int epi, int K, int n_mtiles, int n_rows) {
        TcParams p;
        memset(&p, 0, sizeof p);
        p.epi = epi;
        p.K = K;
        p.n_mtiles = n_mtiles;
        p.n_rows = n_rows;
        p.B = B;
        p.npad = npad;
        p.eps = f.eps;
        p.part = c->tc_part;
        p.count = c->tc_count;
        p.st = c->st;
        p.io = reinterpret_cast<const FrameIO*>(c->io_region);
        p.D = D;
        return p;
    };
    auto go = [&](const CUtensorMap& A, const CUtensorMap& X, const CUtensorMap& N, TcParams& p, int kind,
                  const char* what) -> pm_status {
        if (!plan_tc(p, c->num_sms)) return fail(c, PM_ERR_UNSUPPORTED, std::string("no tensor-core plan for ") + what);
        if ((size_t)p.n_mtiles * p.maxseg * p.npad * 128 > c->tc_part_floats || p.n_mtiles > c->tc_count_max)
            return fail(c, PM_ERR_UNSUPPORTED, std::string("tensor-core scratch too small for ") + what);
        PM_CUDA(launch_tc(A, X, N, p, s, pdl));
        return mark(c, s, kind);
    };
    // the batched GEMV's residual epilogues leave one sum-of-squares partial per CTA instead
    // of one per 128-row tile
    int ss_parts = (D + 1023) / 1024;  // partials of the operand the next normed projection reads
    auto go_mg = [&](TcParams& p, const uint16_t* w, uint64_t w_rows, const uint16_t* xop, int kind,
                     const char* what) -> pm_status {
        p.w = w;
        p.xop = xop;
        if (!plan_mg(p, c->num_sms)) return fail(c, PM_ERR_UNSUPPORTED, std::string("no batched GEMV plan for ") + what);
        if (p.epi == TE_RESIDUAL && p.grid > c->ss_parts_max)
            return fail(c, PM_ERR_UNSUPPORTED, std::string("sum-of-squares scratch too small for ") + what);
        CUtensorMap maps[4];
        if (!mg_tensor_maps(p, w, w_rows, xop, maps))
            return fail(c, PM_ERR_CUDA, std::string("tensor map encoding failed for ") + what);
        PM_CUDA(launch_mg(maps, p, s, pdl));
        if (p.epi == TE_RESIDUAL) ss_parts = p.grid;
        return mark(c, s, kind);
    };
    // weight tensor maps of every projection (each kernel also prefetches the next one's head)
    std::vector<CUtensorMap> mq(f.n_layers), mwo(f.n_layers), mwi(f.n_layers), mwt(f.n_layers);
    for (int l = 0; l < f.n_layers; ++l)
        if (!make_tmap_bf16(&mq[l], c->in_proj[l], D, 3 * D, 128) ||
            !make_tmap_bf16(&mwo[l], c->out_proj[l], D, D, 128) ||
            !make_tmap_bf16(&mwi[l], c->lin_in[l], D, 2 * F, 64) || !make_tmap_bf16(&mwt[l], c->lin_out[l], F, D, 128))
            return fail(c, PM_ERR_CUDA, "tensor map encoding failed (weights)");
    CUtensorMap mh;
    if (!make_tmap_bf16(&mh, c->text_linear, D, f.text_out, 128))
        return fail(c, PM_ERR_CUDA, "tensor map encoding failed (text head)");
    const int head_tiles = (f.text_out + 127) / 128;
    const size_t layer_elems = (size_t)f.B_max * f.H * f.ctx * f.dh;
    for (int l = 0; l < f.n_layers; ++l) {
        uint16_t* kc = c->kv + (size_t)(2 * l + 0) * layer_elems;
        uint16_t* vc = c->kv + (size_t)(2 * l + 1) * layer_elems;
        // RMSNorm1 (folded) + fused QKV + RoPE + KV append
        TcParams p = base(TE_QKV_ROPE, D, 3 * D / 128, 3 * D);
        p.ss_in = c->ss;
        p.ss_parts = ss_parts;
        p.y = c->q;
        p.y_stride = D;
        p.H = f.H;
        p.dh = f.dh;
        p.ctx = f.ctx;
        p.kc = kc;
        p.vc = vc;
        p.rope_tab = c->rope_tab;
        p.nx = next_tc(c, TE_RESIDUAL, D, D / 128, 0, npad);
        p.seq = seq ? 1 : 0;
        p.kv_new = c->seq_kv;
        pm_status ps = mg ? go_mg(p, c->in_proj[l], 3u * D, c->xb, PM_KERNEL_QKV, "in_proj")
                          : go(mq[l], mx, mwo[l], p, PM_KERNEL_QKV, "in_proj");
        if (ps) return ps;
        if (seq) {
            AttnSeqParams aq;
            memset(&aq, 0, sizeof aq);
            aq.q = c->q;
            aq.kc = kc;
            aq.vc = vc;
            aq.kv_new = c->seq_kv;
            aq.o = c->o;
            aq.ob = c->ob;
            aq.part = c->seq_part;
            aq.st = c->st;
            aq.io = reinterpret_cast<const FrameIO*>(c->io_region);
            aq.T = B;
            aq.H = f.H;
            aq.ctx = f.ctx;
            aq.win = f.ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);
            aq.D = D;
            aq.grid = 2 * c->num_sms;
            aq.scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dh));
            PM_CUDA(launch_attn_seq(aq, s, pdl));
            PM_CUDA(launch_seq_commit(aq, s, pdl));
        }
        AttnParams ap;
        memset(&ap, 0, sizeof ap);
        ap.ob = c->ob;
        ap.ob_lo_rows = lo_rows;
        ap.q = c->q;
        ap.kc = kc;
        ap.vc = vc;
        ap.o = c->o;
        ap.part = c->att_part;
        ap.count = c->att_count;
        ap.st = c->st;
        ap.B = B;
        ap.H = f.H;
        ap.ctx = f.ctx;
        ap.S = attn_max_splits(f.ctx);
        ap.win = f.ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);
        attn_plan(ap, c->num_sms);
        ap.D = D;
        ap.scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dh));
        if (!seq) PM_CUDA(launch_attn(ap, s, pdl));
        if ((ms = mark(c, s, PM_KERNEL_ATTENTION))) return ms;
        // W_O + residual; emits bf16(norm2 alpha * y) and per-tile sums of y^2
        p = base(TE_RESIDUAL, D, D / 128, D);
        p.y = c->x;
        p.y_stride = D;
        p.yb = c->xb;
        p.yb_stride = D;
        p.yb_lo_rows = lo_rows;
        p.alpha_next = c->norm2[l];
        p.ss_out = c->ss;
        p.nx = next_tc(c, TE_SWIGLU, D, F / 64, F, npad);
        ps = mg ? go_mg(p, c->out_proj[l], D, c->ob, PM_KERNEL_OUT_PROJ, "out_proj")
                : go(mwo[l], mo, mwi[l], p, PM_KERNEL_OUT_PROJ, "out_proj");
        if (ps) return ps;
        if (!mg) ss_parts = D / 128;
        // RMSNorm2 (folded) + linear_in + SwiGLU -> bf16 s
        p = base(TE_SWIGLU, D, F / 64, F);
        p.ss_in = c->ss;
        p.ss_parts = ss_parts;
        p.split_rows = F;
        p.yb = c->sb;
        p.yb_stride = F;
        p.yb_lo_rows = lo_rows;
        p.nx = next_tc(c, TE_RESIDUAL, F, D / 128, 0, npad);
        ps = mg ? go_mg(p, c->lin_in[l], 2u * F, c->xb, PM_KERNEL_LINEAR_IN, "linear_in")
                : go(mwi[l], mx, mwt[l], p, PM_KERNEL_LINEAR_IN, "linear_in");
        if (ps) return ps;
        // linear_out + residual; emits the next norm's operand
        p = base(TE_RESIDUAL, F, D / 128, D);
        p.y = c->x;
        p.y_stride = D;
        p.yb = c->xb;
        p.yb_stride = D;
        p.yb_lo_rows = lo_rows;
        p.alpha_next = (l + 1 < f.n_layers) ? c->norm1[l + 1] : c->out_norm;
        p.ss_out = c->ss;
        const bool last = l + 1 == f.n_layers;
        p.nx = last ? next_tc(c, TE_HEAD, D, head_tiles, 0, npad)
                    : next_tc(c, TE_QKV_ROPE, D, 3 * D / 128, 0, npad);
        ps = mg ? go_mg(p, c->lin_out[l], D, c->sb, PM_KERNEL_LINEAR_OUT, "linear_out")
                : go(mwt[l], msb, last ? mh : mq[l + 1], p, PM_KERNEL_LINEAR_OUT, "linear_out");
        if (ps) return ps;
        if (!mg) ss_parts = D / 128;
    }
    TcParams p = base(TE_HEAD, D, head_tiles, f.text_out);
    p.ss_in = c->ss;
    p.ss_parts = ss_parts;
    p.h_internal = c->h;
    p.x_resid = c->x;
    p.alpha = c->out_norm;
    p.nx = next_tc(c, TE_QKV_ROPE, D, 3 * D / 128, 0, npad);  // the next frame's first projection
    if (c->text_smp) p.logits_copy = c->slog;
    p.seq = seq ? 1 : 0;
    pm_status hs = mg ? go_mg(p, c->text_linear, f.text_out, c->xb, PM_KERNEL_HEAD, "text_linear")
                      : go(mh, mx, mq[0], p, PM_KERNEL_HEAD, "text_linear");
    if (hs) return hs;
    return record_text_sample(c, B, s, pdl, seq);
}

static pm_status record_frame_tc(pm_ctx* c, int B, cudaStream_t s) { return record_frame_tc_impl(c, B, s, false); }
static pm_status record_prefill(pm_ctx* c, int T, cudaStream_t s) { return record_frame_tc_impl(c, T, s, true); }

static pm_status record_depformer(pm_ctx* c, int B, cudaStream_t s) {
    const pm_config& f = c->cfg;
    const int D = f.D, Dd = f.dep_D, Fd = f.dep_ffn, Q = f.dep_steps;
    if (B == 1 && c->dep_fused && !c->audio_smp) {
        // batch 1, selection by argmax or supplied codes: the whole call as one launch
        PM_CUDA(launch_depth_fused(c->df, c->df_smem, s));
        return PM_OK;
    }
    DepBeginParams bp;
    memset(&bp, 0, sizeof bp);
    bp.dio = reinterpret_cast<const DepIO*>(c->dio_region);
    bp.st = c->st;
    bp.h_internal = c->h;
    bp.dep_sup = c->st.dep_sup;
    bp.B = B;
    bp.D = D;
    bp.Q = Q;
    bp.sup_rows = f.dep_audio_in;
    bp.text_rows = f.dep_text_in;
    PM_CUDA(launch_dep_begin(bp, s, false));
    const size_t dl_elems = (size_t)f.B_max * f.dep_H * Q * f.dep_dh;
    {
        // the input projections of the temporal hidden state for every depth position: they
        // depend only on h, so one launch (a segment per position) instead of one per
        // position on the dependent chain; each position's layer-0 prologue adds the
        // embedding of the code before it
        GemvParams p = base_params(c);
        p.W = c->d_in[0];  // (one position: a plain GEMV)
        p.nseg = Q;
        p.seg_units = Dd;
        for (int q = 0; q < Q; ++q) p.Wseg[q] = c->d_in[q];
        p.K = D;
        p.n_units = Q * Dd;
        p.B = B;
        p.x = c->h;
        p.x_stride = D;
        p.y = c->dzin;
        p.y_stride = Q * Dd;
        pm_status ps = plan(c, p, 1, "depformer input projections");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_PLAIN, E_STORE, U_ROW, p, s, true));
    }
    for (int q = 0; q < Q; ++q) {
        GemvParams p;
        pm_status ps;
        for (int j = 0; j < f.dep_layers; ++j) {
            uint16_t* dkc = c->dkv + (size_t)(2 * j + 0) * dl_elems;
            uint16_t* dvc = c->dkv + (size_t)(2 * j + 1) * dl_elems;
            p = base_params(c);
            p.W = c->d_qkv[j] + (size_t)q * 3 * Dd * Dd;
            p.K = Dd;
            p.n_units = 3 * Dd;
            p.B = B;
            p.x = c->dz;
            p.x_stride = Dd;
            if (j == 0) {
                // input projection + embedding of the previous code, kept as the residual
                p.x = c->dzin + (size_t)q * Dd;
                p.x_stride = Q * Dd;
                p.emb = (q == 0) ? c->d_temb : c->d_aemb[q - 1];
                p.x_out = c->dz;
            }
            p.alpha = c->d_norm1[j];
            p.y = c->dq;
            p.y_stride = Dd;
            p.D = Dd;
            p.H = f.dep_H;
            p.dh = f.dep_dh;
            p.Q = Q;
            p.q = q;
            p.dkc = dkc;
            p.dvc = dvc;
            ps = plan(c, p, 1, "depformer in_proj");
            if (ps) return ps;
            PM_CUDA(launch_gemv(j == 0 ? PRO_RMSNORM_EMB : PRO_RMSNORM, E_DEP_QKV, U_ROW, p, s, true));
            // W_o + residual, with the depth attention computed in its prologue
            p = base_params(c);
            p.W = c->d_o[j] + (size_t)q * Dd * Dd;
            p.K = Dd;
            p.n_units = Dd;
            p.B = B;
            p.x = c->dq;
            p.x_stride = Dd;
            p.y = c->dz;
            p.y_stride = Dd;
            p.H = f.dep_H;
            p.Q = Q;
            p.q = q;
            p.dkc = dkc;
            p.dvc = dvc;
            p.dep_ctx = f.dep_ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);  // keys a position sees
            p.dep_scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dep_dh));
            p.x_in_smem = 1;
            ps = plan(c, p, 1, "depformer out_proj");
            if (ps) return ps;
            PM_CUDA(launch_gemv(PRO_DEPATTN, E_RESIDUAL, U_ROW, p, s, true));
            p = base_params(c);
            p.W = c->d_lin_in[(size_t)j * Q + q];
            p.K = Dd;
            p.n_units = Fd;
            p.split_rows = Fd;
            p.B = B;
            p.x = c->dz;
            p.x_stride = Dd;
            p.alpha = c->d_norm2[j];
            p.y = c->ds;
            p.y_stride = Fd;
            ps = plan(c, p, 2, "depformer linear_in");
            if (ps) return ps;
            PM_CUDA(launch_gemv(PRO_RMSNORM, E_SWIGLU, U_PAIR_SPLIT, p, s, true));
            p = base_params(c);
            p.W = c->d_lin_out[(size_t)j * Q + q];
            p.K = Fd;
            p.n_units = Dd;
            p.B = B;
            p.x = c->ds;
            p.x_stride = Fd;
            p.y = c->dz;
            p.y_stride = Dd;
            ps = plan(c, p, 1, "depformer linear_out");
            if (ps) return ps;
            PM_CUDA(launch_gemv(PRO_PLAIN, E_RESIDUAL, U_ROW, p, s, true));
        }
        p = base_params(c);
        p.W = c->d_heads[q];
        p.K = Dd;
        p.n_units = f.dep_card;
        p.B = B;
        p.x = c->dz;
        p.x_stride = Dd;
        p.y_stride = f.dep_card;
        p.q = q;
        p.Q = Q;
        if (c->audio_smp) p.logits_copy = c->dslog;
        ps = plan(c, p, 1, "depformer head");
        if (ps) return ps;
        PM_CUDA(launch_gemv(PRO_PLAIN, E_DEP_HEAD, U_ROW, p, s, true));
        if (c->audio_smp) {
            // the drawn code replaces the argmax where none is supplied, before position
            // q + 1 embeds it
            SampleParams sp;
            memset(&sp, 0, sizeof sp);
            sp.mode = SM_DEPTH;
            sp.logits = c->dslog;
            sp.ld = f.dep_card;
            sp.V = f.dep_card;
            sp.B = B;
            sp.cfg = c->scfg;
            sp.st = c->st;
            sp.io = reinterpret_cast<const FrameIO*>(c->io_region);
            sp.dio = reinterpret_cast<const DepIO*>(c->dio_region);
            sp.q = q;
            sp.Q = Q;
            sp.n_streams = f.n_streams;
            PM_CUDA(launch_sample(sp, s, true));
        }
    }
    return PM_OK;
}



static pm_status get_graph(pm_ctx* c, std::map<int, cudaGraphExec_t>& cache, int B, record_fn rec,
                           cudaGraphExec_t* out) {
    auto it = cache.find(B);
    if (it != cache.end()) {
        *out = it->second;
        return PM_OK;
    }
    PM_CUDA(cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
    pm_status st = rec(c, B, c->cap);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(c->cap, &g);
    if (st != PM_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamEndCapture");
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGraphInstantiate");
    cache[B] = ex;
    *out = ex;
    return PM_OK;
}

// pinned staging slot for one host->device copy; waits for the slot's previous copy
static pm_status take_slot(pm_ctx* c, uint8_t** host, cudaEvent_t* ev) {
    Staging& sl = c->slots[c->next_slot];
    c->next_slot = (c->next_slot + 1) % kStagingSlots;
    PM_CUDA(cudaEventSynchronize(sl.done));
    *host = sl.host;
    *ev = sl.done;
    return PM_OK;
}

static bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// An output the kernels write: null, or device / managed / host-mapped memory with the
// alignment of the widest store made to it.
static bool output_ok(const void* p, uintptr_t align) {
    if (!p) return true;
    if ((uintptr_t)p & (align - 1)) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
}

// ------------------------------------------------------------------------------------
// ABI
// ------------------------------------------------------------------------------------
static void free_ctx(pm_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    for (auto& kv : c->frame_graphs) cudaGraphExecDestroy(kv.second);
    for (auto& kv : c->dep_graphs) cudaGraphExecDestroy(kv.second);
    for (auto& kv : c->prefill_graphs) cudaGraphExecDestroy(kv.second);
    for (int i = 0; i < kStagingSlots; ++i) {
        if (c->slots[i].done) cudaEventDestroy(c->slots[i].done);
        if (c->slots[i].host) cudaFreeHost(c->slots[i].host);
    }
    if (c->cap) cudaStreamDestroy(c->cap);
    if (c->block) cudaFree(c->block);
    if (c->d_phases) cudaFree(c->d_phases);
    if (c->df_block) cudaFree(c->df_block);
    delete c;
}

extern "C" pm_status pm_create(const pm_config* cfg, const pm_temporal_weights* tw, const pm_depformer_weights* dw,
                               void* kv_cache, void* cuda_stream, pm_ctx** out) {
    if (!out) return PM_ERR_ARG;
    *out = nullptr;
    if (!cfg || !tw || !kv_cache) {
        g_create_err = "pm_create: null config, weights or cache";
        return PM_ERR_ARG;
    }
    if (const char* why = check_config(cfg)) {
        g_create_err = std::string("pm_create: ") + why;
        return PM_ERR_UNSUPPORTED;
    }
    pm_ctx* c = new pm_ctx();
    c->cfg = *cfg;
    const pm_config& f = c->cfg;
    c->has_dep = dw != nullptr && f.dep_layers > 0;
    c->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    c->kv = reinterpret_cast<uint16_t*>(kv_cache);
    cudaError_t last = cudaSuccess;
    auto bail = [&](pm_status st, const char* what) {
        g_create_err = std::string("pm_create: ") + what;
        if (last != cudaSuccess) g_create_err += std::string(": ") + cudaGetErrorString(last);
        cudaGetLastError();
        free_ctx(c);
        return st;
    };
    auto ck = [&](cudaError_t e) {
        last = e;
        return e != cudaSuccess;
    };
    if (ck(cudaGetDevice(&c->device))) return bail(PM_ERR_CUDA, "cudaGetDevice");
    if (ck(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device)))
        return bail(PM_ERR_CUDA, "CUDA call failed");
    if (!aligned16(kv_cache)) return bail(PM_ERR_ARG, "kv_cache not 16-byte aligned");

    // weights
    auto W = [](const void* p) { return reinterpret_cast<const uint16_t*>(p); };
    bool ok = tw->text_emb && tw->out_norm && tw->text_linear && tw->norm1 && tw->in_proj && tw->out_proj &&
              tw->norm2 && tw->linear_in && tw->linear_out;
    if (!ok) return bail(PM_ERR_ARG, "null temporal weight pointer");
    c->tables[0] = W(tw->text_emb);
    for (int k = 1; k < f.n_streams; ++k) {
        if (!tw->audio_emb[k - 1]) return bail(PM_ERR_ARG, "null audio embedding pointer");
        c->tables[k] = W(tw->audio_emb[k - 1]);
    }
    for (int l = 0; l < f.n_layers; ++l) {
        c->norm1.push_back(W(tw->norm1[l]));
        c->in_proj.push_back(W(tw->in_proj[l]));
        c->out_proj.push_back(W(tw->out_proj[l]));
        c->norm2.push_back(W(tw->norm2[l]));
        c->lin_in.push_back(W(tw->linear_in[l]));
        c->lin_out.push_back(W(tw->linear_out[l]));
    }
    c->out_norm = W(tw->out_norm);
    c->text_linear = W(tw->text_linear);
    std::vector<const void*> all = {tw->text_emb, tw->out_norm, tw->text_linear};
    for (int k = 1; k < f.n_streams; ++k) all.push_back(tw->audio_emb[k - 1]);
    for (int l = 0; l < f.n_layers; ++l)
        for (const void* p : {tw->norm1[l], tw->in_proj[l], tw->out_proj[l], tw->norm2[l], tw->linear_in[l],
                              tw->linear_out[l]})
            all.push_back(p);
    if (c->has_dep) {
        const int Q = f.dep_steps, J = f.dep_layers;
        if (!dw->dep_in || !dw->text_emb || (Q > 1 && !dw->audio_emb) || !dw->norm1 || !dw->in_proj ||
            !dw->out_proj || !dw->norm2 || !dw->linear_in || !dw->linear_out || !dw->heads)
            return bail(PM_ERR_ARG, "missing depformer weight array");
        c->d_temb = W(dw->text_emb);
        all.push_back(dw->text_emb);
        for (int q = 0; q < Q; ++q) {
            c->d_in.push_back(W(dw->dep_in[q]));
            c->d_heads.push_back(W(dw->heads[q]));
            all.push_back(dw->dep_in[q]);
            all.push_back(dw->heads[q]);
            if (q < Q - 1) {
                c->d_aemb.push_back(W(dw->audio_emb[q]));
                all.push_back(dw->audio_emb[q]);
            }
        }
        for (int j = 0; j < J; ++j) {
            c->d_norm1.push_back(W(dw->norm1[j]));
            c->d_qkv.push_back(W(dw->in_proj[j]));
            c->d_o.push_back(W(dw->out_proj[j]));
            c->d_norm2.push_back(W(dw->norm2[j]));
            all.insert(all.end(), {dw->norm1[j], dw->in_proj[j], dw->out_proj[j], dw->norm2[j]});
            for (int q = 0; q < Q; ++q) {
                c->d_lin_in.push_back(W(dw->linear_in[(size_t)j * Q + q]));
                c->d_lin_out.push_back(W(dw->linear_out[(size_t)j * Q + q]));
                all.push_back(dw->linear_in[(size_t)j * Q + q]);
                all.push_back(dw->linear_out[(size_t)j * Q + q]);
            }
        }
    }
    for (const void* p : all)
        if (!p || !aligned16(p)) return bail(PM_ERR_ARG, "weight pointer null or not 16-byte aligned");

    // owned device memory: one allocation carved into buffers
    const int BM = f.B_max, S = f.n_streams;
    const int Dd = c->has_dep ? f.dep_D : 0, Fd = c->has_dep ? f.dep_ffn : 0, Q = c->has_dep ? f.dep_steps : 1;
    struct Item {
        void** dst;
        size_t bytes;
    };
    void* p_pos; void* p_first; void* p_ring; void* p_sel; void* p_amax; void* p_hc; void* p_status;
    void* p_damax; void* p_dcount; void* p_dcodes; void* p_dtok; void* p_dsup; void* p_budget;
    void *p_gring, *p_gprov, *p_goff, *p_gin, *p_gtok, *p_gsup, *p_gpos, *p_gsel;
    void* p_io; void* p_dio; void *p_x, *p_q, *p_o, *p_s, *p_h, *p_part, *p_cnt, *p_freq, *p_dz, *p_dq,
        *p_ds, *p_dkv, *p_rtab, *p_xb, *p_ob, *p_sb, *p_ss, *p_tcp, *p_tcc, *p_scfg, *p_slog, *p_dslog,
        *p_sres, *p_apart, *p_skv, *p_dzin;
    // rows of the activation buffers: the batch, or a prefill pass of PM_SEQ_MAX_ROWS frames
    const int RM = BM > PM_SEQ_MAX_ROWS ? BM : PM_SEQ_MAX_ROWS;
    // tensor-core path scratch (batches and prefill passes), sized from the plans of this
    // configuration's projections at every N the path uses
    const int NP = 64;
    size_t tc_part_floats = 16;
    int tc_count_max = 1;
    {
        const int shapes[5][3] = {{TE_QKV_ROPE, f.D, 3 * f.D / 128}, {TE_RESIDUAL, f.D, f.D / 128},
                                  {TE_SWIGLU, f.D, f.ffn / 64}, {TE_RESIDUAL, f.ffn, f.D / 128},
                                  {TE_HEAD, f.D, (f.text_out + 127) / 128}};
        for (int np : {16, 32, 64})
            for (auto& sh : shapes) {
                TcParams t;
                memset(&t, 0, sizeof t);
                t.epi = sh[0];
                t.K = sh[1];
                t.n_mtiles = sh[2];
                t.B = 1;
                t.npad = np;
                if (!plan_tc(t, c->num_sms)) return bail(PM_ERR_UNSUPPORTED, "a tensor-core projection has no plan");
                const size_t need = (size_t)t.n_mtiles * t.maxseg * np * 128;
                if (need > tc_part_floats) tc_part_floats = need;
                if (t.n_mtiles > tc_count_max) tc_count_max = t.n_mtiles;
            }
    }
    // batched GEMV: one sum-of-squares partial per CTA of its residual projections
    int ss_parts_max = 0;
    for (int K : {f.D, f.ffn}) {
        TcParams t;
        memset(&t, 0, sizeof t);
        t.epi = TE_RESIDUAL;
        t.K = K;
        t.n_rows = f.D;
        t.B = 1;
        t.npad = 16;
        if (!plan_mg(t, c->num_sms)) return bail(PM_ERR_UNSUPPORTED, "a batched GEMV projection has no plan");
        if (t.grid > ss_parts_max) ss_parts_max = t.grid;
    }
    c->ss_parts_max = ss_parts_max;
    const size_t ss_floats = std::max((size_t)(f.D / 128) * NP, (size_t)ss_parts_max * 16);
    if (attn_seq_max_chunks(f.ctx) > PM_SEQ_MAX_CHUNKS)
        return bail(PM_ERR_UNSUPPORTED, "ctx too long for the prefill attention");
    c->npad_max = NP;
    c->tc_part_floats = tc_part_floats;
    c->tc_count_max = tc_count_max;
    std::vector<Item> items = {
        {&p_pos, 4u * BM}, {&p_first, 4u * BM}, {&p_ring, 4u * BM * 4 * PM_MAX_STREAMS_DEV},
        {&p_sel, 4u * BM * PM_MAX_STREAMS_DEV}, {&p_amax, 8u * BM}, {&p_hc, 4u * BM}, {&p_status, 16u},
        {&p_damax, 8u * BM}, {&p_dcount, 4u * BM}, {&p_dcodes, 4u * BM * Q}, {&p_dtok, 4u * BM},
        {&p_dsup, 4u * BM * Q}, {&p_budget, 4u},
        {&p_gring, 16u * BM * PM_MAX_STREAMS_DEV}, {&p_gprov, 16u * BM * PM_MAX_STREAMS_DEV}, {&p_goff, 4u * BM},
        {&p_gin, 4u * BM * S}, {&p_gtok, 4u * BM}, {&p_gsup, 4u * BM * Q}, {&p_gpos, 4u * BM},
        {&p_gsel, 4u * BM * PM_MAX_STREAMS_DEV},
        {&p_io, 64u + 4u * RM * S}, {&p_dio, 64u + 4u * BM + 4u * BM * Q},
        {&p_x, 4u * RM * f.D}, {&p_q, 4u * RM * f.D}, {&p_o, 4u * RM * f.D}, {&p_s, 4u * RM * f.ffn},
        {&p_h, 4u * BM * f.D}, {&p_part, 4u * BM * f.H * attn_max_splits(f.ctx) * (f.dh + 2)}, {&p_cnt, 4u * BM * f.H},
        {&p_freq, 8u * (f.dh / 2)}, {&p_rtab, 8u * RM * (f.dh / 2)},
        {&p_xb, 2u * NP * f.D}, {&p_ob, 2u * NP * f.D}, {&p_sb, 2u * NP * f.ffn}, {&p_ss, 4u * ss_floats},
        {&p_tcp, 4u * tc_part_floats}, {&p_tcc, 4u * (size_t)tc_count_max},
        {&p_dz, 4u * BM * (Dd ? Dd : 1)}, {&p_dq, 4u * BM * (Dd ? Dd : 1)},
        {&p_ds, 4u * BM * (Fd ? Fd : 1)}, {&p_dzin, 4u * BM * (Dd ? Dd : 1) * Q},
        {&p_dkv, c->has_dep ? 2u * 2u * f.dep_layers * BM * f.dep_H * Q * f.dep_dh : 16u},
        {&p_scfg, sizeof(SampleCfg)}, {&p_slog, 4u * BM * f.text_out},
        {&p_dslog, c->has_dep ? 4u * BM * f.dep_card : 16u},
        {&p_sres, 4u * PM_SEQ_MAX_ROWS * S},
        {&p_apart, 4u * PM_SEQ_MAX_ROWS * f.H * PM_SEQ_MAX_CHUNKS * PM_SEQ_PART_STRIDE},
        {&p_skv, 2u * 2u * PM_SEQ_MAX_ROWS * f.H * f.dh},
    };
    size_t total = 0;
    for (auto& it : items) total = align_up(total, 256) + align_up(it.bytes, 16);
    total = align_up(total, 256);
    if (ck(cudaMalloc(&c->block, total))) {
        cudaGetLastError();
        return bail(PM_ERR_OOM, "allocation failed");
    }
    c->block_bytes = total;
    if (ck(cudaMemset(c->block, 0, total))) return bail(PM_ERR_CUDA, "cudaMemset");
    size_t off = 0;
    for (auto& it : items) {
        off = align_up(off, 256);
        *it.dst = static_cast<uint8_t*>(c->block) + off;
        off += align_up(it.bytes, 16);
    }
    c->st.pos = (int32_t*)p_pos;
    c->st.first_pos = (int32_t*)p_first;
    c->st.ring = (int32_t*)p_ring;
    c->st.sel = (int32_t*)p_sel;
    c->st.amax = (unsigned long long*)p_amax;
    c->st.head_count = (uint32_t*)p_hc;
    c->st.status = (uint32_t*)p_status;
    c->st.dep_amax = (unsigned long long*)p_damax;
    c->st.dep_count = (uint32_t*)p_dcount;
    c->st.dep_codes = (int32_t*)p_dcodes;
    c->st.dep_tok = (int32_t*)p_dtok;
    c->st.dep_sup = (int32_t*)p_dsup;
    c->st.wait_budget = (const uint32_t*)p_budget;
    c->wait_budget = (uint32_t*)p_budget;
    c->gen_ring = (int32_t*)p_gring;
    c->gen_prov = (int32_t*)p_gprov;
    c->gen_off = (int32_t*)p_goff;
    c->gen_in = (int32_t*)p_gin;
    c->gen_tok = (int32_t*)p_gtok;
    c->gen_sup = (int32_t*)p_gsup;
    c->gen_pos_save = (int32_t*)p_gpos;
    c->gen_sel_save = (int32_t*)p_gsel;
    c->gen_s.assign(BM, 0);
    c->io_region = (uint8_t*)p_io;
    c->dio_region = (uint8_t*)p_dio;
    c->x = (float*)p_x;
    c->q = (float*)p_q;
    c->o = (float*)p_o;
    c->s = (float*)p_s;
    c->h = (float*)p_h;
    c->att_part = (float*)p_part;
    c->att_count = (uint32_t*)p_cnt;
    c->rope_freq = (double*)p_freq;
    c->rope_tab = (float2*)p_rtab;
    c->xb = (uint16_t*)p_xb;
    c->ob = (uint16_t*)p_ob;
    c->sb = (uint16_t*)p_sb;
    c->ss = (float*)p_ss;
    c->tc_part = (float*)p_tcp;
    c->tc_count = (uint32_t*)p_tcc;
    c->dz = (float*)p_dz;
    c->dzin = (float*)p_dzin;
    c->dq = (float*)p_dq;
    c->ds = (float*)p_ds;
    c->dkv = (uint16_t*)p_dkv;
    c->scfg = (SampleCfg*)p_scfg;
    c->slog = (float*)p_slog;
    c->dslog = (float*)p_dslog;
    c->seq_resolved = (int32_t*)p_sres;
    c->seq_part = (float*)p_apart;
    c->seq_kv = (uint16_t*)p_skv;

    // RoPE frequencies f_j = exp(-ln(theta) * 2j / dh), in double
    std::vector<double> freq(f.dh / 2);
    for (int j = 0; j < f.dh / 2; ++j) freq[j] = exp(-log((double)f.rope_theta) * (2.0 * j) / (double)f.dh);
    if (ck(cudaMemcpy(c->rope_freq, freq.data(), 8u * freq.size(), cudaMemcpyHostToDevice)))
        return bail(PM_ERR_CUDA, "CUDA call failed");
    // the full poll budget of the bounded waits
    const uint32_t budget = PM_SPIN_LIMIT;
    if (ck(cudaMemcpy(c->wait_budget, &budget, 4u, cudaMemcpyHostToDevice)))
        return bail(PM_ERR_CUDA, "CUDA call failed");
    // no prior selection anywhere; every generator ring slot unwritten (-2)
    std::vector<int32_t> sel((size_t)BM * PM_MAX_STREAMS_DEV * 4, -2);
    if (ck(cudaMemcpy(c->st.sel, sel.data(), 4u * BM * PM_MAX_STREAMS_DEV, cudaMemcpyHostToDevice)) ||
        ck(cudaMemcpy(c->gen_ring, sel.data(), 16u * BM * PM_MAX_STREAMS_DEV, cudaMemcpyHostToDevice)))
        return bail(PM_ERR_CUDA, "CUDA call failed");

    if (ck(cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking))) return bail(PM_ERR_CUDA, "cudaStreamCreateWithFlags");
    const size_t slot_bytes = 64u + 4u * (size_t)RM * (S + 1 + Q);
    for (int i = 0; i < kStagingSlots; ++i) {
        if (cudaHostAlloc((void**)&c->slots[i].host, align_up(slot_bytes, 64), cudaHostAllocDefault) !=
            cudaSuccess)
            return bail(PM_ERR_OOM, "allocation failed");
        if (ck(cudaEventCreateWithFlags(&c->slots[i].done, cudaEventDisableTiming)))
            return bail(PM_ERR_CUDA, "CUDA call failed");
    }
    // verify every GEMV of the configuration has a plan before accepting it
    {
        GemvParams t;
        memset(&t, 0, sizeof t);
        auto chk = [&](int K, int units, int rpu) {
            t.K = K;
            t.n_units = units;
            return plan_gemv(t, rpu, c->num_sms);
        };
        bool good = chk(f.D, 3 * f.D / 2, 2) && chk(f.D, f.D, 1) && chk(f.D, f.ffn, 2) && chk(f.ffn, f.D, 1) &&
                    chk(f.D, f.text_out, 1);
        if (c->has_dep)
            good = good && chk(f.D, f.dep_D, 1) && chk(f.dep_D, 3 * f.dep_D, 1) && chk(f.dep_D, f.dep_D, 1) &&
                   chk(f.dep_D, f.dep_ffn, 2) && chk(f.dep_ffn, f.dep_D, 1) && chk(f.dep_D, f.dep_card, 1);
        if (!good) return bail(PM_ERR_UNSUPPORTED, "a GEMV shape has no plan");
    }
    // persistent batch-1 frame program: phases of the whole frame, built once
    if ((f.flags & PM_FLAG_FRAME_PROGRAM) && frame_prog_supported(f.D, f.ffn, f.dh)) {
        int coop = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
        std::vector<FPhase> ph;
        int partial_floats = 1;
        const int G = c->num_sms;
        auto gemv = [&](int epi, int unit, int K, int n_units, int split, const uint16_t* W, const float* x,
                        const uint16_t* alpha, float* y, uint16_t* kc, uint16_t* vc) {
            FPhase q;
            memset(&q, 0, sizeof q);
            q.type = PH_GEMV;
            q.epi = epi;
            q.unit = unit;
            q.K = K;
            q.n_units = n_units;
            q.split_rows = split;
            const int rpu = unit == U_ROW ? 1 : 2;
            q.upst = frame_prog_stage_rows(K) / rpu;
            q.W = W;
            q.x = x;
            q.alpha = alpha;
            q.y = y;
            q.kc = kc;
            q.vc = vc;
            const int need = ((n_units + G - 1) / G) * rpu * (K / 1024);
            if (need > partial_floats) partial_floats = need;
            ph.push_back(q);
            return q.upst >= 1;
        };
        bool good = coop != 0;
        FPhase e;
        memset(&e, 0, sizeof e);
        e.type = PH_EMBED;
        ph.push_back(e);
        const size_t layer_elems = (size_t)f.B_max * f.H * f.ctx * f.dh;
        for (int l = 0; l < f.n_layers; ++l) {
            uint16_t* kc = c->kv + (size_t)(2 * l + 0) * layer_elems;
            uint16_t* vc = c->kv + (size_t)(2 * l + 1) * layer_elems;
            good = good && gemv(E_QKV_ROPE, U_PAIR_ADJ, f.D, 3 * f.D / 2, 0, c->in_proj[l], c->x, c->norm1[l], c->q,
                                kc, vc);
            FPhase a;
            memset(&a, 0, sizeof a);
            a.type = PH_ATTN;
            a.kc = kc;
            a.vc = vc;
            ph.push_back(a);
            good = good && gemv(E_RESIDUAL, U_ROW, f.D, f.D, 0, c->out_proj[l], c->o, nullptr, c->x, kc, vc);
            good = good && gemv(E_SWIGLU, U_PAIR_SPLIT, f.D, f.ffn, f.ffn, c->lin_in[l], c->x, c->norm2[l], c->s,
                                kc, vc);
            good = good && gemv(E_RESIDUAL, U_ROW, f.ffn, f.D, 0, c->lin_out[l], c->s, nullptr, c->x, kc, vc);
        }
        good = good && gemv(E_HEAD, U_ROW, f.D, f.text_out, 0, c->text_linear, c->x, c->out_norm, nullptr,
                            nullptr, nullptr);
        const int S = attn_max_splits(f.ctx);
        const size_t smem = frame_prog_smem(partial_floats, S);
        int occ = 0;
        good = good && S <= 64 && smem <= 226u * 1024u && frame_prog_prepare(smem) == cudaSuccess &&
               frame_prog_occupancy(smem, &occ) == cudaSuccess && occ >= 1;
        cudaGetLastError();
        if (good) {
            // counters: one per phase, then the launch's exit and timeout counters
            const size_t n_bar = ph.size() + 2;
            if (ck(cudaMalloc(&c->d_phases, sizeof(FPhase) * ph.size() + 4u * n_bar)))
                return bail(PM_ERR_OOM, "device allocation (frame program)");
            c->prog_bar = reinterpret_cast<uint32_t*>(c->d_phases + ph.size());
            if (ck(cudaMemcpy(c->d_phases, ph.data(), sizeof(FPhase) * ph.size(), cudaMemcpyHostToDevice)) ||
                ck(cudaMemset(c->prog_bar, 0, 4u * n_bar)))
                return bail(PM_ERR_CUDA, "frame program upload");
            FrameProgParams& pp = c->prog_params;
            memset(&pp, 0, sizeof pp);
            pp.ph = c->d_phases;
            pp.n_phases = (int)ph.size();
            pp.st = c->st;
            pp.io = reinterpret_cast<const FrameIO*>(c->io_region);
            for (int k = 0; k < f.n_streams; ++k) {
                pp.tables[k] = c->tables[k];
                pp.rows[k] = (k == 0) ? f.text_in : f.audio_in;
                pp.init_id[k] = (k == 0) ? f.init_text : f.init_audio;
                pp.delays[k] = f.delays[k];
            }
            pp.n_streams = f.n_streams;
            pp.rope_freq = c->rope_freq;
            pp.rope_tab = c->rope_tab;
            pp.x = c->x;
            pp.q = c->q;
            pp.o = c->o;
            pp.h = c->h;
            pp.D = f.D;
            pp.H = f.H;
            pp.dh = f.dh;
            pp.ctx = f.ctx;
            pp.win = f.ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);
            pp.eps = f.eps;
            pp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dh));
            pp.part = c->att_part;
            pp.att_count = c->att_count;
            pp.S = S;
            pp.max_chunks = S;
            pp.partial_floats = partial_floats;
            pp.bar = c->prog_bar;
            c->prog_smem = smem;
            c->prog = true;
        }
    }
    // persistent batch-1 depformer: one cooperative launch of H clusters of 4 CTAs, its own
    // re-laid copies of W_o (head blocks) and linear_out (transposed)
    if (c->has_dep && !(f.flags & PM_FLAG_DEPFORMER_CHAIN) && f.dep_steps <= PM_DF_MAX_Q &&
        f.dep_layers <= PM_DF_MAX_J &&
        depth_fused_supported(f.D, f.dep_D, f.dep_H, f.dep_dh, f.dep_ffn, f.dep_steps, f.dep_card, c->num_sms)) {
        int coop = 0, nclu = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
        const size_t smem = depth_fused_smem();
        const int G = 4 * f.dep_H;
        const bool fits = coop && depth_fused_prepare(smem) == cudaSuccess &&
                          depth_fused_max_clusters(smem, G, &nclu) == cudaSuccess && nclu >= f.dep_H;
        cudaGetLastError();
        if (fits) {
            const int J = f.dep_layers, Qd = f.dep_steps;
            const size_t wo_elems = (size_t)J * Qd * Dd * Dd, wt_elems = (size_t)J * Qd * Fd * Dd;
            const size_t sc_bytes = 4u * ((size_t)Qd * Dd + 2u * f.dep_H * Dd) + 8u * Qd + 16u;
            if (ck(cudaMalloc(&c->df_block, 2u * (wo_elems + wt_elems) + sc_bytes + 256)))
                return bail(PM_ERR_OOM, "device allocation (depformer copies)");
            if (ck(cudaMemset(c->df_block, 0, 2u * (wo_elems + wt_elems) + sc_bytes + 256)))
                return bail(PM_ERR_CUDA, "cudaMemset");
            uint16_t* wo = static_cast<uint16_t*>(c->df_block);
            uint16_t* wt = wo + wo_elems;
            uint8_t* scr = reinterpret_cast<uint8_t*>(wt + wt_elems);
            for (int j = 0; j < J; ++j)
                for (int q = 0; q < Qd; ++q)
                    if (ck(depth_relayout(c->d_o[j] + (size_t)q * Dd * Dd, wo + ((size_t)j * Qd + q) * Dd * Dd,
                                          c->d_lin_out[(size_t)j * Qd + q], wt + ((size_t)j * Qd + q) * Fd * Dd, Dd,
                                          Fd, f.dep_H, 0)))
                        return bail(PM_ERR_CUDA, "depformer weight re-layout");
            DepFusedParams& d = c->df;
            memset(&d, 0, sizeof d);
            d.st = c->st;
            d.dio = reinterpret_cast<const DepIO*>(c->dio_region);
            for (int q = 0; q < Qd; ++q) {
                d.dep_in[q] = c->d_in[q];
                d.heads[q] = c->d_heads[q];
                if (q > 0) d.aemb[q - 1] = c->d_aemb[q - 1];
            }
            d.temb = c->d_temb;
            const size_t dl_elems = (size_t)f.B_max * f.dep_H * Qd * f.dep_dh;
            for (int j = 0; j < J; ++j) {
                d.norm1[j] = c->d_norm1[j];
                d.norm2[j] = c->d_norm2[j];
                d.qkv[j] = c->d_qkv[j];
                for (int q = 0; q < Qd; ++q) d.lin_in[j * Qd + q] = c->d_lin_in[(size_t)j * Qd + q];
                d.dk[j] = c->dkv + (size_t)(2 * j + 0) * dl_elems;
                d.dv[j] = c->dkv + (size_t)(2 * j + 1) * dl_elems;
            }
            d.wo_packed = wo;
            d.wout_t = wt;
            d.dzin = reinterpret_cast<float*>(scr);
            d.part_att = d.dzin + (size_t)Qd * Dd;
            d.part_ffn = d.part_att + (size_t)f.dep_H * Dd;
            d.amax = reinterpret_cast<unsigned long long*>(d.part_ffn + (size_t)f.dep_H * Dd);
            d.bar = reinterpret_cast<uint32_t*>(d.amax + Qd);
            d.G = G;
            d.D = f.D;
            d.Dd = Dd;
            d.H = f.dep_H;
            d.Fd = Fd;
            d.Q = Qd;
            d.J = J;
            d.card = f.dep_card;
            d.n_streams = f.n_streams;
            d.text_rows = f.dep_text_in;
            d.sup_rows = f.dep_audio_in;
            d.dep_win = f.dep_ctx - ((f.flags & PM_FLAG_PINNED_RING) ? 1 : 0);
            d.eps = f.eps;
            d.scale_log2 = (float)(1.4426950408889634 / sqrt((double)f.dep_dh));
            c->df_smem = smem;
            c->dep_fused = true;
        }
    }
    if (ck(gemv_prepare())) return bail(PM_ERR_CUDA, "gemv_prepare()");
    if (ck(sample_prepare())) return bail(PM_ERR_CUDA, "sample_prepare()");
    if (ck(attn_seq_prepare())) return bail(PM_ERR_CUDA, "attn_seq_prepare()");
    if (ck(tc_prepare())) return bail(PM_ERR_CUDA, "tc_prepare");
    if (ck(mg_prepare())) return bail(PM_ERR_CUDA, "mg_prepare");
    if (ck(attn_prepare())) return bail(PM_ERR_CUDA, "attn_prepare");
    if (ck(cudaDeviceSynchronize())) return bail(PM_ERR_CUDA, "cudaDeviceSynchronize()");
    *out = c;
    return PM_OK;
}

extern "C" void pm_destroy(pm_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    cudaStreamSynchronize(c->stream);
    free_ctx(c);
}

extern "C" const char* pm_last_error(const pm_ctx* c) { return c ? c->err.c_str() : g_create_err.c_str(); }

static pm_status set_state(pm_ctx* c, const int32_t* pos, const int32_t* apply, int n, bool reset_gen) {
    SetStateArgs a;
    memset(&a, 0, sizeof a);
    a.st = c->st;
    if (reset_gen) {
        a.gen_ring = c->gen_ring;
        a.gen_prov = c->gen_prov;
        a.gen_off = c->gen_off;
        for (int b = 0; b < n; ++b)
            if (apply[b]) c->gen_s[b] = 0;
    }
    a.n = n;
    for (int b = 0; b < n; ++b) {
        a.pos[b] = pos[b];
        a.apply[b] = apply[b];
    }
    k_set_state<<<n, 32, 0, c->stream>>>(a);
    PM_CUDA(cudaGetLastError());
    return PM_OK;
}

extern "C" pm_status pm_reset(pm_ctx* c, const int32_t* mask) {
    if (!c) return PM_ERR_ARG;
    PM_CUDA(cudaSetDevice(c->device));
    int32_t pos[kMaxB] = {0}, apply[kMaxB];
    for (int b = 0; b < c->cfg.B_max; ++b) apply[b] = mask ? (mask[b] != 0) : 1;
    return set_state(c, pos, apply, c->cfg.B_max, true);
}

extern "C" pm_status pm_set_positions(pm_ctx* c, int B, const int32_t* pos) {
    if (!c) return PM_ERR_ARG;
    if (B < 1 || B > c->cfg.B_max || !pos) return fail(c, PM_ERR_ARG, "pm_set_positions: bad B or pos");
    for (int b = 0; b < B; ++b)
        if (pos[b] < 0) return fail(c, PM_ERR_ARG, "pm_set_positions: negative position");
    PM_CUDA(cudaSetDevice(c->device));
    int32_t apply[kMaxB];
    for (int b = 0; b < B; ++b) apply[b] = 1;
    return set_state(c, pos, apply, B, false);
}

extern "C" pm_status pm_get_positions(pm_ctx* c, int32_t* pos_out) {
    if (!c || !pos_out) return PM_ERR_ARG;
    PM_CUDA(cudaSetDevice(c->device));
    PM_CUDA(cudaMemcpyAsync(pos_out, c->st.pos, 4u * c->cfg.B_max, cudaMemcpyDeviceToHost, c->stream));
    PM_CUDA(cudaStreamSynchronize(c->stream));
    return PM_OK;
}

// ------------------------------------------------------------------------------------
// stream snapshots
// ------------------------------------------------------------------------------------
namespace {
constexpr uint32_t kSnapMagic = 0x4E534D50u;  // "PMSN"
constexpr uint32_t kSnapVersion = 2u;
constexpr size_t kSnapHeader = 2048;          // header bytes before the KV rows
// header layout (bytes): [0, 64) identity and shape, 64 pos, 68 first_pos, 72 n_slots,
// 76 generator offset, [128, 128 + 4 * 4 * PM_MAX_STREAMS_DEV) delay ring, then
// PM_MAX_STREAMS_DEV selections; [1024, 1536) the generator's token ring and [1536, 2048)
// its provided ring ([PM_MAX_STREAMS_DEV][4] each)
constexpr size_t kSnapRing = 128;
constexpr size_t kSnapSel = kSnapRing + 4u * 4u * PM_MAX_STREAMS_DEV;
constexpr size_t kSnapGenRing = 1024;
constexpr size_t kSnapGenProv = kSnapGenRing + 16u * PM_MAX_STREAMS_DEV;
struct SnapIdent {
    uint32_t magic, version;
    int32_t n_layers, H, dh, ctx, n_streams, D;
};
static_assert(kSnapSel + 4u * PM_MAX_STREAMS_DEV <= kSnapGenRing, "snapshot header overflow");
static_assert(kSnapGenProv + 16u * PM_MAX_STREAMS_DEV <= kSnapHeader, "snapshot header overflow");
}  // namespace

extern "C" size_t pm_snapshot_bytes(const pm_config* f) {
    if (!f) return 0;
    return kSnapHeader + (size_t)f->n_layers * 2u * f->H * f->ctx * f->dh * 2u;
}

// one stream's KV rows of slots [0, n) <-> the snapshot's [layer][K/V][head][slot][dh]
static pm_status snap_kv(pm_ctx* c, int b, uint8_t* snap, int n, bool to_snap) {
    const pm_config& f = c->cfg;
    const size_t row = (size_t)f.dh * 2u;
    for (int l = 0; l < f.n_layers; ++l)
        for (int kv = 0; kv < 2; ++kv) {
            uint8_t* cache = reinterpret_cast<uint8_t*>(c->kv) +
                             ((((size_t)(2 * l + kv) * f.B_max + b) * f.H) * f.ctx) * row;
            uint8_t* s = snap + kSnapHeader + ((size_t)(2 * l + kv) * f.H) * n * row;
            if (to_snap)
                PM_CUDA(cudaMemcpy2DAsync(s, n * row, cache, f.ctx * row, n * row, f.H, cudaMemcpyDeviceToDevice,
                                          c->stream));
            else
                PM_CUDA(cudaMemcpy2DAsync(cache, f.ctx * row, s, n * row, n * row, f.H, cudaMemcpyDeviceToDevice,
                                          c->stream));
        }
    return PM_OK;
}

extern "C" pm_status pm_snapshot(pm_ctx* c, int b, void* dst) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (b < 0 || b >= f.B_max || !dst || !aligned16(dst)) return fail(c, PM_ERR_ARG, "pm_snapshot: bad stream or dst");
    PM_CUDA(cudaSetDevice(c->device));
    if (!is_device_ptr(dst)) return fail(c, PM_ERR_ARG, "pm_snapshot: dst must be device memory");
    int32_t pf[2];
    PM_CUDA(cudaStreamSynchronize(c->stream));
    PM_CUDA(cudaMemcpy(&pf[0], c->st.pos + b, 4, cudaMemcpyDeviceToHost));
    PM_CUDA(cudaMemcpy(&pf[1], c->st.first_pos + b, 4, cudaMemcpyDeviceToHost));
    const int n = pf[0] < f.ctx ? pf[0] : f.ctx;
    uint8_t hdr[128];
    memset(hdr, 0, sizeof hdr);
    SnapIdent id{kSnapMagic, kSnapVersion, f.n_layers, f.H, f.dh, f.ctx, f.n_streams, f.D};
    memcpy(hdr, &id, sizeof id);
    const int32_t st4[4] = {pf[0], pf[1], n, c->gen_s[b]};
    memcpy(hdr + 64, st4, sizeof st4);
    uint8_t* d = static_cast<uint8_t*>(dst);
    PM_CUDA(cudaMemcpyAsync(d, hdr, sizeof hdr, cudaMemcpyHostToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(d + kSnapRing, c->st.ring + (size_t)b * 4 * PM_MAX_STREAMS_DEV,
                            4u * 4u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(d + kSnapSel, c->st.sel + (size_t)b * PM_MAX_STREAMS_DEV, 4u * PM_MAX_STREAMS_DEV,
                            cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(d + kSnapGenRing, c->gen_ring + (size_t)b * 4 * PM_MAX_STREAMS_DEV,
                            16u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(d + kSnapGenProv, c->gen_prov + (size_t)b * 4 * PM_MAX_STREAMS_DEV,
                            16u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    pm_status st = snap_kv(c, b, d, n, true);
    if (st) return st;
    PM_CUDA(cudaStreamSynchronize(c->stream));
    return PM_OK;
}

extern "C" pm_status pm_restore(pm_ctx* c, int b, const void* src) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (b < 0 || b >= f.B_max || !src || !aligned16(src)) return fail(c, PM_ERR_ARG, "pm_restore: bad stream or src");
    PM_CUDA(cudaSetDevice(c->device));
    if (!is_device_ptr(src)) return fail(c, PM_ERR_ARG, "pm_restore: src must be device memory");
    PM_CUDA(cudaStreamSynchronize(c->stream));
    uint8_t hdr[128];
    PM_CUDA(cudaMemcpy(hdr, src, sizeof hdr, cudaMemcpyDeviceToHost));
    SnapIdent id;
    memcpy(&id, hdr, sizeof id);
    int32_t st3[4];
    memcpy(st3, hdr + 64, sizeof st3);
    if (id.magic != kSnapMagic || id.version != kSnapVersion)
        return fail(c, PM_ERR_ARG, "pm_restore: not a snapshot");
    if (id.n_layers != f.n_layers || id.H != f.H || id.dh != f.dh || id.ctx != f.ctx || id.n_streams != f.n_streams ||
        id.D != f.D)
        return fail(c, PM_ERR_ARG, "pm_restore: snapshot of another configuration");
    if (st3[0] < 0 || st3[1] < 0 || st3[1] > st3[0] || st3[2] != (st3[0] < f.ctx ? st3[0] : f.ctx) || st3[3] < 0)
        return fail(c, PM_ERR_ARG, "pm_restore: inconsistent snapshot header");
    const uint8_t* s = static_cast<const uint8_t*>(src);
    // The delay ring and the selections become row indices of the embedding tables on the
    // next frame: every entry a later frame can read must be a valid ID, checked here on
    // the host before anything reaches the context.
    {
        int32_t ring[4 * PM_MAX_STREAMS_DEV], sel[PM_MAX_STREAMS_DEV];
        PM_CUDA(cudaMemcpy(ring, s + kSnapRing, sizeof ring, cudaMemcpyDeviceToHost));
        PM_CUDA(cudaMemcpy(sel, s + kSnapSel, sizeof sel, cudaMemcpyDeviceToHost));
        const int pos = st3[0], first = st3[1];
        for (int k = 0; k < f.n_streams; ++k) {
            const int rows = (k == 0) ? f.text_in : f.audio_in;
            // frames pos-3..pos-1 since the first position: the ring slots a delay of up to
            // 3 frames reads on the next frames
            for (int q = pos - 3; q < pos; ++q) {
                if (q < first) continue;
                const int32_t id = ring[(q & 3) * PM_MAX_STREAMS_DEV + k];
                if (id < -1 || id >= rows)
                    return fail(c, PM_ERR_ARG, "pm_restore: snapshot delay ring holds ID " + std::to_string(id) +
                                                   " for stream " + std::to_string(k));
            }
            // a selection is a token the stream selected (or -2: none yet)
            if (sel[k] < -2 || sel[k] >= rows)
                return fail(c, PM_ERR_ARG, "pm_restore: snapshot selection " + std::to_string(sel[k]) +
                                               " for stream " + std::to_string(k));
        }
        // the generator's rings: codes -2 (unwritten) .. rows-1, flags 0 / 1
        int32_t gring[4 * PM_MAX_STREAMS_DEV], gprov[4 * PM_MAX_STREAMS_DEV];
        PM_CUDA(cudaMemcpy(gring, s + kSnapGenRing, sizeof gring, cudaMemcpyDeviceToHost));
        PM_CUDA(cudaMemcpy(gprov, s + kSnapGenProv, sizeof gprov, cudaMemcpyDeviceToHost));
        for (int k = 0; k < f.n_streams; ++k) {
            const int rows = (k == 0) ? f.text_in : f.audio_in;
            for (int j = 0; j < 4; ++j) {
                const int32_t v = gring[k * 4 + j], fl = gprov[k * 4 + j];
                if (v < -2 || v >= rows || (fl != 0 && fl != 1))
                    return fail(c, PM_ERR_ARG, "pm_restore: snapshot generator ring holds " + std::to_string(v) +
                                                   " for stream " + std::to_string(k));
            }
        }
    }
    PM_CUDA(cudaMemcpyAsync(c->st.pos + b, s + 64, 4, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->st.first_pos + b, s + 68, 4, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->st.ring + (size_t)b * 4 * PM_MAX_STREAMS_DEV, s + kSnapRing,
                            4u * 4u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->st.sel + (size_t)b * PM_MAX_STREAMS_DEV, s + kSnapSel, 4u * PM_MAX_STREAMS_DEV,
                            cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->gen_ring + (size_t)b * 4 * PM_MAX_STREAMS_DEV, s + kSnapGenRing,
                            16u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->gen_prov + (size_t)b * 4 * PM_MAX_STREAMS_DEV, s + kSnapGenProv,
                            16u * PM_MAX_STREAMS_DEV, cudaMemcpyDeviceToDevice, c->stream));
    PM_CUDA(cudaMemcpyAsync(c->gen_off + b, s + 76, 4, cudaMemcpyDeviceToDevice, c->stream));
    c->gen_s[b] = st3[3];
    pm_status st = snap_kv(c, b, const_cast<uint8_t*>(s), st3[2], false);
    if (st) return st;
    PM_CUDA(cudaStreamSynchronize(c->stream));
    return PM_OK;
}

// one word of device memory, written in stream order
__global__ void k_set_word(uint32_t* dst, uint32_t v) { *dst = v; }

extern "C" pm_status pm_set_wait_budget(pm_ctx* c, uint32_t polls) {
    if (!c) return PM_ERR_ARG;
    PM_CUDA(cudaSetDevice(c->device));
    k_set_word<<<1, 1, 0, c->stream>>>(c->wait_budget, polls == PM_WAIT_BUDGET_DEFAULT ? (uint32_t)PM_SPIN_LIMIT : polls);
    PM_CUDA(cudaGetLastError());
    return PM_OK;
}

extern "C" pm_status pm_device_status(pm_ctx* c) {
    if (!c) return PM_ERR_ARG;
    PM_CUDA(cudaSetDevice(c->device));
    uint32_t st[4] = {0, 0, 0, 0};
    PM_CUDA(cudaStreamSynchronize(c->stream));
    PM_CUDA(cudaMemcpy(st, c->st.status, sizeof st, cudaMemcpyDeviceToHost));
    PM_CUDA(cudaMemset(c->st.status, 0, 4));
    if (st[0] & PM_DEV_ERR_TIMEOUT) return fail(c, PM_ERR_TIMEOUT, "a device-side wait ran out");
    if (st[0] & PM_DEV_ERR_INVALID_ID) return fail(c, PM_ERR_INVALID_ID, "an ID given in device memory was invalid");
    return PM_OK;
}

extern "C" pm_status pm_frame_step(pm_ctx* c, int B, const int32_t* ids, float* text_logits, float* hidden,
                                   int32_t* text_token) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (B < 1 || B > f.B_max) return fail(c, PM_ERR_ARG, "pm_frame_step: B outside 1..B_max");
    if (!ids) return fail(c, PM_ERR_ARG, "pm_frame_step: ids is null");
    PM_CUDA(cudaSetDevice(c->device));
    // the head writes hidden with 16-byte stores, logits and the token with 4-byte stores
    if (!output_ok(hidden, 16) || !output_ok(text_logits, 4) || !output_ok(text_token, 4))
        return fail(c, PM_ERR_ARG,
                    "pm_frame_step: an output is not device or host-mapped memory, or hidden is not 16-byte aligned");
    const int S = f.n_streams;
    const bool dev_ids = is_device_ptr(ids);
    if (!dev_ids) {
        for (int b = 0; b < B; ++b)
            for (int k = 0; k < S; ++k) {
                const int32_t id = ids[(size_t)b * S + k];
                const int rows = (k == 0) ? f.text_in : f.audio_in;
                if (!(id == PM_ID_FEEDBACK || (id >= -1 && id < rows)))
                    return fail(c, PM_ERR_INVALID_ID, "pm_frame_step: ID " + std::to_string(id) + " at batch " +
                                                          std::to_string(b) + " stream " + std::to_string(k));
            }
    }
    cudaGraphExec_t ex;
    pm_status st = get_graph(c, c->frame_graphs, B, B >= 2 ? record_frame_tc : record_frame, &ex);
    if (st) return st;
    uint8_t* host;
    cudaEvent_t ev;
    st = take_slot(c, &host, &ev);
    if (st) return st;
    FrameIO io;
    memset(&io, 0, sizeof io);
    io.ids = dev_ids ? ids : reinterpret_cast<const int32_t*>(c->io_region + 64);
    io.logits = text_logits;
    io.hidden = hidden;
    io.token = text_token;
    memcpy(host, &io, sizeof io);
    size_t bytes = 64;
    if (!dev_ids) {
        memcpy(host + 64, ids, 4u * B * S);
        bytes += 4u * B * S;
    }
    PM_CUDA(cudaMemcpyAsync(c->io_region, host, bytes, cudaMemcpyHostToDevice, c->stream));
    PM_CUDA(cudaEventRecord(ev, c->stream));
    PM_CUDA(cudaGraphLaunch(ex, c->stream));
    return PM_OK;
}

extern "C" pm_status pm_prefill(pm_ctx* c, int stream, int T, const int32_t* ids, float* text_logits, float* hidden,
                                int32_t* text_token) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (stream < 0 || stream >= f.B_max) return fail(c, PM_ERR_ARG, "pm_prefill: stream outside 0..B_max-1");
    if (T < 1 || !ids) return fail(c, PM_ERR_ARG, "pm_prefill: need T >= 1 and ids");
    PM_CUDA(cudaSetDevice(c->device));
    const int S = f.n_streams;
    const bool dev_ids = is_device_ptr(ids);
    if (!dev_ids)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < S; ++k) {
                const int32_t id = ids[(size_t)t * S + k];
                const int rows = (k == 0) ? f.text_in : f.audio_in;
                if (id < -1 || id >= rows)
                    return fail(c, PM_ERR_INVALID_ID, "pm_prefill: ID " + std::to_string(id) + " at frame " +
                                                          std::to_string(t) + " stream " + std::to_string(k));
            }
    for (int t0 = 0; t0 < T; t0 += PM_SEQ_MAX_ROWS) {
        const int n = T - t0 < PM_SEQ_MAX_ROWS ? T - t0 : PM_SEQ_MAX_ROWS;
        cudaGraphExec_t ex;
        pm_status st = get_graph(c, c->prefill_graphs, n, record_prefill, &ex);
        if (st) return st;
        uint8_t* host;
        cudaEvent_t ev;
        st = take_slot(c, &host, &ev);
        if (st) return st;
        FrameIO io;
        memset(&io, 0, sizeof io);
        io.ids = dev_ids ? ids + (size_t)t0 * S : reinterpret_cast<const int32_t*>(c->io_region + 64);
        io.logits = text_logits;
        io.hidden = hidden;
        io.token = text_token;
        io.seq_stream = stream;
        memcpy(host, &io, sizeof io);
        size_t bytes = 64;
        if (!dev_ids) {
            memcpy(host + 64, ids + (size_t)t0 * S, 4u * n * S);
            bytes += 4u * n * S;
        }
        PM_CUDA(cudaMemcpyAsync(c->io_region, host, bytes, cudaMemcpyHostToDevice, c->stream));
        PM_CUDA(cudaEventRecord(ev, c->stream));
        PM_CUDA(cudaGraphLaunch(ex, c->stream));
    }
    return PM_OK;
}

extern "C" pm_status pm_depformer_step(pm_ctx* c, int B, const float* hidden, const int32_t* text_tok,
                                       const int32_t* supplied, float* logits, int32_t* codes) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (!c->has_dep) return fail(c, PM_ERR_STATE, "pm_depformer_step: context has no depformer");
    if (B < 1 || B > f.B_max) return fail(c, PM_ERR_ARG, "pm_depformer_step: B outside 1..B_max");
    PM_CUDA(cudaSetDevice(c->device));
    const int Q = f.dep_steps;
    if (hidden && !is_device_ptr(hidden)) return fail(c, PM_ERR_ARG, "pm_depformer_step: hidden must be device memory");
    const bool dev_tok = text_tok && is_device_ptr(text_tok);
    const bool dev_sup = supplied && is_device_ptr(supplied);
    if (text_tok && !dev_tok)
        for (int b = 0; b < B; ++b)
            if (text_tok[b] < 0 || text_tok[b] >= f.dep_text_in)
                return fail(c, PM_ERR_INVALID_ID, "pm_depformer_step: text token out of range");
    if (supplied && !dev_sup)
        for (int i = 0; i < B * Q; ++i)
            if (supplied[i] < -1 || supplied[i] >= f.dep_audio_in)
                return fail(c, PM_ERR_INVALID_ID, "pm_depformer_step: supplied code out of range");
    cudaGraphExec_t ex;
    pm_status st = get_graph(c, c->dep_graphs, B, record_depformer, &ex);
    if (st) return st;
    uint8_t* host;
    cudaEvent_t ev;
    st = take_slot(c, &host, &ev);
    if (st) return st;
    uint8_t* dev_tok_buf = c->dio_region + 64;
    uint8_t* dev_sup_buf = c->dio_region + 64 + 4u * f.B_max;
    DepIO io;
    memset(&io, 0, sizeof io);
    io.hidden = hidden ? hidden : c->h;
    io.text_tok = text_tok ? (dev_tok ? text_tok : reinterpret_cast<const int32_t*>(dev_tok_buf)) : nullptr;
    io.supplied = supplied ? (dev_sup ? supplied : reinterpret_cast<const int32_t*>(dev_sup_buf)) : nullptr;
    io.logits = logits;
    io.codes = codes;
    memcpy(host, &io, sizeof io);
    if (text_tok && !dev_tok) memcpy(host + 64, text_tok, 4u * B);
    if (supplied && !dev_sup) memcpy(host + 64 + 4u * f.B_max, supplied, 4u * B * Q);
    const size_t bytes = 64u + 4u * f.B_max + 4u * (size_t)B * Q;
    PM_CUDA(cudaMemcpyAsync(c->dio_region, host, bytes, cudaMemcpyHostToDevice, c->stream));
    PM_CUDA(cudaEventRecord(ev, c->stream));
    PM_CUDA(cudaGraphLaunch(ex, c->stream));
    return PM_OK;
}

extern "C" pm_status pm_generator_step(pm_ctx* c, int B, const int32_t* provided, int32_t* out, int32_t* out_valid,
                                       float* text_logits, float* hidden, float* depth_logits) {
    if (!c) return PM_ERR_ARG;
    const pm_config& f = c->cfg;
    if (!c->has_dep) return fail(c, PM_ERR_STATE, "pm_generator_step: context has no depformer");
    if (f.dep_steps != f.n_streams - 1)
        return fail(c, PM_ERR_UNSUPPORTED, "pm_generator_step: needs one depth position per audio stream");
    if (B < 1 || B > f.B_max) return fail(c, PM_ERR_ARG, "pm_generator_step: B outside 1..B_max");
    PM_CUDA(cudaSetDevice(c->device));
    if (!output_ok(out, 4) || !output_ok(out_valid, 4) || !output_ok(text_logits, 4) || !output_ok(hidden, 16) ||
        !output_ok(depth_logits, 4))
        return fail(c, PM_ERR_ARG,
                    "pm_generator_step: an output is not device or host-mapped memory, or hidden is not 16-byte aligned");
    const int S = f.n_streams, Q = f.dep_steps;
    if (provided) {
        if (is_device_ptr(provided)) return fail(c, PM_ERR_ARG, "pm_generator_step: provided must be host memory");
        for (int b = 0; b < B; ++b)
            for (int k = 0; k < S; ++k) {
                // a provided code is a temporal input and a depth input (or conditioning token)
                const int rows = (k == 0) ? std::min(f.text_in, f.dep_text_in) : std::min(f.audio_in, f.dep_audio_in);
                const int32_t v = provided[(size_t)b * S + k];
                if (!(v == -1 || (v >= 0 && v < rows)))
                    return fail(c, PM_ERR_INVALID_ID, "pm_generator_step: provided code " + std::to_string(v) +
                                                          " at batch " + std::to_string(b) + " stream " + std::to_string(k));
            }
    }
    bool run = false;  // a call where every row is at offset 0 runs no model step
    for (int b = 0; b < B; ++b)
        if (c->gen_s[b] > 0) run = true;
    cudaGraphExec_t fex = nullptr, dex = nullptr;
    if (run) {
        pm_status st = get_graph(c, c->frame_graphs, B, B >= 2 ? record_frame_tc : record_frame, &fex);
        if (st) return st;
        st = get_graph(c, c->dep_graphs, B, record_depformer, &dex);
        if (st) return st;
    }
    GenParams g;
    memset(&g, 0, sizeof g);
    g.st = c->st;
    g.ring = c->gen_ring;
    g.prov = c->gen_prov;
    g.off = c->gen_off;
    g.provided = provided ? reinterpret_cast<const int32_t*>(c->io_region + 64) : nullptr;
    g.in = c->gen_in;
    g.dep_tok = c->gen_tok;
    g.dep_sup = c->gen_sup;
    g.pos_save = c->gen_pos_save;
    g.sel_save = c->gen_sel_save;
    g.out = out;
    g.valid = out_valid;
    g.B = B;
    g.S = S;
    g.Q = Q;
    for (int k = 0; k < S; ++k) {
        g.delays[k] = f.delays[k];
        g.init[k] = (k == 0) ? f.init_text : f.init_audio;
        g.max_delay = std::max(g.max_delay, f.delays[k]);
    }
    g.ran = run ? 1 : 0;
    // the frame's I/O block, the provided codes where a frame's host IDs go
    uint8_t* host;
    cudaEvent_t ev;
    pm_status st = take_slot(c, &host, &ev);
    if (st) return st;
    FrameIO io;
    memset(&io, 0, sizeof io);
    io.ids = c->gen_in;
    io.logits = text_logits;
    io.hidden = hidden;
    io.direct = 1;
    memcpy(host, &io, sizeof io);
    size_t bytes = 64;
    if (provided) {
        memcpy(host + 64, provided, 4u * B * S);
        bytes += 4u * B * S;
    }
    PM_CUDA(cudaMemcpyAsync(c->io_region, host, bytes, cudaMemcpyHostToDevice, c->stream));
    PM_CUDA(cudaEventRecord(ev, c->stream));
    PM_CUDA(launch_gen(0, g, c->stream));
    if (run) {
        PM_CUDA(cudaGraphLaunch(fex, c->stream));
        PM_CUDA(launch_gen(1, g, c->stream));
        st = take_slot(c, &host, &ev);
        if (st) return st;
        DepIO dio;
        memset(&dio, 0, sizeof dio);
        dio.hidden = c->h;
        dio.text_tok = c->gen_tok;
        dio.supplied = c->gen_sup;
        dio.logits = depth_logits;
        memcpy(host, &dio, sizeof dio);
        PM_CUDA(cudaMemcpyAsync(c->dio_region, host, 64, cudaMemcpyHostToDevice, c->stream));
        PM_CUDA(cudaEventRecord(ev, c->stream));
        PM_CUDA(cudaGraphLaunch(dex, c->stream));
    }
    PM_CUDA(launch_gen(2, g, c->stream));
    for (int b = 0; b < B; ++b) c->gen_s[b] += 1;
    return PM_OK;
}

extern "C" pm_status pm_set_sampling(pm_ctx* c, float text_temperature, int text_top_k, float audio_temperature,
                                     int audio_top_k, unsigned long long seed) {
    if (!c) return PM_ERR_ARG;
    const bool ton = text_temperature > 0.0f && text_top_k > 1;
    const bool aon = audio_temperature > 0.0f && audio_top_k > 1;
    if ((ton && text_top_k > PM_SAMPLE_MAX_TOP_K) || (aon && audio_top_k > PM_SAMPLE_MAX_TOP_K))
        return fail(c, PM_ERR_ARG, "pm_set_sampling: top_k above 1024");
    if (!(text_temperature == text_temperature) || !(audio_temperature == audio_temperature))
        return fail(c, PM_ERR_ARG, "pm_set_sampling: temperature is NaN");
    PM_CUDA(cudaSetDevice(c->device));
    c->scfg_host.text_temperature = text_temperature;
    c->scfg_host.text_top_k = text_top_k;
    c->scfg_host.audio_temperature = audio_temperature;
    c->scfg_host.audio_top_k = audio_top_k;
    c->scfg_host.seed = seed;
    // pageable source: the copy is staged before the call returns, ordered on the stream
    PM_CUDA(cudaMemcpyAsync(c->scfg, &c->scfg_host, sizeof(SampleCfg), cudaMemcpyHostToDevice, c->stream));
    if (ton != c->text_smp || aon != c->audio_smp) {
        // the set of launches changes: drop the captured graphs (re-captured on next use)
        PM_CUDA(cudaStreamSynchronize(c->stream));
        for (auto& kv : c->frame_graphs) cudaGraphExecDestroy(kv.second);
        for (auto& kv : c->dep_graphs) cudaGraphExecDestroy(kv.second);
        for (auto& kv : c->prefill_graphs) cudaGraphExecDestroy(kv.second);
        c->frame_graphs.clear();
        c->dep_graphs.clear();
        c->prefill_graphs.clear();
        c->text_smp = ton;
        c->audio_smp = aon;
    }
    return PM_OK;
}

extern "C" pm_status pm_sample(pm_ctx* c, int B, const float* logits, int V, int ld, float temperature, int top_k,
                               unsigned long long seed, long long position, int substep, int32_t* tokens) {
    if (!c) return PM_ERR_ARG;
    if (B < 1 || V < 1 || ld < V) return fail(c, PM_ERR_ARG, "pm_sample: need B >= 1, V >= 1, ld >= V");
    if (!logits || !tokens) return fail(c, PM_ERR_ARG, "pm_sample: null pointer");
    if (!(temperature == temperature)) return fail(c, PM_ERR_ARG, "pm_sample: temperature is NaN");
    if (temperature > 0.0f && top_k > PM_SAMPLE_MAX_TOP_K) return fail(c, PM_ERR_ARG, "pm_sample: top_k above 1024");
    PM_CUDA(cudaSetDevice(c->device));
    if (!is_device_ptr(logits)) return fail(c, PM_ERR_ARG, "pm_sample: logits must be device memory");
    SampleParams sp;
    memset(&sp, 0, sizeof sp);
    sp.mode = SM_PLAIN;
    sp.logits = logits;
    sp.ld = ld;
    sp.V = V;
    sp.B = B;
    sp.temperature = temperature;
    sp.top_k = top_k;
    sp.seed = seed;
    sp.position = position;
    sp.substep = substep;
    sp.tokens = tokens;
    PM_CUDA(launch_sample(sp, c->stream, false));
    return PM_OK;
}

extern "C" pm_status pm_profile_frame(pm_ctx* c, int B, const int32_t* ids, float* text_logits, float* hidden,
                                      int32_t* text_token, float* kernel_ms, int32_t* kernel_kind, int max_launches,
                                      int* n_launches) {
    if (!c) return PM_ERR_ARG;
    if (!kernel_ms || !kernel_kind || !n_launches || max_launches < 0)
        return fail(c, PM_ERR_ARG, "pm_profile_frame: null output array");
    const pm_config& f = c->cfg;
    if (B < 1 || B > f.B_max || !ids) return fail(c, PM_ERR_ARG, "pm_profile_frame: bad B or ids");
    PM_CUDA(cudaSetDevice(c->device));
    const int S = f.n_streams;
    const bool dev_ids = is_device_ptr(ids);
    if (!dev_ids)
        for (int i = 0; i < B * S; ++i) {
            const int rows = (i % S == 0) ? f.text_in : f.audio_in;
            if (!(ids[i] == PM_ID_FEEDBACK || (ids[i] >= -1 && ids[i] < rows)))
                return fail(c, PM_ERR_INVALID_ID, "pm_profile_frame: invalid ID");
        }
    uint8_t* host;
    cudaEvent_t ev;
    pm_status st = take_slot(c, &host, &ev);
    if (st) return st;
    FrameIO io;
    memset(&io, 0, sizeof io);
    io.ids = dev_ids ? ids : reinterpret_cast<const int32_t*>(c->io_region + 64);
    io.logits = text_logits;
    io.hidden = hidden;
    io.token = text_token;
    memcpy(host, &io, sizeof io);
    size_t bytes = 64;
    if (!dev_ids) {
        memcpy(host + 64, ids, 4u * B * S);
        bytes += 4u * B * S;
    }
    PM_CUDA(cudaMemcpyAsync(c->io_region, host, bytes, cudaMemcpyHostToDevice, c->stream));
    PM_CUDA(cudaEventRecord(ev, c->stream));
    std::vector<cudaEvent_t> evs;
    std::vector<int> kinds;
    c->prof_ev = &evs;
    c->prof_kind = &kinds;
    st = (B >= 2 ? record_frame_tc : record_frame)(c, B, c->stream);
    c->prof_ev = nullptr;
    c->prof_kind = nullptr;
    cudaError_t e = cudaStreamSynchronize(c->stream);
    int n = 0;
    if (st == PM_OK && e == cudaSuccess) {
        for (size_t i = 1; i < evs.size() && n < max_launches; ++i, ++n) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, evs[i - 1], evs[i]);
            kernel_ms[n] = ms;
            kernel_kind[n] = kinds[i];
        }
    }
    for (cudaEvent_t x : evs) cudaEventDestroy(x);
    *n_launches = n;
    if (st) return st;
    if (e != cudaSuccess) return cuda_fail(c, e, "pm_profile_frame");
    return PM_OK;
}
