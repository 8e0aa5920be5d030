// Shared device helpers for the sm_103a decode-step kernels: bf16 unpacking, warp
// reductions, mbarrier / bulk-copy / programmatic-dependent-launch PTX wrappers, and the
// device-side state the kernels share.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#ifndef PM_SPIN_LIMIT
// Upper bound on mbarrier try_wait polls before a wait is declared timed out.  Each poll
// may suspend the thread for a short hardware-defined time, so this is well under a
// second of wall time on a healthy GPU and ends every wait.
#define PM_SPIN_LIMIT (1u << 22)
#endif

// streams a frame may carry (text + audio codebooks)
#define PM_MAX_STREAMS_DEV 32
// largest batch a context serves
#define PM_MAX_B_DEV 64

// status bits written by kernels (read back by pm_device_status)
#define PM_DEV_ERR_INVALID_ID 1u
#define PM_DEV_ERR_TIMEOUT 2u

namespace pm {

// ---------------------------------------------------------------------------------
// device-resident per-context state (one allocation, carved on the host)
// ---------------------------------------------------------------------------------
struct DevState {
    int32_t* pos;         // [B_max] absolute position of the next frame
    int32_t* first_pos;   // [B_max] position of the first frame since reset / position set
    int32_t* ring;        // [B_max][4][PM_MAX_STREAMS] resolved IDs of frame p at slot p & 3
    int32_t* sel;         // [B_max][PM_MAX_STREAMS] tokens selected on the stream's last frame (-2 none)
    unsigned long long* amax;  // [B_max] packed (value, index) argmax accumulator for the text head
    uint32_t* head_count;      // [B_max] CTA completion counter of the text head
    uint32_t* status;          // [0] sticky error bits, [1] abort flag of the frame in flight
    unsigned long long* dep_amax;  // [B_max] depth-head argmax accumulator
    uint32_t* dep_count;           // [B_max] depth-head CTA completion counter
    int32_t* dep_codes;            // [B_max][dep_steps] codes selected in the frame in flight
    int32_t* dep_tok;              // [B_max] text token the depformer conditions on
    int32_t* dep_sup;              // [B_max][dep_steps] validated supplied codes (-1 = greedy)
    const uint32_t* wait_budget;   // [1] poll budget of the waits that honour it (PM_SPIN_LIMIT unless lowered)
};

// Sampling settings of a context, device-resident so that a captured graph follows
// pm_set_sampling without re-capture (temperature <= 0 or top_k <= 1: greedy).
struct SampleCfg {
    float text_temperature;
    int text_top_k;
    float audio_temperature;
    int audio_top_k;
    unsigned long long seed;
};

// Pointers the caller supplies per call, read by the kernels from device memory so that a
// captured graph serves every call.
struct FrameIO {
    const int32_t* ids;   // [B][n_streams] (a prefill: [T][n_streams], frames of one stream)
    float* logits;        // [B][text_out] or null (a prefill: its last frame's, [1][text_out])
    float* hidden;        // [B][D] or null (a prefill: its last frame's)
    int32_t* token;       // [B] or null (a prefill: its last frame's)
    int32_t seq_stream;   // a prefill: the stream whose frames the rows are
    int32_t direct;       // 1: ids are the model's inputs as given (the generator's input column,
                          // delays already applied): no delay assembly, delay ring untouched
};

struct DepIO {
    const float* hidden;      // [B][D]
    const int32_t* text_tok;  // [B] or null (use the context's last selection)
    const int32_t* supplied;  // [B][Q] or null (all greedy)
    float* logits;            // [B][Q][card] or null
    int32_t* codes;           // [B][Q] or null
};

// ---------------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// round-to-nearest-even fp32 -> bf16 bits (finite inputs)
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// bf16 pair (hi, lo) with hi + lo = f to about 16 significant bits: hi = RNE(f), lo = RNE(f - hi)
__device__ __forceinline__ uint16_t bf16_lo_part(float f, uint16_t hi) {
    return f32_to_bf16_rne(f - __uint_as_float((uint32_t)hi << 16));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float dot8(const uint4 w, const float* x) {
    float a = bf16lo(w.x) * x[0];
    a = fmaf(bf16hi(w.x), x[1], a);
    a = fmaf(bf16lo(w.y), x[2], a);
    a = fmaf(bf16hi(w.y), x[3], a);
    a = fmaf(bf16lo(w.z), x[4], a);
    a = fmaf(bf16hi(w.z), x[5], a);
    a = fmaf(bf16lo(w.w), x[6], a);
    a = fmaf(bf16hi(w.w), x[7], a);
    return a;
}

// order-preserving map of a float to uint32 (larger float -> larger key)
__device__ __forceinline__ uint32_t float_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// packed argmax key: larger value wins, then the lower index
__device__ __forceinline__ unsigned long long pack_argmax(float v, uint32_t idx) {
    return ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t unpack_argmax_index(unsigned long long k) {
    return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

// ---------------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------------
// mbarrier + bulk copy (TMA engine, 1-D)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase of an mbarrier; false when the poll budget ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < PM_SPIN_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Same with a budget read at run time (a budget of 0 gives up without polling).
__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// The context's wait budget (PM_SPIN_LIMIT where a kernel runs without a context word).
__device__ __forceinline__ uint32_t wait_budget(const DevState& st) {
    return st.wait_budget ? *(const volatile uint32_t*)st.wait_budget : (uint32_t)PM_SPIN_LIMIT;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// global -> shared bulk copy completing on `bar`; dst, src 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

// A bounded wait ran out: record it and raise the frame's abort flag, so the kernels that
// follow in the frame skip their writes and the stream's position does not advance.
__device__ __forceinline__ void timeout_abort(const DevState& st) {
    set_status(st.status, PM_DEV_ERR_TIMEOUT);
    atomicExch(&st.status[1], 1u);
}

}  // namespace pm
