// pm_text_head_noalloc: the final RMSNorm + text head + greedy token of a frame, for
// callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA stream is being
// captured into a graph (allocation is not a capturable operation), real-time audio
// threads that must never block on the allocator (cudaMalloc may synchronise the
// device), and hosts that hand all device memory out of their own pool.  They cannot
// create a pm_ctx, whose set-up allocates its workspaces.  This entry point needs no
// context: the caller passes the inputs and the outputs, and the kernel's scratch (the
// packed argmax accumulator and CTA completion counter of each batch row, plus the small
// struct that carries the output pointers) lives in the file-scope device array below.
//
// The array is PM_NOALLOC_SCRATCH_BYTES large, which bounds the batch to
// PM_NOALLOC_MAX_B rows; every GPU that loads the library holds it until the process
// exits.  All calls share it and it keeps the last call's contents: the accumulators
// are cleared on the device at the start of every call, and calls that overlap on the
// GPU (different streams, no ordering between them) race on it.
#include <string.h>

#include <mutex>

#include "../../include/pm.h"
#include "pm_kernels.h"

namespace pm {
namespace {

constexpr int kMaxB = 64;
constexpr int kMaxDevices = 64;
// layout: [0, 64) FrameIO, [64, 128) status words, then per batch row: argmax key (8 B),
// completion counter, position and selected-token slots written by the shared epilogue
constexpr size_t kOffIo = 0;
constexpr size_t kOffStatus = 64;
constexpr size_t kOffAmax = 128;
constexpr size_t kOffCount = kOffAmax + 8 * kMaxB;
constexpr size_t kOffPos = kOffCount + 4 * kMaxB;
constexpr size_t kOffSel = kOffPos + 4 * kMaxB;
constexpr size_t kScratchBytes = kOffSel + 4 * (size_t)kMaxB * PM_MAX_STREAMS_DEV;

}  // namespace
}  // namespace pm

#define PM_NOALLOC_MAX_B pm::kMaxB
#define PM_NOALLOC_SCRATCH_BYTES 10240
static_assert(pm::kScratchBytes <= PM_NOALLOC_SCRATCH_BYTES, "scratch layout exceeds the array");
static_assert(sizeof(pm::FrameIO) <= pm::kOffStatus - pm::kOffIo, "FrameIO overruns its slot");
static_assert(pm::kOffStatus + 16 <= pm::kOffAmax, "status words overrun their slot");

// Device scratch of the no-allocation text head.  In host code this name is only a
// host-side stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PM_NOALLOC_SCRATCH_BYTES];

namespace pm {
namespace {

// per-device address of g_noalloc_scratch, resolved once with that device current
unsigned char* g_scratch_dev[kMaxDevices] = {};
std::mutex g_setup_mu;

// Copy the call's outcome out of the shared scratch: PM_OK, or PM_ERR_TIMEOUT when a bounded
// wait of the head ran out (its outputs are then incomplete).
__global__ void k_noalloc_end(const unsigned char* scratch, int32_t* status) {
    const uint32_t st = *reinterpret_cast<const volatile uint32_t*>(scratch + kOffStatus);
    *status = (st & PM_DEV_ERR_TIMEOUT) ? (int32_t)PM_ERR_TIMEOUT : (int32_t)PM_OK;
}

// device, managed or host-mapped memory with the given alignment (null allowed when `opt`)
bool gpu_ptr_ok(const void* p, uintptr_t align, bool opt) {
    if (!p) return opt;
    if ((uintptr_t)p & (align - 1)) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
}

// Publish the output pointers and clear the accumulators the head kernel starts from.
__global__ void k_noalloc_begin(unsigned char* scratch, int B, float* logits, float* hidden, int32_t* token) {
    FrameIO* io = reinterpret_cast<FrameIO*>(scratch + kOffIo);
    uint32_t* status = reinterpret_cast<uint32_t*>(scratch + kOffStatus);
    unsigned long long* amax = reinterpret_cast<unsigned long long*>(scratch + kOffAmax);
    uint32_t* count = reinterpret_cast<uint32_t*>(scratch + kOffCount);
    const int t = threadIdx.x;
    if (t == 0) {
        io->ids = nullptr;
        io->logits = logits;
        io->hidden = hidden;
        io->token = token;
        status[0] = 0u;
        status[1] = 0u;  // not aborted
    }
    if (t < B) {
        amax[t] = 0ull;
        count[t] = 0u;
    }
}

pm_status setup_device(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return PM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return PM_ERR_CUDA;
        }
        if (gemv_prepare() != cudaSuccess || cudaMemset(p, 0, PM_NOALLOC_SCRATCH_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return PM_ERR_CUDA;
        }
        g_scratch_dev[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_dev[dev];
    return PM_OK;
}

}  // namespace
}  // namespace pm

extern "C" pm_status pm_text_head_noalloc(int B, int D, int V, const float* residual, const void* out_norm,
                                          const void* text_linear, float eps, float* hidden, float* logits,
                                          int32_t* token, int32_t* status, void* cuda_stream) {
    using namespace pm;
    if (B < 1 || B > PM_NOALLOC_MAX_B) return PM_ERR_UNSUPPORTED;  // beyond the static scratch
    if (!residual || !out_norm || !text_linear || V < 1 || !(eps > 0.f)) return PM_ERR_ARG;
    // inputs are read with 16-byte loads; hidden is written with 16-byte stores, logits,
    // the token and the status word with 4-byte stores
    if (!gpu_ptr_ok(residual, 16, false) || !gpu_ptr_ok(out_norm, 16, false) || !gpu_ptr_ok(text_linear, 16, false) ||
        !gpu_ptr_ok(hidden, 16, true) || !gpu_ptr_ok(logits, 4, true) || !gpu_ptr_ok(token, 4, true) ||
        !gpu_ptr_ok(status, 4, true))
        return PM_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PM_ERR_CUDA;
    }
    int num_sms = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return PM_ERR_CUDA;
    }
    GemvParams p;
    memset(&p, 0, sizeof p);
    p.W = reinterpret_cast<const uint16_t*>(text_linear);
    p.K = D;
    p.n_units = V;
    p.B = B;
    if (!plan_gemv(p, 1, num_sms)) return PM_ERR_UNSUPPORTED;  // D must be a multiple of 256
    unsigned char* scratch = nullptr;
    pm_status st = setup_device(dev, &scratch);
    if (st != PM_OK) return st;
    p.x = residual;
    p.x_stride = D;
    p.alpha = reinterpret_cast<const uint16_t*>(out_norm);
    p.eps = eps;
    p.y_stride = V;
    p.io = reinterpret_cast<const FrameIO*>(scratch + kOffIo);
    p.st.status = reinterpret_cast<uint32_t*>(scratch + kOffStatus);
    p.st.amax = reinterpret_cast<unsigned long long*>(scratch + kOffAmax);
    p.st.head_count = reinterpret_cast<uint32_t*>(scratch + kOffCount);
    p.st.pos = reinterpret_cast<int32_t*>(scratch + kOffPos);
    p.st.sel = reinterpret_cast<int32_t*>(scratch + kOffSel);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(cuda_stream);
    k_noalloc_begin<<<1, kMaxB, 0, s>>>(scratch, B, logits, hidden, token);
    if (cudaGetLastError() != cudaSuccess) return PM_ERR_CUDA;
    if (launch_gemv(PRO_RMSNORM, E_HEAD, U_ROW, p, s, false) != cudaSuccess) {
        cudaGetLastError();
        return PM_ERR_CUDA;
    }
    if (status) {
        k_noalloc_end<<<1, 1, 0, s>>>(scratch, status);
        if (cudaGetLastError() != cudaSuccess) return PM_ERR_CUDA;
    }
    return PM_OK;
}
