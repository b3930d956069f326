// A context-free fp32 entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the moment they run a layer:
// - a serving runtime that reserved all device memory for its own pool at
//   start-up and treats any other allocation as a failure;
// - a latency-critical path where an allocation could block on the device
//   or fail under memory pressure;
// - a plug-in that is handed device pointers but no allocator.
// lin_forward_fp32_static runs the same fp32 kernels as lin_forward (the
// FFMA kernel with the dispatch table's split-K choice, or the GEMV for a few
// rows, which needs no scratch). The split's scratch (tile
// counters, then partial sums) lives in the fixed device array below. Every
// GPU that loads this library holds that array until the process exits.
#include <cuda.h>

#include <mutex>

#include "internal.h"

namespace lin {
namespace {

// Scratch of lin_forward_fp32_static, laid out as a context workspace:
// tile counters first, split-K partial sums after.
static __device__ __align__(256) unsigned char g_static_scratch[LIN_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
// Device address of g_static_scratch per device ordinal, with the context it
// was looked up in: a context created anew (after cudaDeviceReset) loads the
// module again, so the address is looked up again.
struct ScratchAddr {
    CUcontext ctx;
    void* addr;
};
ScratchAddr g_scratch_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (CtxGetCurrentFn) nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(ptr);
    }();
    return fn;
}

// Device address of the scratch array on the current device, looked up with
// that device current. Host code must not use the symbol's host-side name as
// an address.
int scratch_on_current_device(void** out, int* device) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return LIN_ERR_UNSUPPORTED;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return LIN_ERR_CUDA;
    if (!ctx) {
        // No context on this thread yet: cudaSetDevice creates the device's
        // primary context and makes it current.
        if (cudaSetDevice(dev) != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return LIN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& e = g_scratch_addr[dev];
    if (!e.addr || e.ctx != ctx) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr) {
            cudaGetLastError();
            return LIN_ERR_CUDA;
        }
        e.ctx = ctx;
        e.addr = addr;
    }
    *out = e.addr;
    *device = dev;
    return LIN_OK;
}

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + bn && pb < pa + an;
}

}  // namespace
}  // namespace lin

extern "C" int lin_forward_fp32_static(int M, int N, int K, const float* X, const float* W, const float* bias,
                                       float* Y, int epilogue, void* stream) {
    using namespace lin;
    if (M < 0 || N < 0 || K < 0 || (epilogue != LIN_EPI_NONE && epilogue != LIN_EPI_GELU_TANH)) return LIN_ERR_ARG;
    if (M == 0 || N == 0) return LIN_OK;
    if (!Y || (K > 0 && (!X || !W))) return LIN_ERR_ARG;
    const size_t ybytes = (size_t)M * N * sizeof(float);
    if (ranges_overlap(Y, ybytes, X, (size_t)M * K * sizeof(float)) ||
        ranges_overlap(Y, ybytes, W, (size_t)N * K * sizeof(float)) ||
        ranges_overlap(Y, ybytes, bias, bias ? (size_t)N * sizeof(float) : 0))
        return LIN_ERR_ARG;
    if (K > 0 && ((((uintptr_t)X | (uintptr_t)W) % 16) != 0 || ((size_t)K * sizeof(float)) % 16 != 0))
        return LIN_ERR_ALIGN;
    if (((uintptr_t)Y % 4) != 0 || ((uintptr_t)bias % 4) != 0) return LIN_ERR_ALIGN;

    void* scratch = nullptr;
    int dev = -1;
    int rc = scratch_on_current_device(&scratch, &dev);
    if (rc != LIN_OK) return rc;
    int sm = 0;
    if (cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LIN_ERR_CUDA;

    // The table's plan for this shape, as if scratch were unlimited: the same
    // split as lin_forward, so the same bits. A shape whose split needs more
    // than the fixed array is refused, not shrunk (the split fills the SMs, so
    // this happens only on GPUs with far more SMs than 152).
    lin_plan plan;
    rc = lin_plan_query(sm, M, N, K, LIN_PREC_FP32, epilogue, (size_t)1 << 62, &plan);
    if (rc != LIN_OK) return rc;
    if (plan.workspace_bytes > (long long)LIN_STATIC_SCRATCH_BYTES) return LIN_ERR_WORKSPACE;

    Problem p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.X = X;
    p.W = W;
    p.bias = bias;
    p.Y = Y;
    p.epilogue = epilogue;
    p.precision = LIN_PREC_FP32;
    p.stream = static_cast<cudaStream_t>(stream);
    p.workspace = scratch;
    p.workspace_bytes = LIN_STATIC_SCRATCH_BYTES;
    p.dev_status = nullptr;
    p.sm_count = sm;
    p.early_start = false;
    p.early_x = false;
    if (plan.kernel == LIN_KERNEL_FILL) return launch_fill(p);
    if (plan.kernel == LIN_KERNEL_GEMV) return launch_gemv(p, plan);  // no scratch
    if (plan.kernel != LIN_KERNEL_FFMA) return LIN_ERR_UNSUPPORTED;
    if (plan.splits > 1) {
        // The array keeps the previous call's contents: zero the counters this
        // launch uses (the partial sums are fully written before they are read).
        const size_t counter_bytes = (size_t)plan.grid_x * plan.grid_y * sizeof(unsigned);
        if (cudaMemsetAsync(splitk_counters(scratch), 0, counter_bytes, p.stream) != cudaSuccess) return LIN_ERR_CUDA;
    }
    return launch_ffma(p, plan);
}
