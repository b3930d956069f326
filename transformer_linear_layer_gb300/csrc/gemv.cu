// Exact-fp32 linear layer for a handful of rows (M <= 8): the one-row sites.
//
// "Optimizing a GPT-2-class transformer on a GPU", Act II: only the final
// token's logits are needed, and "a dedicated GEMV takes the one-row sites"
// of the routing table. With M <= 8 every weight value feeds at most 8
// products, so the layer is a single pass over W and its time is W's bytes
// over the HBM bandwidth; tiles of 64 or 128 rows would multiply 56-127 rows
// of padding.
//
// * X (M x K fp32) is copied into shared memory once per CTA, padded with
//   zero rows to MR = 1, 2, 4 or 8 (the instantiated row count).
// * Each warp takes one row n of W at a time and reads it whole with 128-bit
//   loads, lane l taking the float4s l, l + 32, ...: consecutive lanes read
//   consecutive 16 bytes, and U = 8 loads per lane are in flight before the
//   first is used (with several CTAs per SM, ~100 KB of W in flight per SM).
// * Lane l accumulates its k's in ascending order into M fp32 sums; the 32
//   lanes' sums are added by a fixed butterfly (xor 16, 8, 4, 2, 1), so the
//   result is bitwise repeatable. Lane 0 adds the bias, applies the accurate
//   tanh-GELU and stores the M outputs of column n.
// * Programmatic dependent launch: W streams before griddepcontrol.wait when
//   the caller allows an early start (W is not the previous call's output), X
//   only when it is not that output either; bias and Y after the wait.
#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

struct GemvArgs {
    int M, N, K;
    const float* X;
    const float* W;
    const float* bias;
    float* Y;
    int early_x;  // X may be read before the dependency wait
};

constexpr int kGemvThreads = 256;
constexpr int kGemvUnroll = 8;  // float4 loads of W in flight per lane

template <int MR, bool GELU>
__global__ void __launch_bounds__(kGemvThreads)
gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) float sx[];  // MR x K
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K4 = a.K >> 2;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (!a.early_x) pdl_wait();
    {
        const float4* x4 = reinterpret_cast<const float4*>(a.X);
        float4* s4 = reinterpret_cast<float4*>(sx);
        // The M rows of X, then zeros up to the padded MR rows.
        for (int i = threadIdx.x; i < MR * K4; i += kGemvThreads)
            s4[i] = i < a.M * K4 ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    const float4* sx4 = reinterpret_cast<const float4*>(sx);

    const int warps_total = gridDim.x * (kGemvThreads / 32);
    bool waited = !a.early_x;
    for (int n = blockIdx.x * (kGemvThreads / 32) + warp; n < a.N; n += warps_total) {
        const float4* w4 = reinterpret_cast<const float4*>(a.W + (size_t)n * a.K);
        float acc[MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[m] = 0.f;
        for (int k0 = lane; k0 < K4; k0 += 32 * kGemvUnroll) {
            float4 wv[kGemvUnroll];
#pragma unroll
            for (int u = 0; u < kGemvUnroll; ++u) {
                const int k = k0 + 32 * u;
                wv[u] = k < K4 ? __ldcs(w4 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kGemvUnroll; ++u) {
                const int k = k0 + 32 * u;
                if (k < K4) {
#pragma unroll
                    for (int m = 0; m < MR; ++m) {
                        const float4 xv = sx4[m * K4 + k];
                        acc[m] = fmaf(wv[u].x, xv.x, acc[m]);
                        acc[m] = fmaf(wv[u].y, xv.y, acc[m]);
                        acc[m] = fmaf(wv[u].z, xv.z, acc[m]);
                        acc[m] = fmaf(wv[u].w, xv.w, acc[m]);
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if (!waited) {
            pdl_wait();  // bias and Y only after the previous kernel has finished
            waited = true;
        }
        if (lane == 0) {
            const float b = a.bias ? __ldg(a.bias + n) : 0.f;
#pragma unroll
            for (int m = 0; m < MR; ++m)
                if (m < a.M) a.Y[(size_t)m * a.N + n] = epilogue<GELU>(acc[m], b);
        }
    }
}

template <int MR, bool GELU>
int launch_mr(const GemvArgs& a, int grid, bool early, cudaStream_t st) {
    auto kern = gemv_kernel<MR, GELU>;
    const size_t smem = (size_t)MR * a.K * sizeof(float);
    static unsigned long long attr_set = 0;  // one attribute call per instantiation and device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIN_ERR_CUDA;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem) != cudaSuccess)
            return LIN_ERR_CUDA;
        attr_set |= bit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = early ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

template <bool GELU>
int launch_gelu(const GemvArgs& a, int rows, int grid, bool early, cudaStream_t st) {
    switch (rows) {
        case 1: return launch_mr<1, GELU>(a, grid, early, st);
        case 2: return launch_mr<2, GELU>(a, grid, early, st);
        case 4: return launch_mr<4, GELU>(a, grid, early, st);
        case 8: return launch_mr<8, GELU>(a, grid, early, st);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_gemv(const Problem& p, const lin_plan& plan) {
    if (p.M < 1 || p.M > kGemvMaxRows || (size_t)plan.bm * p.K * sizeof(float) > (size_t)kGemvMaxSmem)
        return LIN_ERR_UNSUPPORTED;
    GemvArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.X = static_cast<const float*>(p.X);
    a.W = static_cast<const float*>(p.W);
    a.bias = p.bias;
    a.Y = static_cast<float*>(p.Y);
    a.early_x = (p.early_start && p.early_x) ? 1 : 0;
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    return gelu ? launch_gelu<true>(a, plan.bm, plan.grid_x, p.early_start, p.stream)
                : launch_gelu<false>(a, plan.bm, plan.grid_x, p.early_start, p.stream);
}

}  // namespace lin
