// Throughput probe of the exact-fp32 FMA pipe, the roofline of the FFMA
// kernels. The pages quote an fp32 peak from the unit count and the clock
// ("Writing a CUDA matmul that catches cuBLAS": 11.1 TF/s at 1200 MHz on their
// part); the datasheet figure on this device (152 SMs x 128 lanes x 2 FLOP x
// clock) assumes every lane issues an FFMA every cycle. This kernel measures
// what the FMA pipe actually sustains: every thread runs independent fmaf
// chains (enough of them to cover the pipe latency), nothing else.
#include "internal.h"

namespace lin {
namespace {

constexpr int kProbeChains = 8;
constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 4;

__global__ void __launch_bounds__(kProbeThreads)
ffma_probe_kernel(int iters, float b, float c, float* out) {
    float a[kProbeChains];
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) a[j] = (float)(threadIdx.x + j);
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
#pragma unroll
            for (int j = 0; j < kProbeChains; ++j) a[j] = fmaf(a[j], b, c);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) s += a[j];
    // Never true for the arguments the host passes (b < 1, c tiny): the chains
    // stay live without a store per thread.
    if (s == -1.0f) out[0] = s;
}

}  // namespace

int launch_ffma_probe(int sm_count, int iters, float* out, cudaStream_t st, double* flops) {
    const int grid = sm_count * kProbeCtasPerSm;
    if (flops) *flops = 2.0 * kProbeChains * 16.0 * (double)iters * (double)grid * kProbeThreads;
    ffma_probe_kernel<<<grid, kProbeThreads, 0, st>>>(iters, 0.999999f, 1e-7f, out);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace lin
