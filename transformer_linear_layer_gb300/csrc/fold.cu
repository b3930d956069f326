// LayerNorm fold ("Optimizing a GPT-2-class transformer on a GPU", Act II,
// rung 10): a layernorm's scale and shift feed only the linear map after it,
// so they move into that map's weight and bias once, offline, in double:
//   W LN(x) + b = (W diag(gamma)) xhat + (W beta + b),  xhat = (x - mean) / sqrt(var + eps),
//   Wf[n][k] = W[n][k] gamma[k],   bf[n] = b[n] + sum_k W[n][k] beta[k].
// Products of two fp32 values are exact in double; the sum runs in ascending
// k, and each output is rounded once (to nearest even) to its storage type.
#include <cuda_bf16.h>

#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

// bf[n] in double, one thread per row (the fold runs once per weight; the
// order of the sum is the definition's).
__global__ void __launch_bounds__(256) fold_bias_kernel(int N, int K, const float* W, const float* bias,
                                                        const float* beta, float* bias_out) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    double s = bias ? (double)bias[n] : 0.0;
    if (beta) {
        const float* w = W + (size_t)n * K;
        for (int k = 0; k < K; ++k) s = __dadd_rn(s, __dmul_rn((double)w[k], (double)beta[k]));
    }
    bias_out[n] = __double2float_rn(s);
}

template <bool BF16>
__global__ void __launch_bounds__(256) fold_weight_kernel(long long count, int K, const float* W, const float* gamma,
                                                          void* W_out) {
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += step) {
        const double v = __dmul_rn((double)W[i], (double)gamma[i % K]);
        if constexpr (BF16) {
            const __nv_bfloat16 h = __double2bfloat16(v);
            static_cast<__nv_bfloat16*>(W_out)[i] = h;
        } else {
            static_cast<float*>(W_out)[i] = __double2float_rn(v);
        }
    }
}

}  // namespace

int launch_fold_layernorm(int N, int K, const float* W, const float* bias, const float* gamma, const float* beta,
                          void* W_out, float* bias_out, bool bf16, int sm_count, cudaStream_t st) {
    // The bias first: W_out may be W (in place), and the bias reads the unfolded W.
    fold_bias_kernel<<<(N + 255) / 256, 256, 0, st>>>(N, K, W, bias, beta, bias_out);
    if (cudaGetLastError() != cudaSuccess) return LIN_ERR_CUDA;
    const long long count = (long long)N * K;
    long long grid = (count + 255) / 256;
    if (grid > 8LL * sm_count) grid = 8LL * sm_count;
    if (grid < 1) grid = 1;
    if (bf16)
        fold_weight_kernel<true><<<(int)grid, 256, 0, st>>>(count, K, W, gamma, W_out);
    else
        fold_weight_kernel<false><<<(int)grid, 256, 0, st>>>(count, K, W, gamma, W_out);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace lin
