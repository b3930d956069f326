// Device helpers shared by the kernels: the epilogue arithmetic and bf16 I/O.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lin {

// tanh-form GELU in fp32 with the accurate tanhf. The constants are those of
// the tanh approximation in Hendrycks & Gimpel, "Gaussian Error Linear Units";
// the pages evaluate it with tanhf in the GEMM's store ("Writing a CUDA matmul
// that catches cuBLAS", "The residual and GELU go the same way").
__device__ __forceinline__ float gelu_tanh(float s) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    const float k1 = 0.044715f;
    return 0.5f * s * (1.0f + tanhf(k0 * (s + k1 * s * s * s)));
}

template <bool GELU>
__device__ __forceinline__ float epilogue(float acc, float b) {
    float s = acc + b;
    if constexpr (GELU) s = gelu_tanh(s);
    return s;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}

}  // namespace lin
