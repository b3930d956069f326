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

// The same GELU for results that are rounded to bf16: tanh from the hardware
// approximation (tanh.approx.f32, relative error about 2^-11 per the PTX ISA),
// below the bf16 rounding of the result (2^-9 relative); the error it adds to
// GELU(s) is at most |s| * 2^-12.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// The tanh argument is evaluated as s (k0 + k0 k1 s^2), one multiply fewer
// than k0 (s + k1 s^3); the two differ by fp32 rounding only.
__device__ __forceinline__ float gelu_tanh_bf16out(float s) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    const float k0k1 = 0.7978845608028654f * 0.044715f;
    const float hs = 0.5f * s;
    return fmaf(hs, tanh_hw(s * fmaf(k0k1, s * s, k0)), hs);
}

// Slope of the tanh-form GELU (the derivative of 0.5 s (1 + tanh(c (s + a s^3)))):
// 0.5 (1 + t) + 0.5 s (1 - t^2) c (1 + 3 a s^2). BF16OUT: the hardware tanh.
// For bf16 results the same expression is evaluated with fewer operations:
// u = s (c + ca s^2), g' = (0.5 + 0.5 s (1 - t^2)(c + 3ca s^2)) + 0.5 t (fp32
// rounding differences only, far below the bf16 rounding of the result).
template <bool BF16OUT>
__device__ __forceinline__ float gelu_tanh_slope(float s) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    const float a = 0.044715f;
    if constexpr (BF16OUT) {
        const float ca = 0.7978845608028654f * 0.044715f;
        const float s2 = s * s;
        const float t = tanh_hw(s * fmaf(ca, s2, c));
        const float r = (0.5f * s) * fmaf(-t, t, 1.0f) * fmaf(3.0f * ca, s2, c);
        return fmaf(0.5f, t, 0.5f + r);
    } else {
        const float u = c * (s + a * s * s * s);
        const float t = tanhf(u);
        return 0.5f * (1.0f + t) + 0.5f * s * (1.0f - t * t) * c * (1.0f + 3.0f * a * s * s);
    }
}

// Bias add and activation. BF16OUT: the result is rounded to bf16 next (the
// activation may use the hardware tanh).
template <bool GELU, bool BF16OUT = false>
__device__ __forceinline__ float epilogue(float acc, float b) {
    float s = acc + b;
    if constexpr (GELU) s = BF16OUT ? gelu_tanh_bf16out(s) : gelu_tanh(s);
    return s;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Two values rounded to nearest-even bf16 by one paired conversion, lo in the
// low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ---- programmatic dependent launch ----
// Wait until the grids this launch depends on have completed and their memory
// is visible (a no-op when launched without the programmatic attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the dependent grid to be scheduled.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

}  // namespace lin
