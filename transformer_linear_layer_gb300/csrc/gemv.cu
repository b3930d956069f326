// Linear layer for a handful of rows (fp32 / tf32 M <= 8, bf16 M <= 4): the
// one-row sites.
//
// "Optimizing a GPT-2-class transformer on a GPU", Act II: only the final
// token's logits are needed, and the routing table sends the one-row sites
// to a GEMV of their own. With M <= 8 every weight value feeds at most 8
// products, so the layer is a single pass over W and its time is W's bytes
// over the HBM bandwidth; tiles of 64 or 128 rows would multiply 56-127 rows
// of padding.
//
// * X (M x K fp32) is copied into shared memory once per CTA, padded with
//   zero rows to MR = 1, 2, 4 or 8 (the instantiated row count).
// * Each warp takes RPW consecutive rows of W at a time and reads them with
//   16-byte loads, lane l taking the pieces l, l + 32, ... of each row:
//   consecutive lanes read consecutive 16 bytes, and 8 loads per lane are in
//   flight before the first is used (RPW = 2 or 4 when rows are short, so
//   that short rows still fill the 8 slots).
// * Lane l accumulates its k's in ascending order into M fp32 sums; the 32
//   lanes' sums are added by a fixed butterfly (xor 16, 8, 4, 2, 1), so the
//   result is bitwise repeatable. Lane 0 adds the bias, applies the accurate
//   tanh-GELU and stores the M outputs of column n.
// * bf16 (M <= 4): X is widened to fp32 in shared memory, each 16-byte load
//   of W carries 8 values, bf16 x bf16 products are exact in fp32 and the
//   sums are fp32 as on the tensor cores; the result is rounded to bf16 (the
//   GELU then uses the hardware tanh). Up to 4 rows run here through explicit
//   plans; the built-in table sends bf16 here for one row only (measured: from
//   2 rows on the skinny tensor-core kernel streams W faster).
// * Programmatic dependent launch: when the caller allows X to be read early
//   (early start level 2) and X is not the previous call's output, X and then
//   W are read before griddepcontrol.wait; otherwise the kernel waits first.
//   Bias and Y only after the wait.
#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

struct GemvArgs {
    int M, N, K;
    const void* X;     // fp32 or bf16
    const void* W;     // fp32 or bf16
    const float* bias;
    void* Y;           // fp32 or bf16
    const void* R;     // residual added after the activation (M x N in Y's type, may be Y), or null
    int early_x;       // X may be read before the dependency wait
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr int kGemvThreads = 256;
constexpr int kGemvUnroll = 8;  // float4 loads of W in flight per lane

template <int MR, int RPW, bool GELU, bool BF16>
__global__ void __launch_bounds__(kGemvThreads)
gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) float sx[];  // MR x K, fp32
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K4 = a.K >> 2;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (!a.early_x) pdl_wait();
    // The M rows of X (widened to fp32), then zeros up to the padded MR rows.
    if constexpr (BF16) {
        const uint2* x4 = reinterpret_cast<const uint2*>(a.X);  // 4 bf16
        float4* s4 = reinterpret_cast<float4*>(sx);
        for (int i = threadIdx.x; i < MR * K4; i += kGemvThreads) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < a.M * K4) {
                const uint2 q = __ldg(x4 + i);
                v = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
            }
            s4[i] = v;
        }
    } else {
        const float4* x4 = reinterpret_cast<const float4*>(a.X);
        float4* s4 = reinterpret_cast<float4*>(sx);
        for (int i = threadIdx.x; i < MR * K4; i += kGemvThreads)
            s4[i] = i < a.M * K4 ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    const float4* sx4 = reinterpret_cast<const float4*>(sx);
    // 16-byte loads of W: 4 fp32 or 8 bf16 values.
    constexpr int VPL = BF16 ? 8 : 4;
    const int KV = a.K / VPL;

    const int warps_total = gridDim.x * (kGemvThreads / 32);
    constexpr int UPR = kGemvUnroll / RPW;  // load slots per row and lane
    bool waited = !a.early_x;
    for (int n0 = (blockIdx.x * (kGemvThreads / 32) + warp) * RPW; n0 < a.N; n0 += warps_total * RPW) {
        float acc[RPW][MR];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[r][m] = 0.f;
        for (int k0 = lane; k0 < KV; k0 += 32 * UPR) {
            uint4 wv[RPW][UPR];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int n = n0 + r;
                const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.W) +
                                                                   (size_t)n * a.K * (BF16 ? 2 : 4));
#pragma unroll
                for (int u = 0; u < UPR; ++u) {
                    const int k = k0 + 32 * u;
                    wv[r][u] = (n < a.N && k < KV) ? __ldcs(wrow + k) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
#pragma unroll
                for (int u = 0; u < UPR; ++u) {
                    const int k = k0 + 32 * u;
                    if (k < KV) {
                        if constexpr (BF16) {
                            const uint4 q = wv[r][u];
                            const float w0 = bf16_lo(q.x), w1 = bf16_hi(q.x), w2 = bf16_lo(q.y), w3 = bf16_hi(q.y),
                                        w4 = bf16_lo(q.z), w5 = bf16_hi(q.z), w6 = bf16_lo(q.w), w7 = bf16_hi(q.w);
#pragma unroll
                            for (int m = 0; m < MR; ++m) {
                                const float4 xa = sx4[m * K4 + 2 * k], xb = sx4[m * K4 + 2 * k + 1];
                                float t = acc[r][m];
                                t = fmaf(w0, xa.x, t);
                                t = fmaf(w1, xa.y, t);
                                t = fmaf(w2, xa.z, t);
                                t = fmaf(w3, xa.w, t);
                                t = fmaf(w4, xb.x, t);
                                t = fmaf(w5, xb.y, t);
                                t = fmaf(w6, xb.z, t);
                                acc[r][m] = fmaf(w7, xb.w, t);
                            }
                        } else {
                            const uint4 q = wv[r][u];
#pragma unroll
                            for (int m = 0; m < MR; ++m) {
                                const float4 xv = sx4[m * K4 + k];
                                float t = acc[r][m];
                                t = fmaf(__uint_as_float(q.x), xv.x, t);
                                t = fmaf(__uint_as_float(q.y), xv.y, t);
                                t = fmaf(__uint_as_float(q.z), xv.z, t);
                                acc[r][m] = fmaf(__uint_as_float(q.w), xv.w, t);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int m = 0; m < MR; ++m)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
        if (!waited) {
            pdl_wait();  // bias and Y only after the previous kernel has finished
            waited = true;
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int n = n0 + r;
                if (n >= a.N) break;
                const float b = a.bias ? __ldg(a.bias + n) : 0.f;
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    if (m < a.M) {
                        const size_t i = (size_t)m * a.N + n;
                        if constexpr (BF16) {
                            const float res = a.R ? bf16_bits_to_f32(static_cast<const uint16_t*>(a.R)[i]) : 0.f;
                            static_cast<uint16_t*>(a.Y)[i] = f32_to_bf16_bits(epilogue<GELU, true>(acc[r][m], b) + res);
                        } else {
                            const float res = a.R ? static_cast<const float*>(a.R)[i] : 0.f;
                            static_cast<float*>(a.Y)[i] = epilogue<GELU>(acc[r][m], b) + res;
                        }
                    }
                }
            }
        }
    }
}

template <int MR, int RPW, bool GELU, bool BF16>
int launch_mr(const GemvArgs& a, int grid, bool early, cudaStream_t st) {
    auto kern = gemv_kernel<MR, RPW, GELU, BF16>;
    const size_t smem = (size_t)MR * a.K * sizeof(float);
    static std::atomic<unsigned long long> attr_set{0};  // per instantiation: one bit per device
    if (ensure_smem_attr(attr_set, kern, kGemvMaxSmem) != LIN_OK) return LIN_ERR_CUDA;
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

template <int RPW, bool GELU, bool BF16>
int launch_rows(const GemvArgs& a, int rows, int grid, bool early, cudaStream_t st) {
    switch (rows) {
        case 1: return launch_mr<1, RPW, GELU, BF16>(a, grid, early, st);
        case 2: return launch_mr<2, RPW, GELU, BF16>(a, grid, early, st);
        case 4: return launch_mr<4, RPW, GELU, BF16>(a, grid, early, st);
        case 8: return BF16 ? LIN_ERR_UNSUPPORTED : launch_mr<8, RPW, GELU, false>(a, grid, early, st);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

// Rows per warp pass: enough short rows to fill the 8 load slots of a lane.
template <bool GELU, bool BF16>
int launch_rpw(const GemvArgs& a, int rows, int grid, bool early, cudaStream_t st) {
    const int kv = a.K / (BF16 ? 8 : 4);
    int rpw = 1;
    while (rpw < 4 && kv * rpw * 2 <= 32 * kGemvUnroll) rpw *= 2;
    switch (rpw) {
        case 1: return launch_rows<1, GELU, BF16>(a, rows, grid, early, st);
        case 2: return launch_rows<2, GELU, BF16>(a, rows, grid, early, st);
        default: return launch_rows<4, GELU, BF16>(a, rows, grid, early, st);
    }
}

}  // namespace

int launch_gemv(const Problem& p, const lin_plan& plan) {
    const bool bf16 = p.precision == LIN_PREC_BF16;
    if (p.M < 1 || p.M > (bf16 ? kGemvMaxRowsBf16 : kGemvMaxRows) ||
        (size_t)plan.bm * p.K * sizeof(float) > (size_t)kGemvMaxSmem || p.K % (bf16 ? 8 : 4) != 0)
        return LIN_ERR_UNSUPPORTED;
    GemvArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.X = p.X;
    a.W = p.W;
    a.bias = p.bias;
    a.Y = p.Y;
    a.R = p.residual;
    a.early_x = (p.early_start && p.early_x) ? 1 : 0;
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    if (bf16)
        return gelu ? launch_rpw<true, true>(a, plan.bm, plan.grid_x, p.early_start, p.stream)
                    : launch_rpw<false, true>(a, plan.bm, plan.grid_x, p.early_start, p.stream);
    return gelu ? launch_rpw<true, false>(a, plan.bm, plan.grid_x, p.early_start, p.stream)
                : launch_rpw<false, false>(a, plan.bm, plan.grid_x, p.early_start, p.stream);
}

}  // namespace lin
