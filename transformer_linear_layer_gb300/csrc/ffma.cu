// Exact-fp32 linear layer on the CUDA cores (fp32 FFMA, no tensor cores).
//
// The sgemm ladder of "Writing a CUDA matmul that catches cuBLAS" (kernels
// 3-8) and the register-tiled kernels of "What the kernels were short of",
// rebuilt for sm_103a:
//
// * Block tile BM x BN, K step BK; each of 256 threads owns a TM x TN register
//   tile, so per k it reads TM + TN values from shared memory and issues
//   TM * TN FMAs ("Kernels 3-5: reuse, at three levels").
// * Both operands are K-contiguous in global memory (X is M x K, W is N x K),
//   read with 128-bit loads and stored transposed (k-major) in shared memory,
//   so the per-k reads of the register tile are 128-bit shared loads of
//   contiguous m (or n) values ("What the kernels were short of": the
//   transposed, k-major A tile with 128-bit shared reads). A thread's 8 rows
//   are two groups of 4 half a tile apart, so a quarter-warp's 128-bit reads
//   cover 128 contiguous bytes (conflict-free).
// * Double buffering: the next K slice is fetched into registers while the
//   current one is multiplied, and written to the other shared buffer after,
//   one barrier per K step ("Kernel 8: the loop was shaped wrong").
// * Fused epilogue: bias, optional tanh-GELU with the accurate tanhf, fp32
//   store ("The bias add did not need to exist"; "The residual and GELU go the
//   same way", with the feature set as a template parameter).
// * Optional split-K for outputs too small to fill 152 SMs: each CTA sums one
//   K range into the workspace, the last CTA of a tile adds the ranges in order
//   ("One kernel was never going to be enough": split-K when the output is
//   small and K is long).
#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

struct FfmaArgs {
    int M, N, K;
    const float* X;
    const float* W;
    const float* bias;
    float* Y;
    float* ws;
    unsigned* counters;
    int splits;
    int nkb;          // ceil(K / BK)
    int y_aligned16;  // Y's base is 16-byte aligned (vector stores allowed)
};

template <int BM, int BN, int BK, int TM, int TN, bool GELU>
__global__ void __launch_bounds__(256, 2)
ffma_kernel(const FfmaArgs a) {
    constexpr int NT = 256;
    constexpr int TX = BN / TN;  // threads along n
    static_assert((BM / TM) * (BN / TN) == NT, "256 threads");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "128-bit register tiles");
    constexpr int PAD = 4;
    constexpr int A_LD = BM + PAD, B_LD = BN + PAD;
    constexpr int A_VEC = BM * BK / 4 / NT;  // float4 loads per thread per K step
    constexpr int B_VEC = BN * BK / 4 / NT;
    static_assert(A_VEC >= 1 && B_VEC >= 1, "tile too small for 256 threads");
    constexpr int KQ = BK / 4;  // float4 per row of a K slice
    // Register-tile placement: TM rows as TM/4 groups of 4, groups BM/(TM/4) apart.
    constexpr int MG = TM / 4, NG = TN / 4;
    constexpr int M_STRIDE = BM / MG, N_STRIDE = BN / NG;

    __shared__ __align__(16) float As[2][BK][A_LD];
    __shared__ __align__(16) float Bs[2][BK][B_LD];
    __shared__ unsigned s_last;

    const int tid = threadIdx.x;
    const int tx = tid % TX, ty = tid / TX;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int split = blockIdx.z;
    const int kb_begin = (int)((long long)split * a.nkb / a.splits);
    const int kb_end = (int)((long long)(split + 1) * a.nkb / a.splits);

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    float4 ra[A_VEC], rb[B_VEC];
    auto fetch = [&](int kb) {
        const int k0 = kb * BK;
#pragma unroll
        for (int v = 0; v < A_VEC; ++v) {
            const int idx = tid + v * NT, r = idx / KQ, q = idx % KQ;
            const int m = m0 + r, k = k0 + 4 * q;
            ra[v] = (m < a.M && k < a.K) ? __ldg(reinterpret_cast<const float4*>(a.X + (size_t)m * a.K + k))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int v = 0; v < B_VEC; ++v) {
            const int idx = tid + v * NT, r = idx / KQ, q = idx % KQ;
            const int n = n0 + r, k = k0 + 4 * q;
            rb[v] = (n < a.N && k < a.K) ? __ldg(reinterpret_cast<const float4*>(a.W + (size_t)n * a.K + k))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int v = 0; v < A_VEC; ++v) {
            const int idx = tid + v * NT, r = idx / KQ, q = idx % KQ;
            As[buf][4 * q + 0][r] = ra[v].x;
            As[buf][4 * q + 1][r] = ra[v].y;
            As[buf][4 * q + 2][r] = ra[v].z;
            As[buf][4 * q + 3][r] = ra[v].w;
        }
#pragma unroll
        for (int v = 0; v < B_VEC; ++v) {
            const int idx = tid + v * NT, r = idx / KQ, q = idx % KQ;
            Bs[buf][4 * q + 0][r] = rb[v].x;
            Bs[buf][4 * q + 1][r] = rb[v].y;
            Bs[buf][4 * q + 2][r] = rb[v].z;
            Bs[buf][4 * q + 3][r] = rb[v].w;
        }
    };

    if (kb_begin < kb_end) {
        fetch(kb_begin);
        stash(0);
        __syncthreads();
        int buf = 0;
        for (int kb = kb_begin; kb < kb_end; ++kb) {
            if (kb + 1 < kb_end) fetch(kb + 1);
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float av[TM], bv[TN];
#pragma unroll
                for (int gq = 0; gq < MG; ++gq) {
                    const float4 v = *reinterpret_cast<const float4*>(&As[buf][kk][gq * M_STRIDE + ty * 4]);
                    av[4 * gq + 0] = v.x; av[4 * gq + 1] = v.y; av[4 * gq + 2] = v.z; av[4 * gq + 3] = v.w;
                }
#pragma unroll
                for (int gq = 0; gq < NG; ++gq) {
                    const float4 v = *reinterpret_cast<const float4*>(&Bs[buf][kk][gq * N_STRIDE + tx * 4]);
                    bv[4 * gq + 0] = v.x; bv[4 * gq + 1] = v.y; bv[4 * gq + 2] = v.z; bv[4 * gq + 3] = v.w;
                }
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            if (kb + 1 < kb_end) {
                stash(buf ^ 1);
                __syncthreads();
                buf ^= 1;
            }
        }
    }

    // Output coordinates of acc[i][j].
    auto row_of = [&](int i) { return m0 + (i / 4) * M_STRIDE + ty * 4 + (i % 4); };
    auto col_of = [&](int j) { return n0 + (j / 4) * N_STRIDE + tx * 4 + (j % 4); };
    const bool vec_ok = (a.N % 4) == 0 && a.y_aligned16;

    auto store_final = [&](int i, int jg, const float (&v)[4]) {
        const int m = row_of(i);
        const int n = col_of(jg * 4);
        if (m >= a.M) return;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float b = (a.bias && n + e < a.N) ? a.bias[n + e] : 0.f;
            o[e] = epilogue<GELU>(v[e], b);
        }
        float* dst = a.Y + (size_t)m * a.N + n;
        if (vec_ok && n + 3 < a.N) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (n + e < a.N) dst[e] = o[e];
        }
    };

    if (a.splits == 1) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jg = 0; jg < NG; ++jg) {
                const float v[4] = {acc[i][4 * jg], acc[i][4 * jg + 1], acc[i][4 * jg + 2], acc[i][4 * jg + 3]};
                store_final(i, jg, v);
            }
        return;
    }

    // Split-K: partial tile to the workspace, last CTA of the tile reduces.
    float* part = a.ws + (size_t)split * a.M * a.N;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = row_of(i);
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = col_of(j);
            if (n < a.N) __stcg(part + (size_t)m * a.N + n, acc[i][j]);
        }
    }
    __threadfence();
    __syncthreads();
    const int tile_id = blockIdx.y * gridDim.x + blockIdx.x;
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.counters[tile_id], 1u);
        s_last = (prev == (unsigned)(a.splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = row_of(i);
#pragma unroll
        for (int jg = 0; jg < NG; ++jg) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (m < a.M) {
                for (int sp = 0; sp < a.splits; ++sp) {
                    const float* src = a.ws + ((size_t)sp * a.M + m) * a.N;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int n = col_of(jg * 4 + e);
                        if (n < a.N) v[e] += __ldcg(src + n);
                    }
                }
            }
            store_final(i, jg, v);
        }
    }
    if (tid == 0) a.counters[tile_id] = 0u;
}

template <int BM, int BN, int BK, int TM, int TN>
int launch_cfg(const FfmaArgs& a, dim3 grid, cudaStream_t st, bool gelu) {
    if (gelu)
        ffma_kernel<BM, BN, BK, TM, TN, true><<<grid, 256, 0, st>>>(a);
    else
        ffma_kernel<BM, BN, BK, TM, TN, false><<<grid, 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace

int launch_ffma(const Problem& p, const lin_plan& plan) {
    FfmaArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.X = static_cast<const float*>(p.X);
    a.W = static_cast<const float*>(p.W);
    a.bias = p.bias;
    a.Y = static_cast<float*>(p.Y);
    a.splits = plan.splits;
    a.nkb = (p.K + plan.bk - 1) / plan.bk;
    a.y_aligned16 = (reinterpret_cast<uintptr_t>(p.Y) % 16) == 0;
    a.ws = nullptr;
    a.counters = nullptr;
    if (plan.splits > 1) {
        a.ws = splitk_partials(p.workspace);
        a.counters = splitk_counters(p.workspace);
    }
    const dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    switch (plan.variant) {
        case 0: return launch_cfg<128, 128, 16, 8, 8>(a, grid, p.stream, gelu);
        case 1: return launch_cfg<64, 64, 16, 4, 4>(a, grid, p.stream, gelu);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace lin
