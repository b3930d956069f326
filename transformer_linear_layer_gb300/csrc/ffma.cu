// Exact-fp32 linear layer on the CUDA cores (fp32 FFMA, no tensor cores).
//
// The sgemm ladder of "Writing a CUDA matmul that catches cuBLAS" (kernels
// 3-8) and the register-tiled kernels of "What the kernels were short of",
// rebuilt for sm_103a:
//
// * Block tile BM x BN, K step BK; each of 256 threads owns a TM x TN register
//   tile ("Kernels 3-5: reuse, at three levels"). A thread's rows are
//   ty, ty + BM/TM, ... and its columns tx, tx + BN/TN, ...: the B reads of a
//   warp fall in distinct banks, the A reads are broadcasts, and the output
//   stores of a warp are consecutive columns.
// * Shared-memory tiles keep the operands' K-contiguous layout (X is M x K, W
//   is N x K), rows padded to an odd number of 16-byte chunks. A thread reads
//   a float4 of four consecutive k for each of its rows, keeps them in
//   registers, and streams its columns' float4s past them: 4 * TM FMAs per
//   128-bit read of B. Each output still accumulates in ascending k.
// * The K slices stream through a STAGES-deep ring filled with cp.async (16-byte
//   copies that bypass registers, zero-filled past the tensor's edge), so the
//   loads of later slices overlap the arithmetic of the current one - the
//   double buffering of "Kernel 8: the loop was shaped wrong", deeper.
// * Fused epilogue: bias, optional tanh-GELU with the accurate tanhf, fp32
//   store ("The bias add did not need to exist"; "The residual and GELU go the
//   same way", with the feature set as a template parameter).
// * Optional split-K for outputs too small to fill the SMs: each CTA sums one
//   K range into the workspace and the last CTA of a tile adds the ranges in
//   order 0..S-1 ("One kernel was never going to be enough": the page splits
//   K for small outputs with long reductions; "Optimizing a GPT-2-class
//   transformer on a GPU", Act I: fixed-order reduction).
// * Programmatic dependent launch (when the caller allows an early start): the
//   CTAs may start while the previous kernel on the stream drains, loading X
//   and W before griddepcontrol.wait when neither is that kernel's output;
//   bias, Y and the split-K workspace are touched only after the wait.
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
    const float* R;    // residual added after the activation (M x N, may be Y itself), or null
    float* ws;
    unsigned* counters;
    int splits;
    int nkb;           // ceil(K / BK)
    int early_inputs;  // X and W may be read before the dependency wait (not the previous call's output)
    int prefetch;      // otherwise ask the L2 for the first slices of them before the wait
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    // src-size 0 fills the 16 bytes with zeros (rows or K past the tensor).
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int BM, int BN, int BK, int STAGES>
constexpr size_t ffma_smem_bytes() {
    return (size_t)STAGES * (BM + BN) * (BK + 4) * sizeof(float);
}

// Split-K: this CTA's partial tile to the workspace; the last CTA of the tile
// adds the S partials in split order. One gpu-scope fence per CTA (cumulative
// over the barrier) publishes the partials before the arrival count.
template <int TM, int TN, bool GELU, class RowOf, class ColOf>
__device__ __forceinline__ void splitk_epilogue(const FfmaArgs& a, const float (&acc)[TM][TN], RowOf row_of,
                                                ColOf col_of, int tid) {
    __shared__ unsigned s_last;
    const int split = blockIdx.z;
    float* part = a.ws + (size_t)split * a.M * a.N;
#pragma unroll
    for (int r = 0; r < TM; ++r) {
        const int m = row_of(r);
        if (m >= a.M) continue;
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int n = col_of(c);
            if (n < a.N) __stcg(part + (size_t)m * a.N + n, acc[r][c]);
        }
    }
    __syncthreads();
    const int tile_id = blockIdx.y * gridDim.x + blockIdx.x;
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&a.counters[tile_id], 1u);
        const unsigned last = prev == (unsigned)(a.splits - 1);
        if (last) {
            a.counters[tile_id] = 0u;  // re-arm for the next launch
            __threadfence();
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;
    // The thread's TM x TN outputs of SB splits at a time are independent loads
    // (one round trip to the L2 per SB splits), added in split order.
    constexpr int SB = TM * TN <= 16 ? 4 : TM * TN <= 32 ? 2 : 1;
    float bcol[TN];
#pragma unroll
    for (int c = 0; c < TN; ++c) {
        const int n = col_of(c);
        bcol[c] = (a.bias && n < a.N) ? __ldg(a.bias + n) : 0.f;
    }
    float sum[TM][TN];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int c = 0; c < TN; ++c) sum[r][c] = 0.f;
#pragma unroll 1
    for (int sp0 = 0; sp0 < a.splits; sp0 += SB) {
        float t[SB][TM][TN];
#pragma unroll
        for (int b = 0; b < SB; ++b) {
            const int sp = sp0 + b;
#pragma unroll
            for (int r = 0; r < TM; ++r) {
                const int m = row_of(r);
#pragma unroll
                for (int c = 0; c < TN; ++c) {
                    const int n = col_of(c);
                    t[b][r][c] = (sp < a.splits && m < a.M && n < a.N)
                                     ? __ldcg(a.ws + ((size_t)sp * a.M + m) * a.N + n)
                                     : 0.f;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < SB; ++b)
#pragma unroll
            for (int r = 0; r < TM; ++r)
#pragma unroll
                for (int c = 0; c < TN; ++c)
                    if (sp0 + b < a.splits) sum[r][c] += t[b][r][c];
    }
#pragma unroll
    for (int r = 0; r < TM; ++r) {
        const int m = row_of(r);
        if (m >= a.M) continue;
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int n = col_of(c);
            if (n < a.N) {
                const size_t i = (size_t)m * a.N + n;
                a.Y[i] = epilogue<GELU>(sum[r][c], bcol[c]) + (a.R ? a.R[i] : 0.f);
            }
        }
    }
}

template <int BM, int BN, int BK, int TM, int TN, int STAGES, bool GELU, bool SPLIT>
__global__ void __launch_bounds__(256, (BM * BN >= 128 * 128 ? 1 : 2))
ffma_kernel(const FfmaArgs a) {
    constexpr int NT = 256;
    constexpr int TX = BN / TN, TY = BM / TM;  // threads along n and along m
    static_assert(TX * TY == NT, "256 threads");
    constexpr int LD = BK + 4;  // row stride in floats: BK/4 + 1 chunks of 16 bytes (odd)
    static_assert((LD / 4) % 2 == 1, "odd number of 16-byte chunks per row");
    constexpr int CPR = BK / 4;  // 16-byte chunks per row of a K slice
    constexpr int A_CHUNKS = BM * CPR / NT, B_CHUNKS = BN * CPR / NT;
    static_assert(A_CHUNKS >= 1 && B_CHUNKS >= 1 && (BM * CPR) % NT == 0 && (BN * CPR) % NT == 0, "chunks");
    constexpr int STAGE_FLOATS = (BM + BN) * LD;

    extern __shared__ __align__(16) float smem[];

    const int tid = threadIdx.x;
    const int tx = tid % TX, ty = tid / TX;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int split = blockIdx.z;
    const int kb_begin = (int)((long long)split * a.nkb / a.splits);
    const int kb_end = (int)((long long)(split + 1) * a.nkb / a.splits);
    const int nk = kb_end - kb_begin;
    if (tid == 0) pdl_launch_dependents();
    if (!a.early_inputs) {
        // X or W may be the previous kernel's output: read nothing before the
        // wait, but have the L2 fetch the first ring's worth of this CTA's rows
        // (one bulk prefetch per row; no data comes back before the wait).
        if (a.prefetch && nk > 0) {
            const int k0 = kb_begin * BK;
            const int k1 = (kb_begin + STAGES - 1 < kb_end ? kb_begin + STAGES - 1 : kb_end) * BK;
            const unsigned bytes = (unsigned)((k1 < a.K ? k1 : a.K) - k0) * 4u;
            const int r = tid < BM ? m0 + tid : n0 + tid - BM;
            const bool is_x = tid < BM;
            if (tid < BM + BN && r < (is_x ? a.M : a.N) && bytes > 0) {
                const float* src = (is_x ? a.X : a.W) + (size_t)r * a.K + k0;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
            }
        }
        pdl_wait();
    }

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    // Copy K slice `kb` into ring stage `st`. Thread `tid` always copies chunk
    // column tid % CPR of rows tid / CPR + v * RSTEP, so one base pointer per
    // operand and a row stride serve every chunk. K is a multiple of 4, so a
    // chunk is wholly inside or outside the tensor.
    constexpr int RSTEP = NT / CPR;
    static_assert(NT % CPR == 0, "whole rows per pass");
    const int lr = tid / CPR, lc = tid % CPR;
    const float* xbase = a.X + (size_t)(m0 + lr) * a.K + 4 * lc;
    const float* wbase = a.W + (size_t)(n0 + lr) * a.K + 4 * lc;
    const size_t rstride = (size_t)RSTEP * a.K;
    auto load_slice = [&](int kb, int st) {
        const int k0 = kb * BK;
        const bool kok = k0 + 4 * lc < a.K;
        const uint32_t sa = smem_base + (uint32_t)(st * STAGE_FLOATS + lr * LD + 4 * lc) * 4u;
        const uint32_t sb = sa + (uint32_t)(BM * LD) * 4u;
#pragma unroll
        for (int v = 0; v < A_CHUNKS; ++v) {
            const bool ok = kok && m0 + lr + v * RSTEP < a.M;
            cp_async16(sa + (uint32_t)(v * RSTEP * LD) * 4u, ok ? xbase + v * rstride + k0 : a.X, ok);
        }
#pragma unroll
        for (int v = 0; v < B_CHUNKS; ++v) {
            const bool ok = kok && n0 + lr + v * RSTEP < a.N;
            cp_async16(sb + (uint32_t)(v * RSTEP * LD) * 4u, ok ? wbase + v * rstride + k0 : a.W, ok);
        }
    };

    // Prologue: STAGES-1 slices in flight (empty groups keep the counting uniform).
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nk) load_slice(kb_begin + s, s);
        cp_async_commit();
    }
    for (int i = 0; i < nk; ++i) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // slice i landed for every thread; slice i-1's stage is free
        if (i + STAGES - 1 < nk) load_slice(kb_begin + i + STAGES - 1, (i + STAGES - 1) % STAGES);
        cp_async_commit();
        const float* As = smem + (i % STAGES) * STAGE_FLOATS;
        const float* Bs = As + BM * LD;
        // The A values of all TM rows for four consecutive k stay in registers
        // while B's float4 for each column streams past (TM + TN 128-bit shared
        // loads per 4 * TM * TN FMAs).
#pragma unroll
        for (int kq = 0; kq < BK / 4; ++kq) {
            float4 av[TM];
#pragma unroll
            for (int r = 0; r < TM; ++r) av[r] = *reinterpret_cast<const float4*>(As + (ty + r * TY) * LD + 4 * kq);
#pragma unroll
            for (int c = 0; c < TN; ++c) {
                const float4 bv = *reinterpret_cast<const float4*>(Bs + (tx + c * TX) * LD + 4 * kq);
#pragma unroll
                for (int r = 0; r < TM; ++r) {
                    acc[r][c] = fmaf(av[r].x, bv.x, acc[r][c]);
                    acc[r][c] = fmaf(av[r].y, bv.y, acc[r][c]);
                    acc[r][c] = fmaf(av[r].z, bv.z, acc[r][c]);
                    acc[r][c] = fmaf(av[r].w, bv.w, acc[r][c]);
                }
            }
        }
    }
    cp_async_wait<0>();
    // Bias, Y and the split-K workspace only after the previous kernel on the
    // stream has finished (it may have written the bias, or be using the
    // workspace).
    pdl_wait();

    auto row_of = [&](int r) { return m0 + ty + r * TY; };
    auto col_of = [&](int c) { return n0 + tx + c * TX; };

    if constexpr (!SPLIT) {
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int n = col_of(c);
            if (n >= a.N) continue;
            const float b = a.bias ? __ldg(a.bias + n) : 0.f;
#pragma unroll
            for (int r = 0; r < TM; ++r) {
                const int m = row_of(r);
                if (m < a.M) {
                    const size_t i = (size_t)m * a.N + n;
                    a.Y[i] = epilogue<GELU>(acc[r][c], b) + (a.R ? a.R[i] : 0.f);
                }
            }
        }
        return;
    } else {
        splitk_epilogue<TM, TN, GELU>(a, acc, row_of, col_of, tid);
    }
}

template <int BM, int BN, int BK, int TM, int TN, int STAGES>
int launch_cfg(const FfmaArgs& a, dim3 grid, cudaStream_t st, bool gelu, bool early) {
    constexpr size_t smem = ffma_smem_bytes<BM, BN, BK, STAGES>();
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    const bool split = a.splits > 1;
    auto kern = gelu ? (split ? ffma_kernel<BM, BN, BK, TM, TN, STAGES, true, true>
                              : ffma_kernel<BM, BN, BK, TM, TN, STAGES, true, false>)
                     : (split ? ffma_kernel<BM, BN, BK, TM, TN, STAGES, false, true>
                              : ffma_kernel<BM, BN, BK, TM, TN, STAGES, false, false>);
    static std::atomic<unsigned long long> attr_set[4];  // per instantiation: one bit per device
    const int which = (gelu ? 2 : 0) + (split ? 1 : 0);
    if (ensure_smem_attr(attr_set[which], kern, smem) != LIN_OK) return LIN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256, 1, 1);
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

}  // namespace

int launch_ffma(const Problem& p, const lin_plan& plan) {
    FfmaArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.X = static_cast<const float*>(p.X);
    a.W = static_cast<const float*>(p.W);
    a.bias = p.bias;
    a.Y = static_cast<float*>(p.Y);
    a.R = static_cast<const float*>(p.residual);
    a.splits = plan.splits;
    a.nkb = (p.K + plan.bk - 1) / plan.bk;
    a.early_inputs = (p.early_start && p.early_x) ? 1 : 0;
    a.prefetch = p.early_start ? 1 : 0;
    a.ws = nullptr;
    a.counters = nullptr;
    if (plan.splits > 1) {
        a.ws = splitk_partials(p.workspace);
        a.counters = splitk_counters(p.workspace);
    }
    const dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    switch (plan.variant) {
#define LIN_FFMA_CASE(V)                                                                                       \
    case V:                                                                                                    \
        return launch_cfg<kFfmaCfg[V].bm, kFfmaCfg[V].bn, kFfmaCfg[V].bk, kFfmaCfg[V].tm, kFfmaCfg[V].tn,     \
                          kFfmaCfg[V].stages>(a, grid, p.stream, gelu, p.early_start);
        LIN_FFMA_CASE(0)
        LIN_FFMA_CASE(1)
        LIN_FFMA_CASE(2)
        LIN_FFMA_CASE(3)
#undef LIN_FFMA_CASE
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace lin
