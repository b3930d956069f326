// Backward of the linear layer Y = act(X W^T + bias), W stored out x in.
//
// "Writing a CUDA matmul that catches cuBLAS", the backward transpose cases:
// dX = dY W^T and dW = dY^T X for a weight stored in x out, which with W
// stored out x in reads
//   dZ = dY * act'(Z),  dX = dZ W (M x K),  dW = dZ^T X (N x K),  db = sum_m dZ.
// The page folds each transpose into the shared-memory staging, so that each
// transpose case becomes an index map of its own. Here:
// * bf16: the tcgen05 kernel with MN-major operand descriptors (tc.cu).
// * fp32 / tf32: bwd_ffma_kernel below, exact fp32 FFMAs. Both operands are
//   staged as [reduction][output] tiles, so that every thread reads float4s
//   of 4 consecutive output rows and columns (the page's fp32 kernel keeps its
//   A tile k-major so that staging is a plain vector copy): an operand whose reduction index is
//   its row (W in dX; dZ and X in dW) is a straight 16-byte copy, and dZ in dX
//   (reduction index contiguous) is transposed on its way through registers.
// * gelu_backward_kernel: dZ = dY * gelu'(Z), elementwise.
// * colsum kernels: db in two passes (partial sums over fixed row chunks, then
//   the chunks in order), so db is bitwise repeatable.
#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

// ------------------------------------------------------------ gelu backward

template <bool BF16>
__global__ void __launch_bounds__(256) gelu_backward_kernel(long long count, const void* dY, const void* Z, void* dZ) {
    const long long step = (long long)gridDim.x * blockDim.x;
    pdl_wait();  // dY is usually the previous kernel's output
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += step) {
        if constexpr (BF16) {
            const float g = bf16_bits_to_f32(static_cast<const uint16_t*>(dY)[i]);
            const float z = bf16_bits_to_f32(static_cast<const uint16_t*>(Z)[i]);
            static_cast<uint16_t*>(dZ)[i] = f32_to_bf16_bits(g * gelu_tanh_slope<true>(z));
        } else {
            const float g = static_cast<const float*>(dY)[i];
            const float z = static_cast<const float*>(Z)[i];
            static_cast<float*>(dZ)[i] = g * gelu_tanh_slope<false>(z);
        }
    }
}

// ------------------------------------------------------------------ db = sum_m dZ

constexpr int kColRows = 128;  // rows per partial sum

// Pass 1: part[c][n] = sum of dZ[m][n] over rows m in chunk c, ascending m.
template <bool BF16>
__global__ void __launch_bounds__(256) colsum_partial_kernel(int M, int N, const void* dZ, float* part) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int c = blockIdx.y;
    if (n >= N) return;
    const int m0 = c * kColRows, m1 = min(M, m0 + kColRows);
    float s = 0.f;
    for (int m = m0; m < m1; ++m)
        s += BF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(dZ)[(size_t)m * N + n])
                  : static_cast<const float*>(dZ)[(size_t)m * N + n];
    part[(size_t)c * N + n] = s;
}

// Pass 2: db[n] = sum over chunks c in order.
__global__ void __launch_bounds__(256) colsum_final_kernel(int N, int chunks, const float* part, float* db) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s += part[(size_t)c * N + n];
    db[n] = s;
}

// ------------------------------------------------------- fp32 backward GEMMs

// C[i][j] = sum_r A(i, r) B(j, r), C: I x J row-major.
//   WHICH 1 (dX): i = m, j = k, r = n: A = dZ[m][n] (r contiguous), B = W[n][k] (r is the row).
//   WHICH 2 (dW): i = n, j = k, r = m: A = dZ[m][n] (r is the row), B = X[m][k] (r is the row).
struct BwdArgs {
    int I, J, R;
    const float* A;  // dZ
    const float* B;  // W or X
    float* C;        // dX or dW
    int lda;         // row length of dZ (N)
    int ldb;         // row length of B (K; a multiple of 4)
    int a_vec;       // dZ rows are 16-byte aligned (N a multiple of 4): float4 loads
    int splits;      // split-K: CTA z sums reduction stages [z * nst / S, (z + 1) * nst / S)
    float* ws;       // split-K partial sums [S][I][J]
    unsigned* counters;
    const float* Zp; // WHICH 1: the previous layer's pre-activation (I x J): C *= gelu'(Zp); or null
};

constexpr int kBT = 64;   // output tile (I and J)
constexpr int kBR = 16;   // reduction per stage
constexpr int kBTh = 256; // threads: 16 x 16, 4 x 4 outputs each

template <int WHICH>
__global__ void __launch_bounds__(kBTh) bwd_ffma_kernel(const BwdArgs a) {
    __shared__ __align__(16) float As[2][kBR][kBT + 4];
    __shared__ __align__(16) float Bs[2][kBR][kBT + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int i0 = blockIdx.y * kBT, j0 = blockIdx.x * kBT;
    const int nst_all = (a.R + kBR - 1) / kBR;
    const int st_begin = (int)((long long)blockIdx.z * nst_all / a.splits);
    const int st_end = (int)((long long)(blockIdx.z + 1) * nst_all / a.splits);
    const int nst = st_end - st_begin;
    pdl_wait();

    // Each thread stages one float4 of A and one of B per stage.
    float4 ra, rb;
    auto fetch = [&](int st) {
        const int r0 = st * kBR;
        if constexpr (WHICH == 1) {
            // A = dZ[i][r], r contiguous: 4 consecutive r of row i (transposed on store).
            const int i = i0 + tid / 4, r = r0 + 4 * (tid % 4);
            ra = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < a.I) {
                const float* p = a.A + (size_t)i * a.lda + r;
                if (a.a_vec && r + 3 < a.R) ra = *reinterpret_cast<const float4*>(p);
                else {
                    if (r < a.R) ra.x = p[0];
                    if (r + 1 < a.R) ra.y = p[1];
                    if (r + 2 < a.R) ra.z = p[2];
                    if (r + 3 < a.R) ra.w = p[3];
                }
            }
        } else {
            // A(i, r) = dZ[r][i]: 4 consecutive i of row r.
            const int r = r0 + tid / 16, i = i0 + 4 * (tid % 16);
            ra = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < a.R) {
                const float* p = a.A + (size_t)r * a.lda + i;
                if (a.a_vec && i + 3 < a.I) ra = *reinterpret_cast<const float4*>(p);
                else {
                    if (i < a.I) ra.x = p[0];
                    if (i + 1 < a.I) ra.y = p[1];
                    if (i + 2 < a.I) ra.z = p[2];
                    if (i + 3 < a.I) ra.w = p[3];
                }
            }
        }
        // B(j, r) = B[r][j]: 4 consecutive j of row r (both cases).
        const int r = r0 + tid / 16, j = j0 + 4 * (tid % 16);
        rb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < a.R) {
            const float* p = a.B + (size_t)r * a.ldb + j;
            if (j + 3 < a.J) rb = *reinterpret_cast<const float4*>(p);
            else {
                if (j < a.J) rb.x = p[0];
                if (j + 1 < a.J) rb.y = p[1];
                if (j + 2 < a.J) rb.z = p[2];
            }
        }
    };
    auto store = [&](int buf) {
        if constexpr (WHICH == 1) {
            const int il = tid / 4, rl = 4 * (tid % 4);
            As[buf][rl + 0][il] = ra.x;
            As[buf][rl + 1][il] = ra.y;
            As[buf][rl + 2][il] = ra.z;
            As[buf][rl + 3][il] = ra.w;
        } else {
            *reinterpret_cast<float4*>(&As[buf][tid / 16][4 * (tid % 16)]) = ra;
        }
        *reinterpret_cast<float4*>(&Bs[buf][tid / 16][4 * (tid % 16)]) = rb;
    };

    float acc[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;

    if (nst > 0) {
        fetch(st_begin);
        store(0);
    }
    __syncthreads();
    for (int st = 0; st < nst; ++st) {
        const int buf = st & 1;
        if (st + 1 < nst) fetch(st_begin + st + 1);  // the next stage's loads overlap this stage's FMAs
#pragma unroll
        for (int r = 0; r < kBR; ++r) {
            const float4 av = *reinterpret_cast<const float4*>(&As[buf][r][4 * ty]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[buf][r][4 * tx]);
            const float ai[4] = {av.x, av.y, av.z, av.w};
            const float bj[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(ai[p], bj[q], acc[p][q]);
        }
        if (st + 1 < nst) store(buf ^ 1);
        __syncthreads();
    }
    if (a.splits == 1) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int i = i0 + 4 * ty + p;
            if (i >= a.I) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = j0 + 4 * tx + q;
                if (j < a.J) {
                    const size_t o = (size_t)i * a.J + j;
                    a.C[o] = a.Zp ? acc[p][q] * gelu_tanh_slope<false>(a.Zp[o]) : acc[p][q];
                }
            }
        }
        return;
    }
    // Split-K: this CTA's partial tile to the workspace; the last CTA of the
    // tile adds the partials in split order (fixed, so bitwise repeatable).
    __shared__ unsigned s_last;
    float* part = a.ws + (size_t)blockIdx.z * a.I * a.J;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int i = i0 + 4 * ty + p;
        if (i >= a.I) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + 4 * tx + q;
            if (j < a.J) __stcg(part + (size_t)i * a.J + j, acc[p][q]);
        }
    }
    __syncthreads();
    const int tile_id = blockIdx.y * gridDim.x + blockIdx.x;
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&a.counters[tile_id], 1u);
        const unsigned last = prev == (unsigned)(a.splits - 1);
        if (last) {
            a.counters[tile_id] = 0u;  // re-armed for the next launch
            __threadfence();
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;
    // The thread's 4 x 4 outputs of four splits at a time are independent loads
    // (one round trip to the L2 per four splits), added in split order.
    float sum[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[p][q] = 0.f;
#pragma unroll 1
    for (int sp0 = 0; sp0 < a.splits; sp0 += 4) {
        float t[4][4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int i = i0 + 4 * ty + p;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = j0 + 4 * tx + q;
                    t[b][p][q] = (sp0 + b < a.splits && i < a.I && j < a.J)
                                     ? __ldcg(a.ws + (size_t)(sp0 + b) * a.I * a.J + (size_t)i * a.J + j)
                                     : 0.f;
                }
            }
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (sp0 + b < a.splits) sum[p][q] += t[b][p][q];
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int i = i0 + 4 * ty + p;
        if (i >= a.I) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + 4 * tx + q;
            if (j < a.J) {
                const size_t o = (size_t)i * a.J + j;
                a.C[o] = a.Zp ? sum[p][q] * gelu_tanh_slope<false>(a.Zp[o]) : sum[p][q];
            }
        }
    }
}

template <class Kern, class... Args>
int launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool early, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = early ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace

int launch_gelu_backward(long long count, const void* dY, const void* Z, void* dZ, bool bf16, int sm_count,
                         cudaStream_t st, bool early) {
    if (count <= 0) return LIN_OK;
    long long grid = (count + 255) / 256;
    if (grid > 8LL * sm_count) grid = 8LL * sm_count;
    return bf16 ? launch_ex(gelu_backward_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, early, count, dY, Z, dZ)
                : launch_ex(gelu_backward_kernel<false>, dim3((unsigned)grid), dim3(256), 0, st, early, count, dY, Z,
                            dZ);
}

size_t colsum_workspace_bytes(int M, int N) {
    const size_t chunks = ((size_t)M + kColRows - 1) / kColRows;
    return kCounterBytes + align_up(chunks * (size_t)N * sizeof(float), 256);
}

int launch_colsum(int M, int N, const void* dZ, float* db, bool bf16, void* workspace, cudaStream_t st) {
    if (N <= 0) return LIN_OK;
    if (M <= 0) return cudaMemsetAsync(db, 0, (size_t)N * sizeof(float), st) == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
    const int chunks = (M + kColRows - 1) / kColRows;
    float* part = splitk_partials(workspace);
    const dim3 g1((N + 255) / 256, chunks);
    if (bf16)
        colsum_partial_kernel<true><<<g1, 256, 0, st>>>(M, N, dZ, part);
    else
        colsum_partial_kernel<false><<<g1, 256, 0, st>>>(M, N, dZ, part);
    if (cudaGetLastError() != cudaSuccess) return LIN_ERR_CUDA;
    colsum_final_kernel<<<(N + 255) / 256, 256, 0, st>>>(N, chunks, part, db);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

int bwd_ffma_splits(int which, int M, int N, int K, int sm_count, size_t ws_bytes) {
    const int I = which == 1 ? M : N, J = K, R = which == 1 ? N : M;
    const long long tiles = (long long)((I + kBT - 1) / kBT) * ((J + kBT - 1) / kBT);
    const int nst = (R + kBR - 1) / kBR;
    // Fill four resident 256-thread CTAs per SM without a second wave, >= 4
    // reduction stages per split (the page splits K when the output is small and
    // the reduction long).
    const long long slots = 4LL * sm_count;
    int S = tiles >= slots ? 1 : (int)(slots / tiles);
    const int max_s = nst / 4 > 1 ? nst / 4 : 1;
    if (S > max_s) S = max_s;
    if (S < 1) S = 1;
    if (tiles > kMaxSplitTiles) S = 1;
    while (S > 1 && splitk_workspace_bytes(S, I, J) > ws_bytes) --S;
    return S;
}

int launch_bwd_ffma(int which, int M, int N, int K, const float* dZ, const float* B, float* out, int splits,
                    void* workspace, cudaStream_t st, bool early, const float* Zp) {
    BwdArgs a = {};
    a.Zp = which == 1 ? Zp : nullptr;
    a.splits = splits < 1 ? 1 : splits;
    a.ws = a.splits > 1 ? splitk_partials(workspace) : nullptr;
    a.counters = a.splits > 1 ? splitk_counters(workspace) : nullptr;
    a.A = dZ;
    a.B = B;
    a.C = out;
    a.lda = N;
    a.ldb = K;
    a.a_vec = (N % 4 == 0 && (reinterpret_cast<uintptr_t>(dZ) % 16) == 0) ? 1 : 0;
    if (which == 1) {
        a.I = M;
        a.J = K;
        a.R = N;
    } else {
        a.I = N;
        a.J = K;
        a.R = M;
    }
    if (a.I <= 0 || a.J <= 0) return LIN_OK;
    if (a.R <= 0)
        return cudaMemsetAsync(out, 0, (size_t)a.I * a.J * sizeof(float), st) == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
    const dim3 grid((a.J + kBT - 1) / kBT, (a.I + kBT - 1) / kBT, a.splits);
    return which == 1 ? launch_ex(bwd_ffma_kernel<1>, grid, dim3(kBTh), 0, st, early, a)
                      : launch_ex(bwd_ffma_kernel<2>, grid, dim3(kBTh), 0, st, early, a);
}

}  // namespace lin
