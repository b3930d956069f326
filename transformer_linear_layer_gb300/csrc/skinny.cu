// Skinny linear layer, M <= 16, bf16 in, fp32 accumulate, bf16 out.
//
// The workload of "One multiply, one RTX 5090, eight kernels": a batch of 16
// vectors against a 4096 x 4096 weight stored out x in. Each weight value
// feeds only M products, so the kernel is a stream over W and its speed is
// the rate at which W leaves HBM ("Where the time goes": the loads-only probe
// took as long as the full kernel). Design on sm_103a:
//
// * Every W byte is loaded exactly once, by 128-bit non-allocating global
//   loads (ld.global.nc.L1::no_allocate.v4), double-buffered in registers
//   one round ahead so each thread keeps several 16-byte loads in flight.
// * The inner product uses the tensor cores through mma.m16n8k16 (bf16 x
//   bf16 -> fp32): X is the 16 x 16 A operand and a 16 x 8 slab of W^T is
//   the B operand. At M = 16 the FFMA units cannot keep up with HBM
//   (16 FLOP per W byte at ~6.8 TB/s is ~108 TFLOP/s), the tensor cores can.
// * The 8 bf16 a thread loads from one W row (k0+8t .. k0+8t+7, t = lane%4)
//   serve two MMAs directly: the reduction over k does not depend on which
//   k sits in which fragment slot, so slots {2t,2t+1 | 2t+8,2t+9} of MMA 0
//   take k = 8t+{0,1 | 2,3} and those of MMA 1 take 8t+{4,5 | 6,7}; X
//   fragments use the same map (one 16-byte X load per fragment row). This
//   avoids any shared-memory staging of W.
// * Split-K fills the chip ("Filling the chip": Kernel 7 splits the inner
//   dimension of each tile into ranges, one block each). Each CTA owns
//   R = warps*groups*8 rows of W and one K range; partial sums go to the
//   workspace and the last CTA of a tile to arrive adds the ranges in fixed
//   order 0..S-1, then applies bias, GELU and the bf16 store - bitwise
//   repeatable ("Optimizing a GPT-2-class transformer on a GPU", Act I).
#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

struct SkinnyArgs {
    int M, N, K;
    const uint16_t* X;  // bf16 bits, M x K
    const uint16_t* W;  // bf16 bits, N x K
    const float* bias;  // N or nullptr
    uint16_t* Y;        // bf16 bits, M x N
    float* ws;          // splits x M x N partials (splits > 1)
    unsigned* counters; // one per n-tile (splits > 1), zero between launches
    int splits;
    int nchunks;        // ceil(K / 32)
};

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_reused(const uint16_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int WARPS, int G, int U, bool GELU>
__global__ void __launch_bounds__(WARPS * 32)
skinny_kernel(const SkinnyArgs a) {
    constexpr int R = WARPS * G * 8;  // rows of W (output columns) per CTA
    constexpr int NT = WARPS * 32;
    __shared__ float tile[16][R + 1];
    __shared__ unsigned s_last;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n_cta = blockIdx.x * R;
    const int split = blockIdx.y;
    const int c_begin = (int)((long long)split * a.nchunks / a.splits);
    const int c_end = (int)((long long)(split + 1) * a.nchunks / a.splits);

    // This thread's W rows: one per n8 group, row g of the group.
    const uint16_t* wrow[G];
    bool wok[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const int n = n_cta + (warp * G + j) * 8 + g;
        wok[j] = n < a.N;
        wrow[j] = a.W + (size_t)(wok[j] ? n : 0) * (size_t)a.K + 8 * t;
    }
    const bool xa_ok = g < a.M, xb_ok = g + 8 < a.M;
    const uint16_t* xa_row = a.X + (size_t)(xa_ok ? g : 0) * (size_t)a.K + 8 * t;
    const uint16_t* xb_row = a.X + (size_t)(xb_ok ? g + 8 : 0) * (size_t)a.K + 8 * t;

    float acc[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    // K is a multiple of 8, so a thread's 8-element slice is wholly in or out.
    auto load_round = [&](uint4 (&wb)[U][G], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = (c0 + u) * 32;
            const bool kin = (c0 + u < c_end) && (k + 8 * t < a.K);
#pragma unroll
            for (int j = 0; j < G; ++j) wb[u][j] = (kin && wok[j]) ? ld_stream(wrow[j] + k) : zero;
        }
    };
    auto compute_round = [&](const uint4 (&wb)[U][G], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = (c0 + u) * 32;
            const bool kin = (c0 + u < c_end) && (k + 8 * t < a.K);
            const uint4 xa = (kin && xa_ok) ? ld_reused(xa_row + k) : zero;
            const uint4 xb = (kin && xb_ok) ? ld_reused(xb_row + k) : zero;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                mma16816(acc[j], xa.x, xb.x, xa.y, xb.y, wb[u][j].x, wb[u][j].y);
                mma16816(acc[j], xa.z, xb.z, xa.w, xb.w, wb[u][j].z, wb[u][j].w);
            }
        }
    };

    if (c_begin < c_end) {
        uint4 bufA[U][G], bufB[U][G];
        int c = c_begin;
        load_round(bufA, c);
        while (true) {
            if (c + U < c_end) load_round(bufB, c + U);
            compute_round(bufA, c);
            c += U;
            if (c >= c_end) break;
            if (c + U < c_end) load_round(bufA, c + U);
            compute_round(bufB, c);
            c += U;
            if (c >= c_end) break;
        }
    }

    // Accumulator fragment (m16n8 f32): c0,c1 -> row g, cols 2t,2t+1; c2,c3 -> row g+8.
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const int nl = (warp * G + j) * 8 + 2 * t;
        tile[g][nl] = acc[j][0];
        tile[g][nl + 1] = acc[j][1];
        tile[g + 8][nl] = acc[j][2];
        tile[g + 8][nl + 1] = acc[j][3];
    }
    __syncthreads();

    const int M = a.M, N = a.N;
    if (a.splits == 1) {
        for (int idx = threadIdx.x; idx < M * R; idx += NT) {
            const int m = idx / R, nl = idx % R, n = n_cta + nl;
            if (n < N) {
                const float b = a.bias ? a.bias[n] : 0.f;
                a.Y[(size_t)m * N + n] = f32_to_bf16_bits(epilogue<GELU>(tile[m][nl], b));
            }
        }
        return;
    }

    float* part = a.ws + (size_t)split * M * N;
    for (int idx = threadIdx.x; idx < M * R; idx += NT) {
        const int m = idx / R, nl = idx % R, n = n_cta + nl;
        if (n < N) __stcg(part + (size_t)m * N + n, tile[m][nl]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&a.counters[blockIdx.x], 1u);
        s_last = (prev == (unsigned)(a.splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < M * R; idx += NT) {
        const int m = idx / R, nl = idx % R, n = n_cta + nl;
        if (n < N) {
            float s = 0.f;
            for (int sp = 0; sp < a.splits; ++sp) s += __ldcg(a.ws + ((size_t)sp * M + m) * N + n);
            const float b = a.bias ? a.bias[n] : 0.f;
            a.Y[(size_t)m * N + n] = f32_to_bf16_bits(epilogue<GELU>(s, b));
        }
    }
    if (threadIdx.x == 0) a.counters[blockIdx.x] = 0u;  // re-arm for the next launch
}

template <int WARPS, int G, int U>
int launch_cfg(const SkinnyArgs& a, dim3 grid, cudaStream_t st, bool gelu) {
    if (gelu)
        skinny_kernel<WARPS, G, U, true><<<grid, WARPS * 32, 0, st>>>(a);
    else
        skinny_kernel<WARPS, G, U, false><<<grid, WARPS * 32, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace

int launch_skinny(const Problem& p, const lin_plan& plan) {
    SkinnyArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.X = static_cast<const uint16_t*>(p.X);
    a.W = static_cast<const uint16_t*>(p.W);
    a.bias = p.bias;
    a.Y = static_cast<uint16_t*>(p.Y);
    a.splits = plan.splits;
    a.nchunks = (p.K + 31) / 32;
    a.ws = nullptr;
    a.counters = nullptr;
    if (plan.splits > 1) {
        a.ws = splitk_partials(p.workspace);
        a.counters = splitk_counters(p.workspace);
    }
    const dim3 grid(plan.grid_x, plan.grid_y, 1);
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    switch (plan.variant) {
        case 0: return launch_cfg<4, 2, 4>(a, grid, p.stream, gelu);
        case 1: return launch_cfg<8, 1, 4>(a, grid, p.stream, gelu);
        case 2: return launch_cfg<4, 4, 2>(a, grid, p.stream, gelu);
        case 3: return launch_cfg<8, 2, 2>(a, grid, p.stream, gelu);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace lin
