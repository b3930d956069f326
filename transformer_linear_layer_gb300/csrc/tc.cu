// Dense linear layer on the 5th-generation tensor cores: TMA -> shared memory
// -> tcgen05.mma -> TMEM -> fused epilogue. Two arithmetics share one kernel:
//   BF16: bf16 x bf16 products, fp32 accumulate, bf16 output (kind::f16)
//   TF32: fp32 operands whose TF32 part the tensor core multiplies, fp32
//         accumulate and output (kind::tf32)
//
// The pages' tensor-core ladders (WMMA and mma.sync, "Writing a CUDA matmul
// that catches cuBLAS", "Kernel 9" and "Kernel 10"; "One multiply, one RTX
// 5090, eight kernels", "Inside one block") stage K slices in shared memory
// with a copy requested before the current slice is multiplied. On sm_103a
// the same structure is expressed with hardware queues instead of warps:
//
// * One thread of warp 0 issues 2-D TMA copies of a 128-row A tile (X) and a
//   BN-row B tile (W), 128 bytes of K each, into a STAGES-deep ring, each
//   stage guarded by a "full" and an "empty" mbarrier. The copies use the
//   128-byte swizzle, which the tensor core's shared-memory descriptors read
//   directly (the XOR swizzle of "Kernel 10", done by the copy engine).
// * One thread of warp 1 issues tcgen05.mma (M=128, N=BN, K=32 bytes) into a
//   TMEM accumulator of 128 lanes x BN fp32 columns, and tcgen05.commit frees
//   each stage when its MMAs have read it.
// * Warps 2-5 wait for the last commit, read the accumulator with
//   tcgen05.ld (warp w reads TMEM lanes 32*(w%4) .. +31, one output row per
//   thread), add the bias, apply GELU and store ("The bias add did not need to
//   exist": the epilogue already holds the value in a register).
// * Tails: the copy engine fills rows and K beyond the tensor with zeros;
//   stores are predicated on m < M and n < N.
// * Every wait is bounded (iterations and wall clock); a wait that gives up
//   writes LIN_ERR_DEVICE_TIMEOUT to the status word, the CTA skips its
//   stores, drains its own copies and MMAs, frees TMEM and exits.
#include "internal.h"
#include "device_common.cuh"
#include "tc_common.cuh"

namespace lin {
namespace {

struct TcArgs {
    int M, N, K;
    const float* bias;
    void* Y;
    int* status;
    int y_aligned16;  // Y's base is 16-byte aligned (vector stores allowed)
};

template <bool BF16, int BN, int STAGES, bool GELU>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcArgs a) {
    constexpr int BM = 128;
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int BK = 128 / ESZ;                 // K elements per stage (128 bytes)
    constexpr uint32_t A_BYTES = BM * 128;        // 16 KiB
    constexpr uint32_t B_BYTES = BN * 128;
    constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES;
    constexpr int MMAS = 4;                       // 32 bytes of K per MMA
    constexpr uint32_t TMEM_COLS = BN;            // power of two, >= 32
    constexpr uint32_t IDESC = make_idesc(BF16 ? 1u : 2u, BM, BN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "N tile");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int nkb = (a.K + BK - 1) / BK;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);
    const uint32_t accum_bar = smem_u32(bars + 2 * STAGES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum_bar, 1);
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto give_up = [&]() {
        atomicExch(s_abort, 1);
        atomicExch(a.status, (int)LIN_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (*(volatile int*)s_abort || !mbar_wait(empty0 + 8 * s, ph ^ 1)) {
                    give_up();
                    break;
                }
                mbar_expect_tx(full0 + 8 * s, STAGE_TX);
                tma_load_2d(smem_u32(sA + s * A_BYTES), &tmA, full0 + 8 * s, kb * BK, m0);
                tma_load_2d(smem_u32(sB + s * B_BYTES), &tmB, full0 + 8 * s, kb * BK, n0);
                issued = kb + 1;
            }
            if (*(volatile int*)s_abort) {
                // Drain this CTA's own copies still in flight before the CTA exits.
                const int first = issued > STAGES ? issued - STAGES : 0;
                for (int kb = first; kb < issued; ++kb) mbar_wait(full0 + 8 * (kb % STAGES), (kb / STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (*(volatile int*)s_abort || !mbar_wait(full0 + 8 * s, ph)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + s * A_BYTES));
                const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
                for (int kk = 0; kk < MMAS; ++kk)
                    tc_mma<BF16>(tmem_base, ad + 2u * kk, bd + 2u * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
                tc_commit(empty0 + 8 * s);
            }
            tc_commit(accum_bar);
            // Do not reach the teardown before this CTA's MMAs have completed.
            if (!mbar_wait(accum_bar, 0)) give_up();
        }
    } else {
        // ---- epilogue: warps 2..5 ----
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int m = m0 + q * 32 + lane;
        const bool mine = mbar_wait(accum_bar, 0);
        if (!mine) give_up();
        tc_fence_after();
        // tcgen05.ld is warp-collective: the warp proceeds only if every lane saw
        // the accumulator complete and no role of this CTA gave up.
        const bool ok = __all_sync(0xffffffffu, mine && *(volatile int*)s_abort == 0);
        if (ok) {
            const int N = a.N;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int nb = n0 + c * 32;
                if (nb >= N) break;  // warp-uniform
                uint32_t r[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 32), r);
                if (m < a.M) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = nb + j;
                        const float b = (a.bias && n < N) ? __ldg(a.bias + n) : 0.f;
                        v[j] = epilogue<GELU>(__uint_as_float(r[j]), b);
                    }
                    const bool full = nb + 32 <= N;
                    if constexpr (BF16) {
                        uint16_t* dst = static_cast<uint16_t*>(a.Y) + (size_t)m * N + nb;
                        if (full && (N % 8) == 0 && a.y_aligned16) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 o;
                                o.x = pack_bf16x2(v[j], v[j + 1]);
                                o.y = pack_bf16x2(v[j + 2], v[j + 3]);
                                o.z = pack_bf16x2(v[j + 4], v[j + 5]);
                                o.w = pack_bf16x2(v[j + 6], v[j + 7]);
                                *reinterpret_cast<uint4*>(dst + j) = o;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (nb + j < N) dst[j] = f32_to_bf16_bits(v[j]);
                        }
                    } else {
                        float* dst = static_cast<float*>(a.Y) + (size_t)m * N + nb;
                        if (full && (N % 4) == 0 && a.y_aligned16) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (nb + j < N) dst[j] = v[j];
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

template <bool BF16, int BN, int STAGES, bool GELU>
int launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const TcArgs& a, dim3 grid, cudaStream_t st) {
    constexpr size_t smem = STAGES * (128 * 128 + BN * 128) + 1024 + 256;
    auto kern = tc_kernel<BF16, BN, STAGES, GELU>;
    static unsigned long long attr_set = 0;  // one attribute call per instantiation and device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIN_ERR_CUDA;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LIN_ERR_CUDA;
        attr_set |= bit;
    }
    kern<<<grid, kTcThreads, smem, st>>>(ta, tb, a);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

template <bool BF16, bool GELU>
int launch_variant(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const TcArgs& a, dim3 grid,
                   cudaStream_t st) {
    switch (variant) {
        case 0: return launch_cfg<BF16, kTcCfg[0].bn, kTcCfg[0].stages, GELU>(ta, tb, a, grid, st);
        case 1: return launch_cfg<BF16, kTcCfg[1].bn, kTcCfg[1].stages, GELU>(ta, tb, a, grid, st);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}
}  // namespace

bool make_kmajor_map(CUtensorMap* map, const void* base, bool bf16, int rows, int K, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int launch_tc(const Problem& p, const lin_plan& plan) {
    const bool bf16 = p.precision == LIN_PREC_BF16;
    CUtensorMap ta, tb;
    if (!make_kmajor_map(&ta, p.X, bf16, p.M, p.K, 128)) return LIN_ERR_CUDA;
    if (!make_kmajor_map(&tb, p.W, bf16, p.N, p.K, plan.bn)) return LIN_ERR_CUDA;
    TcArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bias = p.bias;
    a.Y = p.Y;
    a.status = p.dev_status;
    a.y_aligned16 = (reinterpret_cast<uintptr_t>(p.Y) % 16) == 0;
    const dim3 grid(plan.grid_x, plan.grid_y, 1);
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    if (bf16)
        return gelu ? launch_variant<true, true>(plan.variant, ta, tb, a, grid, p.stream)
                    : launch_variant<true, false>(plan.variant, ta, tb, a, grid, p.stream);
    return gelu ? launch_variant<false, true>(plan.variant, ta, tb, a, grid, p.stream)
                : launch_variant<false, false>(plan.variant, ta, tb, a, grid, p.stream);
}

}  // namespace lin
