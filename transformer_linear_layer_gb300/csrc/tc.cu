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
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "device_common.cuh"

namespace lin {
namespace {

struct TcArgs {
    int M, N, K;
    const float* bias;
    void* Y;
    int* status;
    int y_aligned16;  // Y's base is 16-byte aligned (vector stores allowed)
};

constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s per wait, then give up
constexpr uint32_t kWaitIters = 1u << 30;               // backstop on iterations

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with parity `parity` to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1; i < kWaitIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (stride
// byte offset), leading byte offset unused for this layout, descriptor
// version 1 (bits 46-47), swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor (kind::f16 / kind::tf32): D fp32 (bits 4-5 = 1),
// A and B format (bits 7-9, 10-12: 1 = bf16, 2 = tf32), both K-major
// (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t make_idesc(uint32_t ab_format, int m, int n) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

template <bool BF16>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    if constexpr (BF16) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

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
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over a rows x K row-major tensor, box = 128 bytes of K x box_rows.
bool make_map(CUtensorMap* map, const void* base, bool bf16, int rows, int K, int box_rows) {
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

int launch_tc(const Problem& p, const lin_plan& plan) {
    const bool bf16 = p.precision == LIN_PREC_BF16;
    CUtensorMap ta, tb;
    if (!make_map(&ta, p.X, bf16, p.M, p.K, 128)) return LIN_ERR_CUDA;
    if (!make_map(&tb, p.W, bf16, p.N, p.K, plan.bn)) return LIN_ERR_CUDA;
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
