// Skinny linear layer (M <= 16, bf16), stream-K over the whole GPU.
//
// Same stream and multiply as the cluster kernel (skinny.cu): TMA copies of W
// tiles and X tiles into a shared-memory ring, tcgen05.mma with W as the
// 128-row operand and the 16-row batch as N, fp32 accumulators in TMEM. What
// differs is the division of work ("Filling the chip": enough blocks for every
// SM; "Optimizing a GPT-2-class transformer on a GPU", Act I: split-K
// combined by a fixed-order reduction):
//
// * The tiles (128 W rows x KBOX*64 K) are numbered t = rb * KT + kb (row
//   block rb, K tile kb) and the P CTAs (one per SM) take equal contiguous
//   runs [p*T/P, (p+1)*T/P). Every SM streams the same number of bytes, and
//   with one CTA per SM the second shared-memory slot stays free for the next
//   layer's kernel to start prefetching its weights early.
// * A run crosses row blocks; each maximal piece inside one row block is a
//   segment. The MMA thread alternates two 16-column TMEM accumulators between
//   segments, so the epilogue of one segment overlaps the next one's MMAs.
// * A segment that covers a whole row block is finished in place. Otherwise
//   its 16 x 128 partial sums go to workspace slot (p + rb) - unique, because
//   runs advance monotonically in both p and rb - and the CTA that brings the
//   row block's arrival count to its number of contributors adds the slots of
//   contributors p_first..p_last in that order, then applies bias and GELU and
//   stores bf16. The result does not depend on which CTA finishes last.
// * Programmatic dependent launch as in the cluster kernel: W copies of the
//   first STAGES tiles are issued before griddepcontrol.wait; X, bias, the
//   workspace and Y are touched only after it.
#include "internal.h"
#include "device_common.cuh"
#include "tc_common.cuh"

namespace lin {
namespace {

struct SkArgs {
    int M, N, K;
    const float* bias;
    uint16_t* Y;
    int* status;
    float* ws;           // slots of M x 128 fp32 partial sums
    unsigned* counters;  // one per row block, zero between launches
    int kt;              // K tiles per row block
    long long T;         // total tiles
    int P;               // CTAs
};

constexpr int kRows = 128;
constexpr int kMP = 16;
constexpr uint32_t kWBox = kRows * 128;  // one 128-byte-wide W box
constexpr uint32_t kXBox = kMP * 128;

constexpr size_t sk_smem_bytes(int stages, int kbox) {
    return 1024 + (size_t)stages * kbox * (kWBox + kXBox) + (2 * stages + 4) * 8 + 32;
}

// CTA owning tile t: the largest p with floor(p*T/P) <= t.
__device__ __forceinline__ int owner_of(long long t, long long T, int P) {
    return (int)(((t + 1) * P - 1) / T);
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int STAGES, int KBOX, bool GELU>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
skinny_sk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const SkArgs a) {
    constexpr uint32_t WB = KBOX * kWBox, XB = KBOX * kXBox;
    constexpr uint32_t TMEM_COLS = 32;  // two 16-column accumulators
    constexpr uint32_t IDESC = make_idesc(1u, kRows, kMP);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem;
    uint8_t* sX = sW + STAGES * WB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sX + STAGES * XB);  // full[S] empty[S] accf[2] acce[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);
    int* s_last = s_abort + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.x;
    const long long t0 = (long long)p * a.T / a.P, t1 = (long long)(p + 1) * a.T / a.P;
    const int ntile = (int)(t1 - t0);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();

    auto give_up = [&]() {
        atomicExch(s_abort, 1);
        atomicExch(a.status, (int)LIN_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---- producer ----
            auto load_w = [&](int i, long long t) {
                const int s = i % STAGES;
                const int rb = (int)(t / a.kt), kb = (int)(t % a.kt);
#pragma unroll
                for (int b = 0; b < KBOX; ++b)
                    tma_load_2d(smem_u32(sW + s * WB + b * kWBox), &tmW, full0 + 8 * s, (kb * KBOX + b) * 64,
                                rb * kRows);
            };
            auto load_x = [&](int i, long long t) {
                const int s = i % STAGES;
                const int kb = (int)(t % a.kt);
#pragma unroll
                for (int b = 0; b < KBOX; ++b)
                    tma_load_2d(smem_u32(sX + s * XB + b * kXBox), &tmX, full0 + 8 * s, (kb * KBOX + b) * 64, 0);
            };
            const int pre = ntile < STAGES ? ntile : STAGES;
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(full0 + 8 * i, WB + XB);
                load_w(i, t0 + i);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) load_x(i, t0 + i);
            int issued = pre;
            for (int i = pre; i < ntile; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (*(volatile int*)s_abort || !mbar_wait(empty0 + 8 * s, ph ^ 1)) {
                    give_up();
                    break;
                }
                mbar_expect_tx(full0 + 8 * s, WB + XB);
                load_w(i, t0 + i);
                load_x(i, t0 + i);
                issued = i + 1;
            }
            if (*(volatile int*)s_abort) {
                const int first = issued > STAGES ? issued - STAGES : 0;
                for (int i = first; i < issued; ++i) mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            int sg = 0;
            bool ok = true;
            for (int i = 0; i < ntile && ok; ++i) {
                const long long t = t0 + i;
                const bool first = (i == 0) || (t % a.kt == 0);
                const bool last = (i + 1 == ntile) || ((t + 1) % a.kt == 0);
                const uint32_t buf = sg & 1;
                if (first && !mbar_wait(acce0 + 8 * buf, ((sg >> 1) & 1) ^ 1)) ok = false;
                const int s = i % STAGES;
                if (ok && (*(volatile int*)s_abort || !mbar_wait(full0 + 8 * s, (i / STAGES) & 1))) ok = false;
                if (!ok) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + buf * kMP;
#pragma unroll
                for (int b = 0; b < KBOX; ++b) {
                    const uint64_t ad = sw128_kmajor_desc(smem_u32(sW + s * WB + b * kWBox));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(sX + s * XB + b * kXBox));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma<true>(d, ad + 2u * kk, bd + 2u * kk, IDESC, (first && b == 0 && kk == 0) ? 0u : 1u);
                }
                tc_commit(empty0 + 8 * s);
                if (last) {
                    tc_commit(accf0 + 8 * buf);
                    ++sg;
                }
            }
            // Do not reach the teardown before this CTA's MMAs have completed.
            if (sg > 0 && !mbar_wait(accf0 + 8 * ((sg - 1) & 1), ((sg - 1) >> 1) & 1)) give_up();
        }
    } else {
        // ---- epilogue warps 2..5: TMEM lanes 32q..32q+31 = W rows of the block ----
        pdl_wait();
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int M = a.M, N = a.N;
        const size_t slot_elems = (size_t)M * kRows;
        int sg = 0;
        long long t = t0;
        while (t < t1) {
            const int rb = (int)(t / a.kt);
            const long long rb_begin = (long long)rb * a.kt, rb_end = rb_begin + a.kt;
            const long long seg_end = t1 < rb_end ? t1 : rb_end;
            const uint32_t buf = sg & 1;
            const bool mine = mbar_wait(accf0 + 8 * buf, (sg >> 1) & 1);
            if (!mine) give_up();
            tc_fence_after();
            float v[kMP];
            const bool ok = __all_sync(0xffffffffu, mine && *(volatile int*)s_abort == 0);
            if (ok) {
                uint32_t r[16];
                tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kMP, r);
#pragma unroll
                for (int m = 0; m < kMP; ++m) v[m] = __uint_as_float(r[m]);
            } else {
#pragma unroll
                for (int m = 0; m < kMP; ++m) v[m] = 0.f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * buf);
            // After a give-up the loop still runs every segment with the same
            // named barriers (its values are zero and the status word is set),
            // so no epilogue warp waits on one that has left.

            const int n = rb * kRows + row;
            const float bn = (a.bias && n < N) ? __ldg(a.bias + n) : 0.f;
            if (t == rb_begin && seg_end == rb_end) {
                // the whole row block is this CTA's
                if (n < N) {
#pragma unroll
                    for (int m = 0; m < kMP; ++m)
                        if (m < M) a.Y[(size_t)m * N + n] = f32_to_bf16_bits(epilogue<GELU>(v[m], bn));
                }
            } else {
                // Publish this segment's partial sums: plain stores by all, then one
                // gpu-scope fence (cumulative over the named barrier) before the
                // arrival count; the last arriver fences again before reading.
                float* part = a.ws + (size_t)(p + rb) * slot_elems;
#pragma unroll
                for (int m = 0; m < kMP; ++m)
                    if (m < M) __stcg(part + m * kRows + row, v[m]);
                epi_bar_sync();
                const int pf = owner_of(rb_begin, a.T, a.P);
                const int pl = owner_of((rb_end < a.T ? rb_end : a.T) - 1, a.T, a.P);
                if (threadIdx.x == 64) {
                    __threadfence();
                    const unsigned prev = atomicAdd(&a.counters[rb], 1u);
                    const int last = prev == (unsigned)(pl - pf);
                    if (last) {
                        a.counters[rb] = 0u;  // re-arm for the next launch
                        __threadfence();
                    }
                    *s_last = last;
                }
                epi_bar_sync();
                if (*(volatile int*)s_last && n < N) {
                    float acc[kMP];
#pragma unroll
                    for (int m = 0; m < kMP; ++m) acc[m] = 0.f;
                    // contributors in fixed order; each one's 16 rows are independent loads
#pragma unroll 2
                    for (int pp = pf; pp <= pl; ++pp) {
                        const float* src = a.ws + (size_t)(pp + rb) * slot_elems + row;
                        float tmp[kMP];
#pragma unroll
                        for (int m = 0; m < kMP; ++m) tmp[m] = (m < M) ? __ldcg(src + m * kRows) : 0.f;
#pragma unroll
                        for (int m = 0; m < kMP; ++m) acc[m] += tmp[m];
                    }
#pragma unroll
                    for (int m = 0; m < kMP; ++m)
                        if (m < M) a.Y[(size_t)m * N + n] = f32_to_bf16_bits(epilogue<GELU>(acc[m], bn));
                }
                epi_bar_sync();  // s_last is reused by the next segment
            }
            ++sg;
            t = seg_end;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int STAGES, int KBOX, bool GELU>
int launch_cfg(const CUtensorMap& tw, const CUtensorMap& tx, const SkArgs& a, bool early, cudaStream_t st) {
    constexpr size_t smem = sk_smem_bytes(STAGES, KBOX);
    auto kern = skinny_sk_kernel<STAGES, KBOX, GELU>;
    static unsigned long long attr_set = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIN_ERR_CUDA;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LIN_ERR_CUDA;
        attr_set |= bit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.P, 1, 1);
    cfg.blockDim = dim3(kSkinnyThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = early ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, tw, tx, a) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

template <int STAGES, int KBOX>
int launch_epi(bool gelu, const CUtensorMap& tw, const CUtensorMap& tx, const SkArgs& a, bool early,
               cudaStream_t st) {
    return gelu ? launch_cfg<STAGES, KBOX, true>(tw, tx, a, early, st)
                : launch_cfg<STAGES, KBOX, false>(tw, tx, a, early, st);
}

}  // namespace

size_t skinny_sk_workspace_bytes(int P, int M, int N, int K, int kbox) {
    const int nrb = (N + kRows - 1) / kRows;
    (void)K;
    (void)kbox;
    return kCounterBytes + align_up((size_t)(P + nrb) * (size_t)M * kRows * sizeof(float), 256);
}

int launch_skinny_sk(const Problem& p, const lin_plan& plan) {
    const SkinnySkCfg c = kSkinnySkCfg[plan.variant];
    CUtensorMap tw, tx;
    if (!make_kmajor_map(&tw, p.W, true, p.N, p.K, kRows)) return LIN_ERR_CUDA;
    if (!make_kmajor_map(&tx, p.X, true, p.M, p.K, kMP)) return LIN_ERR_CUDA;
    SkArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bias = p.bias;
    a.Y = static_cast<uint16_t*>(p.Y);
    a.status = p.dev_status;
    a.counters = splitk_counters(p.workspace);
    a.ws = splitk_partials(p.workspace);
    a.kt = (p.K + 64 * c.kbox - 1) / (64 * c.kbox);
    const int nrb = (p.N + kRows - 1) / kRows;
    a.T = (long long)nrb * a.kt;
    a.P = plan.grid_x;
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    switch (plan.variant) {
        case 0: return launch_epi<kSkinnySkCfg[0].stages, kSkinnySkCfg[0].kbox>(gelu, tw, tx, a, p.early_start, p.stream);
        case 1: return launch_epi<kSkinnySkCfg[1].stages, kSkinnySkCfg[1].kbox>(gelu, tw, tx, a, p.early_start, p.stream);
        case 2: return launch_epi<kSkinnySkCfg[2].stages, kSkinnySkCfg[2].kbox>(gelu, tw, tx, a, p.early_start, p.stream);
        case 3: return launch_epi<kSkinnySkCfg[3].stages, kSkinnySkCfg[3].kbox>(gelu, tw, tx, a, p.early_start, p.stream);
        case 4: return launch_epi<kSkinnySkCfg[4].stages, kSkinnySkCfg[4].kbox>(gelu, tw, tx, a, p.early_start, p.stream);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace lin
