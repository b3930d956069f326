// Skinny linear layer, M <= 16, bf16 in, fp32 accumulate, bf16 out.
//
// The workload of "One multiply, one RTX 5090, eight kernels": a batch of 16
// vectors against a 4096 x 4096 weight stored out x in. Each weight value
// feeds only M products, so the kernel is a stream over W and its speed is the
// rate at which W leaves HBM ("Where the time goes": the loads-only probe took
// as long as the full kernel). The page's kernels request the next K slice
// before multiplying the current one and split K across blocks ("Inside one
// block", "Filling the chip"); on sm_103a:
//
// * Stream: one thread issues 2-D TMA copies of W tiles (128 rows x 128 bytes
//   of K, 16 KiB) and the matching X tile (16 rows x 128 bytes) into a
//   STAGES-deep shared-memory ring, so ~80 KiB of W per CTA are in flight -
//   enough bytes in flight per SM to cover HBM latency (Little's law), which
//   register-staged loads cannot reach at this occupancy.
// * Multiply ("swap AB"): the tensor core computes D = W_tile . X_tile^T with
//   tcgen05.mma M = 128 (W rows), N = 16 (the batch, zero-padded by the copy
//   engine when M < 16), K = 16 per instruction, straight from the swizzled
//   tiles, accumulating in 16 TMEM columns. At M = 16 the FFMA units could
//   not keep up with HBM (16 FLOP per W byte ~ 108 TFLOP/s at 6.8 TB/s).
// * Split-K in a thread-block cluster: the CL CTAs of a cluster share one
//   128-row block of W and take consecutive K ranges. K is always cut into 8
//   segments with their own TMEM accumulators; a CTA adds its segments by a
//   balanced pairwise tree, pushes that partial into the inbox of the CTA that
//   finishes the columns (distributed shared memory), and the finishing CTA
//   adds the CL partials by the same tree, applies bias and GELU and stores
//   bf16. The sum is therefore the same balanced tree over the 8 segments for
//   every cluster size - bitwise identical across split choices and runs (the
//   fixed-order reduction of "Optimizing a GPT-2-class transformer on a GPU",
//   Act I). No global workspace.
// * Programmatic dependent launch: a call's CTAs start as the previous
//   kernel's CTAs leave the SMs and, before griddepcontrol.wait, ask the L2 to
//   fetch this CTA's whole share of W: each of the 128 epilogue threads issues
//   one bulk L2 prefetch of its W row's K range (an L2 prefetch returns nothing
//   to the SM, so it is safe whatever the previous kernel writes). HBM keeps
//   streaming across the call boundary, and after the wait the copies into
//   shared memory hit the L2 (measured: the post-wait stream of a 16 x 4096 x
//   4096 call falls from ~5 us to ~2.4 us; tensor-map prefetches issued by the
//   producer thread did not reach the L2 in time and held back its first
//   copies). When the caller allows it (the host checks that W does not
//   overlap the previous call's output), the W copies of the first STAGES
//   stages go straight to shared memory before the wait, and X too when it is
//   not the previous call's output (independent layers then stream
//   concurrently). Bias, the residual and Y are touched only after the wait.
#include "internal.h"
#include "device_common.cuh"
#include "tc_common.cuh"
#include "timeline.cuh"

namespace lin {
namespace {

#ifdef LIN_TIMELINE
// Timeline stamps per CTA, records numbered in the order the CTAs start
// (consecutive launches follow one another): [0] set up, [1] producer past
// its dependency wait, [2] MMAs complete, [3] done; [16 + i] stage i's
// copies landed (seen by the MMA issuer), i < 160.
__device__ unsigned long long g_timeline_skinny[kTimelineCtas * kTimelineSlots];
__device__ unsigned g_timeline_skinny_next;
#endif

struct SkinnyArgs {
    int M, N, K;
    const float* bias;
    uint16_t* Y;
    const uint16_t* R;  // residual added after the activation (M x N bf16, may be Y itself), or null
    int* status;
    int kblocks;  // ceil(K / (64 * KBOX)): stages of K per 128-row block
    int early_w;  // W may be read before the dependency wait (it is not the previous call's output)
    int early_x;  // X may be read before the dependency wait (implies early_w)
    int prefetch; // ask the L2 for this CTA's share of W before the dependency wait
    const uint16_t* W;  // N x K, for the L2 prefetch (the copies go through the tensor map)
};

constexpr int kSkSegs = 8;    // K segments: the fixed shape of the summation tree
constexpr int kSkRows = 128;  // W rows (outputs) per cluster
constexpr int kSkMP = 16;     // batch rows, padded to the MMA N
constexpr uint32_t kSkWBox = kSkRows * 128;  // one 128-byte-wide box of W
constexpr uint32_t kSkXBox = kSkMP * 128;

// A stage holds KBOX boxes of 64 K each: the boxes of one stage are issued
// together, so each W row is read as a run of KBOX * 128 contiguous bytes
// (DRAM rows stay open across the run). Shared memory: the stage ring, then
// (cluster split) the incoming partial sums of the CL CTAs for the columns
// this CTA finishes, then the mbarriers.
constexpr size_t skinny_smem_bytes(int stages, int kbox, int cl) {
    return 1024 + (size_t)stages * kbox * (kSkWBox + kSkXBox) + (cl > 1 ? (size_t)cl * kSkMP * (kSkRows / cl) * 4 : 0) +
           (2 * stages + 2) * 8 + 16;
}

struct Vec16 {
    float x[kSkMP];
};

__device__ __forceinline__ Vec16 add16(const Vec16& a, const Vec16& b) {
    Vec16 r;
#pragma unroll
    for (int m = 0; m < kSkMP; ++m) r.x[m] = a.x[m] + b.x[m];
    return r;
}

// One segment's sum: its NACC accumulators added pairwise, left to right.
template <int NACC>
__device__ __forceinline__ Vec16 segment_sum(uint32_t lane_base, int ls) {
    Vec16 acc[NACC];
#pragma unroll
    for (int c = 0; c < NACC; ++c) {
        uint32_t r[16];
        tmem_ld16(lane_base + (uint32_t)((ls * NACC + c) * kSkMP), r);
#pragma unroll
        for (int m = 0; m < kSkMP; ++m) acc[c].x[m] = __uint_as_float(r[m]);
    }
    if constexpr (NACC == 1) return acc[0];
    else if constexpr (NACC == 2) return add16(acc[0], acc[1]);
    else if constexpr (NACC == 3) return add16(add16(acc[0], acc[1]), acc[2]);
    else return add16(add16(acc[0], acc[1]), add16(acc[2], acc[3]));
}

// Balanced pairwise tree over N consecutive local segments starting at `first`.
template <int N, int NACC, class NonEmpty>
__device__ __forceinline__ Vec16 tree_of_segments(uint32_t lane_base, int first, NonEmpty nonempty) {
    if constexpr (N == 1) {
        // tcgen05.ld is warp-collective: the condition is the same for all lanes.
        if (nonempty(first)) return segment_sum<NACC>(lane_base, first);
        return Vec16{};
    } else {
        const Vec16 lo = tree_of_segments<N / 2, NACC>(lane_base, first, nonempty);
        const Vec16 hi = tree_of_segments<N / 2, NACC>(lane_base, first + N / 2, nonempty);
        return add16(lo, hi);
    }
}

// Balanced pairwise tree over the partial sums of N consecutive ranks (stride apart).
template <int N>
__device__ __forceinline__ float tree_of_ranks(const float* p, int stride, int first) {
    if constexpr (N == 1)
        return p[first * stride];
    else
        return tree_of_ranks<N / 2>(p, stride, first) + tree_of_ranks<N / 2>(p, stride, first + N / 2);
}

template <int STAGES, int KBOX, int CL, bool GELU>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const SkinnyArgs a) {
    constexpr int NACC = KBOX < 4 ? KBOX : 4;          // independent accumulators (MMA chains) per segment
    constexpr int LSEG = kSkSegs / CL;                 // K segments of this CTA
    constexpr int ACC_COLS = LSEG * NACC * kSkMP;
    constexpr uint32_t TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
    static_assert(kSkSegs % CL == 0 && ACC_COLS <= 512, "segments per CTA");
    constexpr uint32_t IDESC = make_idesc(1u, kSkRows, kSkMP);
    constexpr int COLS = kSkRows / CL;  // output columns this CTA finishes
    constexpr uint32_t WB = KBOX * kSkWBox, XB = KBOX * kSkXBox;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem;
    uint8_t* sX = sW + STAGES * WB;
    float* inbox = reinterpret_cast<float*>(sX + STAGES * XB);  // [CL][kSkMP][COLS] (cluster split)
    uint64_t* bars = reinterpret_cast<uint64_t*>(inbox + (CL > 1 ? CL * kSkMP * COLS : 0));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kSkRows;
    const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
    // Segment s covers K stages [s*kblocks/8, (s+1)*kblocks/8); this CTA owns
    // segments [rank*LSEG, rank*LSEG + LSEG).
    auto seg_begin = [&](int sg) { return (int)((long long)sg * a.kblocks / kSkSegs); };
    const int seg0 = (int)rank * LSEG;
    const int kb0 = seg_begin(seg0);
    const int kb1 = seg_begin(seg0 + LSEG);
    const int nkb = kb1 - kb0;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t accum_bar = smem_u32(bars + 2 * STAGES), inbox_bar = smem_u32(bars + 2 * STAGES + 1);

#ifdef LIN_TIMELINE
    __shared__ unsigned timeline_rec_sh;
    if (threadIdx.x == 0) timeline_rec_sh = atomicAdd(&g_timeline_skinny_next, 1u);
#endif
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum_bar, 1);
        mbar_init(inbox_bar, kSkRows);  // one arrival per W row of the block, from whichever CTA holds it
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Peers may write into this CTA's inbox only after every CTA of the cluster
    // initialised its barriers: arrive now, wait just before the first remote write.
    if constexpr (CL > 1) cluster_arrive_relaxed();
    const uint32_t tmem_base = *tmem_slot;
#ifdef LIN_TIMELINE
    const unsigned trec = timeline_rec_sh;
#endif
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) LIN_STAMP(g_timeline_skinny, trec, 0);

    auto give_up = [&]() {
        atomicExch(s_abort, 1);
        atomicExch(a.status, (int)LIN_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---- producer: W tiles early, X tiles after the dependency wait ----
            auto load_w = [&](int i) {
                const int s = i % STAGES;
#pragma unroll
                for (int b = 0; b < KBOX; ++b)
                    tma_load_2d(smem_u32(sW + s * WB + b * kSkWBox), &tmW, full0 + 8 * s, ((kb0 + i) * KBOX + b) * 64,
                                n0);
            };
            auto load_x = [&](int i) {
                const int s = i % STAGES;
#pragma unroll
                for (int b = 0; b < KBOX; ++b)
                    tma_load_2d(smem_u32(sX + s * XB + b * kSkXBox), &tmX, full0 + 8 * s, ((kb0 + i) * KBOX + b) * 64,
                                0);
            };
            const int pre = nkb < STAGES ? nkb : STAGES;
            if (a.early_w) {
                // W (and X when allowed) straight into the ring; the epilogue
                // threads ask the L2 for the rest of the share meanwhile.
                for (int i = 0; i < pre; ++i) {
                    mbar_expect_tx(full0 + 8 * i, WB + XB);
                    load_w(i);
                    if (a.early_x) load_x(i);
                }
                if (!a.early_x) {
                    pdl_wait();
                    LIN_STAMP(g_timeline_skinny, trec, 1);
                    for (int i = 0; i < pre; ++i) load_x(i);
                }
            } else {
                // Nothing is read before the wait (the epilogue threads ask the
                // L2 for the share meanwhile).
                pdl_wait();
                LIN_STAMP(g_timeline_skinny, trec, 1);
                for (int i = 0; i < pre; ++i) {
                    mbar_expect_tx(full0 + 8 * i, WB + XB);
                    load_w(i);
                    load_x(i);
                }
            }
            int issued = pre;
            for (int i = pre; i < nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (*(volatile int*)s_abort || !mbar_wait(empty0 + 8 * s, ph ^ 1)) {
                    give_up();
                    break;
                }
                mbar_expect_tx(full0 + 8 * s, WB + XB);
                load_w(i);
                load_x(i);
                issued = i + 1;
            }
            if (*(volatile int*)s_abort) {
                const int first = issued > STAGES ? issued - STAGES : 0;
                for (int i = first; i < issued; ++i) mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && nkb > 0) {
            // ---- MMA issuer: box b of every stage accumulates into accumulator b % NACC,
            // so up to NACC MMA chains run side by side ----
            int ls = 0;  // local segment of the current stage
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                while (kb0 + i >= seg_begin(seg0 + ls + 1)) ++ls;
                const bool seg_first = (kb0 + i == seg_begin(seg0 + ls));
                if (*(volatile int*)s_abort || !mbar_wait(full0 + 8 * s, ph)) {
                    give_up();
                    break;
                }
                if (i < 160) LIN_STAMP(g_timeline_skinny, trec, 16 + i);
                tc_fence_after();
#pragma unroll
                for (int b = 0; b < KBOX; ++b) {
                    const uint64_t ad = sw128_kmajor_desc(smem_u32(sW + s * WB + b * kSkWBox));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(sX + s * XB + b * kSkXBox));
                    const uint32_t d = tmem_base + (uint32_t)((ls * NACC + b % NACC) * kSkMP);
                    const bool fresh = seg_first && (b < NACC);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma<true>(d, ad + 2u * kk, bd + 2u * kk, IDESC, (fresh && kk == 0) ? 0u : 1u);
                }
                tc_commit(empty0 + 8 * s);
            }
            tc_commit(accum_bar);
            if (!mbar_wait(accum_bar, 0)) give_up();
            LIN_STAMP(g_timeline_skinny, trec, 2);
        }
    } else {
        // ---- epilogue warps 2..5: TMEM lane quadrant q holds W rows 32q..32q+31 ----
        const int q = warp & 3;
        const int row = q * 32 + lane;
        if (a.prefetch && nkb > 0 && n0 + row < a.N) {
            // This CTA's K range of W row n0 + row to the L2 (16-byte aligned:
            // K * 2 is a multiple of 16 and the range starts on a stage), past
            // the stages that the producer copies before the wait.
            const int early = a.early_w ? (nkb < STAGES ? nkb : STAGES) : 0;
            const int k0 = (kb0 + early) * KBOX * 64;
            const int k1 = kb1 * KBOX * 64 < a.K ? kb1 * KBOX * 64 : a.K;
            if (k1 > k0) {
                const uint16_t* src = a.W + (size_t)(n0 + row) * a.K + k0;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((unsigned)(k1 - k0) * 2u)
                             : "memory");
            }
        }
        pdl_wait();
        const int M = a.M, N = a.N;
        // The bias and residual values this thread adds, fetched while the
        // accumulators fill. Without a cluster split a thread finishes its W row
        // n for every batch row; with one it finishes PER outputs of one column
        // (128 threads, a multiple of the COLS columns this CTA finishes).
        static_assert(CL == 1 || 128 % COLS == 0, "columns per finishing thread");
        constexpr int PER = CL == 1 ? kSkMP : kSkMP * COLS / 128;
        const int t = threadIdx.x - 64;
        const int n_out = CL == 1 ? n0 + row : n0 + (int)rank * COLS + t % COLS;
        auto m_out = [&](int e) { return CL == 1 ? e : (t + 128 * e) / COLS; };
        const float b_out = (a.bias && n_out < N) ? __ldg(a.bias + n_out) : 0.f;
        float r_out[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e)
            r_out[e] = (a.R && m_out(e) < M && n_out < N) ? bf16_bits_to_f32(a.R[(size_t)m_out(e) * N + n_out]) : 0.f;
        Vec16 v = {};
        if (nkb > 0) {
            const bool mine = mbar_wait(accum_bar, 0);
            if (!mine) give_up();
            tc_fence_after();
            if (__all_sync(0xffffffffu, mine && *(volatile int*)s_abort == 0)) {
                // Empty segments (fewer K stages than segments) hold no MMA result: zero.
                const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                v = tree_of_segments<LSEG, NACC>(lane_base, 0, [&](int ls) {
                    return seg_begin(seg0 + ls) < seg_begin(seg0 + ls + 1);
                });
            }
        }
        if constexpr (CL == 1) {
            const int n = n_out;
            if (n < N) {
#pragma unroll
                for (int m = 0; m < kSkMP; ++m)
                    if (m < M) a.Y[(size_t)m * N + n] = f32_to_bf16_bits(epilogue<GELU, true>(v.x[m], b_out) + r_out[m]);
            }
        } else {
            // Push this row's partial sums into the inbox of the CTA that finishes it,
            // then arrive there (release at cluster scope covers the stores).
            cluster_wait();
            const uint32_t owner = (uint32_t)(row / COLS);
            const int col = row % COLS;
            const uint32_t dst = dsmem_map(smem_u32(inbox + ((int)rank * kSkMP) * COLS + col), owner);
#pragma unroll
            for (int m = 0; m < kSkMP; ++m) dsmem_st_f32(dst + (uint32_t)(m * COLS * 4), v.x[m]);
            mbar_arrive_remote(dsmem_map(inbox_bar, owner));
            // Finish this CTA's columns: the CL partial sums added in rank order.
            const bool ok = mbar_wait_cluster(inbox_bar, 0);
            if (!ok) give_up();
            const int c = t % COLS;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int m = m_out(e);
                if (ok && m < M && n_out < N) {
                    const float acc = tree_of_ranks<CL>(inbox + m * COLS + c, kSkMP * COLS, 0);
                    a.Y[(size_t)m * N + n_out] = f32_to_bf16_bits(epilogue<GELU, true>(acc, b_out) + r_out[e]);
                }
            }
        }
    }

    if (threadIdx.x == 64) LIN_STAMP(g_timeline_skinny, trec, 3);
    __syncwarp();
    if constexpr (CL > 1) {
        // Every thread that arrived on the cluster barrier also waits on it.
        if (warp < 2) cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int STAGES, int KBOX, int CL, bool GELU>
int launch_cfg(const CUtensorMap& tw, const CUtensorMap& tx, const SkinnyArgs& a, int grid_x, bool early,
               cudaStream_t st) {
    constexpr size_t smem = skinny_smem_bytes(STAGES, KBOX, CL);
    static_assert(skinny_smem_bytes(STAGES, KBOX, CL) <= 227 * 1024, "shared memory");
    auto kern = skinny_kernel<STAGES, KBOX, CL, GELU>;
    static std::atomic<unsigned long long> attr_set{0};  // per instantiation: one bit per device
    if (ensure_smem_attr(attr_set, kern, smem) != LIN_OK) return LIN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, CL, 1);
    cfg.blockDim = dim3(kSkinnyThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (CL > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = CL;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (early) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, tw, tx, a) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

template <int STAGES, int KBOX, bool GELU>
int launch_split(int splits, const CUtensorMap& tw, const CUtensorMap& tx, const SkinnyArgs& a, int grid_x,
                 bool early, cudaStream_t st) {
    switch (splits) {
        case 1: return launch_cfg<STAGES, KBOX, 1, GELU>(tw, tx, a, grid_x, early, st);
        case 2: return launch_cfg<STAGES, KBOX, 2, GELU>(tw, tx, a, grid_x, early, st);
        case 4: return launch_cfg<STAGES, KBOX, 4, GELU>(tw, tx, a, grid_x, early, st);
        case 8: return launch_cfg<STAGES, KBOX, 8, GELU>(tw, tx, a, grid_x, early, st);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_skinny(const Problem& p, const lin_plan& plan) {
    CUtensorMap tw, tx;
    if (!make_kmajor_map(&tw, p.W, true, p.N, p.K, kSkRows)) return LIN_ERR_CUDA;
    if (!make_kmajor_map(&tx, p.X, true, p.M, p.K, kSkMP)) return LIN_ERR_CUDA;
    SkinnyArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bias = p.bias;
    a.Y = static_cast<uint16_t*>(p.Y);
    a.R = static_cast<const uint16_t*>(p.residual);
    a.status = p.dev_status;
    a.kblocks = (p.K + 64 * kSkinnyCfg[plan.variant].kbox - 1) / (64 * kSkinnyCfg[plan.variant].kbox);
    a.early_w = p.early_w ? 1 : 0;
    a.early_x = p.early_x ? 1 : 0;
    a.prefetch = p.early_start ? 1 : 0;  // useful only when the CTAs can start before the wait ends
    a.W = static_cast<const uint16_t*>(p.W);
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
#define LIN_SKINNY_CASE(V)                                                                                 \
    case V:                                                                                                \
        return gelu ? launch_split<kSkinnyCfg[V].stages, kSkinnyCfg[V].kbox, true>(                   \
                          plan.splits, tw, tx, a, plan.grid_x, p.early_start, p.stream)                    \
                    : launch_split<kSkinnyCfg[V].stages, kSkinnyCfg[V].kbox, false>(                      \
                          plan.splits, tw, tx, a, plan.grid_x, p.early_start, p.stream);
    switch (plan.variant) {
        LIN_SKINNY_CASE(0)
        LIN_SKINNY_CASE(1)
        LIN_SKINNY_CASE(2)
        LIN_SKINNY_CASE(3)
        LIN_SKINNY_CASE(4)
        default: return LIN_ERR_UNSUPPORTED;
    }
#undef LIN_SKINNY_CASE
}

int timeline_copy_skinny(void* dst, size_t bytes, bool clear) {
#ifdef LIN_TIMELINE
    const size_t total = sizeof(unsigned long long) * kTimelineCtas * kTimelineSlots;
    if (dst && bytes > 0 &&
        cudaMemcpyFromSymbol(dst, g_timeline_skinny, bytes < total ? bytes : total) != cudaSuccess)
        return LIN_ERR_CUDA;
    if (clear) {
        void* p = nullptr;
        const unsigned zero = 0;
        if (cudaGetSymbolAddress(&p, g_timeline_skinny) != cudaSuccess || cudaMemset(p, 0, total) != cudaSuccess ||
            cudaMemcpyToSymbol(g_timeline_skinny_next, &zero, sizeof(zero)) != cudaSuccess)
            return LIN_ERR_CUDA;
    }
    return LIN_OK;
#else
    (void)dst;
    (void)bytes;
    (void)clear;
    return LIN_ERR_UNSUPPORTED;
#endif
}

}  // namespace lin
