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
// * Programmatic dependent launch: a CTA may start on an SM as soon as the
//   previous kernel's CTA there has exited, before that whole grid finishes
//   (its prologue overlaps the other SMs' last tiles). Operands
//   are read before griddepcontrol.wait only when neither is that kernel's
//   output; bias and Y always after it.
// * Every wait is bounded (iterations and wall clock); a wait that gives up
//   writes LIN_ERR_DEVICE_TIMEOUT to the status word, the CTA skips its
//   stores, drains its own copies and MMAs, frees TMEM and exits.
#include "internal.h"
#include "device_common.cuh"
#include "tc_common.cuh"
#include "timeline.cuh"

namespace lin {
namespace {

#ifdef LIN_TIMELINE
// Timeline stamps per CTA (blockIdx.x): [0] set up, [1] producer past its
// dependency wait, [2] teardown; per work item j < 32: [8 + 4j] MMAs start
// (accumulator free), [8 + 4j + 1] last MMA and commit issued, [8 + 4j + 2]
// epilogue warp 2 sees the accumulator, [8 + 4j + 3] epilogue warp 2 done,
// [136 + j] epilogue warp 9 done.
__device__ unsigned long long g_timeline_tc[kTimelineCtas * kTimelineSlots];
#endif

struct TcArgs {
    int M, N, K;
    const float* bias;
    void* Y;
    int* status;
    int y_aligned16;     // Y's base is 16-byte aligned (vector stores allowed)
    int bias_aligned16;  // bias is 16-byte aligned (vector loads allowed)
    int early_inputs;    // X and W may be read before the dependency wait (not the previous call's output)
    int prefetch;        // otherwise ask the L2 for the first ring's worth of them before the wait
    int y_tma;           // bf16 Y stored by TMA from 32 x 32 boxes (16-byte aligned rows)
    float* partials;     // stream-K: one 128 x BN fp32 slot per CTA boundary; K split: one per (tile, split)
    unsigned* flags;     // stream-K: 8 hand-over flags per CTA boundary; K split: 8 counters per tile
                         // (zero between launches)
    int ksplits;         // K split (whole tiles, single CTA): each tile's K stages cut in ksplits ranges
    int tail_whole;      // with ksplits > 1: the first tail_whole tiles run whole, only the rest are split
    const void* aux;     // M x N in Y's type (may be Y itself), read in the epilogue, or null:
    int aux_mode;        //   1 adds it after the activation (residual), 2 multiplies by the GELU slope at it
    int aux_vec;         // aux rows are 16-byte aligned (vector loads)
};

// Epilogue staging: each epilogue warp owns a 32 x 32 output tile in shared
// memory, rows padded by 16 bytes so the row-per-lane writes and the
// row-segment reads below are (nearly) free of bank conflicts.
// fp32 outputs pass through in two halves of 16 rows, so both dtypes stage
// about 20 KiB and keep the ring deep.
template <bool BF16>
constexpr int stage_row_bytes() { return BF16 ? 32 * 2 + 16 : 32 * 4 + 16; }
template <bool BF16>
constexpr int stage_rows() { return BF16 ? 32 : 16; }
// Per warp: its rows, plus (bf16) 16 bytes after every 8 rows, which spreads the
// shifted row writes of the unaligned-row store path over the banks.
template <bool BF16>
constexpr int stage_warp_bytes() { return stage_rows<BF16>() * stage_row_bytes<BF16>() + (BF16 ? 64 : 0); }
template <bool BF16>
constexpr int stage_bytes() { return 8 * stage_warp_bytes<BF16>(); }
// Bias staging: each epilogue warp keeps the bias of its BN/2 columns of the
// current tile in shared memory (8 warps x BN/2 floats).
template <int BN>
constexpr int bias_stage_bytes() { return 8 * (BN / 2) * 4; }
// Bytes of one K stage in a CTA: the 128-row A tile and this CTA's W rows
// (all BN of them, or BN/2 for an SM pair).
template <int BN, bool PAIR>
constexpr int tc_stage_bytes() { return 128 * 128 + (PAIR ? BN / 2 : BN) * 128; }
// Ring depth: as many 128-byte K stages as fit beside the staging areas.
template <bool BF16, int BN, bool PAIR>
constexpr int tc_stages() {
    return (227 * 1024 - 2048 - stage_bytes<BF16>() - bias_stage_bytes<BN>()) / tc_stage_bytes<BN, PAIR>() < 8
               ? (227 * 1024 - 2048 - stage_bytes<BF16>() - bias_stage_bytes<BN>()) / tc_stage_bytes<BN, PAIR>()
               : 8;
}
template <bool BF16, int BN, bool PAIR>
constexpr size_t tc_smem_bytes() {
    return 1024 + (size_t)tc_stages<BF16, BN, PAIR>() * tc_stage_bytes<BN, PAIR>() + stage_bytes<BF16>() +
           bias_stage_bytes<BN>() + (2 * tc_stages<BF16, BN, PAIR>() + 4) * 8 + 16;
}

// PAIR: SM-pair MMA. The CTAs run as 2 x 1 clusters and a cluster computes a
// 256 x BN tile with tcgen05.mma.cta_group::2 issued by the even CTA: each CTA
// loads its own 128 rows of X and one half (BN/2 rows) of the W tile into its
// shared memory, the pair's tensor cores read both halves, and each CTA's TMEM
// receives its 128 rows of the accumulator. Per unit of MMA work a CTA stages
// a third less shared-memory data than with a 128 x BN tile of its own (which
// is what bounds the single-CTA form: TMA writes plus tensor-core reads).
// Both CTAs' copies complete the even CTA's "full" barrier; its commits
// release the stage ("empty") and publish the accumulator ("tfull") in both
// CTAs; both CTAs' epilogue warps release the accumulator to its "tempty".
//
// SK: stream-K schedule (single-CTA tiles only). The grid's work is the
// tile-major sequence of (tile, K stage) units; CTA b takes the equal share
// [b * U / G, (b + 1) * U / G), so every SM finishes at the same time however
// the tile count divides the grid. Each share holds at least one tile, so a
// tile is cut at most once, between CTAs b and b + 1: CTA b + 1 computes the
// later K stages first, writes them to the workspace slot of that boundary and
// sets one flag per epilogue warp; CTA b reaches the earlier K stages last,
// waits for the flags, adds the partial sums to its accumulator in that fixed
// order and runs the epilogue (deterministic for a given plan).
//
// LAY: operand layouts (bf16, single-CTA, whole tiles only). 0: both K-major
// (the forward, Y = X W^T). 1: B MN-major (dX = dZ W: A = dZ, B = W read with
// the output column contiguous). 2: A and B MN-major (dW = dZ^T X: A = dZ and
// B = X, both read with the reduction index as the row). The transposes of
// the backward pass are index maps of the TMA boxes and the descriptors'
// major-ness ("Writing a CUDA matmul that catches cuBLAS": keep each operand
// in the layout that makes staging a vector copy, choose the fragment layout
// to match); nothing is transposed in memory. An MN-major stage is one box of
// 64 (MN) x 64 (K rows) per 64 rows or columns of the tile.
// YODD: bf16 Y whose rows are not 16-byte aligned (N not a multiple of 8)
// leaves by the shifted-staging vector stores below (a separate instantiation,
// so that the other paths keep their registers).
template <bool BF16, int BN, bool GELU, bool PAIR, bool SK, int LAY, bool YODD = false>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmY, const TcArgs a) {
    constexpr int STAGES = tc_stages<BF16, BN, PAIR>();
    constexpr int BM = 128;                       // rows per CTA
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int BK = 128 / ESZ;                 // K elements per stage (128 bytes)
    constexpr int BROWS = PAIR ? BN / 2 : BN;     // W rows this CTA loads per stage
    constexpr uint32_t A_BYTES = BM * 128;        // 16 KiB
    constexpr uint32_t B_BYTES = BROWS * 128;
    constexpr uint32_t STAGE_TX = (PAIR ? 2u : 1u) * (A_BYTES + B_BYTES);  // both CTAs' copies for a pair
    constexpr int MMAS = 4;                       // 32 bytes of K per MMA
    constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // two accumulators
    constexpr uint32_t BUF_COLS = BN <= 128 ? BN : 256;          // column offset of the second one
    constexpr bool A_MN = LAY == 2, B_MN = LAY >= 1;
    static_assert(LAY == 0 || (BF16 && !PAIR && !SK), "MN-major operands: bf16, single-CTA tiles");
    constexpr uint32_t IDESC = make_idesc(BF16 ? 1u : 2u, PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
    constexpr int EPI_WARPS = kTcThreads / 32 - 2;  // two per TMEM lane quadrant
    constexpr int HALF = BN / 2;                  // columns per epilogue warp
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "N tile");
    static_assert(EPI_WARPS == 8, "8 epilogue warps");
    static_assert(!(PAIR && SK), "stream-K runs single-CTA tiles");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint8_t* sOut = sB + STAGES * B_BYTES;  // 8 warps x 32 rows x stage_row_bytes
    float* sBiasAll = reinterpret_cast<float*>(sOut + stage_bytes<BF16>());  // 8 warps x BN/2 floats
    uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + stage_bytes<BF16>() + bias_stage_bytes<BN>());
    // bars: full[S] empty[S] tfull[2] tempty[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (a.M + BM - 1) / BM, nt = (a.N + BN - 1) / BN;
    // Work items: single tiles, or (for PAIR) vertical pairs of tiles per cluster.
    const int mu = PAIR ? (mt + 1) / 2 : mt;
    const int ntiles = mu * nt;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;  // issues the MMAs; owns the full and tempty barriers
    const int first_item = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
    const int item_step = PAIR ? (int)cluster_count_x() : (int)gridDim.x;
    auto tile_m0 = [&](int item) { return (PAIR ? 2 * (item % mu) + (int)rank : item % mu) * BM; };
    auto tile_n0 = [&](int item) { return (item / mu) * BN; };
    const int nkb = (a.K + BK - 1) / BK;
    // This CTA's work as segments (tile, K stages [lo, hi)): whole tiles
    // first_item, first_item + item_step, ... or, for SK, its share of units.
    const long long units = (long long)ntiles * nkb;
    const long long u0 = SK ? (long long)blockIdx.x * units / gridDim.x : 0;
    const long long u1 = SK ? (long long)(blockIdx.x + 1) * units / gridDim.x : 0;
    // K split (ksplits > 1, whole single-CTA tiles): the work items are
    // (tile, split) pairs, split-major; each covers K stages
    // [split * nkb / S, (split + 1) * nkb / S) of its tile. With tail_whole > 0
    // (the grid's whole rounds of tiles), the first tail_whole items are whole
    // tiles and only the remaining tiles (the ragged last round) are split, so
    // that their pieces fill the SMs in one short round.
    const int ksplits = (SK || PAIR) ? 1 : a.ksplits;
    const int tail0 = ksplits > 1 ? a.tail_whole : 0;
    int cur_split = 0;  // split of the last segment returned (epilogue); -1 = a whole tile
    auto seg = [&](int j, int& tile, int& lo, int& hi) -> bool {
        if constexpr (SK) {
            const long long t = u0 / nkb + j;
            const long long st = j == 0 ? u0 : t * nkb;
            if (st >= u1) return false;
            const long long en = u1 < (t + 1) * nkb ? u1 : (t + 1) * nkb;
            tile = (int)t;
            lo = (int)(st - t * nkb);
            hi = (int)(en - t * nkb);
            return true;
        } else {
            const int item = first_item + j * item_step;
            if (tail0 > 0 && item < tail0) {
                tile = item;
                cur_split = -1;
                lo = 0;
                hi = nkb;
                return true;
            }
            const int rest = ntiles - tail0;  // tiles split in K
            const int it2 = item - tail0;
            if (it2 >= rest * ksplits) return false;
            tile = tail0 + it2 % rest;
            cur_split = ksplits > 1 ? it2 / rest : -1;
            lo = ksplits > 1 ? (int)((long long)cur_split * nkb / ksplits) : 0;
            hi = ksplits > 1 ? (int)((long long)(cur_split + 1) * nkb / ksplits) : nkb;
            return true;
        }
    };
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, PAIR ? 2 * EPI_WARPS : EPI_WARPS);
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        else
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync_all();  // the peer's barriers exist before any copy, commit or arrival reaches them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) LIN_STAMP(g_timeline_tc, blockIdx.x, 0);

    auto give_up = [&]() {
        atomicExch(s_abort, 1);
        atomicExch(a.status, (int)LIN_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: the K stages of this CTA's tiles, in order ----
            if (!a.early_inputs) {
                // The first ring's worth of operands to L2 while the previous
                // kernel finishes (no data comes back before the wait).
                if (LAY == 0 && a.prefetch) {
                    int t0, l0, h0;
                    if (seg(0, t0, l0, h0)) {
                        const int m0 = tile_m0(t0), nb0 = tile_n0(t0) + (int)rank * BROWS;
                        for (int kb = l0; kb < h0 && kb < l0 + STAGES; ++kb) {
                            if (m0 < a.M) tma_prefetch_l2_2d(&tmA, kb * BK, m0);
                            if (nb0 < a.N) tma_prefetch_l2_2d(&tmB, kb * BK, nb0);
                        }
                    }
                }
                pdl_wait();
            }
            LIN_STAMP(g_timeline_tc, blockIdx.x, 1);
            uint32_t it = 0, issued = 0;
            bool ok = true;
            int tile, lo, hi;
            for (int j = 0; ok && seg(j, tile, lo, hi); ++j) {
                const int m0 = tile_m0(tile), n0 = tile_n0(tile);
                for (int kb = lo; kb < hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (*(volatile int*)s_abort || !mbar_wait(empty0 + 8 * s, ph ^ 1)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    if constexpr (PAIR) {
                        // Both CTAs' copies complete the even CTA's barrier.
                        if (leader) mbar_expect_tx(full0 + 8 * s, STAGE_TX);
                        const uint32_t fb = dsmem_map(full0 + 8 * s, 0);
                        tma_load_2d_pair(smem_u32(sA + s * A_BYTES), &tmA, fb, kb * BK, m0);
                        tma_load_2d_pair(smem_u32(sB + s * B_BYTES), &tmB, fb, kb * BK, n0 + (int)rank * BROWS);
                    } else {
                        mbar_expect_tx(full0 + 8 * s, STAGE_TX);
                        if constexpr (A_MN) {
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j)
                                tma_load_2d(smem_u32(sA + s * A_BYTES + j * 8192), &tmA, full0 + 8 * s, m0 + 64 * j,
                                            kb * BK);
                        } else {
                            tma_load_2d(smem_u32(sA + s * A_BYTES), &tmA, full0 + 8 * s, kb * BK, m0);
                        }
                        if constexpr (B_MN) {
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_2d(smem_u32(sB + s * B_BYTES + j * 8192), &tmB, full0 + 8 * s, n0 + 64 * j,
                                            kb * BK);
                        } else {
                            tma_load_2d(smem_u32(sB + s * B_BYTES), &tmB, full0 + 8 * s, kb * BK, n0);
                        }
                    }
                    issued = it + 1;
                }
            }
            if (*(volatile int*)s_abort && leader) {
                // Drain the copies still in flight before the CTA exits (for a pair,
                // the even CTA's barriers count both CTAs' copies).
                const uint32_t first = issued > (uint32_t)STAGES ? issued - STAGES : 0;
                for (uint32_t i = first; i < issued; ++i) mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---- MMA issuer: accumulators alternate between two TMEM buffers ----
            uint32_t it = 0;
            int j = 0, tile, lo, hi;
            bool ok = true;
            for (; ok && seg(j, tile, lo, hi); ++j) {
                const uint32_t buf = j & 1;
                const bool freed = PAIR ? mbar_wait_cluster(tempty0 + 8 * buf, ((j >> 1) & 1) ^ 1)
                                        : mbar_wait(tempty0 + 8 * buf, ((j >> 1) & 1) ^ 1);
                if (*(volatile int*)s_abort || !freed) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + buf * BUF_COLS;
                if (j < 32) LIN_STAMP(g_timeline_tc, blockIdx.x, 8 + 4 * j);
                for (int kb = lo; kb < hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (*(volatile int*)s_abort || !mbar_wait(full0 + 8 * s, ph)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = A_MN ? sw128_mnmajor_desc(smem_u32(sA + s * A_BYTES))
                                             : sw128_kmajor_desc(smem_u32(sA + s * A_BYTES));
                    const uint64_t bd = B_MN ? sw128_mnmajor_desc(smem_u32(sB + s * B_BYTES))
                                             : sw128_kmajor_desc(smem_u32(sB + s * B_BYTES));
                    // K advance per MMA: 32 bytes of a K-major row, or 16 rows of an MN-major tile.
                    constexpr uint32_t ASTEP = A_MN ? 128u : 2u, BSTEP = B_MN ? 128u : 2u;
                    if constexpr (PAIR) {
#pragma unroll
                        for (int kk = 0; kk < MMAS; ++kk)
                            tc_mma_pair<BF16>(d, ad + 2u * kk, bd + 2u * kk, IDESC, (kb != lo || kk != 0) ? 1u : 0u);
                        tc_commit_pair_mc(empty0 + 8 * s, (uint16_t)0x3);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < MMAS; ++kk)
                            tc_mma<BF16>(d, ad + ASTEP * kk, bd + BSTEP * kk, IDESC, (kb != lo || kk != 0) ? 1u : 0u);
                        tc_commit(empty0 + 8 * s);
                    }
                }
                if constexpr (PAIR)
                    tc_commit_pair_mc(tfull0 + 8 * buf, (uint16_t)0x3);
                else
                    tc_commit(tfull0 + 8 * buf);
                if (j < 32) LIN_STAMP(g_timeline_tc, blockIdx.x, 8 + 4 * j + 1);
            }
            // Do not reach the teardown before this CTA's MMAs have completed.
            if (j > 0) {
                const uint32_t lb = tfull0 + 8 * ((j - 1) & 1), lp = ((j - 1) >> 1) & 1;
                if (!(PAIR ? mbar_wait_cluster(lb, lp) : mbar_wait(lb, lp))) give_up();
            }
        }
    } else {
        // ---- epilogue: warp w reads TMEM lanes 32*(w%4).., columns half (w-2)/4 ----
        pdl_wait();  // Y (and bias) only after the previous kernel on the stream has finished
        const int q = warp & 3;
        const int ew = warp - 2;
        const int c_begin = (ew >> 2) * HALF;
        const int N = a.N;
        float* sBias = sBiasAll + ew * HALF;
        constexpr int CH = HALF / 32;  // 32-column chunks per warp and tile
        // Chunks per round trip to TMEM: one where the registers are needed
        // elsewhere (fp32 staging; the odd-row store path, which spilled with two).
        constexpr int PER = (BF16 && !YODD) ? 2 : 1;
        constexpr int RB = stage_row_bytes<BF16>();
        constexpr int RP = stage_rows<BF16>();
        constexpr int ESZO = BF16 ? 2 : 4;
        constexpr int LPR = 32 * ESZO / 16;  // lanes per row with 16-byte pieces
        uint8_t* st = sOut + ew * stage_warp_bytes<BF16>();

        // One 32 x 32 chunk: bias, activation, convert; lane = row. The values go
        // through this warp's staging tile (rows [h*RP, h*RP + RP) per pass) and
        // leave as whole row segments: consecutive lanes, consecutive addresses
        // (storing each lane's own row from registers scatters every store
        // instruction over 32 rows and was measured slower).
        // `pre`: the chunk's auxiliary pieces, already loaded (see aux_pieces), or null.
        auto emit = [&](const uint32_t (&r)[32], int c, int m0, int n0, const uint4* pre = nullptr) {
            const int col = c_begin + c * 32;
            const int nb = n0 + col;
            if (nb >= N) return;  // warp-uniform
            const bool full = nb + 32 <= N;
            float v[32];
#pragma unroll
            for (int j4 = 0; j4 < 32; j4 += 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(sBias + c * 32 + j4);
                v[j4 + 0] = epilogue<GELU, BF16>(__uint_as_float(r[j4 + 0]), b4.x);
                v[j4 + 1] = epilogue<GELU, BF16>(__uint_as_float(r[j4 + 1]), b4.y);
                v[j4 + 2] = epilogue<GELU, BF16>(__uint_as_float(r[j4 + 2]), b4.z);
                v[j4 + 3] = epilogue<GELU, BF16>(__uint_as_float(r[j4 + 3]), b4.w);
            }
            const int mrow0 = m0 + q * 32;
            // The auxiliary tensor at this lane's row: the residual stream
            // (added), or the previous layer's pre-activation (GELU slope).
            if (a.aux_mode) {
                float t[32];
                bool staged = false;
                if constexpr (BF16) {
                    if (a.y_tma && full && a.aux_vec && mrow0 < a.M) {
                        // Coalesced: four passes of 8 rows x 64 bytes (lane = 16
                        // bytes of a row), through this warp's output box (free once
                        // the previous store has read it), then each lane reads its
                        // own row back. A row per lane straight from global memory
                        // would touch 32 rows per load instruction.
                        uint4 piece[4];
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int r = it * 8 + (lane >> 2), k = lane & 3;
                            if (pre) {
                                piece[it] = pre[it];
                            } else {
                                piece[it] = make_uint4(0u, 0u, 0u, 0u);
                                if (mrow0 + r < a.M)
                                    piece[it] = *reinterpret_cast<const uint4*>(
                                        static_cast<const uint16_t*>(a.aux) + (size_t)(mrow0 + r) * N + nb + 8 * k);
                            }
                        }
                        uint8_t* box = sOut + ew * 2048;
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int r = it * 8 + (lane >> 2), k = lane & 3;
                            *reinterpret_cast<uint4*>(box + r * 64 + ((k ^ ((r >> 1) & 3)) * 16)) = piece[it];
                        }
                        __syncwarp();
                        // Applied 8 values at a time as they come back (fewer live
                        // registers than unpacking the whole row first).
#pragma unroll
                        for (int p16 = 0; p16 < 4; ++p16) {
                            const uint4 w = *reinterpret_cast<const uint4*>(box + lane * 64 + ((p16 ^ ((lane >> 1) & 3)) * 16));
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float lo = __uint_as_float(ws[h] << 16);
                                const float hi = __uint_as_float(ws[h] & 0xffff0000u);
                                float& v0 = v[8 * p16 + 2 * h];
                                float& v1 = v[8 * p16 + 2 * h + 1];
                                if (a.aux_mode == 1) {
                                    v0 += lo;
                                    v1 += hi;
                                } else {
                                    v0 *= gelu_tanh_slope<BF16>(lo);
                                    v1 *= gelu_tanh_slope<BF16>(hi);
                                }
                            }
                        }
                        __syncwarp();  // the box takes this chunk's output next
                        staged = true;
                    }
                }
                const bool row_ok = mrow0 + lane < a.M;
                if (!staged && row_ok) {
                    const size_t rowoff = (size_t)(mrow0 + lane) * N + nb;
                    if (full && a.aux_vec) {
                        if constexpr (BF16) {
                            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.aux) + rowoff);
#pragma unroll
                            for (int p16 = 0; p16 < 4; ++p16) {
                                const uint4 w = src[p16];
                                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    t[8 * p16 + 2 * h] = __uint_as_float(ws[h] << 16);
                                    t[8 * p16 + 2 * h + 1] = __uint_as_float(ws[h] & 0xffff0000u);
                                }
                            }
                        } else {
                            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.aux) + rowoff);
#pragma unroll
                            for (int p4 = 0; p4 < 8; ++p4) {
                                const float4 w = src[p4];
                                t[4 * p4] = w.x;
                                t[4 * p4 + 1] = w.y;
                                t[4 * p4 + 2] = w.z;
                                t[4 * p4 + 3] = w.w;
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            t[j] = 0.f;
                            if (nb + j < N)
                                t[j] = BF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(a.aux)[rowoff + j])
                                            : static_cast<const float*>(a.aux)[rowoff + j];
                        }
                    }
                }
                if (!staged && row_ok) {
                    if (a.aux_mode == 1) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += t[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= gelu_tanh_slope<BF16>(t[j]);
                    }
                }
            }
            if constexpr (BF16) {
                if (a.y_tma) {
                    // Into this warp's 32 x 32 box (64-byte swizzle: conflict-free
                    // row-per-lane writes), then one TMA store, which clips rows
                    // and columns outside Y. The box is reused once the previous
                    // store has read it.
                    if (mrow0 >= a.M) return;
                    uint8_t* box = sOut + ew * 2048;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int p16 = 0; p16 < 4; ++p16) {
                        uint4 o;
                        o.x = pack_bf16x2(v[8 * p16 + 0], v[8 * p16 + 1]);
                        o.y = pack_bf16x2(v[8 * p16 + 2], v[8 * p16 + 3]);
                        o.z = pack_bf16x2(v[8 * p16 + 4], v[8 * p16 + 5]);
                        o.w = pack_bf16x2(v[8 * p16 + 6], v[8 * p16 + 7]);
                        *reinterpret_cast<uint4*>(box + lane * 64 + ((p16 ^ ((lane >> 1) & 3)) * 16)) = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, smem_u32(box), nb, mrow0);
                        bulk_commit();
                    }
                    return;
                }
                if (YODD && full && a.y_aligned16 && (N * ESZO) % 16 != 0) {
                    // Rows that are not 16-byte aligned (N not a multiple of 8, as
                    // in a 50257-word LM head): each lane writes its row into the
                    // staging tile shifted by the row's misalignment s (elements),
                    // so that the row's 16-byte blocks of Y sit on 16-byte
                    // boundaries there; the blocks wholly inside this chunk leave
                    // by vector stores, the few elements of the two partial blocks
                    // one by one.
                    auto row_at = [&](int r) { return st + r * RB + (r >> 3) * 16; };
                    {
                        uint32_t w[17];
#pragma unroll
                        for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                        w[16] = 0u;
                        const long long g = (long long)(mrow0 + lane) * N + nb;
                        const int s = (int)(g & 7);
                        const bool odd = (s & 1) != 0;
                        uint32_t* dst = reinterpret_cast<uint32_t*>(row_at(lane)) + (s >> 1);
                        // odd s: word k holds elements (2k - 1, 2k) of the chunk
                        uint32_t prev = 0u;
#pragma unroll
                        for (int j = 0; j < 17; ++j) {
                            dst[j] = odd ? __byte_perm(prev, w[j], 0x5432) : w[j];
                            prev = w[j];
                        }
                    }
                    __syncwarp();
                    // Whole blocks: rows x blocks 0..3 of the shifted row (block 0
                    // only when the row is aligned).
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int item = it * 32 + lane;
                        const int r = item >> 2, k = item & 3;
                        const int m = mrow0 + r;
                        const long long g = (long long)m * N + nb;
                        const int s = (int)(g & 7);
                        if (m < a.M && (k > 0 || s == 0)) {
                            const uint4 val = *reinterpret_cast<const uint4*>(row_at(r) + 16 * k);
                            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.Y) + (g - s) + 8 * k) = val;
                        }
                    }
                    // Partial blocks: the first 8 - s and the last s elements of a
                    // row with s > 0.
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int item = it * 32 + lane;
                        const int r = item >> 3, idx = item & 7;
                        const int m = mrow0 + r;
                        const long long g = (long long)m * N + nb;
                        const int s = (int)(g & 7);
                        if (m < a.M && s > 0) {
                            const int e = idx < 8 - s ? idx : 24 + idx;
                            static_cast<uint16_t*>(a.Y)[g + e] =
                                *reinterpret_cast<const uint16_t*>(row_at(r) + 2 * (s + e));
                        }
                    }
                    __syncwarp();  // the staging rows are rewritten by the next chunk
                    return;
                }
            }
            const bool vec = full && (N * ESZO) % 16 == 0 && a.y_aligned16;
#pragma unroll
            for (int h = 0; h < 32 / RP; ++h) {
                if (lane / RP == h) {
                    uint8_t* mine_row = st + (lane % RP) * RB;
                    if constexpr (BF16) {
#pragma unroll
                        for (int jj = 0; jj < 32; jj += 8) {
                            uint4 o;
                            o.x = pack_bf16x2(v[jj], v[jj + 1]);
                            o.y = pack_bf16x2(v[jj + 2], v[jj + 3]);
                            o.z = pack_bf16x2(v[jj + 4], v[jj + 5]);
                            o.w = pack_bf16x2(v[jj + 6], v[jj + 7]);
                            *reinterpret_cast<uint4*>(mine_row + jj * 2) = o;
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; jj += 4)
                            *reinterpret_cast<float4*>(mine_row + jj * 4) =
                                make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                    }
                }
                __syncwarp();
                const int rbase = mrow0 + h * RP;
                if (vec) {
                    const int sub = lane % LPR, rsub = lane / LPR;
#pragma unroll
                    for (int r0 = 0; r0 < RP; r0 += 32 / LPR) {
                        const int rr = r0 + rsub;
                        if (rbase + rr < a.M) {
                            const uint4 val = *reinterpret_cast<const uint4*>(st + rr * RB + sub * 16);
                            uint8_t* dst = static_cast<uint8_t*>(a.Y) + ((size_t)(rbase + rr) * N + nb) * ESZO + sub * 16;
                            *reinterpret_cast<uint4*>(dst) = val;
                        }
                    }
                } else {
                    const bool col_ok = nb + lane < N;
#pragma unroll 4
                    for (int rr = 0; rr < RP; ++rr) {
                        if (rbase + rr < a.M && col_ok) {
                            if constexpr (BF16)
                                static_cast<uint16_t*>(a.Y)[(size_t)(rbase + rr) * N + nb + lane] =
                                    *reinterpret_cast<const uint16_t*>(st + rr * RB + lane * 2);
                            else
                                static_cast<float*>(a.Y)[(size_t)(rbase + rr) * N + nb + lane] =
                                    *reinterpret_cast<const float*>(st + rr * RB + lane * 4);
                        }
                    }
                }
                __syncwarp();  // the staging rows are rewritten by the next pass / chunk
            }
        };

        // The coalesced auxiliary pieces of chunk c (the layout emit's staged path
        // reads), loaded ahead so that their latency overlaps other work. Only
        // for whole bf16 chunks whose output leaves by TMA store.
        auto aux_pieces = [&](int c, int m0, int n0, uint4 (&p)[4]) {
            const int nb = n0 + c_begin + c * 32;
            const int mrow0 = m0 + q * 32;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = it * 8 + (lane >> 2), k = lane & 3;
                p[it] = make_uint4(0u, 0u, 0u, 0u);
                if (mrow0 + r < a.M)
                    p[it] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.aux) +
                                                           (size_t)(mrow0 + r) * N + nb + 8 * k);
            }
        };
        auto aux_ahead_ok = [&](int c, int m0, int n0) {
            return BF16 && a.aux_mode && a.y_tma && a.aux_vec && c < CH && m0 + q * 32 < a.M &&
                   n0 + c_begin + c * 32 + 32 <= N;
        };

        // Hand an accumulator buffer back to the MMA issuer (the even CTA's barrier).
        auto release_acc = [&](uint32_t buf) {
            if (PAIR && !leader)
                mbar_arrive_remote(dsmem_map(tempty0 + 8 * buf, 0));
            else
                mbar_arrive(tempty0 + 8 * buf);
        };

        // Stream-K hand-over: this warp's region of a boundary slot, laid out
        // [chunk][column][row] so that lane = row accesses are coalesced.
        auto part_ptr = [&](int boundary) {
            return a.partials + (size_t)boundary * (BM * BN) + (size_t)ew * (CH * 1024);
        };
        auto store_part = [&](const uint32_t (&r)[32], int c) {
            float* dst = part_ptr(blockIdx.x) + c * 1024 + lane;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) __stcg(dst + jj * 32, __uint_as_float(r[jj]));
        };
        auto add_part = [&](uint32_t (&r)[32], int c) {
            const float* src = part_ptr(blockIdx.x + 1) + c * 1024 + lane;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) r[jj] = __float_as_uint(__uint_as_float(r[jj]) + __ldcg(src + jj * 32));
        };
        // K split: this warp's region of the (tile, split) slot, same layout.
        // Slots and counters are numbered from the first split tile.
        auto ks_ptr = [&](int tile_, int split_) {
            return a.partials + (((size_t)(tile_ - tail0) * ksplits + split_) * EPI_WARPS + ew) * (CH * 1024);
        };

        int j = 0, tile, lo, hi;
        for (; seg(j, tile, lo, hi); ++j) {
            const uint32_t buf = j & 1;
            const int m0 = tile_m0(tile), n0 = tile_n0(tile);
            const bool part_out = SK && lo > 0;            // later K stages of a cut tile: hand over
            const bool part_in = SK && lo == 0 && hi < nkb;  // earlier K stages: add the partner's, finish
            const int split = cur_split;
            const bool kpart = ksplits > 1 && split >= 0;  // one K range of a split tile
            // This warp's bias columns of the tile, fetched while the MMAs run.
#pragma unroll
            for (int t = lane; t < HALF; t += 32) {
                const int n = n0 + c_begin + t;
                sBias[t] = (a.bias && n < N) ? __ldg(a.bias + n) : 0.f;
            }
            // The auxiliary tensor's part of this warp's region (one row segment
            // per lane) to L2 while the MMAs run, so that the epilogue's row loads
            // of it hit the L2 instead of waiting on HBM.
            if (a.aux_mode && a.aux_vec) {
                const int arow = m0 + q * 32 + lane, acol = n0 + c_begin;
                const int ncols = N - acol < HALF ? N - acol : HALF;
                if (arow < a.M && ncols > 0) {
                    const char* src = static_cast<const char*>(a.aux) + ((size_t)arow * N + acol) * (BF16 ? 2 : 4);
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src),
                                 "r"((unsigned)ncols * (BF16 ? 2u : 4u))
                                 : "memory");
                }
            }
            __syncwarp();
            // With an auxiliary tensor, chunks go one per round trip to TMEM and
            // the next chunk's pieces are loaded while this one is processed; the
            // first chunk's before the accumulator is ready.
            const bool aux_ahead = !kpart && !SK && a.aux_mode && a.y_tma && a.aux_vec;
            uint4 ahead[4];
            bool have_ahead = false;
            if (aux_ahead && aux_ahead_ok(0, m0, n0)) {
                aux_pieces(0, m0, n0, ahead);
                have_ahead = true;
            }
            const bool mine = PAIR ? mbar_wait_cluster(tfull0 + 8 * buf, (j >> 1) & 1)
                                   : mbar_wait(tfull0 + 8 * buf, (j >> 1) & 1);
            if (!mine) give_up();
            tc_fence_after();
            if (warp == 2 && lane == 0 && j < 32) LIN_STAMP(g_timeline_tc, blockIdx.x, 8 + 4 * j + 2);
            // tcgen05.ld is warp-collective: a warp proceeds only if every lane saw
            // the accumulator complete and no role of this CTA gave up.
            bool ok = __all_sync(0xffffffffu, mine && *(volatile int*)s_abort == 0);
            unsigned* flag = SK ? a.flags + (size_t)(blockIdx.x + (part_in ? 1 : 0)) * 8 + ew : nullptr;
            if (SK && part_in && ok) {
                // The partner (the next CTA) computed the later K stages first.
                bool got = lane == 0 ? wait_flag_set(flag) : true;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) give_up();
                ok = got && ld_acquire_gpu(flag) != 0u;
            }
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BUF_COLS + static_cast<uint32_t>(c_begin);
            bool released = false;
            if (aux_ahead) {
                // One chunk per round trip to TMEM; the next chunk's pieces are
                // loaded before this chunk is processed.
#pragma unroll 1
                for (int c = 0; c < CH && ok; ++c) {
                    uint4 cur[4];
                    const bool have_cur = have_ahead;
#pragma unroll
                    for (int it = 0; it < 4; ++it) cur[it] = ahead[it];
                    have_ahead = aux_ahead_ok(c + 1, m0, n0);
                    if (have_ahead) aux_pieces(c + 1, m0, n0, ahead);
                    uint32_t r0[32];
                    tmem_ld32_async(tbase + c * 32, r0);
                    tmem_wait_ld(r0);
                    if (c + 1 >= CH) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) release_acc(buf);
                        released = true;
                    }
                    emit(r0, c, m0, n0, have_cur ? cur : nullptr);
                }
            }
#pragma unroll 1
            for (int c = 0; c < CH && ok && !aux_ahead; c += PER) {
                uint32_t r0[32], r1[32];
                const bool two = PER == 2 && c + 1 < CH;
                tmem_ld32_async(tbase + c * 32, r0);
                if (two) tmem_ld32_async(tbase + (c + 1) * 32, r1);
                tmem_wait_ld(r0);
                if (two) tmem_wait_ld(r1);
                if (c + PER >= CH) {
                    // Last read of the accumulator: the MMA issuer may reuse it
                    // while this warp converts and stores.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc(buf);
                    released = true;
                }
                if (kpart) {
                    float* dst = ks_ptr(tile, split) + lane;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) __stcg(dst + c * 1024 + jj * 32, __uint_as_float(r0[jj]));
                    if (two) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            __stcg(dst + (c + 1) * 1024 + jj * 32, __uint_as_float(r1[jj]));
                    }
                    continue;
                }
                if constexpr (SK) {
                    if (part_out) {
                        store_part(r0, c);
                        if (two) store_part(r1, c + 1);
                        continue;
                    }
                    if (part_in) {
                        add_part(r0, c);
                        if (two) add_part(r1, c + 1);
                    }
                }
                emit(r0, c, m0, n0);
                if (two) emit(r1, c + 1, m0, n0);
            }
            if (kpart && ok) {
                // Count this region in; the last of the tile's splits adds all of
                // them in split order and finishes the region.
                __threadfence();
                __syncwarp();
                unsigned* cnt = a.flags + (size_t)(tile - tail0) * EPI_WARPS + ew;
                unsigned last = 0;
                if (lane == 0) {
                    last = atomicAdd(cnt, 1u) == (unsigned)(ksplits - 1);
                    if (last) *cnt = 0u;  // re-armed for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
#pragma unroll 1
                    for (int c = 0; c < CH; ++c) {
                        float sum[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) sum[jj] = 0.f;
                        // Two splits' loads in flight per round trip to the L2;
                        // the adds stay in split order.
                        int sp = 0;
#pragma unroll 1
                        for (; sp + 1 < ksplits; sp += 2) {
                            const float* s0 = ks_ptr(tile, sp) + c * 1024 + lane;
                            const float* s1 = ks_ptr(tile, sp + 1) + c * 1024 + lane;
                            float t0[32], t1[32];
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) t0[jj] = __ldcg(s0 + jj * 32);
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) t1[jj] = __ldcg(s1 + jj * 32);
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) sum[jj] += t0[jj];
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) sum[jj] += t1[jj];
                        }
                        if (sp < ksplits) {
                            const float* src = ks_ptr(tile, sp) + c * 1024 + lane;
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) sum[jj] += __ldcg(src + jj * 32);
                        }
                        uint32_t r[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) r[jj] = __float_as_uint(sum[jj]);
                        emit(r, c, m0, n0);
                    }
                }
            }
            if constexpr (SK) {
                if (part_out && ok) {
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) st_release_gpu(flag, 1u);
                }
                if (part_in && ok) {
                    __syncwarp();
                    if (lane == 0) *flag = 0u;  // re-armed for the next launch
                }
            }
            if (lane == 0 && j < 32 && warp == 2) LIN_STAMP(g_timeline_tc, blockIdx.x, 8 + 4 * j + 3);
            if (lane == 0 && j < 32 && warp == 9) LIN_STAMP(g_timeline_tc, blockIdx.x, 136 + j);
            if (!released) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(buf);
            }
            __syncwarp();  // sBias is rewritten for the next tile
        }
        // The TMA stores of this warp have read their box before the CTA releases
        // its shared memory (their global writes complete with the grid).
        if (BF16 && a.y_tma && lane == 0) bulk_wait_read_all();
        __syncwarp();
    }

    __syncwarp();
    tc_fence_before();
    if (threadIdx.x == 64) LIN_STAMP(g_timeline_tc, blockIdx.x, 2);
    // PAIR: neither CTA leaves while the peer's copies or arrivals may still
    // target its shared memory.
    if constexpr (PAIR)
        cluster_sync_all();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

template <bool BF16, int BN, bool GELU, bool PAIR, bool SK, int LAY = 0, bool YODD = false>
int launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const TcArgs& a, int grid, bool early,
               cudaStream_t st) {
    constexpr size_t smem = tc_smem_bytes<BF16, BN, PAIR>();
    static_assert(tc_smem_bytes<BF16, BN, PAIR>() <= 227 * 1024, "shared memory");
    auto kern = tc_kernel<BF16, BN, GELU, PAIR, SK, LAY, YODD>;
    static std::atomic<unsigned long long> attr_set{0};  // per instantiation: one bit per device
    if (ensure_smem_attr(attr_set, kern, smem) != LIN_OK) return LIN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (PAIR) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 2;
        attrs[na].val.clusterDim.y = 1;
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
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, a) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

template <bool BF16, bool GELU>
int launch_variant(int variant, bool sk, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                   const TcArgs& a, int grid, bool early, cudaStream_t st) {
    // Whole tiles of bf16 Y with unaligned rows: the vector-store epilogue.
    const bool yodd = BF16 && a.ksplits <= 1 && !a.y_tma && a.y_aligned16 && (a.N % 8) != 0;
    if (sk) {
        switch (variant) {
            case 0: return launch_cfg<BF16, kTcCfg[0].bn, GELU, false, true>(ta, tb, ty, a, grid, early, st);
            case 1: return launch_cfg<BF16, kTcCfg[1].bn, GELU, false, true>(ta, tb, ty, a, grid, early, st);
            case 2: return launch_cfg<BF16, kTcCfg[2].bn, GELU, false, true>(ta, tb, ty, a, grid, early, st);
            default: return LIN_ERR_UNSUPPORTED;
        }
    }
    switch (variant) {
        case 0:
            if (BF16 && yodd) return launch_cfg<BF16, kTcCfg[0].bn, GELU, false, false, 0, true>(ta, tb, ty, a, grid, early, st);
            return launch_cfg<BF16, kTcCfg[0].bn, GELU, false, false>(ta, tb, ty, a, grid, early, st);
        case 1: return launch_cfg<BF16, kTcCfg[1].bn, GELU, false, false>(ta, tb, ty, a, grid, early, st);
        case 2: return launch_cfg<BF16, kTcCfg[2].bn, GELU, false, false>(ta, tb, ty, a, grid, early, st);
        case 3:
            if (BF16 && yodd) return launch_cfg<BF16, kTcCfg[3].bn, GELU, true, false, 0, true>(ta, tb, ty, a, grid, early, st);
            return launch_cfg<BF16, kTcCfg[3].bn, GELU, true, false>(ta, tb, ty, a, grid, early, st);
        case 4: return launch_cfg<BF16, kTcCfg[4].bn, GELU, true, false>(ta, tb, ty, a, grid, early, st);
        case 5: return launch_cfg<BF16, kTcCfg[5].bn, GELU, true, false>(ta, tb, ty, a, grid, early, st);
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

bool make_out_map_bf16(CUtensorMap* map, void* base, int M, int N) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_mnmajor_map(CUtensorMap* map, const void* base, int rows, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 backward GEMMs on the tensor cores, 128 x 256 single-CTA tiles (K
// split when the tiles are few, the reduction long and no independent
// predecessor on the stream fills the idle SMs instead):
//   which 1: dX (M x K) = dZ (M x N) . W (N x K): A = dZ K-major, B = W MN-major.
//   which 2: dW (N x K) = dZ^T . X (M x K):       A = dZ MN-major, B = X MN-major.
// Rows of dZ, W and X must be 16-byte aligned (N and K multiples of 8).
int launch_tc_backward(const BwdProblem& q) {
    const int Mo = q.which == 1 ? q.M : q.N;  // output rows
    const int No = q.K;                       // output columns
    const int R = q.which == 1 ? q.N : q.M;   // reduction
    CUtensorMap ta, tb, ty;
    if (q.which == 1) {
        if (!make_kmajor_map(&ta, q.dZ, true, q.M, q.N, 128)) return LIN_ERR_CUDA;
        if (!make_mnmajor_map(&tb, q.B, q.N, q.K)) return LIN_ERR_CUDA;
    } else {
        if (!make_mnmajor_map(&ta, q.dZ, q.M, q.N)) return LIN_ERR_CUDA;
        if (!make_mnmajor_map(&tb, q.B, q.M, q.K)) return LIN_ERR_CUDA;
    }
    TcArgs a = {};
    a.M = Mo;
    a.N = No;
    a.K = R;
    a.bias = nullptr;
    a.Y = q.out;
    a.status = q.dev_status;
    a.y_aligned16 = (reinterpret_cast<uintptr_t>(q.out) % 16) == 0;
    a.bias_aligned16 = 0;
    a.early_inputs = q.early_x ? 1 : 0;
    a.prefetch = 0;
    a.partials = nullptr;
    a.flags = nullptr;
    a.aux = q.which == 1 ? q.aux : nullptr;
    a.aux_mode = a.aux ? 2 : 0;
    a.aux_vec = (reinterpret_cast<uintptr_t>(a.aux) % 16) == 0 && (No * 2) % 16 == 0;
    // Small outputs with a long reduction (the weight gradients): split K.
    const long long ntile = (long long)((Mo + 127) / 128) * ((No + 255) / 256);
    a.ksplits = q.ksplit_ok ? tc_ksplits(ntile, (R + 63) / 64, q.sm_count, q.workspace_bytes, kTcCfg[0].bn) : 1;
    if (a.ksplits > 1) {
        a.partials = splitk_partials(q.workspace);
        a.flags = splitk_counters(q.workspace);
    }
    ty = ta;
    a.y_tma = 0;
    if (a.y_aligned16 && No % 8 == 0) {
        if (!make_out_map_bf16(&ty, q.out, Mo, No)) return LIN_ERR_CUDA;
        a.y_tma = 1;
    }
    const long long items = ntile * a.ksplits;
    const int grid = (int)(items < q.sm_count ? items : q.sm_count);
    if (q.which == 1)
        return launch_cfg<true, kTcCfg[0].bn, false, false, false, 1>(ta, tb, ty, a, grid, q.early_start, q.stream);
    return launch_cfg<true, kTcCfg[0].bn, false, false, false, 2>(ta, tb, ty, a, grid, q.early_start, q.stream);
}

int launch_tc(const Problem& p, const lin_plan& plan) {
    const bool bf16 = p.precision == LIN_PREC_BF16;
    if (plan.variant < 0 || plan.variant >= kTcVariants) return LIN_ERR_UNSUPPORTED;
    const bool pair = kTcCfg[plan.variant].pair;
    CUtensorMap ta, tb;
    if (!make_kmajor_map(&ta, p.X, bf16, p.M, p.K, 128)) return LIN_ERR_CUDA;
    if (!make_kmajor_map(&tb, p.W, bf16, p.N, p.K, pair ? plan.bn / 2 : plan.bn)) return LIN_ERR_CUDA;
    TcArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bias = p.bias;
    a.Y = p.Y;
    a.status = p.dev_status;
    a.y_aligned16 = (reinterpret_cast<uintptr_t>(p.Y) % 16) == 0;
    a.bias_aligned16 = (reinterpret_cast<uintptr_t>(p.bias) % 16) == 0;
    a.early_inputs = (p.early_start && p.early_x) ? 1 : 0;
    a.prefetch = p.early_start ? 1 : 0;
    a.aux = p.residual;
    a.aux_mode = p.residual ? 1 : 0;
    a.aux_vec = (reinterpret_cast<uintptr_t>(p.residual) % 16) == 0 && ((size_t)p.N * (bf16 ? 2 : 4)) % 16 == 0;
    const bool sk = plan.splits == 2;
    // Stream-K CTAs wait for their successor's hand-over, so all of them must
    // be resident at once: at most one per SM.
    if (sk && (pair || plan.grid_x > kTcMaxStreamKCtas || plan.grid_x > p.sm_count ||
               p.workspace_bytes < tc_streamk_workspace_bytes(plan.grid_x, plan.bn)))
        return LIN_ERR_UNSUPPORTED;
    a.partials = sk ? splitk_partials(p.workspace) : nullptr;
    a.flags = sk ? splitk_counters(p.workspace) + kTcFlagBase : nullptr;
    a.ksplits = plan.grid_z > 1 ? plan.grid_z : 1;
    a.tail_whole = 0;
    if (a.ksplits > 1) {
        const long long ntile = (long long)((p.M + 127) / 128) * ((p.N + plan.bn - 1) / plan.bn);
        a.tail_whole = (int)tc_tail_whole(ntile, plan.grid_x);
        const long long split_tiles = ntile - a.tail_whole;
        if (sk || pair || split_tiles < 1 || split_tiles > kTcMaxKSplitTiles ||
            p.workspace_bytes < tc_ksplit_workspace_bytes(split_tiles, a.ksplits, plan.bn))
            return LIN_ERR_UNSUPPORTED;
        a.partials = splitk_partials(p.workspace);
        a.flags = splitk_counters(p.workspace);
    }
    // bf16 rows 16-byte aligned: Y leaves by TMA store; otherwise (odd N, as in
    // the LM head) through the staged row-segment stores. The fallback map is a
    // placeholder the kernel never uses.
    CUtensorMap ty = ta;
    a.y_tma = 0;
    if (bf16 && a.y_aligned16 && p.N % 8 == 0) {
        if (!make_out_map_bf16(&ty, p.Y, p.M, p.N)) return LIN_ERR_CUDA;
        a.y_tma = 1;
    }
    const int grid = plan.grid_x;
    const bool gelu = p.epilogue == LIN_EPI_GELU_TANH;
    // Programmatic dependent launch whenever the context allows an early start:
    // a CTA of this grid starts on an SM as soon as the previous kernel's CTA
    // there has exited (prologue, TMEM allocation and, for independent inputs,
    // the first loads overlap the previous kernel's last tiles elsewhere). The
    // kernel waits before its first load unless the inputs are independent.
    const bool early = p.early_start;
    if (bf16)
        return gelu ? launch_variant<true, true>(plan.variant, sk, ta, tb, ty, a, grid, early, p.stream)
                    : launch_variant<true, false>(plan.variant, sk, ta, tb, ty, a, grid, early, p.stream);
    return gelu ? launch_variant<false, true>(plan.variant, sk, ta, tb, ty, a, grid, early, p.stream)
                : launch_variant<false, false>(plan.variant, sk, ta, tb, ty, a, grid, early, p.stream);
}

int timeline_copy_tc(void* dst, size_t bytes, bool clear) {
#ifdef LIN_TIMELINE
    const size_t total = sizeof(unsigned long long) * kTimelineCtas * kTimelineSlots;
    if (dst && bytes > 0 &&
        cudaMemcpyFromSymbol(dst, g_timeline_tc, bytes < total ? bytes : total) != cudaSuccess)
        return LIN_ERR_CUDA;
    if (clear) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_timeline_tc) != cudaSuccess || cudaMemset(p, 0, total) != cudaSuccess)
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
