// Fused self-attention forward of one transformer layer, read straight out of
// the qkv projection's output and written in the layout the output
// projection reads ("Writing a CUDA matmul that catches cuBLAS", section
// "Fusing attention: the score matrix never exists"):
//
//   qkv : (B*T) x 3C bf16, C = H*64; for token t of sequence b and head h,
//         q = qkv[b*T + t][h*64 ..], k at column C + h*64, v at 2C + h*64.
//   out : (B*T) x C bf16, out[b*T + i][h*64 + d] = sum_j p_ij v_j[d],
//         p_ij = softmax over the visible keys j of (q_i . k_j) * scale.
//   lse : optional B x H x T fp32, max_j s_ij + log sum_j exp(s_ij - max).
//
// The page's scheme, kept: a block of queries walks the key blocks holding a
// running row max m and row sum l; when a block raises the max to m', what
// was accumulated is scaled by exp(m - m'), and O is divided by l at the end.
// Causality is the loop bound (a query block visits key blocks up to its own
// diagonal block only), and the score matrix never reaches memory.
//
// On sm_103a (not the page's design, which was written for mma.sync on
// sm_89): a persistent CTA per SM walks work items (sequence, head, block of
// 128 queries), largest causal items first. Its softmax warps form two groups
// that take alternate items, so that one group's softmax runs while the
// other waits for its MMAs, its TMEM loads or its output store.
//   warp 0      TMA: the Q tile (128 x 64, K-major, 128-byte swizzle) of item
//               n into group n % 2's stage, K (128 keys x 64, K-major) and V
//               (128 keys x 64, MN-major: two 64-key boxes) through a 3-deep
//               ring, in item order. Before the dependency wait it asks the L2
//               for its first items' tiles.
//   warps 1, 2  tcgen05.mma, one issuing thread per softmax group: S = Q K^T
//               (M 128, N 128, K 64) into the group's TMEM S buffer (columns
//               0-127 or 128-255), then O += P V (M 128, N 64, K 128) into its
//               O buffer (columns 256-319 or 320-383).
//   warps 4-7,  the two softmax groups: warp w reads TMEM lanes 32*(w%4)..
//   warps 8-11  (its 32 query rows), one thread per row and all 128 keys of a
//               block, so no exchange between warps is needed. Scores are
//               scaled into base-2 units (scale * log2 e) by a packed fp32x2
//               FMA and exponentiated with the hardware ex2; P is rounded to
//               bf16 into the group's shared-memory P buffer in the operand
//               layout of the next MMA. A 32-key chunk that no row of a warp
//               sees (above the causal diagonal, or past T) is neither read
//               nor exponentiated. When a later key block raises a row's max,
//               the warp scales that row's O in TMEM by alpha = 2^(m - m')
//               before the block's P.V adds to it. At an item's end the warp
//               divides O by l, stages its rows as two 32 x 32 bf16 boxes in
//               its part of the P buffer and stores them by TMA through a
//               B x T x C view of the output, which leaves out the rows past a
//               sequence's end.
// Every wait is bounded (about 1 s); a CTA that gives up sets the device
// status word to LIN_ERR_DEVICE_TIMEOUT and leaves its output incomplete.
#include <math.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "timeline.cuh"

namespace lin {
namespace {

// Timeline stamps (timeline build only): record = blockIdx.x; [0] set up,
// [1] producer past its dependency wait, [2] teardown; for the CTA's work item
// n < 16, at 8 + 10 n + k: k 0 Q copy issued, 1 first K/V copy issued, 2 the
// group's MMA issuer saw the first S inputs ready, 3 first S MMAs committed, 4
// the item's softmax group (warp 6 or 10) saw the first S, 5 it released the
// last P, 6 last P.V MMAs committed, 7 warp 6 or 10 saw the last P.V, 8 it
// issued its output store, 9 warp 5 or 9 issued its output store.
__device__ unsigned long long g_timeline_attn[kTimelineCtas * kTimelineSlots];
#define AT_STAMP(n, k) \
    do {                \
        if ((n) < 16) LIN_STAMP(g_timeline_attn, blockIdx.x, 8 + 10 * (n) + (k)); \
    } while (0)

constexpr int kAtBM = 128;                          // query rows per work item
constexpr int kAtBN = 128;                          // keys per block
constexpr int kAtD = 64;                            // head width
constexpr int kAtThreads = 384;                     // warp 0 TMA, warps 1-2 MMA, warps 4-7 and 8-11 softmax
// Register split (setmaxnreg, per warpgroup): launched at kAtLaunchRegs a
// thread, warpgroup 0 (TMA, the two MMA issuers, an idle warp) gives registers back down to
// kAtRegsLow and the two softmax warpgroups take kAtRegsHigh:
// 128 * 72 + 256 * 216 = 64512 = 384 * 168. The host refuses to launch when
// the compiled kernel holds fewer than kAtLaunchRegs registers a thread (the
// increase could then never be granted).
constexpr int kAtLaunchRegs = 168, kAtRegsLow = 72, kAtRegsHigh = 216;
static_assert(128 * kAtRegsLow + 256 * kAtRegsHigh <= kAtThreads * kAtLaunchRegs, "register split");
constexpr int kAtQStages = 2;                       // one Q tile per softmax group
constexpr int kAtKvStages = 3;
constexpr uint32_t kAtQBytes = kAtBM * kAtD * 2;    // 16 KiB
constexpr uint32_t kAtKBytes = kAtBN * kAtD * 2;    // 16 KiB
constexpr uint32_t kAtVBytes = kAtBN * kAtD * 2;    // 16 KiB (two 64-key boxes)
constexpr uint32_t kAtPBytes = kAtBM * kAtBN * 2;   // 32 KiB per group (two 64-key K-major blocks)
constexpr uint32_t kAtTmemCols = 512;               // S of group 0 / 1 in columns 0-127 / 128-255,
constexpr uint32_t kAtOCol = 256;                   // O of group 0 / 1 in columns 256-319 / 320-383
constexpr int kAtBars = 2 * kAtQStages + 2 * kAtKvStages + 8;

constexpr size_t at_smem_bytes() {
    return 1024 + kAtQStages * kAtQBytes + kAtKvStages * (kAtKBytes + kAtVBytes) + 2 * kAtPBytes + kAtBars * 8 + 16;
}
static_assert(at_smem_bytes() <= 227 * 1024, "shared memory");

struct AttnArgs {
    int B, T, H, C;
    int nqb;             // query blocks per sequence
    int items;           // B * H * nqb
    int causal;
    float scale_log2;    // softmax scale times log2(e)
    uint16_t* out;
    float* lse;
    int* status;
};

struct Item {
    int b, h, qb, nkb;   // sequence, head, query block, key blocks to visit
};

// Items are ordered query block major, last block first: in the causal case
// the items with the most key blocks start first.
__device__ __forceinline__ Item at_item(const AttnArgs& a, int i) {
    const int bh_count = a.B * a.H;
    Item it;
    it.qb = a.nqb - 1 - i / bh_count;
    const int bh = i % bh_count;
    it.b = bh / a.H;
    it.h = bh % a.H;
    it.nkb = a.causal ? it.qb + 1 : a.nqb;
    return it;
}

// The CTA's items are blockIdx.x, blockIdx.x + gridDim.x, ... (local index n
// = 0, 1, 2, ...), their key blocks numbered in that order (g = 0, 1, 2, ...:
// the order of the K/V ring). Softmax group grp takes the items with n % 2 ==
// grp; its walker steps over the other group's items.
struct GWalker {
    int i, n, j, g;      // item, local item index, key block within it, CTA block index
    int nkb;             // key blocks of item i
    bool valid;
    __device__ __forceinline__ static int blocks(const AttnArgs& a, int i) {
        return a.causal ? a.nqb - i / (a.B * a.H) : a.nqb;  // query block + 1, or all
    }
    __device__ __forceinline__ void init(const AttnArgs& a, int grp) {
        i = blockIdx.x;
        n = 0;
        j = 0;
        g = 0;
        valid = i < a.items;
        nkb = valid ? blocks(a, i) : 0;
        if (grp == 1 && valid) skip(a);
    }
    // Move to item n + 1 (from the start of item n).
    __device__ __forceinline__ void skip(const AttnArgs& a) {
        g += nkb;
        ++n;
        i += gridDim.x;
        valid = i < a.items;
        nkb = valid ? blocks(a, i) : 0;
    }
    __device__ __forceinline__ void next(const AttnArgs& a) {
        ++j;
        if (j < nkb) {
            ++g;
            return;
        }
        j = 0;
        g -= nkb - 1;  // back to the item's first block
        skip(a);
        if (valid) skip(a);
    }
};

__device__ __forceinline__ float ex2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_hw(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 3-D tiled TMA store of a shared-memory box to (x = column, y = token, z =
// sequence); elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Packed pairs of fp32 (sm_100+ f32x2 arithmetic: one instruction for two
// lanes' worth of values held by one thread) and the three-input max.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Store 32 consecutive fp32 columns of this thread's TMEM lane (the rescale of
// the P.V accumulator), and wait for this thread's TMEM stores.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void regs_release_low() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kAtRegsLow));
}
__device__ __forceinline__ void regs_take_high() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kAtRegsHigh));
}

__global__ void __launch_bounds__(kAtThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmQ32,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const AttnArgs a) {
    constexpr uint32_t IDESC_S = make_idesc(1u, kAtBM, kAtBN);               // Q, K both K-major
    constexpr uint32_t IDESC_O = make_idesc(1u, kAtBM, kAtD, false, true);   // P K-major, V MN-major
    constexpr int QS = kAtQStages, KS = kAtKvStages;
    constexpr int GROUP_WARPS = 4;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                    // Q of group 0 / 1
    uint8_t* sK = sQ + QS * kAtQBytes;
    uint8_t* sV = sK + KS * kAtKBytes;
    uint8_t* sP = sV + KS * kAtVBytes;     // P of group 0 / 1
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * kAtPBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAtBars);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    // bars: qfull[2] qempty[2] kvfull[KS] kvempty[KS] sfull[2] sfree[2] pfull[2] pvfull[2];
    // the per-group barriers count that group's blocks (phase = its block count).
    const uint32_t qfull0 = smem_u32(bars), qempty0 = qfull0 + 8 * QS;
    const uint32_t kvfull0 = qempty0 + 8 * QS, kvempty0 = kvfull0 + 8 * KS;
    const uint32_t sfull0 = kvempty0 + 8 * KS, sfree0 = sfull0 + 16, pfull0 = sfull0 + 32, pvfull0 = sfull0 + 48;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < QS; ++s) {
            mbar_init(qfull0 + 8 * s, 1);
            mbar_init(qempty0 + 8 * s, 1);
        }
        for (int s = 0; s < KS; ++s) {
            mbar_init(kvfull0 + 8 * s, 1);
            mbar_init(kvempty0 + 8 * s, 1);
        }
        for (int grp = 0; grp < 2; ++grp) {
            mbar_init(sfull0 + 8 * grp, 1);
            mbar_init(sfree0 + 8 * grp, GROUP_WARPS);
            mbar_init(pfull0 + 8 * grp, GROUP_WARPS);
            mbar_init(pvfull0 + 8 * grp, 1);
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmQK);
        tma_prefetch_map(&tmQ32);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmO);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kAtTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (threadIdx.x == 0) LIN_STAMP(g_timeline_attn, blockIdx.x, 0);


    auto give_up = [&]() {
        atomicExch(s_abort, 1);
        atomicExch(a.status, (int)LIN_ERR_DEVICE_TIMEOUT);
    };
    auto aborted = [&]() { return *(volatile int*)s_abort != 0; };

    if (warp < 4) regs_release_low();  // warpgroup 0: TMA, MMA and two idle warps
    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: the CTA's items in order; Q of item n to
            // stage n % 2 (its group's), K/V blocks through the ring ----
            // The first items' Q, K and V to L2 while the previous kernel
            // finishes: an L2 prefetch returns nothing to the SM, and the L2 is
            // where all writes meet, so this changes no result whatever that
            // kernel writes. The copies into shared memory wait for it.
            for (int i = blockIdx.x, n = 0; i < a.items && n < 2; i += gridDim.x, ++n) {
                const Item it = at_item(a, i);
                const int row0 = it.b * a.T;
                tma_prefetch_l2_2d(&tmQK, it.h * kAtD, row0 + it.qb * kAtBM);  // rows < B*T: a query block starts inside
                tma_prefetch_l2_2d(&tmQK, a.C + it.h * kAtD, row0);
                tma_prefetch_l2_2d(&tmV, 2 * a.C + it.h * kAtD, row0);
                if (row0 + 64 < a.B * a.T) tma_prefetch_l2_2d(&tmV, 2 * a.C + it.h * kAtD, row0 + 64);
            }
            pdl_wait();  // qkv only after the previous kernel on the stream has finished
            LIN_STAMP(g_timeline_attn, blockIdx.x, 1);
            uint32_t g = 0, nq = 0;  // K/V blocks and Q tiles issued
            bool ok = true;
            for (int i = blockIdx.x; ok && i < a.items; i += gridDim.x) {
                const Item it = at_item(a, i);
                const int row0 = it.b * a.T;
                const uint32_t qs = nq % QS, qph = (nq / QS) & 1;
                if (aborted() || !mbar_wait(qempty0 + 8 * qs, qph ^ 1)) {
                    ok = false;
                    break;
                }
                // Q in four 32-row boxes; group 1 (odd items) takes them in
                // reverse order, so that the TMEM lane quadrant that holds a
                // block's last (causally heaviest) rows in one group holds the
                // first rows in the other, and each SM sub-partition carries one
                // heavy and one light warp.
                mbar_expect_tx(qfull0 + 8 * qs, kAtQBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int quad = (nq & 1) ? 3 - k : k;
                    tma_load_2d(smem_u32(sQ + qs * kAtQBytes + quad * 4096), &tmQ32, qfull0 + 8 * qs, it.h * kAtD,
                                row0 + it.qb * kAtBM + 32 * k);
                }
                AT_STAMP(nq, 0);
                ++nq;
                for (int j = 0; j < it.nkb; ++j) {
                    const uint32_t s = g % KS, ph = (g / KS) & 1;
                    if (aborted() || !mbar_wait(kvempty0 + 8 * s, ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    const int kr = row0 + j * kAtBN;
                    mbar_expect_tx(kvfull0 + 8 * s, kAtKBytes + kAtVBytes);
                    tma_load_2d(smem_u32(sK + s * kAtKBytes), &tmQK, kvfull0 + 8 * s, a.C + it.h * kAtD, kr);
                    tma_load_2d(smem_u32(sV + s * kAtVBytes), &tmV, kvfull0 + 8 * s, 2 * a.C + it.h * kAtD, kr);
                    tma_load_2d(smem_u32(sV + s * kAtVBytes + 8192), &tmV, kvfull0 + 8 * s, 2 * a.C + it.h * kAtD,
                                kr + 64);
                    if (j == 0) AT_STAMP(nq - 1, 1);
                    ++g;
                }
            }
            if (!ok) {
                give_up();
                // Let the copies still in flight land before the CTA exits (the
                // last ring's worth of each barrier is the phase issued last).
                for (uint32_t n = nq > (uint32_t)QS ? nq - QS : 0; n < nq; ++n)
                    mbar_wait(qfull0 + 8 * (n % QS), (n / QS) & 1);
                for (uint32_t n = g > (uint32_t)KS ? g - KS : 0; n < g; ++n)
                    mbar_wait(kvfull0 + 8 * (n % KS), (n / KS) & 1);
            }
        }
    } else if (warp == 1 || warp == 2) {
        if (lane == 0) {
            // ---- MMA issuer of group grp = warp - 1 (one thread per group):
            // S of the group's block into its S buffer, then P.V of that block
            // once its P is in shared memory; every wait blocks on one barrier ----
            const int grp = warp - 1;
            GWalker w;
            w.init(a, grp);
            uint32_t c = 0;  // the group's blocks issued
            bool ok = true;
            while (w.valid) {
                const uint32_t s = w.g % KS, ph = (w.g / KS) & 1;
                if (aborted() || (w.j == 0 && !mbar_wait(qfull0 + 8 * grp, (w.n / QS) & 1)) ||
                    !mbar_wait(kvfull0 + 8 * s, ph) || (c > 0 && !mbar_wait(sfree0 + 8 * grp, (c - 1) & 1))) {
                    ok = false;
                    break;
                }
                if (w.j == 0) AT_STAMP(w.n, 2);
                tc_fence_after();
                const uint64_t qd = sw128_kmajor_desc(smem_u32(sQ + grp * kAtQBytes));
                const uint64_t kd = sw128_kmajor_desc(smem_u32(sK + s * kAtKBytes));
#pragma unroll
                for (int kk = 0; kk < kAtD / 16; ++kk)
                    tc_mma<true>(tmem_base + 128u * grp, qd + 2u * kk, kd + 2u * kk, IDESC_S, kk != 0 ? 1u : 0u);
                tc_commit(sfull0 + 8 * grp);
                if (w.j == 0) AT_STAMP(w.n, 3);
                if (w.j == w.nkb - 1) tc_commit(qempty0 + 8 * grp);  // Q is read by S only

                if (aborted() || !mbar_wait(pfull0 + 8 * grp, c & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t pd = sw128_kmajor_desc(smem_u32(sP + grp * kAtPBytes));
                const uint64_t vd = sw128_mnmajor_desc(smem_u32(sV + s * kAtVBytes));
                // K = 128 keys in 8 steps of 16: P advances 32 bytes within a
                // 64-key block (+2) and 16 KiB between the blocks (+1024); V
                // advances 16 key rows (2 KiB, +128). O accumulates over the
                // item's blocks.
#pragma unroll
                for (int kk = 0; kk < kAtBN / 16; ++kk)
                    tc_mma<true>(tmem_base + kAtOCol + 64u * grp, pd + 1024u * (kk >> 2) + 2u * (kk & 3),
                                 vd + 128u * kk, IDESC_O, (kk != 0 || w.j != 0) ? 1u : 0u);
                tc_commit(pvfull0 + 8 * grp);
                tc_commit(kvempty0 + 8 * s);  // K and V of this block are no longer read
                if (w.j == w.nkb - 1) AT_STAMP(w.n, 6);
                w.next(a);
                ++c;
            }
            if (!ok) give_up();
            // Do not reach the teardown before this group's MMAs have completed.
            if (c > 0) mbar_wait(pvfull0 + 8 * grp, (c - 1) & 1);
            if (!ok) mbar_wait(sfull0 + 8 * grp, c & 1);  // an S issued without its P.V
        }
    } else if (warp >= 4) {
        regs_take_high();
        // ---- softmax and output, two warpgroups working on alternate
        // items; warp w reads TMEM lanes 32*(w%4).. (its 32 query rows), one
        // thread per row, all 128 keys of a block ----
        pdl_wait();  // out and lse only after the previous kernel on the stream has finished
        const int grp = (warp - 4) >> 2;
        const int q = warp & 3;
        const int r = 32 * q + lane;            // TMEM lane = row of S, P and O
        const int qq = grp ? 3 - q : q;         // the warp's query rows: 32 qq .. 32 qq + 31
        const int qr = 32 * qq + lane;          // this thread's query row within the block
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t tS = tmem_base + lane_addr + 128u * grp;
        const uint32_t tO = tmem_base + lane_addr + kAtOCol + 64u * grp;
        uint8_t* sPg = sP + grp * kAtPBytes;
        uint8_t* prow = sPg + (r >> 3) * 1024 + (r & 7) * 128;  // + 16 KiB for keys 64-127
        // Output staging: the warp's rows of the group's P buffer (free once
        // the item's last P.V has completed, until the warp writes its next P):
        // two 32 x 32 boxes (head columns 0-31, 32-63), 64-byte rows with the
        // 64-byte swizzle of the output map (piece v of row i at v ^ ((i >> 1) & 3)).
        uint8_t* obox = sPg + q * 4096;
        const float NEG_INF = -INFINITY;
        const float sl2 = a.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const bool stamper = lane == 0 && q == 2;  // warps 6 and 10

        float m = NEG_INF, l = 0.f;   // running max of the raw scores, running sum
        bool store_pending = false;   // this warp's boxes may still be read by a TMA store
        bool ok = true;
        uint32_t cnt = 0;             // this group's blocks so far
        GWalker w;
        w.init(a, grp);
        while (w.valid) {
            const Item it = at_item(a, w.i);
            const int j = w.j;
            const bool last = j == it.nkb - 1;
            const int qpos = it.qb * kAtBM + qr;
            // Keys visible to this row: kpos < lim. A 32-key chunk that no row
            // of the warp sees is neither read nor exponentiated; one that every
            // row sees whole needs no mask.
            const int lim = a.causal ? min(qpos + 1, a.T) : a.T;
            const int wmax = a.causal ? min(it.qb * kAtBM + 32 * qq + 32, a.T) : a.T;
            const int wmin = a.causal ? min(it.qb * kAtBM + 32 * qq + 1, a.T) : a.T;
            const int k0 = j * kAtBN;

            // 1. the block's 128 raw scores of this row in one round trip to
            //    TMEM (the chunks no row of the warp sees are not read), masked,
            //    and their max (scale > 0 commutes with the max)
            if (!__all_sync(0xffffffffu, !aborted() && mbar_wait(sfull0 + 8 * grp, cnt & 1))) {
                ok = false;
                break;
            }
            if (stamper && j == 0) AT_STAMP(w.n, 4);
            tc_fence_after();
            uint32_t sv[4][32];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                if (k0 + 32 * ch < wmax) tmem_ld32_async(tS + 32u * ch, sv[ch]);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                if (k0 + 32 * ch < wmax) tmem_wait_ld(sv[ch]);
            float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int c0 = k0 + 32 * ch;
                if (c0 >= wmax) continue;
                if (c0 + 32 > wmin) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c0 + c >= lim) sv[ch][c] = __float_as_uint(NEG_INF);
                }
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    mx[ch] = max3(mx[ch], __uint_as_float(sv[ch][c]), __uint_as_float(sv[ch][c + 1]));
            }
            const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = fmaxf(m, mloc);
            const float m_use = m_new == NEG_INF ? 0.f : m_new;  // a row with no visible key so far
            const float alpha = ex2_hw((m - m_use) * sl2);      // 0 at the first block (m = -inf)
            const uint64_t nmbx2 = f2_pack(-m_use * sl2, -m_use * sl2);
            m = m_new;

            // 2. the group's previous P.V has completed: P may be rewritten, and
            //    a later block of the item rescales O by alpha before its P.V
            if (cnt > 0 && j > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(pvfull0 + 8 * grp, (cnt - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                    uint32_t ov[2][32];
                    tmem_ld32_async(tO, ov[0]);
                    tmem_ld32_async(tO + 32u, ov[1]);
                    tmem_wait_ld(ov[0]);
                    tmem_wait_ld(ov[1]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int d = 0; d < 32; ++d) ov[hh][d] = __float_as_uint(__uint_as_float(ov[hh][d]) * alpha);
                        tmem_st32(tO + 32u * hh, ov[hh]);
                    }
                    tmem_wait_st();
                }
            }
            if (store_pending) {
                if (lane == 0) bulk_wait_read_all();  // the boxes have been read out
                __syncwarp();
                store_pending = false;
            }

            // 3. p = 2^(s * scale * log2 e - max) per 32-key chunk, rounded to
            //    bf16 into the group's P buffer (row r: 128-byte rows of two
            //    K-major 64-key blocks, 16-byte pieces swizzled by r % 8)
            uint64_t ls2[2] = {0ull, 0ull};  // packed partial row sums (+0.0f pairs)
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t pk[16];
                if (k0 + 32 * ch < wmax) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[ch][c]), __uint_as_float(sv[ch][c + 1])), sl2x2,
                                         nmbx2),
                                  x0, x1);
                        const float p0 = ex2_hw(x0), p1 = ex2_hw(x1);
                        ls2[(c >> 1) & 1] = f2_add(ls2[(c >> 1) & 1], f2_pack(p0, p1));
                        pk[c >> 1] = pack_bf16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = 0u;
                }
                uint8_t* row = prow + (ch >> 1) * (kAtPBytes / 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int piece = 4 * (ch & 1) + i;
                    *reinterpret_cast<uint4*>(row + ((piece ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            // S has been read, P written: release both
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sfree0 + 8 * grp);
                mbar_arrive(pfull0 + 8 * grp);
            }
            if (stamper && last) AT_STAMP(w.n, 5);
            float la, lb, lc, ld;
            f2_unpack(ls2[0], la, lb);
            f2_unpack(ls2[1], lc, ld);
            l = fmaf(l, alpha, (la + lb) + (lc + ld));

            // 4. the item's last block: wait for its P.V, write O / l (bf16)
            //    by TMA store, and lse
            if (last) {
                if (!__all_sync(0xffffffffu, mbar_wait(pvfull0 + 8 * grp, cnt & 1))) {
                    ok = false;
                    break;
                }
                if (stamper) AT_STAMP(w.n, 7);
                tc_fence_after();
                const float inv = 1.0f / l;
                uint32_t ovv[2][32];
                tmem_ld32_async(tO, ovv[0]);
                tmem_ld32_async(tO + 32u, ovv[1]);
                tmem_wait_ld(ovv[0]);
                tmem_wait_ld(ovv[1]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t* ov = ovv[hh];
                    uint8_t* orow = obox + hh * 2048 + lane * 64;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        *reinterpret_cast<uint4*>(orow + ((v ^ ((lane >> 1) & 3)) << 4)) = make_uint4(
                            pack_bf16x2(__uint_as_float(ov[8 * v]) * inv, __uint_as_float(ov[8 * v + 1]) * inv),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv, __uint_as_float(ov[8 * v + 3]) * inv),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv, __uint_as_float(ov[8 * v + 5]) * inv),
                            pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv, __uint_as_float(ov[8 * v + 7]) * inv));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // Rows past the sequence's end (t >= T) lie outside the map and are not written.
                    const int y = it.qb * kAtBM + 32 * qq;
                    tma_store_3d(&tmO, smem_u32(obox), it.h * kAtD, y, it.b);
                    tma_store_3d(&tmO, smem_u32(obox + 2048), it.h * kAtD + 32, y, it.b);
                    bulk_commit();
                }
                store_pending = true;
                if (a.lse && qpos < a.T)
                    a.lse[((size_t)it.b * a.H + it.h) * a.T + qpos] = (m * sl2 + lg2_hw(l)) * 0.6931471805599453f;
                if (stamper) AT_STAMP(w.n, 8);
                if (lane == 0 && q == 1) AT_STAMP(w.n, 9);  // warps 5 and 9
                m = NEG_INF;
                l = 0.f;
            }
            w.next(a);
            ++cnt;
        }
        if (!ok) give_up();
        if (lane == 0) bulk_wait_read_all();  // the output boxes are read out before the CTA exits
    }

    __syncwarp();
    tc_fence_before();
    if (threadIdx.x == 64) LIN_STAMP(g_timeline_attn, blockIdx.x, 2);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kAtTmemCols);
    }
}

// The driver's tensor-map encoder, looked up once (thread-safe static).
PFN_cuTensorMapEncodeTiled_v12000 at_encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

// The output viewed as B x T x C bf16 (so that a box never crosses into the
// next sequence): box = 32 columns x 32 tokens x 1 sequence, 64-byte swizzle.
bool make_out3_map(CUtensorMap* map, void* base, int B, int T, int C) {
    auto fn = at_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(T) * C * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int launch_attention(const AttnProblem& p) {
    const int C = p.H * kAtD;
    const long long rows = (long long)p.B * p.T;
    CUtensorMap tqk, tv;
    // q and k: 64-column (128-byte) x 128-row boxes of the (B*T) x 3C tensor;
    // v: 64-column x 64-row boxes read MN-major.
    if (!make_kmajor_map(&tqk, p.qkv, true, (int)rows, 3 * C, 128)) return LIN_ERR_CUDA;
    CUtensorMap tq32;  // q in 32-row boxes
    if (!make_kmajor_map(&tq32, p.qkv, true, (int)rows, 3 * C, 32)) return LIN_ERR_CUDA;
    if (!make_mnmajor_map(&tv, p.qkv, (int)rows, 3 * C)) return LIN_ERR_CUDA;
    CUtensorMap to;
    if (!make_out3_map(&to, p.out, p.B, p.T, C)) return LIN_ERR_CUDA;
    AttnArgs a;
    a.B = p.B;
    a.T = p.T;
    a.H = p.H;
    a.C = C;
    a.nqb = (p.T + kAtBM - 1) / kAtBM;
    a.items = p.B * p.H * a.nqb;
    a.causal = p.causal ? 1 : 0;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.out = static_cast<uint16_t*>(p.out);
    a.lse = p.lse;
    a.status = p.dev_status;
    const int grid = a.items < p.sm_count ? a.items : p.sm_count;
    constexpr size_t smem = at_smem_bytes();
    static std::atomic<unsigned long long> attr_set{0};
    if (ensure_smem_attr(attr_set, attn_fwd_kernel, smem) != LIN_OK) return LIN_ERR_CUDA;
    // The register split needs the kernel launched at kAtLaunchRegs a thread
    // (else the softmax warpgroups' increase would wait forever): refuse otherwise.
    static const int regs = []() {
        cudaFuncAttributes fa;
        return cudaFuncGetAttributes(&fa, attn_fwd_kernel) == cudaSuccess ? fa.numRegs : 0;
    }();
    if (regs < kAtLaunchRegs) return LIN_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = p.early_start ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, attn_fwd_kernel, tqk, tq32, tv, to, a) != cudaSuccess) return LIN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

int timeline_copy_attn(void* dst, size_t bytes, bool clear) {
#ifdef LIN_TIMELINE
    const size_t total = sizeof(unsigned long long) * kTimelineCtas * kTimelineSlots;
    if (dst && bytes > 0 &&
        cudaMemcpyFromSymbol(dst, g_timeline_attn, bytes < total ? bytes : total) != cudaSuccess)
        return LIN_ERR_CUDA;
    if (clear) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_timeline_attn) != cudaSuccess || cudaMemset(p, 0, total) != cudaSuccess)
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
