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
// 128 queries), largest causal items first.
//   warp 0      TMA: Q (128 x 64, K-major, 128-byte swizzle) into a 3-deep
//               ring, K (128 keys x 64, K-major) and V (128 keys x 64,
//               MN-major: two 64-key boxes) into a 3-deep ring, up to two
//               items ahead. Before the dependency wait it asks the L2 for its
//               first items' tiles.
//   warp 1      tcgen05.mma: S = Q K^T (M 128, N 128, K 64) into one of two
//               TMEM buffers (columns 0-127, 128-255, alternating blocks), and
//               O += P V (M 128, N 64, K 128) into one of two O buffers
//               (columns 256-319, 320-383, alternating items). It polls its
//               barriers and issues whichever of the next S or the next P.V
//               has its inputs first, up to two S ahead.
//   warps 2-9   softmax and output: warp w reads TMEM lanes 32*(w%4).. (its
//               query rows) and one half of the 128 key columns; the two
//               warps of a row exchange their row maxima (and the previous
//               item's row sums) through shared memory. Scores are scaled into
//               base-2 units (scale * log2 e) by a packed fp32x2 FMA and
//               exponentiated with the hardware ex2; P is rounded to bf16 into
//               shared memory in the operand layout of the next MMA. A 32-key
//               chunk that no row of a warp sees (above the causal diagonal,
//               or past T) is neither read nor exponentiated. When a later key
//               block raises a row's max, the warp scales that row's O in TMEM
//               by alpha = 2^(m - m') before the block's P.V adds to it. An
//               item's output (O / l, bf16) is written during the next block,
//               once its last P.V has completed: through a 32 x 32 box per warp
//               in shared memory and a TMA store of a B x T x C view of the
//               output, which leaves out the rows past a sequence's end.
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
// n < 16, at 8 + 10 n + k: k 0 Q copy issued, 1 first K/V copy issued, 2 MMA
// warp saw the first K/V block land, 3 first S MMAs committed, 4 softmax warp 2
// saw the first S, 5 softmax warp 2 released the last P, 6 last P.V MMAs
// committed, 7 softmax warp 2 saw the last P.V, 8 softmax warp 2 stored its
// rows, 9 softmax warp 9 stored its rows.
__device__ unsigned long long g_timeline_attn[kTimelineCtas * kTimelineSlots];
#define AT_STAMP(n, k) \
    do {                \
        if ((n) < 16) LIN_STAMP(g_timeline_attn, blockIdx.x, 8 + 10 * (n) + (k)); \
    } while (0)

constexpr int kAtBM = 128;                          // query rows per work item
constexpr int kAtBN = 128;                          // keys per block
constexpr int kAtD = 64;                            // head width
constexpr int kAtThreads = 320;                     // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int kAtQStages = 3;
constexpr int kAtKvStages = 3;
constexpr uint32_t kAtQBytes = kAtBM * kAtD * 2;    // 16 KiB
constexpr uint32_t kAtKBytes = kAtBN * kAtD * 2;    // 16 KiB
constexpr uint32_t kAtVBytes = kAtBN * kAtD * 2;    // 16 KiB (two 64-key boxes)
constexpr uint32_t kAtPBytes = kAtBM * kAtBN * 2;   // 32 KiB (two 64-key K-major blocks)
constexpr uint32_t kAtOutBoxBytes = 32 * 32 * 2;    // one softmax warp's 32 x 32 bf16 output box
constexpr uint32_t kAtTmemCols = 512;               // S in columns 0-127 and 128-255 (alternating blocks)
constexpr uint32_t kAtOCol = 256;                   // O of even items in columns 256-319, odd items 320-383
constexpr int kAtRedFloats = 2 * 2 * 2 * 128;      // row maxima and row sums, each [parity][half][row]
constexpr int kAtOkInts = 32;                       // [parity][warp] after maxima, [warp] after sums
constexpr int kAtBars = 2 * kAtQStages + 2 * kAtKvStages + 6;

constexpr size_t at_smem_bytes() {
    return 1024 + kAtQStages * kAtQBytes + kAtKvStages * (kAtKBytes + kAtVBytes) + kAtPBytes + 8 * kAtOutBoxBytes +
           kAtRedFloats * 4 + kAtOkInts * 4 + kAtBars * 8 + 16;
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

// The CTA's key blocks in order: items blockIdx.x, blockIdx.x + gridDim.x, ...
struct Walker {
    int i, n, j;         // item, item count so far, key block within the item
    bool valid;
    Item it;
    __device__ __forceinline__ void init(const AttnArgs& a) {
        i = blockIdx.x;
        n = 0;
        j = 0;
        valid = i < a.items;
        if (valid) it = at_item(a, i);
    }
    __device__ __forceinline__ void next(const AttnArgs& a) {
        if (++j < it.nkb) return;
        j = 0;
        ++n;
        i += gridDim.x;
        valid = i < a.items;
        if (valid) it = at_item(a, i);
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

// Non-blocking test of an mbarrier phase (the MMA thread polls two barriers).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__global__ void __launch_bounds__(kAtThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmO, const AttnArgs a) {
    constexpr uint32_t IDESC_S = make_idesc(1u, kAtBM, kAtBN);               // Q, K both K-major
    constexpr uint32_t IDESC_O = make_idesc(1u, kAtBM, kAtD, false, true);   // P K-major, V MN-major
    constexpr int QS = kAtQStages, KS = kAtKvStages;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + QS * kAtQBytes;
    uint8_t* sV = sK + KS * kAtKBytes;
    uint8_t* sP = sV + KS * kAtVBytes;
    uint8_t* sOut = sP + kAtPBytes;                              // 8 output boxes
    float* red_max = reinterpret_cast<float*>(sOut + 8 * kAtOutBoxBytes);  // [parity][half][row]
    float* red_sum = red_max + 2 * 2 * 128;                      // [parity][half][row]
    int* red_ok = reinterpret_cast<int*>(red_sum + 2 * 2 * 128); // [parity][8]
    uint64_t* bars = reinterpret_cast<uint64_t*>(red_ok + kAtOkInts);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAtBars);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    // bars: qfull[QS] qempty[QS] kvfull[KS] kvempty[KS] sfull[2] sfree[2] pfull pvfull
    // (S buffer b = block g % 2 holds its u = g / 2-th block: phase u of sfull[b], sfree[b])
    const uint32_t qfull0 = smem_u32(bars), qempty0 = qfull0 + 8 * QS;
    const uint32_t kvfull0 = qempty0 + 8 * QS, kvempty0 = kvfull0 + 8 * KS;
    const uint32_t sfull0 = kvempty0 + 8 * KS, sfree0 = sfull0 + 16, pfull = sfull0 + 32, pvfull = sfull0 + 40;
    constexpr int SOFT_WARPS = kAtThreads / 32 - 2;

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
        for (int b = 0; b < 2; ++b) {
            mbar_init(sfull0 + 8 * b, 1);
            mbar_init(sfree0 + 8 * b, SOFT_WARPS);
        }
        mbar_init(pfull, SOFT_WARPS);
        mbar_init(pvfull, 1);
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmQK);
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

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            // The first items' Q, K and V to L2 while the previous kernel
            // finishes: an L2 prefetch returns nothing to the SM, and the L2 is
            // where all writes meet, so this changes no result whatever that
            // kernel writes. The copies into shared memory wait for it.
            for (int i = blockIdx.x, n = 0; i < a.items && n < QS; i += gridDim.x, ++n) {
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
                mbar_expect_tx(qfull0 + 8 * qs, kAtQBytes);
                tma_load_2d(smem_u32(sQ + qs * kAtQBytes), &tmQK, qfull0 + 8 * qs, it.h * kAtD, row0 + it.qb * kAtBM);
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
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: S of blocks g + 1 and g + 2 (two TMEM buffers) may
            // go before P.V of block g, so that they overlap the softmax of
            // block g; whichever has its inputs first is issued first ----
            Walker ws, wp;
            ws.init(a);
            wp.init(a);
            uint32_t gs = 0, gp = 0;
            auto s_ready = [&]() -> bool {
                const uint32_t s = gs % KS, ph = (gs / KS) & 1;
                const uint32_t qs = ws.n % QS, qph = (ws.n / QS) & 1;
                const uint32_t b = gs & 1, u = gs >> 1;  // S buffer and its use
                return (ws.j != 0 || mbar_test(qfull0 + 8 * qs, qph)) && mbar_test(kvfull0 + 8 * s, ph) &&
                       (u == 0 || mbar_test(sfree0 + 8 * b, (u - 1) & 1));
            };
            auto issue_s = [&]() {
                const uint32_t s = gs % KS, qs = ws.n % QS;
                if (ws.j == 0) AT_STAMP(ws.n, 2);
                tc_fence_after();
                const uint64_t qd = sw128_kmajor_desc(smem_u32(sQ + qs * kAtQBytes));
                const uint64_t kd = sw128_kmajor_desc(smem_u32(sK + s * kAtKBytes));
#pragma unroll
                for (int kk = 0; kk < kAtD / 16; ++kk)
                    tc_mma<true>(tmem_base + 128u * (gs & 1), qd + 2u * kk, kd + 2u * kk, IDESC_S, kk != 0 ? 1u : 0u);
                tc_commit(sfull0 + 8 * (gs & 1));
                if (ws.j == 0) AT_STAMP(ws.n, 3);
                if (ws.j == ws.it.nkb - 1) tc_commit(qempty0 + 8 * qs);  // Q is read by S only
                ws.next(a);
                ++gs;
            };
            auto issue_pv = [&]() {
                const uint32_t s = gp % KS;
                tc_fence_after();
                const uint64_t pd = sw128_kmajor_desc(smem_u32(sP));
                const uint64_t vd = sw128_mnmajor_desc(smem_u32(sV + s * kAtVBytes));
                // K = 128 keys in 8 steps of 16: P advances 32 bytes within a
                // 64-key block (+2) and 16 KiB between the blocks (+1024); V
                // advances 16 key rows (2 KiB, +128).
#pragma unroll
                for (int kk = 0; kk < kAtBN / 16; ++kk)
                    tc_mma<true>(tmem_base + kAtOCol + 64u * (wp.n & 1), pd + 1024u * (kk >> 2) + 2u * (kk & 3),
                                 vd + 128u * kk, IDESC_O,
                                 (kk != 0 || wp.j != 0) ? 1u : 0u);  // O accumulates over the item's blocks
                tc_commit(pvfull);
                tc_commit(kvempty0 + 8 * s);  // K and V of this block are no longer read
                if (wp.j == wp.it.nkb - 1) AT_STAMP(wp.n, 6);
                wp.next(a);
                ++gp;
            };
            bool ok = true;
            uint32_t idle = 0;
            unsigned long long t_idle = 0;
            while (wp.valid) {
                if (ws.valid && gs <= gp + 2 && s_ready()) {
                    issue_s();
                    idle = 0;
                } else if (gp < gs && mbar_test(pfull, gp & 1)) {
                    issue_pv();
                    idle = 0;
                } else {
                    // Bounded: give up after kWaitNs without progress.
                    if (idle == 0) t_idle = global_ns();
                    if ((++idle & 255u) == 0u && (aborted() || global_ns() - t_idle > kWaitNs || idle >= kWaitIters)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) give_up();
            // Do not reach the teardown before the last MMAs have completed.
            if (gp > 0) mbar_wait(pvfull, (gp - 1) & 1);
            if (gs > gp) mbar_wait(sfull0 + 8 * ((gs - 1) & 1), ((gs - 1) >> 1) & 1);
        }
    } else {
        // ---- softmax and output: warp w holds TMEM lanes 32*(w%4).., key half (w-2)/4 ----
        pdl_wait();  // out and lse only after the previous kernel on the stream has finished
        const int q = warp & 3, ew = warp - 2, half = ew >> 2;
        const int r = 32 * q + lane;  // query row within the block = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t tS0 = tmem_base + lane_addr + 64u * half;  // + 128 for the odd blocks' S
        const uint32_t tO0 = tmem_base + lane_addr + kAtOCol + 32u * half;  // + 64 for odd items' O
        uint8_t* prow = sP + half * (kAtPBytes / 2) + (r >> 3) * 1024 + (r & 7) * 128;
        // This warp's 32 x 32 output box (rows = its TMEM lanes, columns = its
        // half of the head), 64-byte rows with the 64-byte swizzle of the
        // output tensor map: 16-byte piece v of row i at piece v ^ ((i >> 1) & 3).
        uint8_t* obox = sOut + ew * kAtOutBoxBytes;
        uint8_t* orow = obox + lane * 64;
        const float NEG_INF = -INFINITY;
        const float sl2 = a.scale_log2;

        // The current item: m is its running max of the raw scores, l its
        // running sum (this half's keys). O accumulates in TMEM over the
        // item's blocks; when a block raises the max, the softmax warps scale
        // the accumulated O by alpha before the block's P.V adds to it. The
        // item whose last P.V is still in flight: pit, pm, pl; its output is
        // written during the next block.
        float m = NEG_INF, l = 0.f;
        bool pend = false;
        Item pit = {0, 0, 0, 0};
        float pm = 0.f, pl = 0.f;
        bool ok_local = true;  // every wait since the last exchange succeeded
        bool ok = true;

        // Wait until the P.V of block gprev has completed (O is final for it).
        auto wait_pv = [&](uint32_t gprev) -> bool {
            const bool got = __all_sync(0xffffffffu, ok_local && mbar_wait(pvfull, gprev & 1));
            if (got)
                tc_fence_after();
            else
                ok_local = false;
            return got;
        };
        // O / lt (lt: the row sum of both halves) into the warp's box, stored
        // by TMA; lse.
        auto finish = [&](const Item& e, uint32_t tO, float em, float lt) {
            uint32_t ov[32];
            tmem_ld32_async(tO, ov);
            tmem_wait_ld(ov);
            const float inv = 1.0f / lt;
            if (lane == 0) bulk_wait_read_all();  // the box's previous store has read it
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 4; ++v)
                *reinterpret_cast<uint4*>(orow + ((v ^ ((lane >> 1) & 3)) << 4)) = make_uint4(
                    pack_bf16x2(__uint_as_float(ov[8 * v]) * inv, __uint_as_float(ov[8 * v + 1]) * inv),
                    pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv, __uint_as_float(ov[8 * v + 3]) * inv),
                    pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv, __uint_as_float(ov[8 * v + 5]) * inv),
                    pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv, __uint_as_float(ov[8 * v + 7]) * inv));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // Rows past the sequence's end (t >= T) lie outside the map and are not written.
                tma_store_3d(&tmO, smem_u32(obox), e.h * kAtD + 32 * half, e.qb * kAtBM + 32 * q, e.b);
                bulk_commit();
            }
            const int qpos = e.qb * kAtBM + r;
            if (a.lse && half == 0 && qpos < a.T)
                a.lse[((size_t)e.b * a.H + e.h) * a.T + qpos] = (em * sl2 + lg2_hw(lt)) * 0.6931471805599453f;
        };

        Walker w;
        w.init(a);
        uint32_t g = 0;
        while (w.valid) {
            const Item it = w.it;
            const int j = w.j;
            const bool last = j == it.nkb - 1;
            const int qpos = it.qb * kAtBM + r;
            const int kbase = j * kAtBN + 64 * half;
            const uint32_t tS = tS0 + 128u * (g & 1);
            const uint32_t sb_buf = g & 1, su = g >> 1;  // S buffer and its use
            // Keys visible to this row: kpos < lim. Per 32-key chunk and warp:
            // no row sees it (skipped: not read, not exponentiated), every row
            // sees all of it (no mask), or the mask applies per key.
            const int lim = a.causal ? min(qpos + 1, a.T) : a.T;
            const int wmax = a.causal ? min(it.qb * kAtBM + 32 * q + 32, a.T) : a.T;  // largest lim of the warp
            const int wmin = a.causal ? min(it.qb * kAtBM + 32 * q + 1, a.T) : a.T;   // smallest
            const bool live0 = kbase < wmax, live1 = kbase + 32 < wmax;
            const bool mask0 = kbase + 32 > wmin, mask1 = kbase + 64 > wmin;

            // 1. the block's raw scores: both 32-key chunks of this half in one
            //    round trip to TMEM; the buffer is released right after
            uint32_t sa[32], sb[32];
            bool got = __all_sync(0xffffffffu, ok_local && !aborted() && mbar_wait(sfull0 + 8 * sb_buf, su & 1));
            if (warp == 2 && lane == 0 && j == 0) AT_STAMP(w.n, 4);
            if (got) {
                tc_fence_after();
                if (live0) tmem_ld32_async(tS, sa);
                if (live1) tmem_ld32_async(tS + 32, sb);
                if (live0) tmem_wait_ld(sa);
                if (live1) tmem_wait_ld(sb);
            } else {
                ok_local = false;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfree0 + 8 * sb_buf);
            const bool use0 = got && live0, use1 = got && live1;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (!use0 || (mask0 && kbase + c >= lim)) sa[c] = __float_as_uint(NEG_INF);
                if (!use1 || (mask1 && kbase + 32 + c >= lim)) sb[c] = __float_as_uint(NEG_INF);
            }

            // 2. row max (raw scores; scale > 0 commutes with the max) across
            //    the two halves; the pending item's row sums travel with it
            float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
            if (use0) {
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    mx[(c >> 1) & 1] = max3(mx[(c >> 1) & 1], __uint_as_float(sa[c]), __uint_as_float(sa[c + 1]));
            }
            if (use1) {
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    mx[2 + ((c >> 1) & 1)] =
                        max3(mx[2 + ((c >> 1) & 1)], __uint_as_float(sb[c]), __uint_as_float(sb[c + 1]));
            }
            const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const int par = g & 1;
            red_max[(par * 2 + half) * 128 + r] = mloc;
            red_sum[(par * 2 + half) * 128 + r] = pl;
            if (lane == 0) red_ok[par * 8 + ew] = ok_local ? 1 : 0;
            named_bar_sync(1 + q, 64);
            const float mo = red_max[(par * 2 + (half ^ 1)) * 128 + r];
            const float plt = pl + red_sum[(par * 2 + (half ^ 1)) * 128 + r];
            if (!(red_ok[par * 8 + ew] && red_ok[par * 8 + (ew ^ 4)])) {
                ok = false;
                break;
            }
            const float m_new = fmaxf(m, fmaxf(mloc, mo));
            const float m_use = m_new == NEG_INF ? 0.f : m_new;  // a row with no visible key so far
            const float alpha = ex2_hw((m - m_use) * sl2);      // 0 at the first block (m = -inf)
            const float mb = m_use * sl2;
            m = m_new;

            // 3. p = 2^(s * scale * log2 e - max), rounded to bf16 for P.V
            uint32_t pk[32];
            uint64_t ls2[2] = {0ull, 0ull};  // packed partial row sums (+0.0f pairs)
            const uint64_t sl2x2 = f2_pack(sl2, sl2), nmbx2 = f2_pack(-mb, -mb);
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t* sv = ch == 0 ? sa : sb;
                if (ch == 0 ? use0 : use1) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nmbx2), x0,
                                  x1);
                        const float p0 = ex2_hw(x0), p1 = ex2_hw(x1);
                        ls2[(c >> 1) & 1] = f2_add(ls2[(c >> 1) & 1], f2_pack(p0, p1));
                        pk[16 * ch + (c >> 1)] = pack_bf16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[16 * ch + c] = 0u;
                }
            }
            float la, lb, lc, ld;
            f2_unpack(ls2[0], la, lb);
            f2_unpack(ls2[1], lc, ld);
            l = fmaf(l, alpha, (la + lb) + (lc + ld));

            // 4. the previous block's P.V has completed: the P buffer is free,
            //    and a later block of the item rescales the item's O by alpha
            //    (before this block's P.V adds to it)
            bool fin = false;
            if (j > 0) {
                const uint32_t tO = tO0 + 64u * (w.n & 1);
                if (wait_pv(g - 1) && __any_sync(0xffffffffu, alpha != 1.0f)) {
                    uint32_t ov[32];
                    tmem_ld32_async(tO, ov);
                    tmem_wait_ld(ov);
#pragma unroll
                    for (int d = 0; d < 32; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
                    tmem_st32(tO, ov);
                    tmem_wait_st();
                }
            } else if (pend) {
                fin = wait_pv(g - 1);
                pend = false;
            }

            // 5. P into shared memory: row r's 64 keys of this half as one
            //    128-byte row of a K-major block, 16-byte pieces swizzled by r % 8
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<uint4*>(prow + ((i ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull);
            if (warp == 2 && lane == 0 && last) AT_STAMP(w.n, 5);

            // 6. the previous item's output: its O is final and sits in the other
            //    O buffer, which only the next item's first P.V overwrites, after
            //    every warp has released that item's P (so after this load)
            if (fin) {
                if (warp == 2 && lane == 0) AT_STAMP(w.n - 1, 7);
                finish(pit, tO0 + 64u * ((w.n - 1) & 1), pm, plt);
                if (warp == 2 && lane == 0) AT_STAMP(w.n - 1, 8);
                if (warp == 9 && lane == 0) AT_STAMP(w.n - 1, 9);
            }
            pl = j == 0 ? 0.f : pl;

            if (last) {
                pend = true;
                pit = it;
                pm = m;
                pl = l;
                m = NEG_INF;
                l = 0.f;
            }
            w.next(a);
            ++g;
        }
        if (ok && pend) {
            // The last item: its P.V, then the row sums across the halves.
            const bool got = wait_pv(g - 1);
            if (warp == 2 && lane == 0) AT_STAMP(w.n - 1, 7);
            const int par = g & 1;
            red_sum[(par * 2 + half) * 128 + r] = pl;
            if (lane == 0) red_ok[par * 8 + ew] = ok_local ? 1 : 0;
            named_bar_sync(1 + q, 64);
            const float plt = pl + red_sum[(par * 2 + (half ^ 1)) * 128 + r];
            if (got && red_ok[par * 8 + ew] && red_ok[par * 8 + (ew ^ 4)])
                finish(pit, tO0 + 64u * ((w.n - 1) & 1), pm, plt);
            else
                ok = false;
            if (warp == 2 && lane == 0) AT_STAMP(w.n - 1, 8);
            if (warp == 9 && lane == 0) AT_STAMP(w.n - 1, 9);
        }
        if (!ok || !ok_local) give_up();
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
    if (cudaLaunchKernelEx(&cfg, attn_fwd_kernel, tqk, tv, to, a) != cudaSuccess) return LIN_ERR_CUDA;
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
