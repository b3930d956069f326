// C ABI of the linear-layer library: context, argument validation, the
// per-shape dispatch table and the launches. No host fallback exists: when a
// kernel cannot run, the call returns an error.
//
// Dispatch ("Optimizing a GPT-2-class transformer on a GPU", Act II: route each
// shape to its measured winner; "Writing a CUDA matmul that catches cuBLAS",
// "One kernel was never going to be enough": tile and split chosen per shape):
//   BF16, M <= 16        -> skinny W stream (HBM-bound), split-K inside a
//                           thread-block cluster, reduced through DSMEM
//   BF16, M > 16 ; TF32  -> tcgen05 kernel, N tile chosen for wave efficiency
//   FP32                 -> FFMA kernel; 64x64 tiles + split-K when 128x128
//                           tiles cannot fill the SMs
//   K == 0               -> fill Y = act(bias)
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>
#include <new>

#include "internal.h"
#include "device_common.cuh"

// A measured winner installed for one exact call signature.
struct lin_override {
    int M, N, K, precision, epilogue;
    lin_plan plan;
};

struct lin_ctx {
    int device;
    int sm_count;
    void* workspace;
    size_t workspace_bytes;
    int* dev_status;
    int early_level;   // LIN_OPT_EARLY_START: 0 none, 1 W and bias, 2 also X
    bool programmatic; // LIN_OPT_PROGRAMMATIC_LAUNCH
    bool adaptive;     // LIN_OPT_ADAPTIVE_PLANS
    lin_plan last_plan;
    std::mutex override_mu;
    std::vector<lin_override> overrides;  // consulted by lin_forward before the table
};

namespace lin {
namespace {

template <bool BF16, bool GELU>
__global__ void fill_kernel(int M, int N, const float* bias, const void* R, void* Y) {
    const size_t total = (size_t)M * N;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(i % N);
        const float v = epilogue<GELU>(0.f, bias ? bias[n] : 0.f);
        if constexpr (BF16)
            static_cast<uint16_t*>(Y)[i] =
                f32_to_bf16_bits(v + (R ? bf16_bits_to_f32(static_cast<const uint16_t*>(R)[i]) : 0.f));
        else
            static_cast<float*>(Y)[i] = v + (R ? static_cast<const float*>(R)[i] : 0.f);
    }
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

void plan_common(lin_plan* p, int kernel, int variant) {
    std::memset(p, 0, sizeof(*p));
    p->kernel = kernel;
    p->variant = variant;
    p->splits = 1;
}

int make_skinny(int sm, int variant, int splits, int M, int N, int K, size_t /*ws*/, lin_plan* p) {
    if (variant < 0 || variant >= kSkinnyVariants || M > 16 || M < 1 || N < 1 || K < 1) return LIN_ERR_UNSUPPORTED;
    const SkinnyCfg c = kSkinnyCfg[variant];
    const int tiles = ceil_div(N, 128);
    const int kblocks = ceil_div(K, 64 * c.kbox);
    int S = splits;
    if (S <= 0) {
        // Cluster split-K: the largest power of two (<= 8, the portable cluster
        // size) keeping the grid within the CTAs the SMs hold at once (one per SM,
        // two for the small ring), with >= 2 K stages per CTA.
        const long long slots = variant == kSkinnyTwoPerSm ? 2LL * sm : (long long)sm;
        S = 1;
        while (S < 8 && (long long)tiles * S * 2 <= slots && 2 * S <= kblocks) S *= 2;
    }
    if (S != 1 && S != 2 && S != 4 && S != 8) return LIN_ERR_UNSUPPORTED;
    plan_common(p, LIN_KERNEL_SKINNY, variant);
    p->bm = 16;
    p->bn = 128;
    p->bk = 64 * c.kbox;
    p->splits = S;
    p->stages = c.stages;
    p->grid_x = tiles;
    p->grid_y = S;
    p->grid_z = 1;
    p->threads = kSkinnyThreads;
    p->workspace_bytes = 0;
    return LIN_OK;
}

// `min_steps`: the fewest K steps of 32 a split keeps (4 for a call that runs
// alone; a call that overlaps an independent predecessor passes more, see run()).
int make_ffma(int sm, int variant, int splits, int M, int N, int K, size_t ws, lin_plan* p, int min_steps = 4) {
    if (M < 1 || N < 1 || K < 1) return LIN_ERR_UNSUPPORTED;
    if (variant < 0) {
        // 128x128 tiles when they give at least one full wave, else 64x64 + split-K.
        // The 128x128 tiles take K in steps of 64 over 3 stages (variant 2):
        // half the barriers of steps of 32 (4096^3: 50.2 -> 53.2 TF/s).
        const long long big = (long long)ceil_div(M, kFfmaCfg[0].bm) * ceil_div(N, kFfmaCfg[0].bn);
        variant = big >= sm ? 2 : 1;
    }
    if (variant >= kFfmaVariants) return LIN_ERR_UNSUPPORTED;
    const FfmaCfg c = kFfmaCfg[variant];
    const int gx = ceil_div(N, c.bn), gy = ceil_div(M, c.bm);
    const int tiles = gx * gy;
    const int nkb = ceil_div(K, c.bk);
    int S = splits;
    if (S <= 0) {
        // Fill the resident slots (one 128x128 CTA per SM, two 64x64 CTAs per
        // SM) without starting a second wave, keeping >= 4 K steps per split
        // (measured on the GPT-2 M = 128 shapes: qkv 22 -> 17 us, fc1 29 -> 23 us
        // against rounding the split up to one CTA per SM).
        const int slots = (variant == 1 || variant == 3) ? 2 * sm : sm;  // resident CTAs
        S = tiles >= slots ? 1 : slots / tiles;
        // A short reduction is not split (256^3, 8 steps: 9.8 us whole against
        // 12.1 us in two halves, measured as isolated calls).
        const int max_s = nkb >= 16 && nkb / min_steps > 1 ? nkb / min_steps : 1;
        if (S > max_s) S = max_s;
        if (S < 1) S = 1;
        while (S > 1 && splitk_workspace_bytes(S, M, N) > ws) --S;
    }
    if (S > nkb) S = nkb;
    if (tiles > kMaxSplitTiles) S = 1;
    plan_common(p, LIN_KERNEL_FFMA, variant);
    p->bm = c.bm;
    p->bn = c.bn;
    p->bk = c.bk;
    p->splits = S;
    p->grid_x = gx;
    p->grid_y = gy;
    p->grid_z = S;
    p->threads = 256;
    p->workspace_bytes = (long long)splitk_workspace_bytes(S, M, N);
    return LIN_OK;
}

// GEMV (FP32 / TF32 M <= 8, BF16 M <= 4): X padded to 1, 2, 4 or 8 rows in shared memory;
// `width` CTAs of 8 warps (0 = as many as fit on the SMs at once, by shared
// memory and by threads) take the rows of W in turn.
int gemv_rows(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }
bool gemv_fits(int M, int K, bool bf16) {
    return M >= 1 && M <= (bf16 ? kGemvMaxRowsBf16 : kGemvMaxRows) && K % (bf16 ? 8 : 4) == 0 &&
           (size_t)gemv_rows(M) * K * sizeof(float) <= (size_t)kGemvMaxSmem;
}
int make_gemv(int sm, int width, int M, int N, int K, bool bf16, lin_plan* p) {
    if (N < 1 || K < 1 || !gemv_fits(M, K, bf16)) return LIN_ERR_UNSUPPORTED;
    const int rows = gemv_rows(M);
    const long long smem = (long long)rows * K * 4 + 1024;
    long long per_sm = (228 * 1024) / smem;
    if (per_sm > 8) per_sm = 8;  // 2048 threads per SM
    if (per_sm < 1) per_sm = 1;
    long long grid = width > 0 ? width : (long long)sm * per_sm;
    const long long need = ((long long)N + 7) / 8;  // one row per warp and pass
    if (grid > need) grid = need;
    plan_common(p, LIN_KERNEL_GEMV, 0);
    p->bm = rows;
    p->bn = 8;
    p->bk = 0;
    p->splits = 1;
    p->stages = 0;
    p->grid_x = (int)grid;
    p->grid_y = 1;
    p->grid_z = 1;
    p->threads = 256;
    p->workspace_bytes = 0;
    return LIN_OK;
}

// Persistent tcgen05 kernel: `width` CTAs walk the 128 x BN output tiles
// (0 = one CTA per SM) in static round robin; pair variants walk 256 x BN
// tiles with one 2-CTA cluster (an SM pair) per tile (grid rounded down to
// even). `stream_k` (single-CTA variants, at least one tile per CTA): every CTA
// takes an equal share of the (tile, K stage) sequence instead (splits = 2).
// Default, from the measured M = 8192 GPT-2 shapes, the LM head and
// 4096^3 / 8192^3:
// * SM pair when each tile runs at least 64 K stages (K >= 4096 bf16 or 2048
//   tf32): there the pair's lighter shared-memory traffic wins (8192^3 bf16
//   1.91 vs 1.62 PF/s); with shorter K its per-tile synchronisation costs
//   more than it saves.
// * Otherwise whole single-CTA tiles, the N tile minimising rounds_eff(BN) x
//   r(BN), where rounds_eff is the mean of the average and the maximum tiles
//   per CTA (a back-to-back caller overlaps part of a ragged last round with
//   its next call) and r = 1, 0.9, 0.75 for BN = 256, 192, 128 is the measured
//   time of one round relative to BN = 256 (A is reloaded for every N tile, so
//   narrow tiles are slower per column).
// * Never stream-K by default: on the M = 8192 GPT-2 shapes it measured slower
//   than whole tiles both back to back (where the SMs that a ragged last round
//   frees start the next call early) and with the early start off (the cut
//   tiles' hand-over sits on the critical path). Explicit plans reach it.
int make_tc(int sm, int variant, int width, bool stream_k, int M, int N, int K, int esz, lin_plan* p,
            size_t ksplit_ws = 0) {
    if (M < 1 || N < 1 || K < 1 || width < 0) return LIN_ERR_UNSUPPORTED;
    const long long w0 = width > 0 ? width : sm;
    if (variant < 0) {
        // SM pairs for long K, unless the single-CTA tiles are so few that a K
        // split (below) is what fills the SMs.
        const long long tiles256 = (long long)ceil_div(M, 128) * ceil_div(N, 256);
        const bool want_pair = ceil_div(K, 128 / esz) >= 64 && !(ksplit_ws > 0 && tiles256 * 2 <= sm);
        double best = 0.0;
        for (int v = 0; v < kTcVariants; ++v) {
            if (kTcCfg[v].pair != want_pair) continue;
            const int bn = kTcCfg[v].bn;
            const long long items =
                (long long)(want_pair ? ceil_div(ceil_div(M, 128), 2) : ceil_div(M, 128)) * ceil_div(N, bn);
            long long slots = w0;
            if (want_pair) slots = slots / 2 > 0 ? slots / 2 : 1;
            const double avg = (double)items / (double)slots;
            const double mx = (double)((items + slots - 1) / slots);
            const double rel = bn == 256 ? 1.0 : bn == 192 ? 0.9 : 0.75;
            const double cost = 0.5 * (avg + mx) * rel;
            if (variant < 0 || cost < best) {
                best = cost;
                variant = v;
            }
        }
    }
    if (variant >= kTcVariants) return LIN_ERR_UNSUPPORTED;
    const bool pair = kTcCfg[variant].pair;
    const long long items = (long long)(pair ? ceil_div(ceil_div(M, 128), 2) : ceil_div(M, 128)) *
                            ceil_div(N, kTcCfg[variant].bn);
    long long w = w0;
    if (pair) {
        if (stream_k) return LIN_ERR_UNSUPPORTED;
        w = (w / 2 < items ? w / 2 : items) * 2;
        if (w < 2) w = 2;
    } else if (w > items) {
        w = items;
    }
    if (stream_k && (items < w || w > kTcMaxStreamKCtas)) return LIN_ERR_UNSUPPORTED;
    plan_common(p, LIN_KERNEL_TC, variant);
    p->bm = 128;
    p->bn = kTcCfg[variant].bn;
    p->bk = 0;  // 128 bytes of K: 64 bf16 or 32 fp32
    p->splits = stream_k ? 2 : 1;
    p->stages = 0;  // derived in the kernel from the shared-memory budget
    p->grid_x = (int)w;
    p->grid_y = 1;
    p->grid_z = 1;
    p->threads = kTcThreads;
    p->workspace_bytes = stream_k ? (long long)tc_streamk_workspace_bytes((int)w, p->bn) : 0;
    // Few tiles with a long K (and room in the workspace): split K so that
    // the (tile, split) items fill the SMs; grid_z = splits.
    if (!pair && !stream_k && ksplit_ws > 0) {
        const int S = tc_ksplits(items, ceil_div(K, 128 / esz), sm, ksplit_ws, p->bn);
        if (S > 1) {
            const long long w2 = width > 0 ? width : sm;
            p->grid_z = S;
            p->grid_x = (int)(items * S < w2 ? items * S : w2);
            p->workspace_bytes = (long long)tc_ksplit_workspace_bytes(items, S, p->bn);
        }
        // A ragged last round (more tiles than CTAs) is not split by default:
        // measured on GB300 as isolated calls, splitting the last round's tiles
        // in K was slower than running them whole (8192 x 768 x 768: 20.7 against
        // 13.8 us; 8192 x 3072 x 768 with GELU: 43.0 against 36.3 us; 8192 x 768 x
        // 3072: 37.6 against 36.5 us): the split pieces' partial sums pass through
        // the L2 and the last piece's reduction sits on the critical path.
        // Explicit plans (grid_z > 1 with more tiles than CTAs) still run it.
    }
    return LIN_OK;
}

bool valid_enums(int epilogue, int precision) {
    return (epilogue == LIN_EPI_NONE || epilogue == LIN_EPI_GELU_TANH) &&
           (precision == LIN_PREC_FP32 || precision == LIN_PREC_TF32 || precision == LIN_PREC_BF16);
}

int plan_default(int sm, int M, int N, int K, int precision, size_t ws, lin_plan* p) {
    if (M == 0 || N == 0) {
        plan_common(p, LIN_KERNEL_NONE, 0);
        return LIN_OK;
    }
    if (K == 0) {
        plan_common(p, LIN_KERNEL_FILL, 0);
        p->grid_x = ceil_div((long long)M * N, 256) < 4 * sm ? ceil_div((long long)M * N, 256) : 4 * sm;
        p->grid_y = p->grid_z = 1;
        p->threads = 256;
        return LIN_OK;
    }
    switch (precision) {
        case LIN_PREC_BF16:
            // The GEMV only for one row and at most one 128-row tile of W per
            // SM; measured back to back, the skinny tensor-core kernel wins
            // everywhere else (4 x 50257 x 768: 12.1 against 41.5 us; one row
            // of 50257: 11.9 against 14.3 us; one row of 2304: 1.9 against 1.3 us).
            if (M == 1 && ceil_div(N, 128) <= sm && gemv_fits(M, K, true)) return make_gemv(sm, 0, M, N, K, true, p);
            // More row tiles than SMs: the 6 x 1 ring (two CTAs per SM) without a
            // split, so the tiles run in fewer waves (measured on the last
            // token's logits, 50257 rows: 15.7 -> 12.1 us). Otherwise the 5 x 1
            // ring split over a cluster (two CTAs per SM): the next call's CTAs
            // start beside this call's and stream their W into L2 meanwhile.
            if (M <= 16) return make_skinny(sm, ceil_div(N, 128) > sm ? 1 : kSkinnyTwoPerSm, 0, M, N, K, ws, p);
            return make_tc(sm, -1, 0, false, M, N, K, 2, p, ws);
        case LIN_PREC_TF32:
            // A few rows are a weight stream: the exact-fp32 GEMV is as fast as
            // any tensor-core tile there, and more accurate than TF32.
            if (gemv_fits(M, K, false)) return make_gemv(sm, 0, M, N, K, false, p);
            return make_tc(sm, -1, 0, false, M, N, K, 4, p, ws);
        default:
            if (gemv_fits(M, K, false)) return make_gemv(sm, 0, M, N, K, false, p);
            return make_ffma(sm, -1, 0, M, N, K, ws, p);
    }
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + bn && pb < pa + an;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Output range of the last launch on each stream (process-wide): a kernel
// that starts before its predecessor finishes may prefetch W only when W does
// not overlap what that predecessor writes.
struct LastOut {
    cudaStream_t stream;
    uintptr_t lo, hi;
};
std::mutex g_last_mu;
LastOut g_last[64];
int g_last_n = 0;

struct Range {
    const void* p;
    size_t bytes;
};

// Which inputs may be read before the dependency wait: *w_ok for W and bias,
// *x_ok for X (each false when it overlaps the previous output on `st`).
// Records Y as this stream's newest output.
void early_reads_ok(cudaStream_t st, Range w, Range bias, Range x, Range y, bool* w_ok, bool* x_ok, bool* known) {
    auto hits = [](const LastOut& o, Range r) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(r.p), hi = lo + r.bytes;
        return r.p && r.bytes && lo < o.hi && o.lo < hi;
    };
    std::lock_guard<std::mutex> lk(g_last_mu);
    *w_ok = *x_ok = true;
    *known = false;
    int slot = -1;
    for (int i = 0; i < g_last_n; ++i)
        if (g_last[i].stream == st) {
            *w_ok = !hits(g_last[i], w) && !hits(g_last[i], bias);
            *x_ok = !hits(g_last[i], x);
            *known = true;
            slot = i;
            break;
        }
    if (slot < 0) {
        if (g_last_n < 64) {
            slot = g_last_n++;
        } else {
            slot = 0;  // table full: forget the oldest entry's stream, stay safe for this one
            *w_ok = *x_ok = false;
        }
    }
    g_last[slot].stream = st;
    g_last[slot].lo = reinterpret_cast<uintptr_t>(y.p);
    g_last[slot].hi = g_last[slot].lo + y.bytes;
}

// Record `y` as the last output on stream `st` (for a call whose last kernel
// writes a different range than its main output).
void note_output(cudaStream_t st, Range y) {
    std::lock_guard<std::mutex> lk(g_last_mu);
    for (int i = 0; i < g_last_n; ++i)
        if (g_last[i].stream == st) {
            g_last[i].lo = reinterpret_cast<uintptr_t>(y.p);
            g_last[i].hi = g_last[i].lo + y.bytes;
            return;
        }
}

int check_plan_fits(const lin_plan& p, int M, int N, int K, int precision) {
    switch (p.kernel) {
        case LIN_KERNEL_NONE: return (M == 0 || N == 0) ? LIN_OK : LIN_ERR_UNSUPPORTED;
        case LIN_KERNEL_FILL: return (K == 0 && p.grid_x > 0) ? LIN_OK : LIN_ERR_UNSUPPORTED;
        case LIN_KERNEL_SKINNY: {
            if (precision != LIN_PREC_BF16 || M > 16 || K == 0) return LIN_ERR_UNSUPPORTED;
            if (p.variant < 0 || p.variant >= kSkinnyVariants) return LIN_ERR_UNSUPPORTED;
            if (p.splits != 1 && p.splits != 2 && p.splits != 4 && p.splits != 8) return LIN_ERR_UNSUPPORTED;
            if (p.grid_x != ceil_div(N, 128) || p.grid_y != p.splits) return LIN_ERR_UNSUPPORTED;
            return LIN_OK;
        }
        case LIN_KERNEL_FFMA: {
            if (precision != LIN_PREC_FP32 || K == 0) return LIN_ERR_UNSUPPORTED;
            if (p.variant < 0 || p.variant >= kFfmaVariants || p.splits < 1) return LIN_ERR_UNSUPPORTED;
            const FfmaCfg c = kFfmaCfg[p.variant];
            if (p.bk != c.bk || p.grid_x != ceil_div(N, c.bn) || p.grid_y != ceil_div(M, c.bm) ||
                p.grid_z != p.splits || p.splits > ceil_div(K, c.bk) ||
                (p.splits > 1 && (long long)p.grid_x * p.grid_y > kMaxSplitTiles))
                return LIN_ERR_UNSUPPORTED;
            return LIN_OK;
        }
        case LIN_KERNEL_TC: {
            if (precision == LIN_PREC_FP32 || K == 0) return LIN_ERR_UNSUPPORTED;
            if (p.variant < 0 || p.variant >= kTcVariants || (p.splits != 1 && p.splits != 2))
                return LIN_ERR_UNSUPPORTED;
            const bool pair = kTcCfg[p.variant].pair;
            const long long items = (long long)(pair ? ceil_div(ceil_div(M, 128), 2) : ceil_div(M, 128)) *
                                    ceil_div(N, kTcCfg[p.variant].bn);
            const long long ctas = pair ? 2 * items : items * (p.grid_z > 1 ? p.grid_z : 1);
            if (p.bn != kTcCfg[p.variant].bn || p.grid_x < 1 || p.grid_x > ctas || p.grid_y != 1 ||
                (pair && p.grid_x % 2 != 0))
                return LIN_ERR_UNSUPPORTED;
            if (p.splits == 2 &&
                (pair || p.grid_x > kTcMaxStreamKCtas ||
                 p.workspace_bytes < (long long)tc_streamk_workspace_bytes(p.grid_x, p.bn)))
                return LIN_ERR_UNSUPPORTED;
            if (p.grid_z > 1) {  // K split (of every tile, or of the tiles past the whole rounds)
                const long long tiles = (long long)ceil_div(M, 128) * ceil_div(N, p.bn);
                const long long split_tiles = tiles - tc_tail_whole(tiles, p.grid_x);
                if (pair || p.splits != 1 || p.grid_z > 16 || split_tiles < 1 || split_tiles > kTcMaxKSplitTiles ||
                    ceil_div(K, precision == LIN_PREC_BF16 ? 64 : 32) < p.grid_z ||
                    p.workspace_bytes < (long long)tc_ksplit_workspace_bytes(split_tiles, p.grid_z, p.bn))
                    return LIN_ERR_UNSUPPORTED;
            } else if (p.grid_z != 1) {
                return LIN_ERR_UNSUPPORTED;
            }
            return LIN_OK;
        }
        case LIN_KERNEL_GEMV: {
            if (K == 0 || !gemv_fits(M, K, precision == LIN_PREC_BF16)) return LIN_ERR_UNSUPPORTED;
            if (p.bm != gemv_rows(M) || p.grid_x < 1 || p.grid_y != 1 || p.grid_z != 1) return LIN_ERR_UNSUPPORTED;
            return LIN_OK;
        }
        default: return LIN_ERR_UNSUPPORTED;
    }
}

int run(lin_ctx* ctx, const lin_plan& plan_in, int M, int N, int K, const void* X, const void* W, const float* bias,
        void* Y, int epilogue, int precision, void* stream, bool adaptive, const void* R = nullptr) {
    lin_plan plan = plan_in;
    if (!ctx || M < 0 || N < 0 || K < 0 || !valid_enums(epilogue, precision)) return LIN_ERR_ARG;
    if (M == 0 || N == 0) return plan.kernel == LIN_KERNEL_NONE ? LIN_OK : LIN_ERR_UNSUPPORTED;
    if (!Y || (K > 0 && (!X || !W))) return LIN_ERR_ARG;
    const size_t ein = precision == LIN_PREC_BF16 ? 2 : 4;
    const size_t eout = ein;
    const size_t ybytes = (size_t)M * N * eout;
    if (overlaps(Y, ybytes, X, (size_t)M * K * ein) || overlaps(Y, ybytes, W, (size_t)N * K * ein) ||
        overlaps(Y, ybytes, bias, bias ? (size_t)N * 4 : 0))
        return LIN_ERR_ARG;
    if (R && R != Y && overlaps(Y, ybytes, R, ybytes)) return LIN_ERR_ARG;  // in place, or apart
    if (K > 0 && (((uintptr_t)X | (uintptr_t)W) % 16 != 0 || ((size_t)K * ein) % 16 != 0)) return LIN_ERR_ALIGN;
    if ((((uintptr_t)Y | (uintptr_t)R) % eout) != 0 || ((uintptr_t)bias % 4) != 0) return LIN_ERR_ALIGN;
    const int fit = check_plan_fits(plan, M, N, K, precision);
    if (fit != LIN_OK) return fit;
    if ((size_t)plan.workspace_bytes > ctx->workspace_bytes) return LIN_ERR_WORKSPACE;

    DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    Problem p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.X = X;
    p.W = W;
    p.bias = bias;
    p.Y = Y;
    p.residual = R;
    p.epilogue = epilogue;
    p.precision = precision;
    p.stream = static_cast<cudaStream_t>(stream);
    p.workspace = ctx->workspace;
    p.workspace_bytes = ctx->workspace_bytes;
    p.dev_status = ctx->dev_status;
    p.sm_count = ctx->sm_count;
    bool w_ok = false, x_ok = false, known = false;
    early_reads_ok(p.stream, Range{W, (size_t)N * K * ein}, Range{bias, bias ? (size_t)N * 4 : 0},
                   Range{X, (size_t)M * K * ein}, Range{Y, ybytes}, &w_ok, &x_ok, &known);
    p.early_start = ctx->programmatic;
    p.early_w = p.early_start && ctx->early_level >= 1 && w_ok;
    p.early_x = p.early_w && ctx->early_level >= 2 && x_ok;
    // An independent call right after another call on this stream overlaps it:
    // the skinny stream then needs no K split to fill the SMs (the concurrent
    // calls do), and skipping the split saves its reduction.
    // The two-per-SM ring keeps its variant (the same summation order, so the
    // same bits) and takes the split that leaves one CTA slot per SM to the
    // neighbouring call (measured on 16 x 4096 x 4096: cluster 4 5.4 us per
    // call back to back against 7.2 us for cluster 8); the deep rings drop the
    // split altogether.
    if (adaptive && ctx->adaptive && known && p.early_x && plan.kernel == LIN_KERNEL_SKINNY && plan.splits > 1) {
        lin_plan narrow;
        int S = 1;
        if (plan.variant == kSkinnyTwoPerSm) {
            const long long tiles = ceil_div(N, 128), kblocks = ceil_div(K, 64);
            while (S < 8 && tiles * S * 2 <= ctx->sm_count && 2 * S <= kblocks) S *= 2;
        }
        if (S < plan.splits && make_skinny(ctx->sm_count, plan.variant, S, M, N, K, ctx->workspace_bytes, &narrow) == LIN_OK)
            plan = narrow;
    }
    // Likewise a tensor-core K split (measured: it helps an isolated call and
    // costs a back-to-back one).
    if (adaptive && ctx->adaptive && known && p.early_x && plan.kernel == LIN_KERNEL_TC && plan.grid_z > 1) {
        lin_plan whole;
        if (make_tc(ctx->sm_count, -1, 0, false, M, N, K, precision == LIN_PREC_BF16 ? 2 : 4, &whole) == LIN_OK)
            plan = whole;
    }
    // And the FFMA split: back to back, the next call's CTAs fill the SMs that
    // a split would, so a split must now pay for its reduction with a long K
    // (>= 24 steps of 32 each; measured on the GPT-2 M = 128 layers: proj
    // 8.6 -> 4.1 us, qkv 14.7 -> 11.9 us, fc2 keeps a split of 4).
    // Without a split, wide outputs of a few rows take 128 x 64 tiles (two CTAs
    // per SM; measured back to back at M = 128, K = 768: N = 2304 10.5 -> 9.4 us,
    // N = 3072 14.3 -> 13.4 us; N = 768 unchanged).
    if (adaptive && ctx->adaptive && known && p.early_x && plan.kernel == LIN_KERNEL_FFMA && plan.splits > 1) {
        lin_plan fewer;
        if (make_ffma(ctx->sm_count, -1, 0, M, N, K, ctx->workspace_bytes, &fewer, 24) == LIN_OK) {
            plan = fewer;
            lin_plan wide;
            if (plan.splits == 1 && plan.variant == 1 && M <= 128 && N >= 2048 &&
                make_ffma(ctx->sm_count, 3, 1, M, N, K, ctx->workspace_bytes, &wide) == LIN_OK)
                plan = wide;
        }
    }
    ctx->last_plan = plan;
    switch (plan.kernel) {
        case LIN_KERNEL_FILL: return launch_fill(p);
        case LIN_KERNEL_SKINNY: return launch_skinny(p, plan);
        case LIN_KERNEL_FFMA: return launch_ffma(p, plan);
        case LIN_KERNEL_TC: return launch_tc(p, plan);
        case LIN_KERNEL_GEMV: return launch_gemv(p, plan);
        default: return LIN_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_fill(const Problem& p) {
    const long long total = (long long)p.M * p.N;
    int grid = (int)((total + 255) / 256);
    if (grid > 4 * p.sm_count) grid = 4 * p.sm_count;
    if (grid < 1) grid = 1;
    const bool bf16 = p.precision == LIN_PREC_BF16, gelu = p.epilogue == LIN_EPI_GELU_TANH;
    const void* R = p.residual;
    if (bf16 && gelu) fill_kernel<true, true><<<grid, 256, 0, p.stream>>>(p.M, p.N, p.bias, R, p.Y);
    else if (bf16) fill_kernel<true, false><<<grid, 256, 0, p.stream>>>(p.M, p.N, p.bias, R, p.Y);
    else if (gelu) fill_kernel<false, true><<<grid, 256, 0, p.stream>>>(p.M, p.N, p.bias, R, p.Y);
    else fill_kernel<false, false><<<grid, 256, 0, p.stream>>>(p.M, p.N, p.bias, R, p.Y);
    return cudaGetLastError() == cudaSuccess ? LIN_OK : LIN_ERR_CUDA;
}

}  // namespace lin

extern "C" {

int lin_abi_version(void) { return LIN_ABI_VERSION; }

int lin_timeline(int kernel, void* host_dst, size_t bytes, int clear) {
    if ((host_dst == nullptr) != (bytes == 0)) return LIN_ERR_ARG;
    switch (kernel) {
        case LIN_KERNEL_TC: return lin::timeline_copy_tc(host_dst, bytes, clear != 0);
        case LIN_KERNEL_SKINNY: return lin::timeline_copy_skinny(host_dst, bytes, clear != 0);
        case LIN_TIMELINE_ATTENTION: return lin::timeline_copy_attn(host_dst, bytes, clear != 0);
        default: return LIN_ERR_ARG;
    }
}

const char* lin_strerror(int status) {
    switch (status) {
        case LIN_OK: return "success";
        case LIN_ERR_ARG: return "invalid argument (NULL pointer, negative size, unknown enum, or Y overlapping an input)";
        case LIN_ERR_ALIGN: return "misaligned operand (X and W need 16-byte alignment and K*element size a multiple of 16)";
        case LIN_ERR_WORKSPACE: return "plan needs more workspace than the context holds";
        case LIN_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
        case LIN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait; its output is incomplete";
        case LIN_ERR_UNSUPPORTED: return "the plan's kernel cannot run this shape or precision";
        default: return "unknown status";
    }
}

int lin_create(lin_ctx** out, int device, size_t max_workspace_bytes) {
    if (!out) return LIN_ERR_ARG;
    *out = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        cudaGetLastError();
        return LIN_ERR_CUDA;
    }
    lin::DeviceGuard guard(device);
    if (!guard.ok) return LIN_ERR_CUDA;
    lin_ctx* c = new (std::nothrow) lin_ctx();
    if (!c) return LIN_ERR_CUDA;
    c->device = device;
    c->early_level = 0;
    c->programmatic = true;
    c->adaptive = true;
    std::memset(&c->last_plan, 0, sizeof(c->last_plan));
    c->workspace_bytes = max_workspace_bytes ? max_workspace_bytes : ((size_t)64 << 20);
    if (cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaMalloc(&c->workspace, c->workspace_bytes) != cudaSuccess ||
        cudaMemset(c->workspace, 0, c->workspace_bytes) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&c->dev_status), sizeof(int)) != cudaSuccess ||
        cudaMemset(c->dev_status, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        if (c->workspace) cudaFree(c->workspace);
        if (c->dev_status) cudaFree(c->dev_status);
        delete c;
        cudaGetLastError();
        return LIN_ERR_CUDA;
    }
    *out = c;
    return LIN_OK;
}

int lin_destroy(lin_ctx* ctx) {
    if (!ctx) return LIN_OK;
    int rc = LIN_OK;
    {
        lin::DeviceGuard guard(ctx->device);
        if (cudaDeviceSynchronize() != cudaSuccess) rc = LIN_ERR_CUDA;
        cudaFree(ctx->workspace);
        cudaFree(ctx->dev_status);
    }
    delete ctx;
    return rc;
}

int lin_ctx_last_plan(const lin_ctx* ctx, lin_plan* out) {
    if (!ctx || !out) return LIN_ERR_ARG;
    *out = ctx->last_plan;
    return LIN_OK;
}

int lin_set_option(lin_ctx* ctx, int option, long long value) {
    if (!ctx) return LIN_ERR_ARG;
    switch (option) {
        case LIN_OPT_EARLY_START:
            if (value < 0 || value > 2) return LIN_ERR_ARG;
            ctx->early_level = (int)value;
            return LIN_OK;
        case LIN_OPT_ADAPTIVE_PLANS:
            if (value != 0 && value != 1) return LIN_ERR_ARG;
            ctx->adaptive = value != 0;
            return LIN_OK;
        case LIN_OPT_PROGRAMMATIC_LAUNCH:
            if (value != 0 && value != 1) return LIN_ERR_ARG;
            ctx->programmatic = value != 0;
            return LIN_OK;
        default: return LIN_ERR_ARG;
    }
}

int lin_ctx_info(const lin_ctx* ctx, int* device, int* sm_count, size_t* workspace_bytes) {
    if (!ctx) return LIN_ERR_ARG;
    if (device) *device = ctx->device;
    if (sm_count) *sm_count = ctx->sm_count;
    if (workspace_bytes) *workspace_bytes = ctx->workspace_bytes;
    return LIN_OK;
}

int lin_plan_query(int sm_count, int M, int N, int K, int precision, int epilogue, size_t workspace_bytes,
                   lin_plan* out) {
    if (!out || sm_count < 1 || M < 0 || N < 0 || K < 0 || !lin::valid_enums(epilogue, precision)) return LIN_ERR_ARG;
    return lin::plan_default(sm_count, M, N, K, precision, workspace_bytes, out);
}

int lin_plan_check(const lin_plan* plan, int M, int N, int K, int precision, size_t workspace_bytes) {
    if (!plan || M < 0 || N < 0 || K < 0 || !lin::valid_enums(0, precision)) return LIN_ERR_ARG;
    if (M == 0 || N == 0) return plan->kernel == LIN_KERNEL_NONE ? LIN_OK : LIN_ERR_UNSUPPORTED;
    const int fit = lin::check_plan_fits(*plan, M, N, K, precision);
    if (fit != LIN_OK) return fit;
    return (size_t)plan->workspace_bytes > workspace_bytes ? LIN_ERR_WORKSPACE : LIN_OK;
}

int lin_plan_make(int sm_count, int kernel, int variant, int splits, int M, int N, int K, int precision,
                  lin_plan* out) {
    if (!out || sm_count < 1 || M < 0 || N < 0 || K < 0 || !lin::valid_enums(0, precision)) return LIN_ERR_ARG;
    const size_t unlimited = (size_t)1 << 62;
    switch (kernel) {
        case LIN_KERNEL_SKINNY:
            if (precision != LIN_PREC_BF16) return LIN_ERR_UNSUPPORTED;
            return lin::make_skinny(sm_count, variant, splits, M, N, K, unlimited, out);
        case LIN_KERNEL_FFMA:
            if (precision != LIN_PREC_FP32) return LIN_ERR_UNSUPPORTED;
            return lin::make_ffma(sm_count, variant, splits, M, N, K, unlimited, out);
        case LIN_KERNEL_TC:
            if (precision == LIN_PREC_FP32) return LIN_ERR_UNSUPPORTED;
            // splits >= 0: CTAs walking whole tiles (0 = one per SM); -1: stream-K with
            // one CTA per SM; -c (c >= 2): stream-K with c CTAs.
            return lin::make_tc(sm_count, variant, splits >= 0 ? splits : (splits == -1 ? 0 : -splits), splits < 0,
                                M, N, K, precision == LIN_PREC_BF16 ? 2 : 4, out);
        case LIN_KERNEL_GEMV:  // splits = CTAs (0 = as many as fit)
            return lin::make_gemv(sm_count, splits > 0 ? splits : 0, M, N, K, precision == LIN_PREC_BF16, out);
        case LIN_KERNEL_NONE:
        case LIN_KERNEL_FILL:
            return lin::plan_default(sm_count, M, N, K, precision, unlimited, out);
        default: return LIN_ERR_ARG;
    }
}

namespace {

// lin_forward and lin_forward_residual: an installed plan for the call
// signature, else the built-in table (adapted to the call's neighbour).
int forward_dispatch(lin_ctx* ctx, int M, int N, int K, const void* X, const void* W, const float* bias,
                     const void* R, void* Y, int epilogue, int precision, void* stream) {
    if (!ctx || M < 0 || N < 0 || K < 0 || !lin::valid_enums(epilogue, precision)) return LIN_ERR_ARG;
    lin_plan plan;
    bool installed = false;
    {
        std::lock_guard<std::mutex> lk(ctx->override_mu);  // copy the entry; launch outside the lock
        for (const lin_override& o : ctx->overrides)
            if (o.M == M && o.N == N && o.K == K && o.precision == precision && o.epilogue == epilogue) {
                plan = o.plan;
                installed = true;
                break;
            }
    }
    if (installed) return lin::run(ctx, plan, M, N, K, X, W, bias, Y, epilogue, precision, stream, false, R);
    const int rc = lin::plan_default(ctx->sm_count, M, N, K, precision, ctx->workspace_bytes, &plan);
    if (rc != LIN_OK) return rc;
    return lin::run(ctx, plan, M, N, K, X, W, bias, Y, epilogue, precision, stream, true, R);
}

}  // namespace

int lin_forward(lin_ctx* ctx, int M, int N, int K, const void* X, const void* W, const float* bias, void* Y,
                int epilogue, int precision, void* stream) {
    return forward_dispatch(ctx, M, N, K, X, W, bias, nullptr, Y, epilogue, precision, stream);
}

int lin_forward_residual(lin_ctx* ctx, int M, int N, int K, const void* X, const void* W, const float* bias,
                         const void* R, void* Y, int epilogue, int precision, void* stream) {
    if (!R && M > 0 && N > 0) return LIN_ERR_ARG;
    return forward_dispatch(ctx, M, N, K, X, W, bias, R, Y, epilogue, precision, stream);
}

int lin_set_plan_override(lin_ctx* ctx, int M, int N, int K, int precision, int epilogue, const lin_plan* plan) {
    if (!ctx || M < 0 || N < 0 || K < 0 || !lin::valid_enums(epilogue, precision)) return LIN_ERR_ARG;
    if (plan) {  // a refused plan leaves the table as it was
        const int fit = lin::check_plan_fits(*plan, M, N, K, precision);
        if (fit != LIN_OK) return fit;
        if ((size_t)plan->workspace_bytes > ctx->workspace_bytes) return LIN_ERR_WORKSPACE;
    }
    std::lock_guard<std::mutex> lk(ctx->override_mu);
    auto& v = ctx->overrides;
    for (size_t i = 0; i < v.size(); ++i)
        if (v[i].M == M && v[i].N == N && v[i].K == K && v[i].precision == precision && v[i].epilogue == epilogue) {
            v.erase(v.begin() + (long)i);
            break;
        }
    if (plan) v.push_back(lin_override{M, N, K, precision, epilogue, *plan});
    return LIN_OK;
}

int lin_clear_plan_overrides(lin_ctx* ctx) {
    if (!ctx) return LIN_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->override_mu);
    ctx->overrides.clear();
    return LIN_OK;
}

namespace {

// Shared checks of the two backward GEMMs: returns LIN_OK and fills q, or an error.
int backward_setup(lin_ctx* ctx, int which, int M, int N, int K, const void* dZ, const void* B, void* out,
                   int precision, void* stream, lin::BwdProblem* q) {
    using namespace lin;
    if (!ctx || M < 0 || N < 0 || K < 0 || !valid_enums(0, precision)) return LIN_ERR_ARG;
    const size_t esz = precision == LIN_PREC_BF16 ? 2 : 4;
    const int Mo = which == 1 ? M : N;
    const size_t out_bytes = (size_t)Mo * K * esz;
    if (Mo == 0 || K == 0) return LIN_OK;
    if (!out || (M > 0 && N > 0 && (!dZ || !B))) return LIN_ERR_ARG;
    const size_t dz_bytes = (size_t)M * N * esz;
    const size_t b_bytes = (size_t)(which == 1 ? N : M) * K * esz;
    if (overlaps(out, out_bytes, dZ, dz_bytes) || overlaps(out, out_bytes, B, b_bytes)) return LIN_ERR_ARG;
    if ((((uintptr_t)dZ | (uintptr_t)B | (uintptr_t)out) % 16) != 0 || ((size_t)K * esz) % 16 != 0) return LIN_ERR_ALIGN;
    if (precision == LIN_PREC_BF16 && ((size_t)N * esz) % 16 != 0) return LIN_ERR_ALIGN;  // dZ rows by TMA
    q->which = which;
    q->M = M;
    q->N = N;
    q->K = K;
    q->dZ = dZ;
    q->B = B;
    q->out = out;
    q->stream = static_cast<cudaStream_t>(stream);
    q->dev_status = ctx->dev_status;
    q->sm_count = ctx->sm_count;
    bool w_ok = false, x_ok = false, known = false;
    early_reads_ok(q->stream, Range{B, b_bytes}, Range{nullptr, 0}, Range{dZ, dz_bytes}, Range{out, out_bytes}, &w_ok,
                   &x_ok, &known);
    q->early_start = ctx->programmatic;
    q->early_x = q->early_start && ctx->early_level >= 1 && w_ok && ctx->early_level >= 2 && x_ok;
    q->workspace = ctx->workspace;
    q->workspace_bytes = ctx->workspace_bytes;
    // Right after an independent call the two overlap (early start) and fill
    // the SMs together: a K split would only add its round trip.
    q->ksplit_ok = !(ctx->adaptive && known && q->early_x);
    q->aux = nullptr;
    return LIN_OK;
}

int backward_run(const lin::BwdProblem& q, int precision, lin_ctx* ctx) {
    using namespace lin;
    const int R = q.which == 1 ? q.N : q.M;
    const int Mo = q.which == 1 ? q.M : q.N;
    if (R == 0)
        return cudaMemsetAsync(q.out, 0, (size_t)Mo * q.K * (precision == LIN_PREC_BF16 ? 2 : 4), q.stream) == cudaSuccess
                   ? LIN_OK
                   : LIN_ERR_CUDA;
    if (precision == LIN_PREC_BF16) return launch_tc_backward(q);
    const int S = bwd_ffma_splits(q.which, q.M, q.N, q.K, ctx->sm_count, ctx->workspace_bytes);
    return launch_bwd_ffma(q.which, q.M, q.N, q.K, static_cast<const float*>(q.dZ), static_cast<const float*>(q.B),
                           static_cast<float*>(q.out), S, ctx->workspace, q.stream, q.early_start,
                           static_cast<const float*>(q.aux));
}

}  // namespace

int lin_backward_data(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* W, void* dX, int precision,
                      void* stream) {
    lin::BwdProblem q;
    q.which = 0;
    const int rc = backward_setup(ctx, 1, M, N, K, dZ, W, dX, precision, stream, &q);
    if (rc != LIN_OK || q.which == 0) return rc;
    lin::DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    return backward_run(q, precision, ctx);
}

int lin_backward_data_gelu(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* W, const void* Zp,
                           void* dX, int precision, void* stream) {
    lin::BwdProblem q;
    q.which = 0;
    if (!ctx || !lin::valid_enums(0, precision)) return LIN_ERR_ARG;
    const size_t esz = precision == LIN_PREC_BF16 ? 2 : 4;
    const size_t bytes = (size_t)(M > 0 ? M : 0) * (K > 0 ? K : 0) * esz;
    if (bytes > 0 && !Zp) return LIN_ERR_ARG;
    if (Zp != dX && lin::overlaps(Zp, bytes, dX, bytes)) return LIN_ERR_ARG;  // in place, or apart
    if ((uintptr_t)Zp % esz != 0) return LIN_ERR_ALIGN;
    const int rc = backward_setup(ctx, 1, M, N, K, dZ, W, dX, precision, stream, &q);
    if (rc != LIN_OK || q.which == 0) return rc;
    q.aux = Zp;
    lin::DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    return backward_run(q, precision, ctx);
}

int lin_backward_weight(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* X, void* dW, float* db,
                        int precision, void* stream) {
    using namespace lin;
    lin::BwdProblem q;
    q.which = 0;
    int rc = backward_setup(ctx, 2, M, N, K, dZ, X, dW, precision, stream, &q);
    if (rc != LIN_OK) return rc;
    if (db) {
        if ((uintptr_t)db % 4 != 0) return LIN_ERR_ALIGN;
        const size_t esz = precision == LIN_PREC_BF16 ? 2 : 4;
        if (overlaps(db, (size_t)N * 4, dZ, (size_t)M * N * esz) || overlaps(db, (size_t)N * 4, X, (size_t)M * K * esz) ||
            overlaps(db, (size_t)N * 4, dW, (size_t)N * K * esz))
            return LIN_ERR_ARG;
        if (M > 0 && N > 0 && colsum_workspace_bytes(M, N) > ctx->workspace_bytes) return LIN_ERR_WORKSPACE;
    }
    lin::DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    if (q.which != 0) {
        rc = backward_run(q, precision, ctx);
        if (rc != LIN_OK) return rc;
    }
    if (db && N > 0) {
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        rc = launch_colsum(M, N, dZ, db, precision == LIN_PREC_BF16, ctx->workspace, st);
        if (rc != LIN_OK) return rc;
        note_output(st, Range{db, (size_t)N * 4});
    }
    return LIN_OK;
}

int lin_gelu_backward(lin_ctx* ctx, long long count, const void* dY, const void* Z, void* dZ, int precision,
                      void* stream) {
    using namespace lin;
    if (!ctx || count < 0 || !valid_enums(0, precision)) return LIN_ERR_ARG;
    if (count == 0) return LIN_OK;
    if (!dY || !Z || !dZ) return LIN_ERR_ARG;
    const size_t esz = precision == LIN_PREC_BF16 ? 2 : 4;
    const size_t bytes = (size_t)count * esz;
    if (overlaps(dZ, bytes, Z, bytes)) return LIN_ERR_ARG;  // dZ may overwrite dY in place
    if ((((uintptr_t)dY | (uintptr_t)Z | (uintptr_t)dZ) % esz) != 0) return LIN_ERR_ALIGN;
    DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool w_ok = false, x_ok = false, known = false;
    early_reads_ok(st, Range{Z, bytes}, Range{nullptr, 0}, Range{dY, bytes}, Range{dZ, bytes}, &w_ok, &x_ok, &known);
    return launch_gelu_backward(count, dY, Z, dZ, precision == LIN_PREC_BF16, ctx->sm_count, st,
                                ctx->programmatic);
}

int lin_fold_layernorm(lin_ctx* ctx, int N, int K, const float* W, const float* bias, const float* gamma,
                       const float* beta, void* W_out, float* bias_out, int precision, void* stream) {
    using namespace lin;
    if (!ctx || N < 0 || K < 0 || !valid_enums(0, precision)) return LIN_ERR_ARG;
    if (N == 0) return LIN_OK;
    if (!W_out || !bias_out || (K > 0 && (!W || !gamma))) return LIN_ERR_ARG;
    const size_t eout = precision == LIN_PREC_BF16 ? 2 : 4;
    const size_t wbytes = (size_t)N * K * 4, wobytes = (size_t)N * K * eout;
    // In place: W_out = W (fp32 storage) and bias_out = bias are allowed; no other overlap.
    if (!(W_out == W && eout == 4) && overlaps(W_out, wobytes, W, wbytes)) return LIN_ERR_ARG;
    if (overlaps(W_out, wobytes, gamma, (size_t)K * 4) || overlaps(W_out, wobytes, beta, beta ? (size_t)K * 4 : 0) ||
        overlaps(W_out, wobytes, bias, bias ? (size_t)N * 4 : 0) || overlaps(W_out, wobytes, bias_out, (size_t)N * 4))
        return LIN_ERR_ARG;
    if (bias_out != bias && overlaps(bias_out, (size_t)N * 4, bias, bias ? (size_t)N * 4 : 0)) return LIN_ERR_ARG;
    if (overlaps(bias_out, (size_t)N * 4, W, wbytes) || overlaps(bias_out, (size_t)N * 4, gamma, (size_t)K * 4) ||
        overlaps(bias_out, (size_t)N * 4, beta, beta ? (size_t)K * 4 : 0))
        return LIN_ERR_ARG;
    if ((((uintptr_t)W | (uintptr_t)bias | (uintptr_t)gamma | (uintptr_t)beta | (uintptr_t)bias_out) % 4) != 0 ||
        ((uintptr_t)W_out % eout) != 0)
        return LIN_ERR_ALIGN;
    DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rc = launch_fold_layernorm(N, K, W, bias, gamma, beta, W_out, bias_out, precision == LIN_PREC_BF16,
                                         ctx->sm_count, st);
    if (rc == LIN_OK) {
        note_output(st, Range{W_out, wobytes});
    }
    return rc;
}

int lin_forward_plan(lin_ctx* ctx, const lin_plan* plan, int M, int N, int K, const void* X, const void* W,
                     const float* bias, void* Y, int epilogue, int precision, void* stream) {
    if (!plan) return LIN_ERR_ARG;
    return lin::run(ctx, *plan, M, N, K, X, W, bias, Y, epilogue, precision, stream, false);
}

int lin_probe_ffma(lin_ctx* ctx, int iters, float* out, double* flops, void* stream) {
    if (!ctx || iters < 1 || !out) return LIN_ERR_ARG;
    if ((uintptr_t)out % 4 != 0) return LIN_ERR_ALIGN;
    lin::DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    return lin::launch_ffma_probe(ctx->sm_count, iters, out, static_cast<cudaStream_t>(stream), flops);
}

int lin_attention_forward(lin_ctx* ctx, int B, int T, int H, int D, const void* qkv, void* out, float* lse,
                          int causal, float scale, void* stream) {
    using namespace lin;
    if (!ctx || B < 0 || T < 0 || H < 0 || D < 0 || (causal != 0 && causal != 1)) return LIN_ERR_ARG;
    if (!(scale >= 0.f) || isinf(scale)) return LIN_ERR_ARG;  // NaN, negative or infinite
    if (B == 0 || T == 0 || H == 0) return LIN_OK;
    if (D != 64) return LIN_ERR_UNSUPPORTED;
    const long long rows = (long long)B * T;
    const long long nqb = (T + 127) / 128;
    if (rows > INT_MAX || (long long)H * D * 3 > INT_MAX || (long long)B * H * nqb > INT_MAX) return LIN_ERR_UNSUPPORTED;
    if (!qkv || !out) return LIN_ERR_ARG;
    const size_t C = (size_t)H * D;
    const size_t in_bytes = (size_t)rows * 3 * C * 2, out_bytes = (size_t)rows * C * 2;
    const size_t lse_bytes = lse ? (size_t)B * H * T * 4 : 0;
    if (overlaps(out, out_bytes, qkv, in_bytes) || overlaps(lse, lse_bytes, qkv, in_bytes) ||
        overlaps(lse, lse_bytes, out, out_bytes))
        return LIN_ERR_ARG;
    if ((((uintptr_t)qkv | (uintptr_t)out) % 16) != 0 || ((uintptr_t)lse % 4) != 0) return LIN_ERR_ALIGN;
    DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    AttnProblem p;
    p.B = B;
    p.T = T;
    p.H = H;
    p.qkv = qkv;
    p.out = out;
    p.lse = lse;
    p.causal = causal != 0;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    p.stream = static_cast<cudaStream_t>(stream);
    p.dev_status = ctx->dev_status;
    p.sm_count = ctx->sm_count;
    p.early_start = ctx->programmatic;
    // Its output is a later call's input: note it for the early-read checks.
    bool w_ok = false, x_ok = false, known = false;
    early_reads_ok(p.stream, Range{nullptr, 0}, Range{nullptr, 0}, Range{qkv, in_bytes}, Range{out, out_bytes}, &w_ok,
                   &x_ok, &known);
    return launch_attention(p);
}

int lin_check_device(lin_ctx* ctx, void* stream) {
    if (!ctx) return LIN_ERR_ARG;
    lin::DeviceGuard guard(ctx->device);
    if (!guard.ok) return LIN_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LIN_ERR_CUDA;
    int status = 0;
    if (cudaMemcpy(&status, ctx->dev_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LIN_ERR_CUDA;
    if (status != 0) {
        if (cudaMemset(ctx->dev_status, 0, sizeof(int)) != cudaSuccess) return LIN_ERR_CUDA;
        return status;
    }
    return LIN_OK;
}

}  // extern "C"
