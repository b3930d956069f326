// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/lin.h"

namespace lin {

// Everything one launch needs; filled by the C ABI layer after validation.
struct Problem {
    int M = 0, N = 0, K = 0;
    const void* X = nullptr;
    const void* W = nullptr;
    const float* bias = nullptr;
    void* Y = nullptr;
    // Residual added after the activation: M x N in Y's type, Y itself (in
    // place) or not overlapping Y; null for none. Read after the dependency
    // wait, like Y.
    const void* residual = nullptr;
    int epilogue = 0;   // lin_epilogue
    int precision = 0;  // lin_precision
    cudaStream_t stream = nullptr;
    // context resources
    void* workspace = nullptr;    // split-K partials (float) followed by tile counters (unsigned)
    size_t workspace_bytes = 0;
    int* dev_status = nullptr;    // device status word (LIN_ERR_DEVICE_TIMEOUT when a wait gave up)
    int sm_count = 0;
    // early_start: launch as a programmatic dependent of the previous kernel on
    // the stream (the CTAs may start before it finishes; nothing is read before
    // griddepcontrol.wait unless early_w / early_x say so; L2 prefetches of the
    // operands may be issued before it). early_w: W and bias do not overlap that
    // kernel's output and may be read before the wait; early_x: neither does X.
    // Y is written only after the wait.
    bool early_start = false;
    bool early_w = false;
    bool early_x = false;
};

// Workspace layout for split-K: a fixed block of per-tile arrival counters at
// the start (zero between launches: the last CTA of a tile re-arms its counter),
// then the partial sums [split][M][N] in fp32. The counters never move, so no
// launch's partial sums can overwrite another launch's counters.
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
constexpr size_t kCounterBytes = 64 * 1024;
constexpr int kMaxSplitTiles = (int)(kCounterBytes / sizeof(unsigned));
inline size_t splitk_workspace_bytes(int splits, int M, int N) {
    return splits > 1 ? kCounterBytes + align_up((size_t)splits * (size_t)M * (size_t)N * sizeof(float), 256) : 0;
}
inline unsigned* splitk_counters(void* ws) { return static_cast<unsigned*>(ws); }
inline float* splitk_partials(void* ws) { return reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes); }

// Tile configurations per kernel family (variant ids in lin_plan).
struct SkinnyCfg { int stages, kbox; };           // 128 W rows per cluster; splits = cluster size
constexpr int kSkinnyVariants = 5;
// Ring (stages x boxes of 64 K): 0 = 3 x 4 (~200 KB, one CTA per SM), 1 = 6 x 1
// (~110 KB), 2 = 3 x 2, 3 = 4 x 3, 4 = 5 x 1 (~99 KB with the cluster inbox:
// two CTAs per SM, so a call's CTAs can start while the previous call's run).
constexpr SkinnyCfg kSkinnyCfg[kSkinnyVariants] = {{3, 4}, {6, 1}, {3, 2}, {4, 3}, {5, 1}};
constexpr int kSkinnyTwoPerSm = 4;                 // the variant two CTAs of which fit on an SM
constexpr int kSkinnyThreads = 192;                // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

struct FfmaCfg { int bm, bn, bk, tm, tn, stages; };  // 256 threads each
constexpr int kFfmaVariants = 4;
// 0: 128 x 128, K steps of 32, 4 stages (one CTA per SM); 1: 64 x 64 (two per
// SM); 2: 128 x 128 with K steps of 64 in 3 stages (half the barriers);
// 3: 128 x 64 (two per SM: more warps to hide the shared-memory latency).
constexpr FfmaCfg kFfmaCfg[kFfmaVariants] = {
    {128, 128, 32, 8, 8, 4}, {64, 64, 32, 4, 4, 4}, {128, 128, 64, 8, 8, 3}, {128, 64, 32, 8, 4, 4}};

struct TcCfg { int bn; bool pair; };              // BM = 128 per CTA, BK = 128 bytes of K; ring depth from smem
constexpr int kTcVariants = 6;                     // pair: 2 x 1 clusters, SM-pair MMAs on 256 x BN tiles
constexpr TcCfg kTcCfg[kTcVariants] = {{256, false}, {128, false}, {192, false},
                                       {256, true}, {128, true}, {192, true}};
constexpr int kTcThreads = 320;                    // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
// Stream-K hand-over flags of the tcgen05 kernel: 8 per CTA boundary, in the
// counter block from this index on (zero between launches: the reader clears
// them). TC plans: splits = 1 whole tiles per CTA, 2 = stream-K.
constexpr int kTcFlagBase = 8192;
constexpr int kTcMaxStreamKCtas = (int)(kCounterBytes / sizeof(unsigned) - kTcFlagBase) / 8;
inline size_t tc_streamk_workspace_bytes(int ctas, int bn) {
    return kCounterBytes + align_up((size_t)ctas * 128 * (size_t)bn * sizeof(float), 256);
}
// K split of the tcgen05 kernel (plan.grid_z = splits > 1, whole single-CTA
// tiles): one 128 x BN fp32 slot per (tile, split), 8 counters per tile from
// index 0 of the counter block.
constexpr int kTcMaxKSplitTiles = kTcFlagBase / 8;
inline size_t tc_ksplit_workspace_bytes(long long tiles, int splits, int bn) {
    return kCounterBytes + align_up((size_t)tiles * splits * 128 * (size_t)bn * sizeof(float), 256);
}
// A K-split plan whose tiles outnumber its CTAs runs the grid's whole rounds
// of tiles unsplit and splits only the rest (the ragged last round): the
// number of tiles that run whole.
inline long long tc_tail_whole(long long tiles, int grid) { return tiles > grid ? tiles / grid * grid : 0; }
// Splits for a grid of `tiles` tiles with `nkb` K stages on `sm` SMs: enough
// (tile, split) items to fill the SMs once, >= 32 K stages per split, and only
// when the tiles alone fill at most half of the SMs. Measured on GB300: the
// weight gradient of the GPT-2 fc1 layer (72 tiles, 128 stages) 50.4 -> 37.7 us
// as an isolated call; a 1024^3 layer (16 stages) only got slower.
inline int tc_ksplits(long long tiles, int nkb, int sm, size_t ws_bytes, int bn) {
    if (tiles < 1 || tiles * 2 > sm || tiles > kTcMaxKSplitTiles) return 1;
    int S = (int)(sm / tiles);
    if (S > nkb / 32) S = nkb / 32;
    if (S > 16) S = 16;
    while (S > 1 && tc_ksplit_workspace_bytes(tiles, S, bn) > ws_bytes) --S;
    return S < 2 ? 1 : S;
}

// GEMV for a handful of rows (fp32 / tf32 M <= 8, bf16 M <= 4): X padded to
// 1, 2, 4 or 8 rows (plan.bm) lives in shared memory as fp32, so rows x K x 4
// bytes must fit.
constexpr int kGemvMaxRows = 8;
constexpr int kGemvMaxRowsBf16 = 4;
constexpr int kGemvMaxSmem = 96 * 1024;

// Raise a kernel's dynamic shared-memory limit on the current device, once per
// device ordinal below 64 (one bit each in `done`; higher ordinals set it on
// every call). Launches from several host threads may race to the first call:
// both then set the same value, and the mask is only read and or-ed atomically.
template <class Kernel>
int ensure_smem_attr(std::atomic<unsigned long long>& done, Kernel kern, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIN_ERR_CUDA;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return LIN_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LIN_ERR_CUDA;
    if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return LIN_OK;
}

// Launchers (return LIN_OK or LIN_ERR_*). They assume the plan was validated.
int launch_fill(const Problem& p);
int launch_skinny(const Problem& p, const lin_plan& plan);
int launch_ffma(const Problem& p, const lin_plan& plan);
int launch_tc(const Problem& p, const lin_plan& plan);
int launch_gemv(const Problem& p, const lin_plan& plan);

// Backward (training) GEMMs of the layer: which 1: dX = dZ W (M x K);
// which 2: dW = dZ^T X (N x K). B is W (which 1) or X (which 2).
struct BwdProblem {
    int which = 0;
    int M = 0, N = 0, K = 0;       // the forward layer's sizes
    const void* dZ = nullptr;      // M x N
    const void* B = nullptr;       // W (N x K) or X (M x K)
    void* out = nullptr;           // dX (M x K) or dW (N x K)
    cudaStream_t stream = nullptr;
    int* dev_status = nullptr;
    int sm_count = 0;
    bool early_start = false;      // programmatic launch: may start (not read) before the previous kernel finishes
    bool early_x = false;          // and read dZ and B before it finishes
    void* workspace = nullptr;     // context workspace (K split of small outputs)
    size_t workspace_bytes = 0;
    bool ksplit_ok = false;        // no independent call before it on the stream to overlap with
    const void* aux = nullptr;     // which 1: the previous layer's pre-activation (M x K): out *= gelu'(aux); or null
};
int launch_tc_backward(const BwdProblem& q);

// Fused self-attention forward (attn.cu): bf16 q, k, v read from the qkv
// projection's (B*T) x 3C output, heads of 64, output (B*T) x C bf16, row
// log-sum-exp (B x H x T fp32) when lse is not null.
struct AttnProblem {
    int B = 0, T = 0, H = 0;
    const void* qkv = nullptr;
    void* out = nullptr;
    float* lse = nullptr;
    bool causal = true;
    float scale = 0.f;             // softmax scale (> 0)
    cudaStream_t stream = nullptr;
    int* dev_status = nullptr;
    int sm_count = 0;
    bool early_start = false;      // programmatic launch (nothing is read before the dependency wait)
};
int launch_attention(const AttnProblem& p);

// Kernel timelines (timeline build only, see timeline.cuh): copy up to `bytes`
// of the stamp array to host memory at `dst` (if not null), then zero it (if
// `clear`). LIN_ERR_UNSUPPORTED in the library build.
int timeline_copy_tc(void* dst, size_t bytes, bool clear);
int timeline_copy_skinny(void* dst, size_t bytes, bool clear);
int timeline_copy_attn(void* dst, size_t bytes, bool clear);
int bwd_ffma_splits(int which, int M, int N, int K, int sm_count, size_t ws_bytes);
int launch_bwd_ffma(int which, int M, int N, int K, const float* dZ, const float* B, float* out, int splits,
                    void* workspace, cudaStream_t st, bool early, const float* Zp = nullptr);
int launch_gelu_backward(long long count, const void* dY, const void* Z, void* dZ, bool bf16, int sm_count,
                         cudaStream_t st, bool early);
size_t colsum_workspace_bytes(int M, int N);
int launch_colsum(int M, int N, const void* dZ, float* db, bool bf16, void* workspace, cudaStream_t st);

// fp32 FMA throughput probe: sm_count x 4 CTAs of 256 threads, each running
// independent fmaf chains for `iters` x 16 steps; *flops = the FLOPs launched.
int launch_ffma_probe(int sm_count, int iters, float* out, cudaStream_t st, double* flops);

int launch_fold_layernorm(int N, int K, const float* W, const float* bias, const float* gamma, const float* beta,
                          void* W_out, float* bias_out, bool bf16, int sm_count, cudaStream_t st);

}  // namespace lin
