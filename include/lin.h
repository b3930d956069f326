/*
 * lin.h - C ABI of a GB300 (sm_103a) library for the transformer linear layer
 *
 *     Y = act(X . W^T + bias)
 *
 * X is M x K row-major (one row per token / batch vector), W is N x K
 * row-major ("out x in", the way PyTorch stores a linear layer's weight), Y
 * is M x N row-major. Output (m, n) is the inner product of row m of X and
 * row n of W ("One multiply, one RTX 5090, eight kernels", section "The
 * multiply"). The bias (length N, optional) and the activation are applied in
 * the store of the product ("Writing a CUDA matmul that catches cuBLAS",
 * sections "The bias add did not need to exist" and "The residual and GELU go
 * the same way"). The activation is the identity or the tanh form of GELU,
 * 0.5 s (1 + tanh(sqrt(2/pi) (s + 0.044715 s^3))), applied to (sum + bias).
 *
 * All pointers to X, W, bias and Y are DEVICE pointers on the context's
 * device, owned by the caller. Every call is asynchronous on the given CUDA
 * stream (a cudaStream_t passed as void*, NULL = legacy default stream) and
 * returns after the work is enqueued; no call synchronises except
 * lin_check_device. No call ever computes on the host: when the GPU path
 * cannot run the call returns an error.
 *
 * Status codes: 0 on success, a negative LIN_ERR_* otherwise; lin_strerror
 * gives a message. No C++ exception crosses this boundary.
 */
#ifndef LIN_H
#define LIN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LIN_ABI_VERSION 1

#if defined(__GNUC__)
#define LIN_API __attribute__((visibility("default")))
#else
#define LIN_API
#endif

/* Arithmetic of the multiply.
 * FP32: fp32 X, W, Y; fp32 fused multiply-add on the CUDA cores (exact fp32
 *       products, fp32 sums) - the path of the sgemm ladder ("Writing a CUDA
 *       matmul that catches cuBLAS", "Kernel 8: the loop was shaped wrong").
 * TF32: fp32 X, W, Y; tensor-core products of the operands' TF32 parts with
 *       fp32 accumulation ("Writing a CUDA matmul that catches cuBLAS",
 *       "Kernel 9: the silicon I had not touched").
 * BF16: bf16 X, W, Y; fp32 bias; tensor-core bf16 products with fp32
 *       accumulation, output rounded to nearest-even bf16 ("One multiply, one
 *       RTX 5090, eight kernels", "From 748 to 29 microseconds"). */
typedef enum {
    LIN_PREC_FP32 = 0,
    LIN_PREC_TF32 = 1,
    LIN_PREC_BF16 = 2
} lin_precision;

/* Activation applied after the bias. */
typedef enum {
    LIN_EPI_NONE = 0,
    LIN_EPI_GELU_TANH = 1
} lin_epilogue;

typedef enum {
    LIN_OK = 0,
    LIN_ERR_ARG = -1,            /* NULL pointer, negative size, unknown enum, Y aliasing an input */
    LIN_ERR_ALIGN = -2,          /* X or W not 16-byte aligned, or K * element size not a multiple of 16 */
    LIN_ERR_WORKSPACE = -3,      /* an explicit plan needs more workspace than the context holds */
    LIN_ERR_CUDA = -4,           /* a CUDA runtime call or kernel launch failed */
    LIN_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up a bounded wait and skipped its work */
    LIN_ERR_UNSUPPORTED = -6     /* the plan's kernel cannot run this shape / precision */
} lin_status;

/* Kernels a plan can name. */
typedef enum {
    LIN_KERNEL_NONE = 0,   /* M == 0 or N == 0: nothing to do */
    LIN_KERNEL_FILL = 1,   /* K == 0: Y = act(bias) (or act(0)) */
    LIN_KERNEL_SKINNY = 2, /* M <= 16, BF16: W stream on the tensor cores, split-K in a cluster (no workspace) */
    LIN_KERNEL_FFMA = 3,   /* FP32: register-tiled FFMA, optional split-K */
    LIN_KERNEL_TC = 4,     /* TF32 / BF16: TMA + tcgen05 + TMEM, fused epilogue */
    LIN_KERNEL_GEMV = 5    /* FP32 / TF32 M <= 8, BF16 M <= 4 (the table: BF16 one row only): one pass over W in fp32 FMAs */
} lin_kernel;

/* One launch configuration, chosen by the dispatch table or given explicitly.
 * splits > 1 is split-K: each CTA sums one range of K into the workspace and
 * the last CTA to finish a tile adds the ranges in fixed order (0, 1, ...),
 * so results are bitwise repeatable ("Optimizing a GPT-2-class transformer on
 * a GPU", Act I, split-K combined by a fixed-order reduction). */
typedef struct {
    int kernel;   /* lin_kernel */
    int variant;  /* kernel-specific tile configuration id. TC: 0, 1, 2 = one CTA
                   * per 128 x 256 / 128 / 192 tile; 3, 4, 5 = SM pairs (2-CTA
                   * clusters issuing cta_group::2 MMAs) per 256 x 256 / 128 / 192
                   * tile. SKINNY and FFMA: see the kernels' sources. */
    int bm, bn, bk;
    int splits;   /* >= 1 */
    int stages;   /* shared-memory pipeline depth (TC), 0 otherwise */
    int grid_x, grid_y, grid_z; /* TC: grid_z = K splits (1 = none; the splits of a tile
                                 * are added in order by the last one to finish) */
    int threads;
    long long workspace_bytes; /* bytes of context workspace the launch uses */
} lin_plan;

typedef struct lin_ctx lin_ctx; /* opaque; owned by the library */

/* Create a context on CUDA device `device`. Allocates `max_workspace_bytes`
 * of device workspace (0 = a default of 64 MiB) for split-K partial sums and
 * tile counters, plus one device status word. Returns LIN_ERR_CUDA when the
 * device cannot be used. *out is NULL on failure. */
LIN_API int lin_create(lin_ctx** out, int device, size_t max_workspace_bytes);

/* Free a context and its workspace (synchronises the device first). NULL is
 * accepted. */
LIN_API int lin_destroy(lin_ctx* ctx);

/* Y = act(X . W^T + bias), chosen kernel per the dispatch table.
 *   M, N, K   : sizes, each >= 0 (M == 0 or N == 0 does nothing; K == 0 gives
 *               Y = act(bias) or act(0)).
 *   X         : M x K row-major; fp32 for FP32/TF32, bf16 for BF16.
 *   W         : N x K row-major (out x in), same element type as X.
 *   bias      : N fp32 values, or NULL for no bias.
 *   Y         : M x N row-major; fp32 for FP32/TF32, bf16 for BF16. Must not
 *               overlap X, W or bias.
 *   epilogue  : lin_epilogue.   precision : lin_precision.
 *   stream    : cudaStream_t (as void*).
 * X and W must be 16-byte aligned and K * element size a multiple of 16
 * (LIN_ERR_ALIGN otherwise); bias 4-byte aligned; Y aligned to its element.
 * One context must not run two calls at the same time (they share the
 * workspace): use one context per stream.
 * Back-to-back calls: with LIN_OPT_EARLY_START at 2 (off by default; see
 * that option for when it is safe), a call whose inputs (X, W, bias) overlap
 * none of the previous call's output on the same stream is launched as a
 * programmatic dependent of that call, reads its inputs before the previous
 * kernel has finished and writes Y only after it. For such a call the built-in
 * plan may also drop its K split (the skinny kernel's cluster split, the
 * tensor-core K split, an FFMA split over a short K), so that consecutive
 * independent calls fill the SMs together; see LIN_OPT_ADAPTIVE_PLANS.
 * lin_plan_query returns the plan of an isolated call. */
LIN_API int lin_forward(lin_ctx* ctx, int M, int N, int K, const void* X, const void* W,
                const float* bias, void* Y, int epilogue, int precision, void* stream);

/* Y = act(X . W^T + bias) + R: the residual add in the GEMM's store
 * ("Optimizing a GPT-2-class transformer on a GPU", Act II, rung 10, where
 * the bias, the activation and the residual add stop being kernels of their
 * own; "Writing a CUDA matmul that catches cuBLAS", "The residual and GELU go
 * the same way"). A
 * transformer block's x = x + proj(h) is this call with R = Y = x.
 *   R : M x N row-major, Y's element type; added after the activation, in
 *       fp32, with one rounding of the sum to Y's type. R may be Y itself (in
 *       place) and must otherwise not overlap Y; NULL is LIN_ERR_ARG (use
 *       lin_forward). Aligned to its element.
 * Everything else as lin_forward (same dispatch, installed plans included). */
LIN_API int lin_forward_residual(lin_ctx* ctx, int M, int N, int K, const void* X, const void* W,
                                 const float* bias, const void* R, void* Y, int epilogue, int precision,
                                 void* stream);

/* LayerNorm fold ("Optimizing a GPT-2-class transformer on a GPU", Act II,
 * rung 10: since LayerNorm's scale and shift reach the output only through
 * the linear layer after it, they can be moved into that layer's weight and
 * bias once, ahead of time, in double). With
 * LN(x) = gamma * xhat + beta, xhat = (x - mean) / sqrt(var + eps):
 *   W LN(x) + bias = W_out xhat + bias_out,
 *   W_out[n][k] = W[n][k] * gamma[k],  bias_out[n] = bias[n] + sum_k W[n][k] * beta[k].
 *   W        : N x K fp32 (device), the layer's weight (out x in).
 *   bias     : N fp32 or NULL (zero).   gamma : K fp32.   beta : K fp32 or NULL (zero).
 *   W_out    : N x K in the storage type of `precision` (fp32 for FP32/TF32,
 *              bf16 for BF16); may be W itself for fp32 storage (in place).
 *   bias_out : N fp32; may be bias itself.
 * Products and the sum (ascending k) in double; each output rounded once to
 * nearest even. Other overlaps: LIN_ERR_ARG; pointers aligned to their
 * elements (LIN_ERR_ALIGN). Asynchronous on `stream`. */
LIN_API int lin_fold_layernorm(lin_ctx* ctx, int N, int K, const float* W, const float* bias, const float* gamma,
                               const float* beta, void* W_out, float* bias_out, int precision, void* stream);

/* Same, with an explicit launch configuration (for tuning and for tests that
 * must reach one kernel). The plan is validated; LIN_ERR_UNSUPPORTED if its
 * kernel cannot run the shape, LIN_ERR_WORKSPACE if it needs more workspace
 * than the context holds. */
LIN_API int lin_forward_plan(lin_ctx* ctx, const lin_plan* plan, int M, int N, int K, const void* X,
                     const void* W, const float* bias, void* Y, int epilogue, int precision,
                     void* stream);

/* The dispatch table, on the host only (no GPU needed): the plan lin_forward
 * would use for this shape on a device with `sm_count` SMs and a workspace of
 * `workspace_bytes`. Returns LIN_ERR_ARG for invalid sizes or enums. */
LIN_API int lin_plan_query(int sm_count, int M, int N, int K, int precision, int epilogue,
                   size_t workspace_bytes, lin_plan* out);

/* Check a plan against a shape on the host (no GPU needed): LIN_OK when
 * lin_forward_plan would accept it in a context with `workspace_bytes` of
 * workspace, else the status it would return (LIN_ERR_UNSUPPORTED: the kernel
 * cannot run this shape / precision with this grid; LIN_ERR_WORKSPACE; or
 * LIN_ERR_ARG for a NULL plan, negative sizes or an unknown precision).
 * Limits that depend on the device (stream-K CTAs at most one per SM) are
 * checked when the call is launched. */
LIN_API int lin_plan_check(const lin_plan* plan, int M, int N, int K, int precision, size_t workspace_bytes);

/* Fill *out with the default plan of a kernel family for a shape (host only),
 * for sweeps: kernel = lin_kernel, variant = tile configuration, splits = 0
 * lets the table choose the split. For LIN_KERNEL_TC, splits counts CTAs
 * instead: >= 0 CTAs walking whole tiles (0 = one per SM); -1 stream-K with
 * one CTA per SM; -c (c >= 2) stream-K with c CTAs (single-CTA variants, at
 * least one tile per CTA; the plan's splits is then 2 and it needs workspace
 * for one 128 x BN fp32 slot per CTA). For LIN_KERNEL_GEMV, splits is the
 * CTA count (0 = as many as fit at once). Returns LIN_ERR_UNSUPPORTED when the
 * kernel cannot run the shape. */
LIN_API int lin_plan_make(int sm_count, int kernel, int variant, int splits, int M, int N, int K,
                  int precision, lin_plan* out);

/* ---- Backward (training) ----
 * The backward pass of the same layer ("Writing a CUDA matmul that catches
 * cuBLAS", the backward transpose cases: dX = dY W^T and dW = dY^T X for a
 * weight stored in x out; here W is stored out x in):
 *   dZ = dY * act'(Z)           (lin_gelu_backward, or dZ = dY for no activation)
 *   dX = dZ . W      (M x K)    (lin_backward_data)
 *   dW = dZ^T . X    (N x K)    (lin_backward_weight, with db = sum over rows of dZ)
 * Operands are in the precision's input type and results in its output type
 * (bf16 for LIN_PREC_BF16, fp32 otherwise; db is always fp32). BF16 runs on
 * the tensor cores with the transposes folded into the operands' shared-memory
 * layout (nothing is transposed in memory); FP32 and TF32 run exact fp32
 * FFMAs. Results are bitwise repeatable. Calls are asynchronous on `stream`
 * and follow lin_forward's early-start rules. */

/* dX (M x K) = dZ (M x N) . W (N x K), all row-major. dZ, W and dX 16-byte
 * aligned; K * element size a multiple of 16; for BF16 also N * 2 (the rows
 * of dZ are read by TMA). dX must not overlap dZ or W. N == 0 gives zeros. */
LIN_API int lin_backward_data(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* W, void* dX,
                              int precision, void* stream);

/* dW (N x K) = dZ^T . X (dZ: M x N, X: M x K), and db[n] = sum_m dZ[m][n]
 * in fp32 when db is not NULL (two passes over fixed row chunks, in order;
 * uses the context workspace: LIN_ERR_WORKSPACE when it is too small). The
 * alignment rules of lin_backward_data apply to dZ, X and dW; db is 4-byte
 * aligned. M == 0 gives zeros. */
LIN_API int lin_backward_weight(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* X, void* dW,
                                float* db, int precision, void* stream);

/* dZ = dY * gelu'(Z) elementwise over `count` values, Z the pre-activation
 * (act's input) of the forward; the slope of the tanh form used by the
 * forward. dZ may be dY (in place) but not Z. */
LIN_API int lin_gelu_backward(lin_ctx* ctx, long long count, const void* dY, const void* Z, void* dZ,
                              int precision, void* stream);

/* dX carried through the previous layer's GELU in the same pass: when this
 * layer's input was X = gelu(Zp) (Zp the previous layer's pre-activation),
 *   dZp = (dZ . W) * gelu'(Zp)      (M x K),
 * i.e. lin_backward_data followed by lin_gelu_backward, with the slope
 * applied in the GEMM's store instead of a second pass over M x K.
 *   Zp : M x K row-major in the precision's storage type; dZp may be Zp
 *        itself (in place) and must otherwise not overlap it.
 * Everything else as lin_backward_data. */
LIN_API int lin_backward_data_gelu(lin_ctx* ctx, int M, int N, int K, const void* dZ, const void* W,
                                   const void* Zp, void* dZp, int precision, void* stream);

/* Measured dispatch ("Optimizing a GPT-2-class transformer on a GPU", Act II:
 * route each shape to its measured winner). Install `plan` as the context's
 * choice for lin_forward calls with exactly these sizes, precision and
 * epilogue (checked like lin_forward_plan; LIN_ERR_UNSUPPORTED or
 * LIN_ERR_WORKSPACE when it cannot run the shape in this context; a refused
 * plan leaves any earlier entry in place). A NULL plan removes the entry
 * (LIN_OK whether or not there was one). The plan is copied; entries are
 * guarded by a lock, so installing while another thread calls lin_forward is
 * safe. lin_forward consults these entries before the
 * built-in table and runs an installed plan as given (no adaptive change for
 * back-to-back calls). The Python package's autotuner measures candidates and
 * installs winners through this call. */
LIN_API int lin_set_plan_override(lin_ctx* ctx, int M, int N, int K, int precision, int epilogue,
                                  const lin_plan* plan);

/* Remove every installed plan of the context. */
LIN_API int lin_clear_plan_overrides(lin_ctx* ctx);

/* Synchronise `stream`, read and clear the context's device status word.
 * Returns LIN_ERR_DEVICE_TIMEOUT if any kernel since the last check gave up
 * a bounded wait (its output is then incomplete), LIN_ERR_CUDA on a CUDA
 * error, LIN_OK otherwise. */
LIN_API int lin_check_device(lin_ctx* ctx, void* stream);

/* Context options (lin_set_option).
 * LIN_OPT_PROGRAMMATIC_LAUNCH (default 1): calls are launched as programmatic
 *   dependents of the previous kernel on their stream: a call's CTAs may start
 *   on SMs as the previous kernel's CTAs leave them, set up (barriers, tensor
 *   memory, descriptors) and ask the L2 cache to fetch their first operand
 *   tiles, and then wait (griddepcontrol.wait) until that kernel has finished
 *   and its writes are visible before they read anything. An L2 prefetch
 *   returns no data to the kernel and L2 is where all writes meet, so this
 *   changes no result whatever the previous kernel writes. 0 = plain stream
 *   order (the CTAs start only after all earlier work has finished).
 * LIN_OPT_EARLY_START (default 0): which operands may be READ before the
 *   previous kernel on the stream has finished (needs programmatic launch).
 *   0: none; every call reads its operands only after all earlier work on the
 *      stream, like any stream-ordered library.
 *   1: W and bias may be read before that kernel has finished. X is read, and
 *      Y written, only after it.
 *   2: as 1, and X may be read early too.
 *   The library only sees its own calls: it drops the early reads of W / bias
 *   (and X) by itself when they overlap the previous library call's output on
 *   that stream, but it cannot see other work. Use 1 only when no other work on
 *   the stream writes the next call's W or bias between two library calls (an
 *   optimizer step does), and 2 only when nothing but library calls write its X
 *   either (a framework kernel that produces X, such as a layernorm, does).
 *   With 2, a call that overlaps an independent predecessor may also narrow its
 *   plan (LIN_OPT_ADAPTIVE_PLANS).
 * LIN_OPT_ADAPTIVE_PLANS (default 1): a call that overlaps an independent
 *   predecessor on its stream (early start level 2) may drop
 *   the K split of its built-in plan: the neighbouring call then fills the SMs
 *   the split would. A split changes the order of the fp32 sums, so with this
 *   option on, the last bits of a result can depend on the call before it on
 *   the stream (never beyond the precision's tolerance). 0 = the plan of a
 *   call depends only on its sizes, precision and epilogue, so identical
 *   inputs give identical bits whatever ran before. Installed plans
 *   (lin_set_plan_override) and lin_forward_plan are never adapted. */
typedef enum {
    LIN_OPT_EARLY_START = 1,
    LIN_OPT_ADAPTIVE_PLANS = 2,
    LIN_OPT_PROGRAMMATIC_LAUNCH = 3
} lin_option;

/* The plan of the last call launched through this context (host value, no
 * GPU call): lin_forward may refine the dispatch table's plan for a call that
 * overlaps its predecessor. LIN_ERR_ARG if ctx or out is NULL; a context with
 * no call yet reports LIN_KERNEL_NONE. */
LIN_API int lin_ctx_last_plan(const lin_ctx* ctx, lin_plan* out);

/* Set a context option. LIN_ERR_ARG for an unknown option or value. */
LIN_API int lin_set_option(lin_ctx* ctx, int option, long long value);

/* SM count and device ordinal of a context (host values, no GPU call). */
LIN_API int lin_ctx_info(const lin_ctx* ctx, int* device, int* sm_count, size_t* workspace_bytes);

/* Throughput probe of the exact-fp32 FMA pipe (the roofline of the FFMA
 * kernels; the pages derive their fp32 peak from unit counts and the clock,
 * "Writing a CUDA matmul that catches cuBLAS", opening section). Launches, on
 * `stream`, the context's SM count x 4 CTAs of 256 threads, each thread
 * running 8 independent fmaf chains for iters x 16 steps, and nothing else;
 * *flops (if not NULL) receives the FLOPs launched (2 per fmaf). The caller
 * times the launch (CUDA events on `stream`). `out`: a device float the
 * kernel writes only in a case that cannot occur, which keeps the chains
 * live. Returns LIN_ERR_ARG for iters < 1 or a NULL out. */
LIN_API int lin_probe_ffma(lin_ctx* ctx, int iters, float* out, double* flops, void* stream);

/* Static message for a status code. */
LIN_API const char* lin_strerror(int status);

/* LIN_ABI_VERSION of the loaded library. */
LIN_API int lin_abi_version(void);

/* Kernel timeline (measurement aid; "One multiply, one RTX 5090, eight
 * kernels", "Where the time goes", times parts of a kernel separately to see
 * where its time goes). In the separate timeline build of this library
 * (compiled with -DLIN_TIMELINE), the tcgen05 kernel and the skinny kernel
 * record %globaltimer nanoseconds at fixed points of each CTA's schedule into
 * device arrays of LIN_TIMELINE_CTAS x LIN_TIMELINE_SLOTS unsigned 64-bit
 * values (0 = point not reached):
 *   kernel LIN_KERNEL_TC, record = blockIdx.x: [0] set up, [1] producer past
 *     its dependency wait, [2] teardown; for work item j < 32: [8 + 4j] MMAs
 *     start (accumulator free), [8 + 4j + 1] last MMA and commit issued,
 *     [8 + 4j + 2] epilogue warp 2 sees the accumulator, [8 + 4j + 3]
 *     epilogue warp 2 done, [136 + j] epilogue warp 9 done;
 *   kernel LIN_KERNEL_SKINNY, records in the order CTAs start (consecutive
 *     launches follow one another): [0] set up, [1] producer past its
 *     dependency wait, [2] MMAs complete, [3] done, [16 + i] stage i landed;
 *   kernel LIN_TIMELINE_ATTENTION (lin_attention_forward), record =
 *     blockIdx.x: [0] set up, [1] producer past its dependency wait, [2]
 *     teardown; for the CTA's work item n < 16, at 8 + 10n + k: k = 0 Q copy
 *     issued, 1 first K/V copy issued, 2 MMA warp saw the first K/V land, 3
 *     first S MMAs committed, 4 softmax warp 2 saw the first S, 5 it released
 *     the last P, 6 last P.V MMAs committed, 7 softmax warp 2 saw the last
 *     P.V, 8 softmax warp 2 stored its rows, 9 softmax warp 9 stored its rows.
 * lin_timeline copies the first `bytes` of that kernel's array to `host_dst`
 * (synchronously; both NULL/0 to skip the copy), then zeroes the array (and
 * the skinny record counter) if `clear` is non-zero. A stamped launch is
 * identical to the library build's in everything else. Returns
 * LIN_ERR_UNSUPPORTED in the library build, LIN_ERR_ARG for another kernel
 * id or a NULL/non-zero mismatch of host_dst and bytes. */
#define LIN_TIMELINE_ATTENTION 16
#define LIN_TIMELINE_CTAS 1024
#define LIN_TIMELINE_SLOTS 192
LIN_API int lin_timeline(int kernel, void* host_dst, size_t bytes, int clear);

/* Size of the fixed device array behind lin_forward_fp32_static. */
#define LIN_STATIC_SCRATCH_BYTES (8u << 20)

/* The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory when they run the layer, for example:
 * - runtimes that reserve all device memory for their own pool at start-up
 *   and treat any other allocation as a failure;
 * - latency-critical paths where an allocation could block on the device or
 *   fail under memory pressure;
 * - plug-ins that are handed device pointers but no allocator.
 *
 * Y = act(X . W^T + bias) in fp32 on the CURRENT device, with the same
 * kernel and split-K choice as lin_forward(..., LIN_PREC_FP32, ...) (the FFMA
 * kernel, or the GEMV for M <= 8, which needs no scratch), but with no
 * context. It calls no cudaMalloc or cudaFree: the split-K counters and
 * partial sums live in one fixed array of LIN_STATIC_SCRATCH_BYTES (8 MiB),
 * a static device variable of this library that every GPU which loads the
 * library holds until the process exits. Arguments, layouts and alignment
 * rules are those of lin_forward; X, W, bias and Y are caller-owned device
 * pointers.
 *
 * Limits and caveats:
 * - The split is the one lin_forward would take, so the result is bitwise
 *   that of lin_forward. A shape whose split needs more scratch than the
 *   array holds returns LIN_ERR_WORKSPACE (nothing is launched); the split
 *   fills the SMs, so its scratch grows with the SM count (about 5 MB on 152
 *   SMs) and not with the shape.
 * - The first call on a device (and the first after that device's context
 *   was created anew) looks up the array's device address; make that first
 *   call before any stream capture.
 * - Every call shares the one array, and the array keeps the last call's
 *   contents. The call zeroes the counters it uses on `stream` before its
 *   kernel.
 * - Calls whose kernels overlap on the GPU (other streams, or other threads
 *   without ordering) race on the array: order them on one stream. */
LIN_API int lin_forward_fp32_static(int M, int N, int K, const float* X, const float* W,
                                    const float* bias, float* Y, int epilogue, void* stream);

/* Fused self-attention forward, the step between the qkv projection and the
 * output projection ("Writing a CUDA matmul that catches cuBLAS", section
 * "Fusing attention: the score matrix never exists": q, k and v are read
 * straight from the projection's output, a running row max and sum replace
 * the stored score matrix, and causality is the loop bound). For sequence b,
 * head h and query token i:
 *   s_ij  = (q_i . k_j) * scale over the visible keys j (j <= i when causal,
 *           all j < T otherwise),
 *   out[b*T + i][h*64 + d] = sum_j exp(s_ij - m_i) v_j[d] / l_i,
 *   m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i),
 *   lse[(b*H + h)*T + i] = m_i + log(l_i)            (when lse is not NULL).
 *   qkv : DEVICE, (B*T) x 3C bf16 row-major, C = H*D; token t of sequence b is
 *         row b*T + t, holding q, k, v at column offsets 0, C, 2C and head h
 *         at h*D within each (the layout of the qkv linear layer's output).
 *   out : DEVICE, (B*T) x C bf16 row-major (the output projection's input);
 *         must not overlap qkv or lse.
 *   lse : DEVICE fp32 B x H x T, or NULL (the softmax statistics a backward
 *         pass rebuilds the probabilities from).
 *   D   : head width; 64 only (LIN_ERR_UNSUPPORTED otherwise).
 *   causal: 1 (decoder attention) or 0.
 *   scale: softmax scale > 0; 0 selects 1/sqrt(D).
 * Arithmetic: bf16 q, k products accumulated in fp32 on the tensor cores,
 * softmax in fp32 (base-2 exponent of the scaled scores, hardware ex2),
 * probabilities rounded to bf16 for the product with v (fp32 accumulation),
 * output rounded to nearest-even bf16. qkv and out must be 16-byte aligned
 * (LIN_ERR_ALIGN), lse 4-byte aligned; B*T < 2^31. B, T or H == 0: nothing to
 * do. Asynchronous on `stream`; launched as a programmatic dependent of the
 * previous kernel (when LIN_OPT_PROGRAMMATIC_LAUNCH is on) but reads qkv and
 * writes out / lse only after that kernel has finished (before that it only
 * asks the L2 cache for its first tiles, which returns no data to the
 * kernel). LIN_ERR_UNSUPPORTED also when the library was compiled so that
 * the kernel holds fewer registers a thread than its warp-specialised
 * register split needs (it then launches nothing). */
LIN_API int lin_attention_forward(lin_ctx* ctx, int B, int T, int H, int D, const void* qkv, void* out, float* lse,
                                  int causal, float scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIN_H */
