/*
 * CPU oracle for the transformer linear layer. TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library; the product path never does.
 *
 * What it computes (written from the definition, one output at a time):
 *
 *   Y[m][n] = act( sum_{k=0}^{K-1} X[m][k] * W[n][k]  +  bias[n] )
 *
 * - X is M x K row-major, W is N x K row-major ("out x in", the way PyTorch
 *   stores a linear layer's weight), Y is M x N row-major. Output (m, n) is
 *   the inner product of row m of X and row n of W
 *   ("One multiply, one RTX 5090, eight kernels", section "The multiply").
 * - The sum is accumulated in double, in ascending k, one scalar at a time.
 *   Inputs are the fp32 values the GPU receives (bf16 inputs arrive here
 *   widened exactly); each product of two fp32 values is exact in double.
 * - bias (length N, may be absent) is added before the activation
 *   ("Writing a CUDA matmul that catches cuBLAS", sections "The bias add did
 *   not need to exist" and "The residual and GELU go the same way").
 * - act is the identity or the tanh form of GELU,
 *     gelu(s) = 0.5 s (1 + tanh( sqrt(2/pi) (s + 0.044715 s^3) )),
 *   evaluated in double with libm tanh. The pages name GELU and its tanhf
 *   evaluation but print no formula; this form and its constants are those of
 *   Hendrycks and Gimpel, "Gaussian Error Linear Units" (2016).
 *
 * The backward of the same layer (dZ, dX, dW, db), the fused residual, the
 * LayerNorm fold, the dX carried through a GELU and the self-attention that
 * reads the qkv projection are defined further down.
 *
 * OpenMP splits the (m, n) outputs across threads; each output's k order is
 * fixed, so the result does not depend on the thread count.
 * Build with -ffp-contract=off so no multiply-add is fused and x86 and Arm
 * hosts produce identical bits.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double oracle_gelu_tanh(double s)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * s * (1.0 + tanh(c * (s + 0.044715 * s * s * s)));
}

static double one_output(int64_t K, const float* xrow, const float* wrow,
                         const float* bias, int64_t n, int gelu)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += (double)xrow[k] * (double)wrow[k];
    if (bias)
        s += (double)bias[n];
    if (gelu)
        s = oracle_gelu_tanh(s);
    return s;
}

/* Full output. X: M*K, W: N*K, bias: N or NULL, Y: M*N (double). */
void oracle_linear(int64_t M, int64_t N, int64_t K, const float* X, const float* W,
                   const float* bias, int gelu, double* Y, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = one_output(K, X + m * K, W + n * K, bias, n, gelu);
    (void)nthreads;
}

/* Selected outputs (ms[i], ns[i]) for i < count, into Y[i]. */
void oracle_linear_entries(int64_t count, const int64_t* ms, const int64_t* ns,
                           int64_t K, const float* X, const float* W,
                           const float* bias, int gelu, double* Y, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < count; ++i)
        Y[i] = one_output(K, X + ms[i] * K, W + ns[i] * K, bias, ns[i], gelu);
    (void)nthreads;
}

/* gelu over an array (for the activation's own pins). */
void oracle_gelu_array(int64_t count, const double* in, double* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = oracle_gelu_tanh(in[i]);
}

/*
 * Backward of Y = act(Z), Z = X W^T + bias (the definitions written out).
 * The pages' backward pass ("Writing a CUDA matmul that catches cuBLAS",
 * the section on the backward transpose cases) needs dX = dY W^T and
 * dW = dY^T X for a weight stored in x out; with W stored out x in as here:
 *
 *   dZ[m][n] = dY[m][n] * act'(Z[m][n])      (act' = 1, or the GELU slope)
 *   dX[m][k] = sum_n dZ[m][n] * W[n][k]      (M x K)
 *   dW[n][k] = sum_m dZ[m][n] * X[m][k]      (N x K)
 *   db[n]    = sum_m dZ[m][n]
 *
 * Sums in double, in ascending order of the summed index, one output at a
 * time. The slope of the tanh-form GELU g(z) = 0.5 z (1 + tanh u),
 * u = c (z + a z^3), c = sqrt(2/pi), a = 0.044715, is
 *   g'(z) = 0.5 (1 + tanh u) + 0.5 z (1 - tanh^2 u) c (1 + 3 a z^2).
 */
double oracle_gelu_tanh_grad(double z)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double a = 0.044715;
    const double t = tanh(c * (z + a * z * z * z));
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * c * (1.0 + 3.0 * a * z * z);
}

/* dZ from dY and the layer's own inputs (Z recomputed in double).
   dY: M*N, dZ: M*N (double). */
void oracle_backward_dz(int64_t M, int64_t N, int64_t K, const float* X, const float* W,
                        const float* bias, const float* dY, int gelu, double* dZ, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const double g = (double)dY[m * N + n];
            dZ[m * N + n] = gelu ? g * oracle_gelu_tanh_grad(one_output(K, X + m * K, W + n * K, bias, n, 0)) : g;
        }
    (void)nthreads;
}

/* dZ from dY and a given pre-activation Z (fp32 values): M*N each. */
void oracle_gelu_backward(int64_t count, const float* dY, const float* Z, double* dZ)
{
    for (int64_t i = 0; i < count; ++i)
        dZ[i] = (double)dY[i] * oracle_gelu_tanh_grad((double)Z[i]);
}

/* dX = dZ W. dZ: M*N, W: N*K (fp32 values), dX: M*K (double). */
void oracle_backward_dx(int64_t M, int64_t N, int64_t K, const float* dZ, const float* W, double* dX,
                        int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n)
                s += (double)dZ[m * N + n] * (double)W[n * K + k];
            dX[m * K + k] = s;
        }
    (void)nthreads;
}

/* dW = dZ^T X and db = column sums of dZ. dZ: M*N, X: M*K (fp32 values),
   dW: N*K, db: N or NULL (double). */
void oracle_backward_dw(int64_t M, int64_t N, int64_t K, const float* dZ, const float* X, double* dW,
                        double* db, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double s = 0.0;
            for (int64_t m = 0; m < M; ++m)
                s += (double)dZ[m * N + n] * (double)X[m * K + k];
            dW[n * K + k] = s;
        }
    if (db) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t m = 0; m < M; ++m)
                s += (double)dZ[m * N + n];
            db[n] = s;
        }
    }
    (void)nthreads;
}

/* gelu slope over an array (for its own pins). */
void oracle_gelu_grad_array(int64_t count, const double* in, double* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = oracle_gelu_tanh_grad(in[i]);
}

/*
 * Residual add in the GEMM's store ("Optimizing a GPT-2-class transformer on
 * a GPU", Act II, rung 10, where the bias, the activation and the residual
 * add stop being kernels of their own; "Writing a CUDA matmul that catches
 * cuBLAS", "The residual and GELU go the same way"):
 *
 *   Y[m][n] = act(Z[m][n]) + R[m][n],   Z = X W^T + bias,
 *
 * R (M x N, fp32 values) is the residual stream, added after the activation
 * (the transformer's x + sublayer(x); the pages give no order, the
 * activation-free case is the one a GPT block uses).
 */
void oracle_linear_residual(int64_t M, int64_t N, int64_t K, const float* X, const float* W,
                            const float* bias, const float* R, int gelu, double* Y, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = one_output(K, X + m * K, W + n * K, bias, n, gelu) + (double)R[m * N + n];
    (void)nthreads;
}

/*
 * LayerNorm over the last axis (the definition, in double):
 *   mean = (1/K) sum_k x[k],  var = (1/K) sum_k (x[k] - mean)^2,
 *   xhat[k] = (x[k] - mean) / sqrt(var + eps),
 *   out[k] = gamma[k] xhat[k] + beta[k]   (gamma / beta NULL: xhat alone).
 * Sums in ascending k. X: M*K fp32 values, out: M*K double.
 */
void oracle_layernorm(int64_t M, int64_t K, const float* X, const float* gamma, const float* beta,
                      double eps, double* out)
{
    for (int64_t m = 0; m < M; ++m) {
        const float* x = X + m * K;
        double mean = 0.0, var = 0.0;
        for (int64_t k = 0; k < K; ++k) mean += (double)x[k];
        mean /= (double)K;
        for (int64_t k = 0; k < K; ++k) var += ((double)x[k] - mean) * ((double)x[k] - mean);
        var /= (double)K;
        const double inv = 1.0 / sqrt(var + eps);
        for (int64_t k = 0; k < K; ++k) {
            double v = ((double)x[k] - mean) * inv;
            if (gamma) v *= (double)gamma[k];
            if (beta) v += (double)beta[k];
            out[m * K + k] = v;
        }
    }
}

/*
 * LayerNorm fold (Act II, rung 10: LayerNorm's scale and shift reach the
 * output only through the next linear layer, so they can be moved into its
 * weight and bias once, ahead of time, in double). With
 * LN(x) = gamma * xhat + beta,
 *   W LN(x) + b = (W diag(gamma)) xhat + (W beta + b), so
 *   Wf[n][k] = W[n][k] * gamma[k],   bf[n] = b[n] + sum_k W[n][k] * beta[k]
 * (ascending k; bias or beta NULL count as zero). W: N*K, gamma, beta: K
 * (fp32 values); Wf: N*K, bf: N (double).
 */
void oracle_fold_layernorm(int64_t N, int64_t K, const float* W, const float* bias, const float* gamma,
                           const float* beta, double* Wf, double* bf)
{
    for (int64_t n = 0; n < N; ++n) {
        double s = bias ? (double)bias[n] : 0.0;
        for (int64_t k = 0; k < K; ++k) {
            Wf[n * K + k] = (double)W[n * K + k] * (double)gamma[k];
            if (beta) s += (double)W[n * K + k] * (double)beta[k];
        }
        bf[n] = s;
    }
}

/*
 * dX of a layer whose input is the GELU of the previous layer's
 * pre-activation Zp (X = gelu(Zp)), carried through that GELU in the same
 * pass: dZp[m][k] = (sum_n dZ[m][n] W[n][k]) * gelu'(Zp[m][k]).
 * dZ: M*N, W: N*K, Zp: M*K (fp32 values); dZp: M*K (double).
 */
void oracle_backward_dx_gelu(int64_t M, int64_t N, int64_t K, const float* dZ, const float* W,
                             const float* Zp, double* dZp, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(static) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n)
                s += (double)dZ[m * N + n] * (double)W[n * K + k];
            dZp[m * K + k] = s * oracle_gelu_tanh_grad((double)Zp[m * K + k]);
        }
    (void)nthreads;
}

/*
 * Causal or full self-attention of one transformer layer, read straight out
 * of the qkv projection's output ("Writing a CUDA matmul that catches
 * cuBLAS", section "Fusing attention: the score matrix never exists": the
 * fused kernel indexes q, k and v in the (B, T, 3C) projection; one head is a
 * fixed column offset).
 *
 *   qkv: (B*T) x 3C fp32 values, C = H*D; for token t of sequence b and head h
 *        q = qkv[b*T + t][h*D .. h*D + D), k at column C + h*D, v at 2C + h*D.
 *   out: (B*T) x C (double), out[b*T + i][h*D + d] = sum_j p_ij v_j[d] with
 *        p_ij = exp(s_ij - m_i) / l_i,  s_ij = (q_i . k_j) * scale,
 *        m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i),
 *        over the keys j visible to query i: j <= i when causal, else all T.
 *   lse: B*H*T (double, may be NULL), lse[(b*H + h)*T + i] = m_i + log(l_i).
 *
 * This is the definition written out (two passes over a row of scores, all
 * in double, each sum in ascending index order); the pages compute the same
 * result with a running max and sum, which changes only the rounding.
 */
void oracle_attention(int64_t B, int64_t T, int64_t H, int64_t D, const float* qkv, int causal, double scale,
                      double* out, double* lse, int nthreads)
{
    const int64_t C = H * D, ld = 3 * C;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(3) schedule(static) num_threads(nthreads)
#endif
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < T; ++i) {
                const float* q = qkv + (b * T + i) * ld + h * D;
                const int64_t nj = causal ? i + 1 : T;
                double m = -INFINITY;
                for (int64_t j = 0; j < nj; ++j) {
                    const float* k = qkv + (b * T + j) * ld + C + h * D;
                    double s = 0.0;
                    for (int64_t d = 0; d < D; ++d) s += (double)q[d] * (double)k[d];
                    s *= scale;
                    if (s > m) m = s;
                }
                double l = 0.0;
                double* o = out + (b * T + i) * C + h * D;
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t j = 0; j < nj; ++j) {
                    const float* k = qkv + (b * T + j) * ld + C + h * D;
                    const float* v = qkv + (b * T + j) * ld + 2 * C + h * D;
                    double s = 0.0;
                    for (int64_t d = 0; d < D; ++d) s += (double)q[d] * (double)k[d];
                    const double e = exp(s * scale - m);
                    l += e;
                    for (int64_t d = 0; d < D; ++d) o[d] += e * (double)v[d];
                }
                for (int64_t d = 0; d < D; ++d) o[d] /= l;
                if (lse) lse[(b * H + h) * T + i] = m + log(l);
            }
    (void)nthreads;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
