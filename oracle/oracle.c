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
 *   stores a linear layer's weight), Y is M x N row-major. Each output is the
 *   dot product of one row of X with one row of W
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

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
