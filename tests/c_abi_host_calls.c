/* A C99 caller of the library's host-only entry points: it compiles against
 * include/lin.h as plain C, links against the built library and runs without
 * a GPU. Prints one line per check and exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "lin.h"

#define CHECK(cond, what)                                   \
    do {                                                    \
        if (!(cond)) {                                      \
            printf("FAIL %s\n", what);                      \
            return 1;                                       \
        }                                                   \
        printf("ok %s\n", what);                            \
    } while (0)

int main(void) {
    lin_plan p;
    lin_ctx* ctx = NULL;
    CHECK(lin_abi_version() == LIN_ABI_VERSION, "abi version");
    CHECK(strlen(lin_strerror(LIN_ERR_ALIGN)) > 0, "strerror");
    CHECK(lin_plan_query(152, 16, 4096, 4096, LIN_PREC_BF16, LIN_EPI_NONE, (size_t)64 << 20, &p) == LIN_OK &&
              p.kernel == LIN_KERNEL_SKINNY,
          "skinny layer routed to the skinny kernel");
    CHECK(lin_plan_check(&p, 16, 4096, 4096, LIN_PREC_BF16, (size_t)64 << 20) == LIN_OK, "its plan checks");
    CHECK(lin_plan_query(152, 8192, 2304, 768, LIN_PREC_BF16, LIN_EPI_GELU_TANH, (size_t)64 << 20, &p) == LIN_OK &&
              p.kernel == LIN_KERNEL_TC,
          "wide bf16 layer routed to the tensor-core kernel");
    CHECK(lin_plan_make(152, LIN_KERNEL_FFMA, 1, 3, 128, 768, 768, LIN_PREC_FP32, &p) == LIN_OK && p.splits == 3,
          "explicit FFMA plan");
    CHECK(lin_plan_check(&p, 128, 768, 768, LIN_PREC_FP32, 0) == LIN_ERR_WORKSPACE, "split needs workspace");
    CHECK(lin_plan_query(152, -1, 1, 1, LIN_PREC_FP32, LIN_EPI_NONE, 0, &p) == LIN_ERR_ARG, "negative size refused");
    CHECK(lin_forward(NULL, 1, 1, 1, NULL, NULL, NULL, NULL, LIN_EPI_NONE, LIN_PREC_FP32, NULL) == LIN_ERR_ARG,
          "null context refused");
    CHECK(lin_attention_forward(NULL, 1, 128, 12, 64, NULL, NULL, NULL, 1, 0.0f, NULL) == LIN_ERR_ARG,
          "attention: null context refused");
    CHECK(lin_create(&ctx, 0, 0) != LIN_OK || ctx != NULL, "create fails cleanly or succeeds");
    if (ctx) lin_destroy(ctx);
    return 0;
}
