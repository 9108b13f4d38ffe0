/* A plain C99 client of the library: it includes only ctx_attn.h, links the
 * shared library and calls the host-side entry points, so that the boundary
 * is shown to be usable without C++, CUDA headers or Python.  Nothing here
 * needs a GPU: the attention calls below are invalid and must be refused
 * before anything is launched.  Exit status 0 = every check held. */
#include <stdio.h>
#include <string.h>

#include "ctx_attn.h"

static int failures = 0;
#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            ++failures;                                               \
        }                                                             \
    } while (0)

int main(void) {
    /* array_split chunking of 1001 rows into 4 chunks: 251, 250, 250, 250 */
    int off[5] = {0};
    CHECK(ctx_chunk_offsets(1001, 4, off) == CTX_OK);
    CHECK(off[0] == 0 && off[1] == 251 && off[2] == 501 && off[3] == 751 && off[4] == 1001);
    CHECK(ctx_chunk_offsets(3, 4, off) == CTX_ERR_INVALID_ARG); /* empty chunks */

    /* the backward always needs a workspace; invalid sizes give 0 */
    CHECK(ctx_attn_workspace_size(1, 32760, 24, 24, 128, 8, 0) > 0);
    CHECK(ctx_attn_workspace_size(1, 1024, 24, 4, 256, 2, 0) > 0);
    CHECK(ctx_attn_workspace_size(1, 1024, 24, 5, 128, 2, 0) == 0); /* Hq % Hkv != 0 */
    CHECK(ctx_attn_workspace_size(1, 4, 1, 1, 64, 5, 0) == 0);      /* P > S */

    CHECK(ctx_exchange_padded_len(1001, 2, 2) == 1004);
    CHECK(ctx_exchange_padded_len(65536, 4, 2) == 65536);

    /* launch plan of the 24/4-head D=256 causal model at 1024 tokens */
    ctx_launch_plan_t plan;
    CHECK(ctx_attn_launch_plan(1, 1024, 24, 4, 256, 2, NULL, 1, &plan) == CTX_OK);
    CHECK(plan.fwd_ctas == 8 * 24 && plan.fwd_head_major == 1 && plan.bwd_group_split >= 1);
    CHECK(ctx_attn_launch_plan(1, 1024, 24, 4, 96, 2, NULL, 1, &plan) == CTX_ERR_UNSUPPORTED);

    const char* s = ctx_status_string(CTX_ERR_TIMEOUT);
    CHECK(s != NULL && strlen(s) > 0);

    /* invalid calls are refused before any launch */
    float lse[8];
    ctx_tensor_t t;
    memset(&t, 0, sizeof t);
    CHECK(ctx_attn_fwd(NULL, NULL, NULL, 1, NULL, CTX_LAYOUT_BSHD, 0, 0.0f, NULL, lse, NULL, 0,
                       CTX_FLAG_NONE, NULL) == CTX_ERR_INVALID_ARG);
    t.data = (void*)(uintptr_t)4096;
    t.B = 1; t.S = 8; t.H = 1; t.D = 96; /* head dimension 96 is not built */
    CHECK(ctx_attn_fwd(&t, &t, &t, 1, NULL, CTX_LAYOUT_BSHD, 0, 0.0f, &t, lse, NULL, 0,
                       CTX_FLAG_NONE, NULL) != CTX_OK);
    CHECK(ctx_seq_head_exchange(NULL, NULL, 2, 2, 0, CTX_LAYOUT_BSHD, NULL) == CTX_ERR_INVALID_ARG);

    if (failures == 0) printf("abi client ok\n");
    return failures == 0 ? 0 : 1;
}
