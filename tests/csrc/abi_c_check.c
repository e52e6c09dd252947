/* Plain C99 client of the q4adamw C ABI (no GPU calls): the header must
 * compile as C, the library must link, and the host-only entry points must
 * answer as include/q4adamw.h states.  Prints "ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "q4adamw.h"

#define CHECK(c)                                                 \
    do {                                                         \
        if (!(c)) {                                              \
            printf("failed: %s (line %d)\n", #c, __LINE__);       \
            return 1;                                            \
        }                                                        \
    } while (0)

int main(void) {
    q4adamw_tensor_t t;
    int64_t q = 0, s = 0, tot = 0, ws = 0;
    float levels[16], thr[15];
    q4adamw_header_t h;

    CHECK(q4adamw_version() == Q4ADAMW_STATE_FORMAT);
    CHECK(strcmp(q4adamw_strerror(Q4_OK), "ok") == 0);
    CHECK(q4adamw_strerror(12345) != NULL);

    memset(&t, 0, sizeof t);
    t.numel = 128 * 1000;
    t.rows = 1;
    CHECK(q4adamw_state_bytes(&t, 1, Q4_RECIPE_ZIP_SR, &q, &s, &tot) == Q4_OK);
    CHECK(q == 128 * 1000 && s == 8 * 1000 && tot == q + s);           /* 1.0625 B/param */
    CHECK(q4adamw_workspace_bytes(&t, 1, Q4_RECIPE_ZE_EDEN, &ws) == Q4_OK && ws > 0 && ws % 256 == 0);
    CHECK(q4adamw_workspace_bytes(&t, 1, 99, &ws) == Q4_ERECIPE);
    t.numel = -1;
    CHECK(q4adamw_workspace_bytes(&t, 1, Q4_RECIPE_ZIP_SR, &ws) == Q4_ESHAPE);

    CHECK(q4adamw_codebook(0, levels, thr) == Q4_OK);
    CHECK(levels[0] == -1.0f && levels[7] == 0.0f && levels[15] == 1.0f);
    CHECK(q4adamw_codebook(1, levels, NULL) == Q4_OK && levels[0] == 0.0f && levels[15] == 1.0f);
    CHECK(q4adamw_codebook(2, levels, NULL) == Q4_OK && levels[0] > 0.0f);
    CHECK(q4adamw_codebook(5, levels, thr) == Q4_ERECIPE);

    memset(&h, 0, sizeof h);
    CHECK(q4adamw_header_check(&h, Q4_RECIPE_ZIP_SR) == Q4_EVERSION);
    CHECK(q4adamw_header_check(NULL, Q4_RECIPE_ZIP_SR) == Q4_EINVAL);

    /* validation happens before any device work: bad arguments never reach CUDA */
    CHECK(q4adamw_step(NULL, -1, 1e-3f, 0.9f, 0.999f, 1e-8f, 0.1f, 1, 0, 0, 0, NULL, 0, NULL) == Q4_EINVAL);
    CHECK(q4adamw_step_clip(NULL, 0, 1e-3f, 0.9f, 0.999f, 1e-8f, 0.1f, 1, 0, 0, 0, 0.0f, NULL, NULL, 0, NULL) ==
          Q4_EINVAL);
    CHECK(q4adamw_draws(0, 0, 0, 0, 0, 4, NULL, NULL) == Q4_EINVAL);
    CHECK(q4adamw_set_stage_wait_limit(-1) == Q4_EINVAL);
    CHECK(q4adamw_set_stage_wait_limit(1000) == Q4_OK && q4adamw_set_stage_wait_limit(0) == Q4_OK);
    CHECK(q4adamw_step_noalloc_status(NULL, NULL) == Q4_EINVAL);
    printf("ok\n");
    return 0;
}
