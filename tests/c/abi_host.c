/* A plain C caller of the library's host-only entry points: the header
 * compiles as C, the symbols link, and configuration errors come back as
 * status codes with a message (no GPU work is launched). */
#include <stdio.h>
#include <string.h>

#include "ep.h"

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                                \
        }                                                            \
    } while (0)

int main(void) {
    CHECK(strstr(ep_version(), "sm_103a") != NULL);
    CHECK(strcmp(ep_status_name(EP_ERR_CAPACITY), "EP_ERR_CAPACITY") == 0);
    /* one message: 16-byte header, H codes, H/128 scales, rounded to 16 */
    CHECK(ep_ll_message_bytes(7168) == 7408);
    CHECK(ep_fp8_row_bytes(7168) == 7392);
    CHECK(ep_ll_size_hint(128, 7168, 16, 256) > 0);
    CHECK(ep_ll_size_hint(0, 7168, 16, 256) == 0);
    /* E not a multiple of R is refused before any CUDA call */
    ep_config bad = {3, 8, 2, 4, 128, 2, 1};
    ep_ctx* ctx = NULL;
    CHECK(ep_ctx_create(&bad, &ctx) == EP_ERR_INVALID_ARG);
    CHECK(ctx == NULL);
    CHECK(strlen(ep_last_error()) > 0);
    CHECK(ep_ctx_check(NULL, NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_ctx_set_expert_alignment(NULL, 8) == EP_ERR_INVALID_ARG);
    printf("c abi ok\n");
    return 0;
}
