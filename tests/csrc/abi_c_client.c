/*
 * A plain C99 client of include/pod.h: checks that the header compiles as C
 * and that a host-only plan can be made, inspected, switched and destroyed
 * through the ABI alone (no device memory is touched: num_sms is given and
 * no workspace is bound). Prints "ok" and returns 0 on success.
 */
#include <stdio.h>
#include <string.h>

#include "pod.h"

#define CHECK(call)                                                              \
    do {                                                                         \
        pod_status st_ = (call);                                                 \
        if (st_ != POD_OK) {                                                     \
            printf("%s -> %d: %s\n", #call, (int)st_, pod_last_error());         \
            return 1;                                                            \
        }                                                                        \
    } while (0)

int main(void)
{
    /* prefill: one request, 5 queries over 9 keys; decode: two requests */
    const int32_t p_q[2] = {0, 5}, p_kv[2] = {0, 3}, p_idx[3] = {2, 0, 1}, p_last[1] = {1};
    const int32_t d_q[3] = {0, 1, 2}, d_kv[3] = {0, 2, 3}, d_idx[3] = {3, 4, 5};
    const int32_t d_last[2] = {4, 2};
    pod_handle h = NULL;
    size_t need = 0;
    CHECK(pod_plan(p_q, p_kv, p_idx, p_last, 1, 4, d_q, d_kv, d_idx, d_last, 2, 6,
                   8, 2, 64, 4, 1, -1, 0.0f, POD_BF16, 0, 8, NULL, 0, NULL, &h, &need));
    if (!h || need == 0 || pod_workspace_size(h) != need) {
        printf("bad workspace size %zu\n", need);
        return 1;
    }
    int32_t kvl[2] = {0, 0};
    int64_t n = 0;
    CHECK(pod_plan_table(h, 6, kvl, 2, &n));
    if (n != 1 || kvl[0] != 9) {
        printf("prefill kv_len %d (count %lld), want 9\n", kvl[0], (long long)n);
        return 1;
    }
    CHECK(pod_plan_table(h, 7, kvl, 2, &n));
    if (n != 2 || kvl[0] != 8 || kvl[1] != 2) {
        printf("decode kv_len %d %d, want 8 2\n", kvl[0], kvl[1]);
        return 1;
    }
    CHECK(pod_plan_set_kv_layout(h, 1, 0));
    CHECK(pod_plan_set_logits_transform(h, 30.0f, NULL));
    CHECK(pod_plan_set_logits_transform(h, 0.0f, NULL));
    CHECK(pod_plan_set_prefill_mask(h, NULL, 0));
    CHECK(pod_plan_set_rope(h, 1.0f, 10000.0f));
    if (pod_workspace_size(h) <= need) {
        printf("RoPE did not grow the workspace\n");
        return 1;
    }
    CHECK(pod_plan_set_rope(h, 0.0f, 0.0f));
    if (pod_plan_set_kv_layout(h, 2, 0) != POD_ERR_INVALID_ARG || strlen(pod_last_error()) == 0) {
        printf("layout 2 was not refused\n");
        return 1;
    }
    /* an invalid page table is refused with a message, not a crash */
    const int32_t bad_idx[3] = {2, 0, 7};
    pod_handle h2 = NULL;
    if (pod_plan(p_q, p_kv, bad_idx, p_last, 1, 4, NULL, NULL, NULL, NULL, 0, 0, 8, 2, 64, 4, 1,
                 -1, 0.0f, POD_BF16, 0, 8, NULL, 0, NULL, &h2, NULL) != POD_ERR_INVALID_ARG ||
        h2 != NULL) {
        printf("out-of-pool page index was not refused\n");
        return 1;
    }
    CHECK(pod_destroy(h));
    printf("ok\n");
    return 0;
}
