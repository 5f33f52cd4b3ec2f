/* Host-only use of libccl.so from plain C (no GPU needed): the planner, the
 * settings and the step-mode traffic counters, and a call rejected by argument
 * validation before anything is launched.  Prints "c abi host ok" and exits 0
 * when every check holds. */
#include <stdio.h>
#include <string.h>

#include "ccl.h"

static int failures = 0;

static void check(int ok, const char *what)
{
    if (!ok) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

int main(void)
{
    size_t off[3], len[3];
    int32_t tab[2 * 3 * 4 * 3];
    unsigned long long sent[4];
    ccl_config_t cfg;
    int i;

    check(ccl_version() >= 10100, "version");

    /* 10 elements over 3 ranks: the first 10 mod 3 = 1 chunk takes the extra one */
    check(ccl_plan_chunks(10, 3, off, len) == CCL_OK, "plan_chunks");
    check(off[0] == 0 && off[1] == 4 && off[2] == 7 && len[0] == 4 && len[1] == 3 && len[2] == 3, "partition");

    /* ReduceScatter step 0: rank i sends chunk i and adds chunk i-1 arriving from rank i-1 */
    check(ccl_plan_ring_schedule(4, tab) == CCL_OK, "plan_ring_schedule");
    for (i = 0; i < 4; ++i)
        check(tab[i * 3] == i && tab[i * 3 + 1] == (i + 3) % 4 && tab[i * 3 + 2] == (i + 3) % 4, "schedule step 0");

    memset(&cfg, 0xff, sizeof cfg);
    check(ccl_get_config(&cfg) == CCL_OK, "get_config");
    check(cfg.mode_override == -1 && cfg.trace == 0 && cfg.check == 0 && cfg.host_path == CCL_HOST_PATH_STAGED &&
              cfg.default_bucket_bytes == CCL_DEFAULT_BUCKET_BYTES,
          "default settings");
    check(ccl_set_host_path(CCL_HOST_PATH_DIRECT) == CCL_OK && ccl_get_config(&cfg) == CCL_OK &&
              cfg.host_path == CCL_HOST_PATH_DIRECT,
          "direct host path");
    check(ccl_set_host_path(7) == CCL_ERR_INVALID_ARG && ccl_set_host_path(CCL_HOST_PATH_STAGED) == CCL_OK,
          "host path setter validates");
    check(ccl_set_mode_override(CCL_MODE_STEP) == CCL_OK, "force step mode");
    check(ccl_set_default_bucket_bytes(1u << 20) == CCL_OK, "bucket size");
    check(ccl_get_config(&cfg) == CCL_OK && cfg.mode_override == CCL_MODE_STEP &&
              cfg.default_bucket_bytes == (1u << 20),
          "settings changed");
    check(ccl_set_mode_override(5) == CCL_ERR_INVALID_ARG, "bad mode rejected");
    check(ccl_set_default_bucket_bytes(3) == CCL_ERR_INVALID_ARG, "bad bucket size rejected");
    check(ccl_set_mode_override(-1) == CCL_OK && ccl_set_default_bucket_bytes(0) == CCL_OK, "settings restored");
    check(ccl_get_config(&cfg) == CCL_OK && cfg.mode_override == -1 &&
              cfg.default_bucket_bytes == CCL_DEFAULT_BUCKET_BYTES,
          "settings back to defaults");

    check(ccl_step_sent(4, sent, 1) == CCL_OK && sent[0] == 0 && sent[3] == 0, "no step traffic yet");
    check(ccl_step_sent(0, sent, 1) == CCL_ERR_INVALID_ARG, "step_sent validates nranks");

    /* rejected before any launch: no ranks */
    check(ccl_allreduce(NULL, NULL, 0, 16, CCL_FP32, CCL_SUM, CCL_MODE_FUSED, 0) == CCL_ERR_INVALID_ARG,
          "allreduce validation");
    check(ccl_status_string(CCL_ERR_OVERLAP) != NULL, "status string");

    if (failures)
        return 1;
    printf("c abi host ok\n");
    return 0;
}
