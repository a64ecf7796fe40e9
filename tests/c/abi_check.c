/*
 * A plain C99 user of the qgemm C-ABI: includes the header, takes the address
 * of every entry point (so each must link), and calls the host-only ones.
 * Built and run by tests/test_abi.py; no GPU is needed.
 */
#include <stdio.h>
#include <string.h>

#include "qgemm.h"

typedef void (*any_fn)(void);

int main(void)
{
    const any_fn fns[] = {
        (any_fn)qgemm_status_string, (any_fn)qgemm_packed_bytes, (any_fn)qgemm_pack_weights,
        (any_fn)qgemm_plan, (any_fn)qgemm_plan_workspace_bytes, (any_fn)qgemm_plan_bind,
        (any_fn)qgemm_run, (any_fn)qgemm_run_multi, (any_fn)qgemm_plan_destroy,
        (any_fn)qgemm_plan_set_pdl, (any_fn)qgemm_plan_route, (any_fn)qgemm_route_name,
        (any_fn)qgemm_launch_count, (any_fn)qgemm_device_status, (any_fn)qgemm_selftest_timeout,
        (any_fn)qgemm_pair_packed_bytes, (any_fn)qgemm_pack_pair, (any_fn)qgemm_plan_set_epilogue,
        (any_fn)qgemm_run_ex, (any_fn)qgemm_plan_force_route, (any_fn)qgemm_run_noalloc,
        (any_fn)qgemm_plan_set_tensor_scale,
    };
    for (size_t i = 0; i < sizeof fns / sizeof fns[0]; ++i)
        if (!fns[i])
            return 10;
    if (strcmp(qgemm_status_string(QGEMM_OK), "ok") != 0)
        return 11;
    if (qgemm_packed_bytes(256, 512, QGEMM_INT4) != (size_t)2 * 8 * 4352)
        return 12;
    if (qgemm_packed_bytes(256, 512, QGEMM_FP8) != (size_t)2 * 8 * 8448)
        return 13;
    if (qgemm_pair_packed_bytes(8, 512, QGEMM_INT5) != qgemm_packed_bytes(16, 512, QGEMM_INT5))
        return 14;
    if (qgemm_packed_bytes(16, 100, QGEMM_INT4) != 0)
        return 15;
    if (qgemm_plan_destroy(NULL) != QGEMM_OK)
        return 16;
    if (qgemm_run(NULL, NULL, 1, NULL, NULL) != QGEMM_ERR_INVALID_ARG)
        return 17;
    if (strcmp(qgemm_route_name(-1), "none") != 0)
        return 18;
    printf("abi ok\n");
    return 0;
}
