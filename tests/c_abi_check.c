/* Plain-C caller of libssd.so (no Python, no torch): argument errors come
 * back synchronously before anything touches a GPU, so this runs on a
 * machine without one.  Compiled and run by tests/test_abi_host.py. */
#include <stdio.h>
#include <string.h>

#include "ssd.h"

#define EXPECT(call, want)                                                        \
    do {                                                                          \
        const ssd_status got_ = (call);                                           \
        if (got_ != (want)) {                                                     \
            printf("FAIL line %d: %s -> %d (%s), want %d\n", __LINE__, #call,      \
                   (int)got_, ssd_status_string(got_), (int)(want));              \
            return 1;                                                             \
        }                                                                         \
    } while (0)

int main(void) {
    /* fake, 16-byte aligned device addresses: the checks reject the call first */
    const void *x = (const void *)0x1000, *B = (const void *)0x2000, *C = (const void *)0x3000;
    const float *dt = (const float *)0x4000, *A = (const float *)0x5000;
    void *y = (void *)0x6000;
    const int cu_bad[3] = {0, 5, 3};
    const int cu_start[2] = {1, 5};
    ssd_dt_transform tr = {NULL, 1, 0.5f, 0.1f}; /* dt_min > dt_max */

    if (strncmp(ssd_status_string(SSD_OK), "SSD_OK", 6) != 0) return 1;
    EXPECT(ssd_scan_fwd(NULL, dt, A, B, C, NULL, SSD_BF16, 1, 256, 4, 64, 64, 1, 64, NULL, y,
                        NULL, NULL, 0, 0),
           SSD_ERR_INVALID_ARG);
    EXPECT(ssd_scan_fwd(x, dt, A, B, C, NULL, SSD_BF16, 1, 256, 6, 64, 64, 4, 64, NULL, y, NULL,
                        NULL, 0, 0),
           SSD_ERR_INVALID_ARG);
    EXPECT(ssd_scan_fwd(x, dt, A, B, C, NULL, SSD_BF16, 1, 256, 4, 64, 512, 1, 64, NULL, y,
                        NULL, NULL, 0, 0),
           SSD_ERR_UNSUPPORTED);
    EXPECT(ssd_scan_fwd_dt(SSD_ALGO_AUTO, x, dt, A, B, C, NULL, &tr, SSD_BF16, 1, 256, 4, 64,
                           64, 1, 64, NULL, y, NULL, NULL, 0, 0),
           SSD_ERR_INVALID_ARG);
    EXPECT(ssd_scan_fwd_varlen(SSD_ALGO_AUTO, x, dt, A, B, C, NULL, NULL, NULL, SSD_BF16, 2,
                               cu_bad, (const int *)0x7000, 4, 64, 64, 1, 64, NULL, y, NULL,
                               NULL, 0, 0),
           SSD_ERR_INVALID_ARG);
    EXPECT(ssd_scan_fwd_varlen(SSD_ALGO_AUTO, x, dt, A, B, C, NULL, NULL, NULL, SSD_BF16, 1,
                               cu_start, (const int *)0x7000, 4, 64, 64, 1, 64, NULL, y, NULL,
                               NULL, 0, 0),
           SSD_ERR_INVALID_ARG);
    EXPECT(ssd_state_update_fused((void *)0x8000, SSD_BF16, x, dt, A, B, C, NULL, NULL, NULL,
                                  SSD_F32, 2, 4, 16, 16, 1, y, 0),
           SSD_ERR_UNSUPPORTED);
    if (ssd_scan_workspace_bytes(0, 256, 4, 64, 64, 1, 64) != (size_t)-1) return 1;
    if (ssd_scan_fused_workspace_bytes(1, 256, 4, 64, 64, 1, 64, SSD_F32, 1) != 0) return 1;
    EXPECT(ssd_debug_inject_fault((ssd_fault)9, 0), SSD_ERR_INVALID_ARG);
    EXPECT(ssd_debug_inject_fault(SSD_FAULT_NONE, 0), SSD_OK);
    if (ssd_scan_kernel_launches(1, 256, 6, 64, 64, 4, 64, SSD_BF16) != -1) return 1;
    /* fp8 inputs: the widened copies need a workspace; decode takes no fp8 */
    EXPECT(ssd_scan_fwd(x, dt, A, B, C, NULL, SSD_FP8_E4M3, 1, 256, 4, 64, 64, 1, 64, NULL, y,
                        NULL, NULL, 0, 0),
           SSD_ERR_WORKSPACE);
    EXPECT(ssd_state_update((float *)0x8000, x, dt, A, B, C, NULL,
                            SSD_FP8_E4M3, 2, 4, 16, 16, 1, y, 0),
           SSD_ERR_UNSUPPORTED);
    EXPECT(ssd_fp8_e4m3_to_bf16(NULL, y, 16, 0), SSD_ERR_INVALID_ARG);
    EXPECT(ssd_fp8_e4m3_to_bf16(NULL, NULL, 0, 0), SSD_OK);
    /* the exchange of a sequence split over GPUs */
    EXPECT(ssd_range_log_decay(NULL, A, NULL, 1, 16, 4, (float *)0x9000, 0), SSD_ERR_INVALID_ARG);
    EXPECT(ssd_chain_states((const float *)0x9000, NULL, NULL, 2, 1, 4, 8, 8, (float *)0xa000, 0),
           SSD_ERR_INVALID_ARG);
    printf("c abi ok\n");
    return 0;
}
