// placeholder: tensor-core path not built yet
#include "launch.h"
SsdTcPlan ssd_tc_plan(int, int, int, int, int, int, int) { SsdTcPlan p{}; p.supported = false; p.launches = 1; return p; }
cudaError_t ssd_launch_scan_tc(const SsdTcPlan &, const void *, const float *, const float *,
                               const void *, const void *, const float *, const float *, void *,
                               float *, int, int, int, int, int, int, void *, unsigned int *,
                               cudaStream_t) { return cudaErrorNotSupported; }
