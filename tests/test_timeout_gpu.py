"""The bounded device-side waits, made to run out on purpose without any
GPU fault: a host-set test hook makes one barrier of the tensor-core scan
kernel wait for an arrival that never comes, so the wait for it ends at a
short limit; the CTA then lets its issued copies and tensor-core products
complete, frees its tensor memory and exits.
The host reads SSD_ERR_TIMEOUT from the device error word, and the next call
on the same context is correct."""
import pytest

import state_space_model_chunked_gb300 as ssd
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, rel, scan_on_gpu, scan_oracle

pytestmark = pytest.mark.gpu

TC = 2
TIMEOUT = 4   # SSD_ERR_TIMEOUT


@pytest.mark.parametrize("L", [128, 640])
def test_withheld_signal_times_out_then_next_call_is_correct(L):
    inp = gen.scan_inputs(1, L, 2, 64, 128, 1, "bf16", seed=4 + L, random_init=True)
    ssd.last_device_error()                           # start from a clear error word
    ssd.debug_inject_fault(ssd.FAULT_WITHHOLD_SIGNAL, 2_000_000)   # 2 ms limit
    try:
        scan_on_gpu(inp, "bf16", 128, TC)             # outputs undefined
    finally:
        ssd.debug_inject_fault(ssd.FAULT_NONE, 0)
    with pytest.raises(ssd.SsdError) as err:
        ssd.last_device_error()
    assert err.value.code == TIMEOUT
    ssd.last_device_error()                           # read once, then clear
    y, f = scan_on_gpu(inp, "bf16", 128, TC)
    yr, fr = scan_oracle(inp)
    assert rel(y, yr) <= TOL["bf16"] and rel(f, fr) <= TOL["bf16"]
    ssd.last_device_error()
