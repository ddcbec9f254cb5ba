"""GPU: the failure path of a device wait, made to run out on purpose.

Every wait in the kernels is bounded; a wait that runs out records
UA_DEVICE_WAIT_TIMEOUT in the device status word and the kernel winds down
(the warps that share barriers stop together, the loads already issued are
waited for, and it returns).  The test hook ua_test_set_wait_limit gives the
decode kernel's main-loop waits 1 ns, so that the first wait that does not
find its data already there gives up: the tiny mixed batch then reports the
timeout, faults nothing and stops nothing, and the same call with the normal
limit right after matches the fp64 oracle.  No arrival is skipped and no
wait is unbounded; only the limit is short.
"""
import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 0x2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_varlen_attention_gb300 import build_lib
    build_lib.build()
    import paged_varlen_attention_gb300 as ua
    ua.load_library()
    ua.device_status()
    yield
    ua.set_test_wait_limit(0)
    assert ua.device_status() == 0


def test_short_wait_limit_reports_timeout_and_the_next_call_is_correct():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = W.config_batch(1, poison=True)           # decode kernel only
    dev = to_device(b)
    ua.set_test_wait_limit(1)
    try:
        out = torch.zeros_like(dev["q"])
        run_gpu(b, dev=dev, out=out)
        torch.cuda.synchronize()                 # the kernel returned; nothing faulted
        code = ua.device_status()
    finally:
        ua.set_test_wait_limit(0)
    assert code & WAIT_TIMEOUT, f"status {code:#x}: no wait ran out"
    assert ua.device_status() == 0               # read and cleared
    got = run_gpu(b, dev=dev)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "after a timed-out call")
    assert ua.device_status() == 0
