"""The bounded-wait path: a wait that cannot complete gives up after its limit, the kernel records
TQ_ERR_TIMEOUT in the device status word and returns, and the context stays usable.

The self-test kernel waits, with a 2 ms limit instead of the kernels' 4 s, on an mbarrier nothing
arrives on (kind 0) and on a grid barrier no CTA reaches (kind 1) - the two wait forms of the
decode, decode-step and prefill kernels.  Nothing faults, traps or hangs: both waits are bounded by
the global timer."""
import time

import numpy as np
import pytest
import torch

import ternary_weight_quantized_unpack_b300 as tq
from tq_testlib import LinearCase, check_tolerance

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_wait_runs_out(kind):
    assert tq.tq_device_status() == 0
    ws = torch.empty(256, dtype=torch.uint8, device="cuda") if kind == 1 else None
    t0 = time.perf_counter()
    tq.tq_selftest_wait(kind, 2_000_000, ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert tq.tq_device_status() == 6          # TQ_ERR_TIMEOUT, recorded by the kernel
    assert tq.tq_device_status() == 0          # the read cleared it
    assert elapsed < 2.0                       # the short limit, not the kernels' 4 s
    # the context is still usable: an ordinary call afterwards is correct and records nothing
    case = LinearCase(71, kind, 96, 512, 128, tq.TQ_PACK_2BIT, 2)
    y = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    y_ref, A = case.oracle()
    check_tolerance(y.cpu().numpy(), y_ref, A)
    assert np.all(np.isfinite(y.cpu().numpy()))
