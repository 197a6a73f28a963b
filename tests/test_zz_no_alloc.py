"""tq_gemv_noalloc (scratch in the library's fixed device array) against tq_gemv (caller workspace):
two calls in a row on the shared scratch, each within the tolerance of the workspace path and of the
oracle; oversize shapes are refused before any launch."""
import numpy as np
import pytest
import torch

import ternary_weight_quantized_unpack_b300 as tq
from tq_testlib import LinearCase, check_tolerance, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("packing", [tq.TQ_PACK_B3, tq.TQ_PACK_2BIT])
def test_noalloc_matches_workspace_gemv(packing):
    cases = [LinearCase(41, 1, 640, 2560, 128, packing, 3), LinearCase(41, 2, 640, 2560, 128, packing, 3)]
    # two calls in a row through the same scratch, then the workspace path
    y_na = [tq.tq_gemv_noalloc(c.desc, c.codes, c.scales, c.x) for c in cases]
    y_ws = [tq.tq_gemv(c.desc, c.codes, c.scales, c.x) for c in cases]
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    rows = sample_rows(640, 64, seed=3)
    for c, a, b in zip(cases, y_na, y_ws):
        y_ref, A = c.oracle(rows)
        a_np, b_np = a.cpu().numpy(), b.cpu().numpy()
        check_tolerance(a_np[:, rows], b_np[:, rows], A, what="noalloc vs tq_gemv")
        check_tolerance(a_np[:, rows], y_ref, A, what="noalloc vs oracle")
        assert np.array_equal(a_np, b_np)  # same kernels, same plan: identical


def test_noalloc_rejects_oversize():
    d = tq.desc(64, 32768, 128, tq.TQ_PACK_2BIT)  # K = 32768 at batch 16 needs more than 1 MiB
    assert tq.tq_gemv_workspace_bytes(d, 16) > 1 << 20
    t = torch.empty(16, dtype=torch.int32, device="cuda")  # never read: the size check comes first
    with pytest.raises(tq.TQError) as err:
        tq.tq_gemv_noalloc(d, t, t, torch.empty((16, 8), dtype=torch.bfloat16, device="cuda"))
    assert err.value.status == 7  # TQ_ERR_WORKSPACE
