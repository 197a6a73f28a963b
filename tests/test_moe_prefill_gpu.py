"""tq_moe_gemm (the expert layer at prefill sizes, grouped tensor-core GEMM) against the oracle.

The same checks as the decode-time expert layer: routing exact, gates within 1e-6, h within the bound
propagated through SwiGLU from the per-linear bound, the down + combine stage within the plain bound
on the GPU's own h, y end to end within the propagated bound.  The FP16 operands (x~ and the
transformed h) round at 2^-11 relative, inside the 1e-3 budget of each stage."""
import numpy as np
import pytest
import torch

import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from test_moe_gpu import MoeCase, check_case

pytestmark = pytest.mark.gpu


class GemmCase(MoeCase):
    def run(self):
        y, idx, gate, h = tq.tq_moe_gemm(self.gu, self.dn, self.E, self.topk, self.gu_codes, self.gu_scales,
                                         self.d_codes, self.d_scales, self.logits.cuda(), self.x_host.cuda(),
                                         want_h=True)
        torch.cuda.synchronize()
        assert tq.tq_device_status() == 0
        return y.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy(), h.cpu().numpy()


@pytest.mark.parametrize("packing", [tq.TQ_PACK_B3, tq.TQ_PACK_2BIT])
def test_moe_gemm_small_every_token(packing):
    """16 experts, top-4, H 256, F 128, 300 tokens: experts with 0 to ~150 tokens, partial row tiles."""
    case = GemmCase(41, 16, 256, 128, 64, packing, 300, topk=4)
    check_case(case, range(300))


def test_moe_gemm_full_size_sampled():
    """256 experts, top-8, hidden 2048, expert FFN 512, group 64, base-3, 256 tokens; 16 tokens checked
    (their 128 expert rows against the oracle), the routing of all 256 exactly."""
    m = inputs.MOE
    case = GemmCase(inputs.seed_of(3) + 256, m["E"], m["H"], m["F"], m["group"], m["packing"], 256, m["topk"])
    tokens = sorted(set([0, 255] + list(np.random.Generator(np.random.PCG64(7)).choice(256, 14, replace=False))))
    check_case(case, tokens)


def test_moe_gemm_matches_decode_layer_and_is_deterministic():
    """The prefill layer and the decode-time layer compute the same function: on the same inputs their
    outputs agree within the sum of their bounds (checked above against the oracle) - here to a
    relative 2e-3 of the output scale; two prefill calls are bit-identical."""
    case = GemmCase(43, 16, 256, 128, 64, tq.TQ_PACK_B3, 64, topk=4)
    y1, idx1, g1, _ = case.run()
    y2, idx2, g2, _ = case.run()
    assert np.array_equal(y1, y2) and np.array_equal(idx1, idx2)
    yd, idxd, gd, _ = MoeCase.run(case)
    assert np.array_equal(idx1, idxd)
    scale = np.abs(yd).max()
    assert np.max(np.abs(y1 - yd)) <= 2e-3 * scale
