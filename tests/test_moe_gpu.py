"""tq_moe_route / tq_moe_gemv against the oracle.

Routing indices are compared bit for bit and gates to 1e-6.  The expert outputs are checked stage by
stage: h = silu(g) * u against the oracle's h with the per-output bound propagated through SwiGLU;
the down projection + combine against the oracle applied to the GPU's own h and gates (the plain
1e-3 * A + 1e-5 bound); and y end to end against the oracle with the bound propagated from h."""
import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import check_tolerance, moe_bounds

pytestmark = pytest.mark.gpu


class MoeCase:
    def __init__(self, seed, E, H, F, group, packing, T, topk=8, fwht_block=128):
        self.seed, self.E, self.H, self.F, self.group, self.packing = seed, E, H, F, group, packing
        self.T, self.topk, self.fwht_block = T, topk, fwht_block
        self.gu = tq.desc(2 * F, H, group, packing, fwht_block)
        self.dn = tq.desc(H, F, group, packing, fwht_block)
        P_H, P_F = O.row_pitch_words(H, packing), O.row_pitch_words(F, packing)
        dev = "cuda"
        self.gu_codes = torch.empty((E, 2 * F, P_H), dtype=torch.int32, device=dev)
        self.d_codes = torch.empty((E, H, P_F), dtype=torch.int32, device=dev)
        self.gu_scales = torch.empty((E, 2 * F, H // group), dtype=torch.float16, device=dev)
        self.d_scales = torch.empty((E, H, F // group), dtype=torch.float16, device=dev)
        for e in range(E):
            tq.tq_pack(self.gu, inputs.trits(seed, 4 * e, 2 * F, H, device=dev), codes=self.gu_codes[e])
            tq.tq_pack(self.dn, inputs.trits(seed, 4 * e + 2, H, F, device=dev), codes=self.d_codes[e])
            self.gu_scales[e] = inputs.scales(seed, 4 * e + 1, 2 * F, H // group, device=dev)
            self.d_scales[e] = inputs.scales(seed, 4 * e + 3, H, F // group, device=dev)
        self.logits = inputs.router_logits(seed, 0, T, E)
        self.x_host = inputs.activations(seed, 1, T, H)

    def host_expert(self, e):
        H, F, G = self.H, self.F, self.group
        gt = inputs.trits(self.seed, 4 * e, 2 * F, H).numpy()
        dt = inputs.trits(self.seed, 4 * e + 2, H, F).numpy()
        gs = inputs.scales(self.seed, 4 * e + 1, 2 * F, H // G).numpy()
        ds = inputs.scales(self.seed, 4 * e + 3, H, F // G).numpy()
        return O.pack(gt, self.packing), gs, O.pack(dt, self.packing), ds, O.dequant(dt, ds, G)

    def run(self):
        y, idx, gate, h = tq.tq_moe_gemv(self.gu, self.dn, self.E, self.topk, self.gu_codes, self.gu_scales,
                                         self.d_codes, self.d_scales, self.logits.cuda(), self.x_host.cuda(),
                                         want_h=True)
        torch.cuda.synchronize()
        assert tq.tq_device_status() == 0
        return y.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy(), h.cpu().numpy()


def check_case(case: MoeCase, tokens):
    y, idx, gate, h = case.run()
    idx_ref, gate_ref = O.moe_route(case.logits.numpy(), case.topk)
    assert np.array_equal(idx, idx_ref), "routing indices differ"
    assert np.max(np.abs(gate - gate_ref)) <= 1e-6
    tokens = np.asarray(tokens)
    experts = sorted(set(idx_ref[tokens].reshape(-1).tolist()))
    host = {e: case.host_expert(e) for e in experts}
    out = O.moe_layer(case.logits.numpy()[tokens], case.x_host.float().numpy()[tokens], None, None, None, None,
                      case.H, case.F, case.group, case.packing, case.topk, case.fwht_block,
                      experts={e: host[e][:4] for e in experts})
    hb, A_e2e, extra = moe_bounds(out, {e: host[e][4] for e in experts}, case.fwht_block)
    # h: per-output bound propagated through silu(g) * u
    hg = h[tokens]
    assert np.all(np.abs(hg - out["h"]) <= hb), f"h worst ratio {np.max(np.abs(hg - out['h']) / hb):.3f}"
    # down + combine on the GPU's own h and gates: plain bound
    y_loc, A_loc = O.moe_down_from_h(hg, idx[tokens], gate[tokens].astype(np.float64),
                                     {e: host[e][2:4] for e in experts}, case.F, case.group, case.packing,
                                     case.fwht_block)
    check_tolerance(y[tokens], y_loc, A_loc, what="y (down stage)")
    # end to end: the down bound plus the h bound carried through FWHT and |W_d|, plus gate error
    check_tolerance(y[tokens], out["y"], A_e2e, extra=extra, what="y (end to end)")


@pytest.mark.parametrize("T", list(inputs.MOE["tokens"]))
def test_moe_expert_layer(T):
    """256 experts, top-8, hidden 2048, expert FFN 512, group 64, base-3, tokens 1 / 8 / 64."""
    m = inputs.MOE
    case = MoeCase(inputs.seed_of(3) + T, m["E"], m["H"], m["F"], m["group"], m["packing"], T, m["topk"])
    check_case(case, list(range(T)))   # every token


@pytest.mark.parametrize("packing", [tq.TQ_PACK_B3, tq.TQ_PACK_2BIT])
def test_moe_small(packing):
    case = MoeCase(31, 16, 256, 128, 64, packing, 5, topk=4)
    check_case(case, range(5))


def test_moe_route_ties_and_order():
    logits = np.random.Generator(np.random.PCG64(0)).standard_normal((6, 256)).astype(np.float32)
    logits[1, [9, 3, 200]] = 5.0
    logits[2, :] = -1.5
    logits[3, 255] = 30.0
    idx, gate = tq.tq_moe_route(torch.from_numpy(logits).cuda(), 8)
    idx_ref, gate_ref = O.moe_route(logits, 8)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert np.max(np.abs(gate.cpu().numpy() - gate_ref)) <= 1e-6
    assert idx_ref[1, :3].tolist() == [3, 9, 200] and idx_ref[2].tolist() == list(range(8))


def test_moe_repeat_and_graph_replay_deterministic():
    """The fused combine is done by whichever CTA finishes a token's last slot, adding the slots in
    slot order: repeated calls (the per-token counts reset themselves) and a CUDA-graph replay give
    bit-identical outputs.  Also a batch with more tokens than shared-memory assignments would not
    matter here (T = 64)."""
    m = inputs.MOE
    case = MoeCase(inputs.seed_of(3) + 99, m["E"], m["H"], m["F"], m["group"], m["packing"], 64, m["topk"])
    logits, x = case.logits.cuda(), case.x_host.cuda()
    ws = torch.empty(tq.tq_moe_workspace_bytes(64, m["E"], m["topk"], m["H"], m["F"]), dtype=torch.uint8, device="cuda")
    y = torch.empty((64, m["H"]), dtype=torch.float32, device="cuda")
    idx = torch.empty((64, m["topk"]), dtype=torch.int32, device="cuda")
    gate = torch.empty((64, m["topk"]), dtype=torch.float32, device="cuda")

    def call():
        tq.tq_moe_gemv(case.gu, case.dn, m["E"], m["topk"], case.gu_codes, case.gu_scales, case.d_codes,
                       case.d_scales, logits, x, topk_idx=idx, topk_gate=gate, y=y, workspace=ws)

    call()
    torch.cuda.synchronize()
    first = y.clone()
    for _ in range(3):
        y.fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        assert torch.equal(y, first)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    assert torch.equal(y, first)
