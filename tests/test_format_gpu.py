"""tq_pack / tq_unpack / tq_fwht on the GPU against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs

pytestmark = pytest.mark.gpu

PACKINGS = [tq.TQ_PACK_B3, tq.TQ_PACK_2BIT]


@pytest.mark.parametrize("packing", PACKINGS)
@pytest.mark.parametrize("N,K", [(1, 1), (3, 19), (5, 21), (2, 80), (7, 128), (33, 1000), (64, 5120), (9, 17408)])
def test_pack_unpack_bit_exact(packing, N, K):
    t = inputs.trits(7, N + K, N, K)
    d = tq.desc(N, K, 128, packing)
    codes = tq.tq_pack(d, t.cuda())
    ref = O.pack(t.numpy(), packing)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), ref)
    back, bad = tq.tq_unpack(d, codes)
    assert int(bad.item()) == 0
    assert torch.equal(back.cpu(), t)
    assert tq.tq_device_status() == 0


@pytest.mark.parametrize("packing", PACKINGS)
def test_pack_full_size_layer(packing):
    """The largest decode matrix (FFN 17408 x 5120), all words compared."""
    N, K = 17408, 5120
    t = inputs.trits(2000, 4, N, K)
    codes = tq.tq_pack(tq.desc(N, K, 128, packing), t.cuda())
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), O.pack(t.numpy(), packing))


@pytest.mark.parametrize("packing", PACKINGS)
def test_unpack_counts_invalid_words(packing):
    N, K = 6, 100
    t = inputs.trits(3, 1, N, K).numpy()
    codes = O.pack(t, packing)
    if packing == tq.TQ_PACK_B3:
        codes[0, 1] = 3 ** 20
        codes[2, 3] = 0xFFFFFFFF
        codes[5, 0] = 3 ** 20 + 12345
    else:
        codes[0, 1] = 0xFFFFFFFF
        codes[4, 2] = 0x55555557
        codes[5, 7] = 0xC0000000  # a padding word, still validated
    n_bad_ref = O.unpack(codes, K, packing)[1]
    assert n_bad_ref == 3
    dev = torch.from_numpy(codes.view(np.int32)).cuda()
    back, bad = tq.tq_unpack(tq.desc(N, K, 128, packing), dev)
    assert int(bad.item()) == n_bad_ref
    assert tq.tq_device_status() == 4   # TQ_ERR_INVALID_CODE
    assert tq.tq_device_status() == 0  # cleared by the read


def test_pack_rejects_out_of_range_trit():
    t = torch.zeros((2, 40), dtype=torch.int8)
    t[1, 7] = 2
    tq.tq_pack(tq.desc(2, 40), t.cuda())
    assert tq.tq_device_status() == 4


@pytest.mark.parametrize("rows,K", [(1, 128), (3, 1024), (16, 5120), (2, 17408)])
def test_fwht_fp32(rows, K):
    x = inputs.activations(5, rows, rows, K, outlier_frac=0.005)
    out = tq.tq_fwht(x.cuda()).cpu().numpy().astype(np.float64)
    xr = x.float().numpy().astype(np.float64)
    ref = O.block_fwht(xr, 128)
    # 7 butterfly stages and one scaling in fp32: error <= 8 * 2^-24 * sum|x_block| / sqrt(128)
    blk_abs = np.repeat(np.abs(xr).reshape(rows, -1, 128).sum(axis=2), 128, axis=1) / math.sqrt(128)
    assert np.all(np.abs(out - ref) <= 8 * 2.0 ** -24 * blk_abs + 1e-30)


def test_fwht_fp16_and_range():
    x = inputs.activations(6, 0, 4, 1024)
    out = tq.tq_fwht(x.cuda(), out_fp16=True).cpu().numpy().astype(np.float64)
    ref = O.block_fwht(x.float().numpy(), 128)
    assert np.all(np.abs(out - ref) <= 2.0 ** -11 * np.abs(ref) + 8 * 2.0 ** -24 * 40 + 2.0 ** -25)
    assert tq.tq_device_status() == 0
    big = torch.full((1, 128), 60000.0, dtype=torch.bfloat16)
    tq.tq_fwht(big.cuda(), out_fp16=True)   # first output is sqrt(128) * 60000: beyond FP16
    assert tq.tq_device_status() == 8
