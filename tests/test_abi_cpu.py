"""The C ABI without a GPU: the library loads, exports every declared entry point, computes sizes,
and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tq.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = tq.lib()
    names = declared_symbols()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, f"declared in tq.h but not exported: {missing}"
    # and the binding wraps each one under the same name
    assert all(hasattr(tq, n) for n in names), [n for n in names if not hasattr(tq, n)]


@pytest.mark.parametrize("packing", [tq.TQ_PACK_B3, tq.TQ_PACK_2BIT, tq.TQ_PACK_3BIT])
@pytest.mark.parametrize("K", [1, 20, 21, 128, 1000, 1024, 2048, 512, 5120, 17408])
def test_sizes_match_oracle(packing, K):
    for N in (1, 7, 1024):
        for group in (64, 128):
            d = tq.desc(N, K, group, packing)
            assert tq.tq_row_pitch_words(d) == O.row_pitch_words(K, packing)
            assert tq.tq_packed_bytes(d) == O.packed_bytes(N, K, packing)
            assert tq.tq_scale_bytes(d) == O.scale_bytes(N, K, group)


def test_invalid_descriptors():
    assert tq.tq_row_pitch_words(tq.desc(0, 128)) == 0
    assert tq.tq_packed_bytes(tq.desc(4, 128, packing=4)) == 0
    # 3-bit codes: the decode GEMV takes batch 1..16 with the same workspace as the ternary packings
    # (x^ halves, then 40 groups x 12 floats rounded to 256 bytes); the other contractions do not
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 128, packing=tq.TQ_PACK_3BIT), 1) == 512
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 5120, packing=tq.TQ_PACK_3BIT), 8) == 5120 * 8 * 2 + 2048
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 128, packing=tq.TQ_PACK_3BIT), 17) == 0
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 100, packing=tq.TQ_PACK_3BIT), 1) == 0
    assert tq.tq_gemm_workspace_bytes(tq.desc(4, 128, packing=tq.TQ_PACK_3BIT), 16) == 0
    # FP8 prefill: E4M3 operands (M x K, N x K bytes), per-row float factors of x, int exponents and
    # float factors of W, each 256-byte aligned; 3-bit codes and a K off the 128-grid are refused
    assert tq.tq_gemm_fp8_workspace_bytes(tq.desc(300, 1024), 77) == 77 * 1024 + 300 * 1024 + 512 + 2 * 1280
    assert tq.tq_gemm_fp8_workspace_bytes(tq.desc(300, 1024, packing=tq.TQ_PACK_3BIT), 77) == 0
    assert tq.tq_gemm_fp8_workspace_bytes(tq.desc(300, 1000), 77) == 0
    assert tq.tq_gemm_fp8_workspace_bytes(tq.desc(300, 1024), 0) == 0
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 100), 1) == 0        # K not a multiple of 128
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 128, group=32), 1) == 0
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 128), 17) == 0        # batch above 16
    # workspace = the transformed activations (K x batch halves) and one row of floats per group
    assert tq.tq_gemv_workspace_bytes(tq.desc(4, 128), 1) == 256 + 256
    assert tq.tq_gemv_workspace_bytes(tq.desc(5120, 17408), 16) == 17408 * 16 * 2 + 11008  # 136 x 20 floats, 256-rounded
    assert tq.tq_gemv_workspace_bytes(tq.desc(64, 128 * 4096), 16) == 0        # activations of a CTA too large
    assert tq.tq_gemv_workspace_bytes(tq.desc(64, 128, flags=2), 1) == 0        # unknown flag
    assert tq.tq_gemv_workspace_bytes(tq.desc(64, 128, flags=tq.TQ_STATIC_WEIGHTS), 1) == 512
    assert tq.tq_moe_workspace_bytes(1, 257, 8, 2048, 512) == 0
    assert tq.tq_moe_workspace_bytes(8, 256, 8, 2048, 512) > 0
    assert tq.tq_moe_gemm_workspace_bytes(256, 256, 8, 2048, 512) > 256 * 3 * 2048 * 512 * 2  # decoded experts
    assert tq.tq_moe_gemm_workspace_bytes(256, 256, 8, 2000, 512) == 0   # H not a multiple of 256
    assert tq.tq_moe_gemm_workspace_bytes(256, 256, 8, 2048, 64) == 0    # 2F not a multiple of 256


def _call(name, *args):
    return getattr(tq.lib(), name)(*args)


def test_host_validation_before_launch():
    """Errors are returned synchronously from the host checks; nothing reaches the device."""
    d = tq.desc(64, 256)
    bd = ctypes.byref(d)
    A16 = 0x10000  # a fake, 16-byte-aligned address: never dereferenced because validation fails first
    assert _call("tq_pack", None, A16, A16, None) == 1
    assert _call("tq_pack", bd, None, A16, None) == 1
    assert _call("tq_pack", bd, A16, A16 + 4, None) == 3
    assert _call("tq_unpack", bd, A16 + 8, A16, None, None) == 3
    assert _call("tq_fwht", A16, A16, 0, 4, 200, 128, None) == 2        # K not a multiple of the block
    assert _call("tq_fwht", A16, A16, 0, 4, 256, 64, None) == 2         # block 64 unsupported
    assert _call("tq_fwht", A16 + 2, A16, 0, 4, 256, 128, None) == 3
    assert _call("tq_gemv", bd, A16, A16, A16, 0, A16, A16, 1 << 20, None) == 1      # batch 0
    assert _call("tq_gemv", bd, A16, A16, A16, 17, A16, A16, 1 << 20, None) == 1     # batch 17
    assert _call("tq_gemv", bd, A16, A16, A16, 1, A16, A16 + 16, 1 << 20, None) == 3  # workspace not 256-aligned
    assert _call("tq_gemv", bd, A16, A16, A16, 1, A16, A16, 16, None) == 7           # workspace too small
    huge = tq.desc(64, 128 * 4096)
    assert _call("tq_gemv", ctypes.byref(huge), A16, A16, A16, 16, A16, A16, 1 << 20, None) == 2
    bad_flags = tq.desc(64, 256, flags=4)
    assert _call("tq_gemv", ctypes.byref(bad_flags), A16, A16, A16, 1, A16, A16, 1 << 20, None) == 1
    bad_group = tq.desc(64, 256, group=96)
    assert _call("tq_gemv", ctypes.byref(bad_group), A16, A16, A16, 1, A16, A16, 1 << 20, None) == 2
    assert _call("tq_gemm", bd, A16, A16, A16, 0, A16, A16, 1 << 30, None) == 1
    assert _call("tq_moe_route", A16, 4, 300, 8, A16, A16, None) == 2
    assert _call("tq_moe_route", A16, 4, 256, 9, A16, A16, None) == 2
    gu, dn = tq.desc(1024, 2048, 64), tq.desc(2048, 512, 64)
    bad_dn = tq.desc(2048, 256, 64)  # down K must equal F = gate_up N / 2
    args = [256, 8] + [A16] * 6 + [1, A16, A16, None, A16, A16, 1 << 30, None]
    assert _call("tq_moe_gemv", ctypes.byref(gu), ctypes.byref(bad_dn), *args) == 1
    args_small_ws = [256, 8] + [A16] * 6 + [1, A16, A16, None, A16, A16, 64, None]
    assert _call("tq_moe_gemv", ctypes.byref(gu), ctypes.byref(dn), *args_small_ws) == 7
    assert _call("tq_quantize", bd, None, A16, A16, None) == 1
    assert _call("tq_quantize", ctypes.byref(tq.desc(64, 200)), A16, A16, A16, None) == 2     # K not a multiple of 128
    assert _call("tq_quantize", ctypes.byref(tq.desc(64, 256, group=32)), A16, A16, A16, None) == 2
    assert _call("tq_quantize", ctypes.byref(tq.desc(64, 256, flags=1)), A16, A16, A16, None) == 1
    assert _call("tq_quantize", ctypes.byref(tq.desc(64, 128 * 2048)), A16, A16, A16, None) == 2  # row too long
    assert _call("tq_quantize", bd, A16 + 8, A16, A16, None) == 3
    assert _call("tq_quantize", bd, A16, A16, A16 + 1, None) == 3
    assert _call("tq_selftest_wait", 2, 1000000, A16, None) == 1         # unknown kind
    assert _call("tq_selftest_wait", 0, 0, None, None) == 1              # limit not positive
    assert _call("tq_selftest_wait", 0, 2 * 10 ** 9, None, None) == 1    # limit above 1 s
    assert _call("tq_selftest_wait", 1, 1000000, None, None) == 1        # kind 1 needs the counter
    assert _call("tq_selftest_wait", 1, 1000000, A16 + 16, None) == 3    # counter not 256-aligned


def test_status_strings_and_version():
    assert tq.tq_version() >= 1
    for s in range(9):
        assert tq.tq_status_str(s) and tq.tq_status_str(s) != "unknown status"
    assert tq.tq_status_str(99) == "unknown status"


def test_last_cuda_error_without_device():
    """Without a usable device a compute call returns TQ_ERR_CUDA and the CUDA code is kept for the caller."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    tq.tq_last_cuda_error()  # clear
    d = tq.desc(64, 256)
    A16 = 0x10000
    assert _call("tq_pack", ctypes.byref(d), A16, A16, None) == 5
    assert tq.tq_last_cuda_error() != 0
    assert tq.tq_last_cuda_error() == 0   # read clears it
