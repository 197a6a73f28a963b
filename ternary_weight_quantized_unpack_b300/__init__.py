"""Python binding of libtq (include/tq.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  It checks nothing the library does
not check itself, allocates output / workspace tensors with torch when the caller does not pass
them, passes raw device pointers and the current CUDA stream, and raises TQError on a non-OK status.
All compute runs in libtq's CUDA kernels; there is no CPU path.  If libtq.so has not been built
the import still succeeds, but the first call raises (build it with
``python -m ternary_weight_quantized_unpack_b300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libtq.so")

TQ_PACK_B3 = 1
TQ_PACK_2BIT = 2
TQ_PACK_3BIT = 3
TQ_STATIC_WEIGHTS = 1

STATUS = {0: "TQ_OK", 1: "TQ_ERR_INVALID_ARG", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_MISALIGNED",
          4: "TQ_ERR_INVALID_CODE", 5: "TQ_ERR_CUDA", 6: "TQ_ERR_TIMEOUT", 7: "TQ_ERR_WORKSPACE", 8: "TQ_ERR_RANGE"}


class TQError(RuntimeError):
    def __init__(self, status: int, where: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        detail = f" (cudaError {cuda_error})" if cuda_error else ""
        super().__init__(f"{where}: {STATUS.get(status, status)}{detail}")


class tq_desc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("K", ctypes.c_int32), ("group", ctypes.c_int32),
                ("packing", ctypes.c_int32), ("fwht_block", ctypes.c_int32), ("flags", ctypes.c_int32)]

    def __repr__(self):
        return (f"tq_desc(N={self.N}, K={self.K}, group={self.group}, packing={self.packing}, "
                f"fwht_block={self.fwht_block}, flags={self.flags})")


def desc(N: int, K: int, group: int = 128, packing: int = TQ_PACK_B3, fwht_block: int = 128,
         flags: int = 0) -> tq_desc:
    return tq_desc(N, K, group, packing, fwht_block, flags)


TQ_SEQ_X_BF16 = 0
TQ_SEQ_X_PREV = 1
TQ_SEQ_X_SWIGLU_PREV = 2
TQ_SEQ_X_RMS_PREV = 3


class tq_seq_call(ctypes.Structure):
    _fields_ = [("d", tq_desc), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("x_src", ctypes.c_int32),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_D = ctypes.POINTER(tq_desc)
_SIGS = {
    "tq_row_pitch_words": (_SZ, [_D]),
    "tq_packed_bytes": (_SZ, [_D]),
    "tq_scale_bytes": (_SZ, [_D]),
    "tq_pack": (_I, [_D, _P, _P, _P]),
    "tq_unpack": (_I, [_D, _P, _P, _P, _P]),
    "tq_fwht": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "tq_quantize": (_I, [_D, _P, _P, _P, _P]),
    "tq_gemv_workspace_bytes": (_SZ, [_D, _I]),
    "tq_gemv": (_I, [_D, _P, _P, _P, _I, _P, _P, _SZ, _P]),
    "tq_gemv_noalloc": (_I, [_D, _P, _P, _P, _I, _P, _P]),
    "tq_gemv_kernel_count": (_I, [_D, _I]),
    "tq_moe_route": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "tq_moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "tq_moe_gemv": (_I, [_D, _D, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tq_moe_gemm_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "tq_moe_gemm": (_I, [_D, _D, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tq_gemm_workspace_bytes": (_SZ, [_D, _I]),
    "tq_gemm": (_I, [_D, _P, _P, _P, _I, _P, _P, _SZ, _P]),
    "tq_gemm_fp8_workspace_bytes": (_SZ, [_D, _I]),
    "tq_gemm_fp8": (_I, [_D, _P, _P, _P, _I, _P, _P, _SZ, _P]),
    "tq_seq_create": (_I, [ctypes.POINTER(tq_seq_call), _I, _I, ctypes.POINTER(ctypes.c_void_p)]),
    "tq_seq_workspace_bytes": (_SZ, [_P]),
    "tq_seq_upload": (_I, [_P, _P, _SZ]),
    "tq_seq_run": (_I, [_P, _P, _P]),
    "tq_seq_kernel_count": (_I, [_P]),
    "tq_seq_destroy": (None, [_P]),
    "tq_selftest_wait": (_I, [_I, ctypes.c_longlong, _P, _P]),
    "tq_device_status": (_I, [ctypes.POINTER(ctypes.c_int32)]),
    "tq_status_str": (ctypes.c_char_p, [_I]),
    "tq_last_cuda_error": (_I, []),
    "tq_version": (_I, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not built: run python -m ternary_weight_quantized_unpack_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors passed to libtq must be contiguous CUDA tensors"
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise TQError(status, where, lib().tq_last_cuda_error() if status == 5 else 0)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


# ---- sizes ----------------------------------------------------------------------------------------

def tq_row_pitch_words(d: tq_desc) -> int:
    return lib().tq_row_pitch_words(ctypes.byref(d))


def tq_packed_bytes(d: tq_desc) -> int:
    return lib().tq_packed_bytes(ctypes.byref(d))


def tq_scale_bytes(d: tq_desc) -> int:
    return lib().tq_scale_bytes(ctypes.byref(d))


def tq_gemv_workspace_bytes(d: tq_desc, batch: int) -> int:
    return lib().tq_gemv_workspace_bytes(ctypes.byref(d), batch)


def tq_gemv_kernel_count(d: tq_desc, batch: int) -> int:
    return lib().tq_gemv_kernel_count(ctypes.byref(d), batch)


def tq_gemm_workspace_bytes(d: tq_desc, M: int) -> int:
    return lib().tq_gemm_workspace_bytes(ctypes.byref(d), M)


def tq_gemm_fp8_workspace_bytes(d: tq_desc, M: int) -> int:
    return lib().tq_gemm_fp8_workspace_bytes(ctypes.byref(d), M)


def tq_moe_workspace_bytes(T: int, E: int, topk: int, H: int, F: int) -> int:
    return lib().tq_moe_workspace_bytes(T, E, topk, H, F)


# ---- compute --------------------------------------------------------------------------------------

def tq_pack(d: tq_desc, trits: torch.Tensor, codes: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int8 trits [N, K] -> int32 tensor [N, P] holding the uint32 code words."""
    if codes is None:
        codes = torch.empty((d.N, tq_row_pitch_words(d)), dtype=torch.int32, device=trits.device)
    _check(lib().tq_pack(ctypes.byref(d), _ptr(trits), _ptr(codes), _stream(stream)), "tq_pack")
    return codes


def tq_unpack(d: tq_desc, codes: torch.Tensor, trits: torch.Tensor | None = None,
              invalid_words: torch.Tensor | None = None, stream=None):
    """codes [N, P] -> (int8 trits [N, K], int32 [1] count of invalid words)."""
    if trits is None:
        trits = torch.empty((d.N, d.K), dtype=torch.int8, device=codes.device)
    if invalid_words is None:
        invalid_words = torch.empty(1, dtype=torch.int32, device=codes.device)
    _check(lib().tq_unpack(ctypes.byref(d), _ptr(codes), _ptr(trits), _ptr(invalid_words), _stream(stream)),
           "tq_unpack")
    return trits, invalid_words


def tq_quantize(d: tq_desc, w: torch.Tensor, codes: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                stream=None):
    """bf16 W [N, K] -> (int32 codes [N, P], fp16 scales [N, K / group]): rotate, absmean-scale, ternarize, pack."""
    assert w.dtype == torch.bfloat16 and w.is_contiguous()
    if codes is None:
        codes = torch.empty((d.N, tq_row_pitch_words(d)), dtype=torch.int32, device=w.device)
    if scales is None:
        scales = torch.empty((d.N, -(-d.K // d.group)), dtype=torch.float16, device=w.device)
    _check(lib().tq_quantize(ctypes.byref(d), _ptr(w), _ptr(codes), _ptr(scales), _stream(stream)), "tq_quantize")
    return codes, scales


def tq_fwht(x: torch.Tensor, out_fp16: bool = False, block: int = 128, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """bf16 [rows, K] -> block-Hadamard transform, float32 (or fp16) [rows, K]."""
    rows, K = x.shape
    if out is None:
        out = torch.empty((rows, K), dtype=torch.float16 if out_fp16 else torch.float32, device=x.device)
    _check(lib().tq_fwht(_ptr(x), _ptr(out), int(out_fp16), rows, K, block, _stream(stream)), "tq_fwht")
    return out


def tq_gemv(d: tq_desc, codes, scales, x, y=None, workspace=None, stream=None) -> torch.Tensor:
    """y[b, n] = sum_k s t x~ ; x bf16 [batch, K] -> y float32 [batch, N]."""
    batch = x.shape[0]
    if y is None:
        y = torch.empty((batch, d.N), dtype=torch.float32, device=x.device)
    nbytes = tq_gemv_workspace_bytes(d, batch)
    if workspace is None:
        workspace = _ws(nbytes, x.device)
    _check(lib().tq_gemv(ctypes.byref(d), _ptr(codes), _ptr(scales), _ptr(x), batch, _ptr(y), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream)), "tq_gemv")
    return y


def tq_gemv_noalloc(d: tq_desc, codes, scales, x, y=None, stream=None) -> torch.Tensor:
    """tq_gemv with the scratch in the library's fixed device array (no workspace argument)."""
    batch = x.shape[0]
    if y is None:
        y = torch.empty((batch, d.N), dtype=torch.float32, device=x.device)
    _check(lib().tq_gemv_noalloc(ctypes.byref(d), _ptr(codes), _ptr(scales), _ptr(x), batch, _ptr(y),
                                 _stream(stream)), "tq_gemv_noalloc")
    return y


def tq_moe_route(logits: torch.Tensor, topk: int = 8, idx=None, gate=None, stream=None):
    T, E = logits.shape
    if idx is None:
        idx = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    if gate is None:
        gate = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    _check(lib().tq_moe_route(_ptr(logits), T, E, topk, _ptr(idx), _ptr(gate), _stream(stream)), "tq_moe_route")
    return idx, gate


def tq_moe_gemv(gate_up: tq_desc, down: tq_desc, E: int, topk: int, gu_codes, gu_scales, d_codes, d_scales,
                router_logits, x, topk_idx=None, topk_gate=None, h_out=None, y=None, workspace=None,
                want_h: bool = False, stream=None):
    """Routed SwiGLU expert layer.  Returns (y [T, H], idx [T, k], gate [T, k], h [T, k, F] or None)."""
    T, H = x.shape
    F = down.K
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if h_out is None and want_h:
        h_out = torch.empty((T, topk, F), dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=dev)
    nbytes = tq_moe_workspace_bytes(T, E, topk, H, F)
    if workspace is None:
        workspace = _ws(nbytes, dev)
    _check(lib().tq_moe_gemv(ctypes.byref(gate_up), ctypes.byref(down), E, topk, _ptr(gu_codes), _ptr(gu_scales),
                             _ptr(d_codes), _ptr(d_scales), _ptr(router_logits), _ptr(x), T, _ptr(topk_idx),
                             _ptr(topk_gate), _ptr(h_out), _ptr(y), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "tq_moe_gemv")
    return y, topk_idx, topk_gate, h_out


def tq_moe_gemm(gate_up: tq_desc, down: tq_desc, E: int, topk: int, gu_codes, gu_scales, d_codes, d_scales,
                router_logits, x, topk_idx=None, topk_gate=None, h_out=None, y=None, workspace=None,
                want_h: bool = False, stream=None):
    """Routed SwiGLU expert layer at prefill sizes (grouped tensor-core GEMM).  Same arguments and
    returns as tq_moe_gemv."""
    T, H = x.shape
    F = down.K
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if h_out is None and want_h:
        h_out = torch.empty((T, topk, F), dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=dev)
    nbytes = tq_moe_gemm_workspace_bytes(T, E, topk, H, F)
    if workspace is None:
        workspace = _ws(nbytes, dev)
    _check(lib().tq_moe_gemm(ctypes.byref(gate_up), ctypes.byref(down), E, topk, _ptr(gu_codes), _ptr(gu_scales),
                             _ptr(d_codes), _ptr(d_scales), _ptr(router_logits), _ptr(x), T, _ptr(topk_idx),
                             _ptr(topk_gate), _ptr(h_out), _ptr(y), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "tq_moe_gemm")
    return y, topk_idx, topk_gate, h_out


def tq_moe_gemm_workspace_bytes(T: int, E: int, topk: int, H: int, F: int) -> int:
    return lib().tq_moe_gemm_workspace_bytes(T, E, topk, H, F)


def tq_gemm(d: tq_desc, codes, scales, x, y=None, workspace=None, stream=None) -> torch.Tensor:
    """Prefill: x bf16 [M, K] -> y bf16 [M, N]."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, d.N), dtype=torch.bfloat16, device=x.device)
    nbytes = tq_gemm_workspace_bytes(d, M)
    if workspace is None:
        workspace = _ws(nbytes, x.device)
    _check(lib().tq_gemm(ctypes.byref(d), _ptr(codes), _ptr(scales), _ptr(x), M, _ptr(y), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream)), "tq_gemm")
    return y


def tq_gemm_fp8(d: tq_desc, codes, scales, x, y=None, workspace=None, stream=None) -> torch.Tensor:
    """Prefill with FP8 E4M3 operands: x bf16 [M, K] -> y bf16 [M, N]."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, d.N), dtype=torch.bfloat16, device=x.device)
    nbytes = tq_gemm_fp8_workspace_bytes(d, M)
    if workspace is None:
        workspace = _ws(nbytes, x.device)
    _check(lib().tq_gemm_fp8(ctypes.byref(d), _ptr(codes), _ptr(scales), _ptr(x), M, _ptr(y), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "tq_gemm_fp8")
    return y


# ---- decode step: a chain of GEMVs in one launch ---------------------------------------------------

def tq_seq_create(calls, batch: int) -> ctypes.c_void_p:
    """calls: sequence of (desc, codes, scales, x_src, x or None, y) -> opaque plan handle."""
    arr = (tq_seq_call * len(calls))()
    for i, (d, codes, scales, x_src, x, y) in enumerate(calls):
        arr[i] = tq_seq_call(d, _ptr(codes), _ptr(scales), x_src, _ptr(x), _ptr(y))
    h = ctypes.c_void_p()
    _check(lib().tq_seq_create(arr, len(calls), batch, ctypes.byref(h)), "tq_seq_create")
    return h


def tq_seq_workspace_bytes(plan) -> int:
    return lib().tq_seq_workspace_bytes(plan)


def tq_seq_upload(plan, workspace: torch.Tensor):
    _check(lib().tq_seq_upload(plan, _ptr(workspace), workspace.numel() * workspace.element_size()), "tq_seq_upload")


def tq_seq_run(plan, workspace: torch.Tensor, stream=None):
    _check(lib().tq_seq_run(plan, _ptr(workspace), _stream(stream)), "tq_seq_run")


def tq_seq_kernel_count(plan) -> int:
    return lib().tq_seq_kernel_count(plan)


def tq_seq_destroy(plan):
    lib().tq_seq_destroy(plan)


class SeqPlan:
    """A decode step (a chain of 2-bit or base-3 GEMVs) prepared once and run with one launch per call of run().

    calls: list of (desc, codes, scales, x_src, x, y) as tq_seq_call; the tensors are kept alive by
    the plan.  The workspace is allocated here with torch unless one is given."""

    def __init__(self, calls, batch: int, workspace: torch.Tensor | None = None):
        self._keep = [t for c in calls for t in c[1:] if isinstance(t, torch.Tensor)]
        self.handle = tq_seq_create(calls, batch)
        nbytes = tq_seq_workspace_bytes(self.handle)
        self.workspace = workspace if workspace is not None else _ws(nbytes, calls[0][1].device)
        tq_seq_upload(self.handle, self.workspace)

    def run(self, stream=None):
        tq_seq_run(self.handle, self.workspace, stream)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.tq_seq_destroy(h)
            self.handle = None


def tq_selftest_wait(kind: int, limit_ns: int, workspace: torch.Tensor | None = None, stream=None):
    """Run the bounded-wait self-test (see include/tq.h); the timeout shows in tq_device_status()."""
    _check(lib().tq_selftest_wait(kind, limit_ns, _ptr(workspace) if workspace is not None else None,
                                  _stream(stream)), "tq_selftest_wait")


def tq_device_status() -> int:
    v = ctypes.c_int32(0)
    _check(lib().tq_device_status(ctypes.byref(v)), "tq_device_status")
    return v.value


def tq_status_str(status: int) -> str:
    return lib().tq_status_str(status).decode()


def tq_last_cuda_error() -> int:
    """cudaError_t code behind the last TQ_ERR_CUDA returned in this thread (0 if none); clears it."""
    return lib().tq_last_cuda_error()


def tq_version() -> int:
    return lib().tq_version()
