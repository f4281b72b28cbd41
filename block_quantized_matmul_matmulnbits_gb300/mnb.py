"""ctypes binding of libmnb.so (C ABI in include/mnb.h).

Argument marshalling only: every function here takes torch tensors (or raw
device addresses as ints, or None), passes their device pointers and sizes to
the C entry point of the same name, and raises ``MnbError`` on a non-zero
status.  No arithmetic of the operation happens in Python, and there is no
fallback: if the library has not been built the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmnb.so")

MNB_OK = 0
MNB_ERR_ARG = -1
MNB_ERR_UNSUPPORTED = -2
MNB_ERR_ALIGN = -3
MNB_ERR_CUDA = -4
MNB_ERR_DEVICE_TIMEOUT = -5
MNB_ERR_NO_DEVICE = -6

ROUTE_NONE, ROUTE_GEMV, ROUTE_GEMM, ROUTE_FILL = 0, 1, 2, 3
MODE_AUTO, MODE_FORCE_GEMV, MODE_FORCE_GEMM = 0, 1, 2
FLAG_EARLY_WEIGHTS = 1

# Every symbol include/mnb.h declares (checked against the header by the tests).
EXPORTS = ("mnb_create", "mnb_destroy", "mnb_run", "mnb_run_bias", "mnb_run_qlora", "mnb_run_multi", "mnb_transpose_dq_weight", "mnb_run_q8x", "mnb_quantize_x", "mnb_check_wait_timeout", "mnb_plan", "mnb_last_route", "mnb_sync_status",
           "mnb_status_str", "mnb_dequant", "mnb_lora_down", "mnb_run_noalloc", "mnb_noalloc_max_rows")


class MnbDesc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("bits", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_rank", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("gemv_max_m", ctypes.c_int32), ("flags", ctypes.c_int32)]


class MnbPlanInfo(ctypes.Structure):
    _fields_ = [("route", ctypes.c_int32), ("lora_kernel", ctypes.c_int32), ("grid_x", ctypes.c_int32),
                ("grid_y", ctypes.c_int32), ("block_threads", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
                ("k_splits", ctypes.c_int32), ("tokens_per_cta", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class MnbProjection(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zp", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class MnbError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_str(code)} ({code})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libmnb.so (raises if it is missing: there is no other compute path)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libmnb.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                                   "or python -m block_quantized_matmul_matmulnbits_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.mnb_create.argtypes = [ctypes.POINTER(MnbDesc), ctypes.POINTER(P)]
            L.mnb_create.restype = ctypes.c_int
            L.mnb_destroy.argtypes = [P]
            L.mnb_destroy.restype = None
            L.mnb_run.argtypes = [P, P, P, P, P, P, P, I32, P, P, I64, I64, P]
            L.mnb_run.restype = ctypes.c_int
            L.mnb_run_bias.argtypes = [P, P, P, P, P, P, P, I32, P, P, P, I64, I64, P]
            L.mnb_run_bias.restype = ctypes.c_int
            L.mnb_run_qlora.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I32, P, P, P, I64, I64, P]
            L.mnb_run_qlora.restype = ctypes.c_int
            L.mnb_run_multi.argtypes = [P, P, ctypes.POINTER(MnbProjection), ctypes.c_int32, I64, I64, P]
            L.mnb_run_multi.restype = ctypes.c_int
            L.mnb_transpose_dq_weight.argtypes = [P, P, P, I64, I64, I32, I32, I32, P, P, P]
            L.mnb_transpose_dq_weight.restype = ctypes.c_int
            L.mnb_run_q8x.argtypes = [P, P, P, P, P, P, P, I32, P, P, P, I64, I64, P]
            L.mnb_run_q8x.restype = ctypes.c_int
            L.mnb_quantize_x.argtypes = [P, I64, I64, P, P, P]
            L.mnb_quantize_x.restype = ctypes.c_int
            L.mnb_check_wait_timeout.argtypes = [I64, P]
            L.mnb_check_wait_timeout.restype = ctypes.c_int
            L.mnb_plan.argtypes = [P, I64, I64, I32, I32, ctypes.POINTER(MnbPlanInfo)]
            L.mnb_plan.restype = ctypes.c_int
            L.mnb_last_route.argtypes = [P]
            L.mnb_last_route.restype = ctypes.c_int
            L.mnb_sync_status.argtypes = [P, P]
            L.mnb_sync_status.restype = ctypes.c_int
            L.mnb_status_str.argtypes = [ctypes.c_int]
            L.mnb_status_str.restype = ctypes.c_char_p
            L.mnb_dequant.argtypes = [P, P, P, I64, I64, I32, I32, P, I32, P]
            L.mnb_dequant.restype = ctypes.c_int
            L.mnb_lora_down.argtypes = [P, P, P, I64, I64, I32, P]
            L.mnb_lora_down.restype = ctypes.c_int
            L.mnb_run_noalloc.argtypes = [P, P, P, P, P, P, P, I32, P, I64, I64, P]
            L.mnb_run_noalloc.restype = ctypes.c_int
            L.mnb_noalloc_max_rows.argtypes = []
            L.mnb_noalloc_max_rows.restype = I64
            _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, what: str):
    if code != MNB_OK:
        raise MnbError(code, what)


def status_str(code: int) -> str:
    return lib().mnb_status_str(code).decode()


def mnb_status_str(code: int) -> str:
    return status_str(code)


def mnb_create(N: int, K: int, bits: int = 4, block_size: int = 32, max_rank: int = 32,
               mode: int = MODE_AUTO, gemv_max_m: int = 0, flags: int = 0) -> ctypes.c_void_p:
    d = MnbDesc(N, K, bits, block_size, max_rank, mode, gemv_max_m, flags)
    h = ctypes.c_void_p()
    _check(lib().mnb_create(ctypes.byref(d), ctypes.byref(h)), "mnb_create")
    return h


def mnb_destroy(h) -> None:
    lib().mnb_destroy(h)


def mnb_run(h, X, Wq, scales, zp, A, B, rank: int, Y, T_ws, batch: int, M: int, stream=None) -> None:
    _check(lib().mnb_run(h, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank,
                         _ptr(Y), _ptr(T_ws), batch, M, _stream(stream)), "mnb_run")


def mnb_run_bias(h, X, Wq, scales, zp, A, B, rank: int, bias, Y, T_ws, batch: int, M: int, stream=None) -> None:
    _check(lib().mnb_run_bias(h, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank, _ptr(bias),
                              _ptr(Y), _ptr(T_ws), batch, M, _stream(stream)), "mnb_run_bias")


def mnb_run_qlora(h, X, Wq, scales, zp, Aq, A_scales, A_zp, Bq, B_scales, B_zp, rank: int, bias, Y, T_ws,
                  batch: int, M: int, stream=None) -> None:
    _check(lib().mnb_run_qlora(h, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(Aq), _ptr(A_scales), _ptr(A_zp),
                               _ptr(Bq), _ptr(B_scales), _ptr(B_zp), rank, _ptr(bias), _ptr(Y), _ptr(T_ws), batch, M,
                               _stream(stream)), "mnb_run_qlora")


def mnb_run_multi(h, X, projections, batch: int, M: int, stream=None) -> None:
    """projections: sequence of (N, Wq, scales, zp, bias, Y); Wq None = empty weight."""
    arr = (MnbProjection * len(projections))()
    for i, (N, Wq, scales, zp, bias, Y) in enumerate(projections):
        arr[i] = MnbProjection(N, _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(bias), _ptr(Y))
    _check(lib().mnb_run_multi(h, _ptr(X), arr, len(projections), batch, M, _stream(stream)), "mnb_run_multi")


def mnb_transpose_dq_weight(w_q, w_scale, w_zp, bits: int, blocked: bool = True, block_size: int = 32):
    """numpy in, numpy out (host): DequantizeLinear weight w_q [K, N] (uint8 codes), w_scale
    (FP16 bits, [K/32, N] or one value), w_zp (uint8 like w_scale, or None) -> (Wq, scales, zp)
    in the MatMulNBits layout."""
    import numpy as np
    w_q = np.ascontiguousarray(w_q, dtype=np.uint8)
    K, N = w_q.shape
    w_scale = np.ascontiguousarray(w_scale, dtype=np.uint16)
    w_zp = None if w_zp is None else np.ascontiguousarray(w_zp, dtype=np.uint8)
    Wq = np.empty((N, K // block_size, block_size * bits // 8), dtype=np.uint8)
    scales = np.empty((N, K // block_size), dtype=np.uint16)
    zp = np.empty((N, K // block_size), dtype=np.uint8)
    addr = lambda a: None if a is None else a.ctypes.data
    _check(lib().mnb_transpose_dq_weight(addr(w_q), addr(w_scale), addr(w_zp), K, N, bits, block_size,
                                         1 if blocked else 0, addr(Wq), addr(scales), addr(zp)),
           "mnb_transpose_dq_weight")
    return Wq, scales, zp


def mnb_run_q8x(h, X, Wq, scales, zp, A, B, rank: int, bias, Y, T_ws, batch: int, M: int, stream=None) -> None:
    _check(lib().mnb_run_q8x(h, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank, _ptr(bias),
                             _ptr(Y), _ptr(T_ws), batch, M, _stream(stream)), "mnb_run_q8x")


def mnb_check_wait_timeout(limit_cycles: int, stream=None) -> None:
    _check(lib().mnb_check_wait_timeout(limit_cycles, _stream(stream)), "mnb_check_wait_timeout")


def mnb_quantize_x(X, Mt: int, K: int, Xq, Xs, stream=None) -> None:
    _check(lib().mnb_quantize_x(_ptr(X), Mt, K, _ptr(Xq), _ptr(Xs), _stream(stream)), "mnb_quantize_x")


def mnb_run_noalloc(h, X, Wq, scales, zp, A, B, rank: int, Y, batch: int, M: int, stream=None) -> None:
    """mnb_run for callers that cannot allocate device memory: T lives in the
    library's own fixed device array (at most mnb_noalloc_max_rows() token
    rows with an adapter; concurrent calls on the GPU race on it)."""
    _check(lib().mnb_run_noalloc(h, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank,
                                 _ptr(Y), batch, M, _stream(stream)), "mnb_run_noalloc")


def mnb_noalloc_max_rows() -> int:
    return int(lib().mnb_noalloc_max_rows())


def mnb_plan(h, batch: int, M: int, rank: int = 0, sm_count: int = 0) -> dict:
    info = MnbPlanInfo()
    _check(lib().mnb_plan(h, batch, M, rank, sm_count, ctypes.byref(info)), "mnb_plan")
    return info.as_dict()


def mnb_last_route(h) -> int:
    return lib().mnb_last_route(h)


def mnb_sync_status(h, stream=None) -> int:
    return lib().mnb_sync_status(h, _stream(stream))


def mnb_dequant(Wq, scales, zp, N: int, K: int, bits: int, W16, variant: int = 0, block_size: int = 32,
                stream=None) -> None:
    _check(lib().mnb_dequant(_ptr(Wq), _ptr(scales), _ptr(zp), N, K, bits, block_size, _ptr(W16), variant,
                             _stream(stream)), "mnb_dequant")


def mnb_lora_down(X, A, T, Mt: int, K: int, rank: int = 32, stream=None) -> None:
    _check(lib().mnb_lora_down(_ptr(X), _ptr(A), _ptr(T), Mt, K, rank, _stream(stream)), "mnb_lora_down")


class Projection:
    """One quantized projection (owns an mnb handle); the call a user makes.

    ``proj(X, Wq, scales, zp=None, A=None, B=None)`` allocates Y (and the T
    scratch when an adapter is given) with torch and runs mnb_run on the
    current stream.  X is [batch, M, K] or [M, K] fp16 on the GPU.
    """

    def __init__(self, N: int, K: int, bits: int = 4, max_rank: int = 32, mode: int = MODE_AUTO,
                 gemv_max_m: int = 0, flags: int = 0):
        self.N, self.K, self.bits = N, K, bits
        self.h = mnb_create(N, K, bits, 32, max_rank, mode, gemv_max_m, flags)

    def __call__(self, X, Wq, scales, zp=None, A=None, B=None, out=None, T_ws=None, stream=None, bias=None):
        import torch
        batch, M = (X.shape[0], X.shape[1]) if X.dim() == 3 else (1, X.shape[0])
        rank = 0 if A is None else int(A.shape[1])
        if out is None:
            shape = (batch, M, self.N) if X.dim() == 3 else (M, self.N)
            out = torch.empty(shape, dtype=torch.float16, device=X.device)
        if rank and T_ws is None:
            T_ws = torch.empty((batch * M, rank), dtype=torch.float16, device=X.device)
        mnb_run_bias(self.h, X, Wq, scales, zp, A, B, rank, bias, out, T_ws, batch, M, stream)
        return out

    @property
    def last_route(self) -> int:
        return mnb_last_route(self.h)

    def close(self):
        if self.h is not None:
            mnb_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
