"""CPU oracle for the block-quantized MatMulNBits product (+ rank-r LoRA).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) may import
this package.  The CUDA library never loads it and shares no code with it.

The arithmetic lives in ``mnb_oracle.c`` (plain C, binary64); this module only
builds that file with gcc and marshals numpy arrays into it.  Every function
follows the plain definition:

* dequant  ``w = (q - zp) * scale`` -- "Fuse DQ->MatMulNBits for shared
  initializers and skip outer-scope weights" (onnxruntime PR 33800),
  Description and repro (DequantizeLinear then MatMul);
* ``Y = X * w^T + (X * A) * B^T`` with an empty adapter giving the base only --
  "[WebGPU] Fuse rank-32 quantized LoRA with MatMulNBits" (onnxruntime PR
  33370), commit message adding the MatMulNBitsLoRA operator, and its
  Description.

Pins for each function (tests/test_oracle_pins.py) check it against things
other than itself: numpy's float16 cast, hand-written golden fixtures,
closed forms, exact rational brute force and numpy matmul identities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mnb_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.mnb_ref_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.mnb_ref_f16_to_f64.restype = ctypes.c_double
            lib.mnb_ref_f64_to_f16.argtypes = [ctypes.c_double]
            lib.mnb_ref_f64_to_f16.restype = ctypes.c_uint16
            for name in ("mnb_ref_unpack", "mnb_ref_pack"):
                getattr(lib, name).argtypes = [P, I64, I64, I, I, P]
                getattr(lib, name).restype = I
            for name in ("mnb_ref_dequant", "mnb_ref_dequant_f16"):
                getattr(lib, name).argtypes = [P, P, P, I64, I64, I, I, P]
                getattr(lib, name).restype = I
            lib.mnb_ref_lora_down.argtypes = [P, P, I64, I64, I, P]
            lib.mnb_ref_lora_down.restype = I
            lib.mnb_ref_run.argtypes = [P, P, P, P, P, P, I, I64, I64, I64, I, I, I, P, P, P]
            lib.mnb_ref_run_bias.argtypes = [P, P, P, P, P, P, I, P, I64, I64, I64, I, I, I, P, P, P]
            lib.mnb_ref_run_bias.restype = I
            lib.mnb_ref_run_qlora.argtypes = [P, P, P, P, P, P, P, P, P, P, I, P, I64, I64, I64, I, I, I, P, P, P]
            lib.mnb_ref_run_qlora.restype = I
            lib.mnb_ref_quantize_x.argtypes = [P, I64, I64, I, P, P]
            lib.mnb_ref_quantize_x.restype = I
            lib.mnb_ref_run_q8x.argtypes = [P, P, P, P, P, P, I, P, I64, I64, I64, I, I, I, P, P, P]
            lib.mnb_ref_run_q8x.restype = I
            lib.mnb_ref_run.restype = I
            lib.mnb_ref_threads.argtypes = []
            lib.mnb_ref_threads.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def threads() -> int:
    """Host threads the oracle's parallel loop uses."""
    return int(_load().mnb_ref_threads())


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.array([lib.mnb_ref_f16_to_f64(int(b)) for b in flat], dtype=np.float64)
    return out.reshape(np.shape(bits))


def f64_to_f16_bits(vals: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(vals, dtype=np.float64).ravel()
    out = np.array([lib.mnb_ref_f64_to_f16(float(v)) for v in flat], dtype=np.uint16)
    return out.reshape(np.shape(vals))


def unpack(Wq: np.ndarray, N: int, K: int, bits: int, block: int = 32) -> np.ndarray:
    """Codes q[N, K] (uint8) from the packed weight bytes."""
    Wq = _c(Wq, np.uint8)
    q = np.empty((N, K), dtype=np.uint8)
    _check(_load().mnb_ref_unpack(_ptr(Wq), N, K, bits, block, _ptr(q)), "unpack")
    return q


def pack(q: np.ndarray, bits: int, block: int = 32) -> np.ndarray:
    """Packed weight bytes [N, K/block, block*bits/8] from codes q[N, K]."""
    q = _c(q, np.uint8)
    N, K = q.shape
    Wq = np.empty((N, K // block, block * bits // 8), dtype=np.uint8)
    _check(_load().mnb_ref_pack(_ptr(q), N, K, bits, block, _ptr(Wq)), "pack")
    return Wq


def dequant(Wq, scales, zp, N, K, bits, block=32) -> np.ndarray:
    """Exact dequantized weight w[N, K] in binary64."""
    Wq, scales, zp = _c(Wq, np.uint8), _c(scales, np.uint16), _c(zp, np.uint8)
    W = np.empty((N, K), dtype=np.float64)
    _check(_load().mnb_ref_dequant(_ptr(Wq), _ptr(scales), _ptr(zp), N, K, bits, block, _ptr(W)), "dequant")
    return W


def dequant_f16(Wq, scales, zp, N, K, bits, block=32) -> np.ndarray:
    """The dequantized weight rounded once to FP16, as uint16 bit patterns [N, K]."""
    Wq, scales, zp = _c(Wq, np.uint8), _c(scales, np.uint16), _c(zp, np.uint8)
    W16 = np.empty((N, K), dtype=np.uint16)
    _check(_load().mnb_ref_dequant_f16(_ptr(Wq), _ptr(scales), _ptr(zp), N, K, bits, block, _ptr(W16)),
           "dequant_f16")
    return W16


def lora_down(X, A) -> np.ndarray:
    """T = X * A in binary64; X [Mt, K] and A [K, r] given as FP16 bit patterns."""
    X, A = _c(X, np.uint16), _c(A, np.uint16)
    Mt, K = X.shape
    r = A.shape[1]
    T = np.empty((Mt, r), dtype=np.float64)
    _check(_load().mnb_ref_lora_down(_ptr(X), _ptr(A), Mt, K, r, _ptr(T)), "lora_down")
    return T


def run(X, Wq, scales, zp, A, B, N, K, bits, block=32, round_t=False, bias=None):
    """Y = X * dequant(Wq)^T (+ (X*A) * B^T) (+ bias broadcast over rows).

    X: [Mt, K] FP16 bit patterns (uint16); A [K, r], B [N, r] FP16 bits or None;
    bias: [N] FP16 bits or None.
    Returns (Y16 bits [Mt, N], Y64 [Mt, N], bound [Mt, N]) where bound is the
    sum of absolute products that scales the FP16 tolerance.
    """
    X = _c(X, np.uint16)
    Wq, scales, zp = _c(Wq, np.uint8), _c(scales, np.uint16), _c(zp, np.uint8)
    rank = 0 if (A is None or B is None) else int(np.shape(A)[1])
    A = _c(A, np.uint16) if rank else None
    B = _c(B, np.uint16) if rank else None
    Mt = X.shape[0]
    Y16 = np.empty((Mt, N), dtype=np.uint16)
    Y64 = np.empty((Mt, N), dtype=np.float64)
    bound = np.empty((Mt, N), dtype=np.float64)
    bias = _c(bias, np.uint16) if bias is not None else None
    rc = _load().mnb_ref_run_bias(_ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank, _ptr(bias),
                                  Mt, N, K, bits, block, 1 if round_t else 0,
                                  _ptr(Y16), _ptr(Y64), _ptr(bound))
    _check(rc, "run")
    return Y16, Y64, bound


def run_qlora(X, Wq, scales, zp, Aq, A_scales, A_zp, Bq, B_scales, B_zp, N, K, bits, block=32, round_t=False,
              bias=None):
    """Y with INT8 block-32 adapters given as 8-bit MatMulNBits weights:
    Aq [r, K/block, block] u8 (+ A_scales, A_zp [r, K/block]) for the down
    projection, Bq [N, r/block, block] u8 (+ B_scales, B_zp [N, r/block]) for
    the up projection; zero points None = 128.  Aq None = no adapter.
    Returns (Y16 bits, Y64, bound) as ``run``."""
    X = _c(X, np.uint16)
    Wq, scales, zp = _c(Wq, np.uint8), _c(scales, np.uint16), _c(zp, np.uint8)
    rank = 0 if Aq is None else int(np.shape(Aq)[0])
    Aq, A_scales, A_zp = _c(Aq, np.uint8), _c(A_scales, np.uint16), _c(A_zp, np.uint8)
    Bq, B_scales, B_zp = _c(Bq, np.uint8), _c(B_scales, np.uint16), _c(B_zp, np.uint8)
    Mt = X.shape[0]
    Y16 = np.empty((Mt, N), dtype=np.uint16)
    Y64 = np.empty((Mt, N), dtype=np.float64)
    bound = np.empty((Mt, N), dtype=np.float64)
    bias = _c(bias, np.uint16) if bias is not None else None
    rc = _load().mnb_ref_run_qlora(_ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(Aq), _ptr(A_scales), _ptr(A_zp),
                                   _ptr(Bq), _ptr(B_scales), _ptr(B_zp), rank, _ptr(bias), Mt, N, K, bits, block,
                                   1 if round_t else 0, _ptr(Y16), _ptr(Y64), _ptr(bound))
    _check(rc, "run_qlora")
    return Y16, Y64, bound


def quantize_x(X, block=32):
    """Per-block int8 activation codes and binary32 scales of X [Mt, K] (FP16
    bits): (Xq int8 [Mt, K], Xs float32 [Mt, K/block])."""
    X = _c(X, np.uint16)
    Mt, K = X.shape
    Xq = np.empty((Mt, K), dtype=np.int8)
    Xs = np.empty((Mt, K // block), dtype=np.float32)
    _check(_load().mnb_ref_quantize_x(_ptr(X), Mt, K, block, _ptr(Xq), _ptr(Xs)), "quantize_x")
    return Xq, Xs


def run_q8x(X, Wq, scales, zp, A, B, N, K, bits, block=32, round_t=False, bias=None):
    """The int8-activation product (per-block int8 X, integer block dots);
    arguments and returns as ``run``."""
    X = _c(X, np.uint16)
    Wq, scales, zp = _c(Wq, np.uint8), _c(scales, np.uint16), _c(zp, np.uint8)
    rank = 0 if (A is None or B is None) else int(np.shape(A)[1])
    A = _c(A, np.uint16) if rank else None
    B = _c(B, np.uint16) if rank else None
    Mt = X.shape[0]
    Y16 = np.empty((Mt, N), dtype=np.uint16)
    Y64 = np.empty((Mt, N), dtype=np.float64)
    bound = np.empty((Mt, N), dtype=np.float64)
    bias = _c(bias, np.uint16) if bias is not None else None
    rc = _load().mnb_ref_run_q8x(_ptr(X), _ptr(Wq), _ptr(scales), _ptr(zp), _ptr(A), _ptr(B), rank, _ptr(bias),
                                 Mt, N, K, bits, block, 1 if round_t else 0, _ptr(Y16), _ptr(Y64), _ptr(bound))
    _check(rc, "run_q8x")
    return Y16, Y64, bound
