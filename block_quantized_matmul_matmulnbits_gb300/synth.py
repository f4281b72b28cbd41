"""Seeded synthetic inputs for the block-quantized matmul.

This module draws random inputs and nothing else: it holds none of the
operation's arithmetic (no unpacking, dequantization or products), so the
tests can feed the same arrays to the CUDA library and to the CPU oracle.

Value recipes follow the workloads of "[WebGPU] Fuse rank-32 quantized LoRA
with MatMulNBits" (onnxruntime PR 33370: INT4 block-32 base weights, FP16
rank-32 adapters) and the tied lm_head of "Fuse DQ->MatMulNBits for shared
initializers and skip outer-scope weights" (onnxruntime PR 33800: INT8 codes
with per-block uint8 zero points):

* packed codes are uniform random bytes, so every 4-bit or 8-bit code is
  uniform over [0, 2^bits) (half-open bounds);
* scales are uniform reals in the given range, rounded once to FP16;
* zero points are uniform integers in an inclusive range, or absent (the
  operator then uses 2^(bits-1));
* X is N(0, 1) rounded to FP16; LoRA A [K, r] and B [N, r] are N(0, 0.02^2)
  rounded to FP16; a "partial" adapter has columns r/2 .. r-1 of A and B zero.

FP16 arrays are returned as uint16 bit patterns (numpy float16 ``view``).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import numpy as np

SEED_BASE = 0x4D4E42
BLOCK = 32
LORA_RANK = 32


@dataclass
class Inputs:
    X: np.ndarray                 # uint16 [batch, M, K] (FP16 bits)
    Wq: np.ndarray                # uint8 [N, K/32, 32*bits/8]
    scales: np.ndarray            # uint16 [N, K/32] (FP16 bits)
    zp: Optional[np.ndarray]      # uint8 [N, K/32] or None (default zero point)
    A: Optional[np.ndarray]       # uint16 [K, r] or None
    B: Optional[np.ndarray]       # uint16 [N, r] or None
    batch: int
    M: int
    N: int
    K: int
    bits: int

    @property
    def rank(self) -> int:
        return 0 if self.A is None else int(self.A.shape[1])

    @property
    def X2d(self) -> np.ndarray:
        return self.X.reshape(self.batch * self.M, self.K)


def _f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype(np.float16)).view(np.uint16)


def make_inputs(*, M: int, K: int, N: int, bits: int = 4, seed: int,
                batch: int = 1,
                zp_range: Optional[Tuple[int, int]] = None,
                scale_range: Tuple[float, float] = (0.005, 0.02),
                rank: int = 0, lora_std: float = 0.02, partial: bool = False,
                x_std: float = 1.0) -> Inputs:
    """Draw one seeded problem.  ``zp_range`` is inclusive; None = default zp."""
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // BLOCK
    bpb = BLOCK * bits // 8
    Wq = rng.integers(0, 256, size=(N, nb, bpb), dtype=np.uint8)
    scales = _f16_bits(rng.uniform(scale_range[0], scale_range[1], size=(N, nb)))
    zp = None
    if zp_range is not None:
        zp = rng.integers(zp_range[0], zp_range[1] + 1, size=(N, nb), dtype=np.uint8)
    X = _f16_bits(rng.standard_normal(size=(batch, M, K)) * x_std)
    A = B = None
    if rank:
        A64 = rng.standard_normal(size=(K, rank)) * lora_std
        B64 = rng.standard_normal(size=(N, rank)) * lora_std
        if partial:
            A64[:, rank // 2:] = 0.0
            B64[:, rank // 2:] = 0.0
        A, B = _f16_bits(A64), _f16_bits(B64)
    return Inputs(X=X, Wq=Wq, scales=scales, zp=zp, A=A, B=B, batch=batch, M=M, N=N, K=K, bits=bits)


@dataclass
class QLoRA:
    """INT8 block-32 adapters as 8-bit MatMulNBits weights."""
    Aq: np.ndarray                # uint8 [r, K/32, 32]   down projection, rank rows along K
    A_scales: np.ndarray          # uint16 [r, K/32] (FP16 bits)
    A_zp: Optional[np.ndarray]    # uint8 [r, K/32] or None (default 128)
    Bq: np.ndarray                # uint8 [N, r/32, 32]   up projection, N rows along the rank
    B_scales: np.ndarray          # uint16 [N, r/32]
    B_zp: Optional[np.ndarray]    # uint8 [N, r/32] or None

    @property
    def rank(self) -> int:
        return int(self.Aq.shape[0])


def make_qlora(*, K: int, N: int, seed: int, rank: int = LORA_RANK, zp: bool = True,
               scale_range: Tuple[float, float] = (1e-4, 3e-4)) -> QLoRA:
    """Seeded INT8 adapters: uniform codes over [0, 256), FP16 scales uniform in
    ``scale_range`` (dequantized values of the size of the FP16 adapters'
    N(0, 0.02^2)), zero points uniform over [120, 136] or absent.  Drawn from
    their own stream."""
    rng = np.random.Generator(np.random.PCG64([seed, 0x51A]))
    Aq = rng.integers(0, 256, size=(rank, K // BLOCK, BLOCK), dtype=np.uint8)
    A_scales = _f16_bits(rng.uniform(scale_range[0], scale_range[1], size=(rank, K // BLOCK)))
    A_zp = rng.integers(120, 137, size=(rank, K // BLOCK), dtype=np.uint8) if zp else None
    Bq = rng.integers(0, 256, size=(N, rank // BLOCK, BLOCK), dtype=np.uint8)
    B_scales = _f16_bits(rng.uniform(scale_range[0], scale_range[1], size=(N, rank // BLOCK)))
    B_zp = rng.integers(120, 137, size=(N, rank // BLOCK), dtype=np.uint8) if zp else None
    return QLoRA(Aq=Aq, A_scales=A_scales, A_zp=A_zp, Bq=Bq, B_scales=B_scales, B_zp=B_zp)


def make_bias(N: int, seed: int, std: float = 0.5) -> np.ndarray:
    """A seeded FP16 bias [N] (bit patterns), drawn from its own stream so the
    other inputs of the same seed are unchanged."""
    rng = np.random.Generator(np.random.PCG64([seed, 0xB1A5]))
    return _f16_bits(rng.standard_normal(size=N) * std)


# Named workloads (shapes and value ranges of the five configurations).

def tiny(M: int, rank: int, seed_offset: int = 0) -> Inputs:
    """M in {1, 4}, K = N = 256, INT4, default zero point, optional rank-32 adapter."""
    return make_inputs(M=M, K=256, N=256, bits=4, seed=SEED_BASE + 0 + seed_offset, rank=rank)


def decode_4096(rank: int = LORA_RANK, partial: bool = False, seed_offset: int = 0, M: int = 1) -> Inputs:
    """M = 1, K = N = 4096, INT4 with explicit uint8 zero points in [0, 15]."""
    return make_inputs(M=M, K=4096, N=4096, bits=4, seed=SEED_BASE + 1 + seed_offset,
                       zp_range=(0, 15), rank=rank, partial=partial)


def prefill_4096(M: int = 1024, batch: int = 1, rank: int = LORA_RANK, seed_offset: int = 0) -> Inputs:
    """M = 1024 (or batch 2 x 512), K = N = 4096, INT4, default zero point 8."""
    return make_inputs(M=M, K=4096, N=4096, bits=4, seed=SEED_BASE + 2 + seed_offset, batch=batch, rank=rank)


def lm_head(K: int, N: int, seed_offset: int = 0, M: int = 1) -> Inputs:
    """INT8 tied-embedding lm_head: zero points in [120, 136], scales in [0.001, 0.01]."""
    return make_inputs(M=M, K=K, N=N, bits=8, seed=SEED_BASE + 3 + seed_offset,
                       zp_range=(120, 136), scale_range=(0.001, 0.01))


def mlp_up(M: int, rank: int = 0, seed_offset: int = 0) -> Inputs:
    """K = 4096, N = 14336 up-projection sweep, INT4, default zero point."""
    return make_inputs(M=M, K=4096, N=14336, bits=4, seed=SEED_BASE + 4 + seed_offset, rank=rank)
