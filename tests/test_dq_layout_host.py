"""The DequantizeLinear -> MatMulNBits layout rewrite (mnb_transpose_dq_weight),
host code in libmnb: checked against the oracle's packing of the transposed
codes, and end to end against numpy's DequantizeLinear followed by MatMul."""
import json
import os

import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import mnb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float16)).view(np.uint16)


def dq_weight(K, N, bits, blocked, with_zp, seed):
    rng = np.random.default_rng(seed)
    w_q = rng.integers(0, 1 << bits, size=(K, N), dtype=np.uint8)
    shape = (K // 32, N) if blocked else (1,)
    w_scale = f16(rng.uniform(0.001, 0.05, size=shape))
    w_zp = rng.integers(0, 1 << bits, size=shape, dtype=np.uint8) if with_zp else None
    return w_q, w_scale, w_zp


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("blocked,with_zp", [(True, True), (True, False), (False, True), (False, False)])
def test_layout_matches_oracle_packing_of_the_transpose(bits, blocked, with_zp):
    K, N = 128, 40
    w_q, w_scale, w_zp = dq_weight(K, N, bits, blocked, with_zp, seed=bits * 10 + blocked * 2 + with_zp)
    Wq, scales, zp = mnb.mnb_transpose_dq_weight(w_q, w_scale, w_zp, bits, blocked)
    assert np.array_equal(Wq, oracle.pack(np.ascontiguousarray(w_q.T), bits))
    s_ref = w_scale.T if blocked else np.full((N, K // 32), w_scale[0], np.uint16)
    assert np.array_equal(scales, s_ref)
    z_ref = (w_zp.T if blocked else np.full((N, K // 32), w_zp[0], np.uint8)) if with_zp else np.zeros((N, K // 32))
    assert np.array_equal(zp, z_ref)


@pytest.mark.parametrize("bits,blocked", [(4, True), (8, False), (2, True)])
def test_matmulnbits_of_the_rewrite_is_dq_then_matmul(bits, blocked):
    """X * DequantizeLinear(w_q) (numpy, fp64) equals the oracle's MatMulNBits
    product on the rewritten weight, to fp64 rounding."""
    K, N, M = 96, 24, 3
    w_q, w_scale, w_zp = dq_weight(K, N, bits, blocked, True, seed=70 + bits)
    Wq, scales, zp = mnb.mnb_transpose_dq_weight(w_q, w_scale, w_zp, bits, blocked)
    s = w_scale.view(np.float16).astype(np.float64)
    z = w_zp.astype(np.float64)
    if blocked:
        s, z = np.repeat(s, 32, axis=0), np.repeat(z, 32, axis=0)
    W = (w_q.astype(np.float64) - z) * s                      # DequantizeLinear, [K, N]
    X = f16(np.random.default_rng(71).standard_normal((M, K)))
    ref = X.view(np.float16).astype(np.float64) @ W
    _, Y64, bound = oracle.run(X, Wq, scales, zp, None, None, N, K, bits)
    assert np.all(np.abs(Y64 - ref) <= 1e-12 * bound)


def test_dq_repro_per_tensor_closed_form():
    """The page's repro weight (all-zero uint8 [64, 32], per-tensor scale 0.02,
    zero point 3) rewritten: every output is -3 * fp16(0.02) * sum_k x_k."""
    cfg = json.load(open(os.path.join(GOLDEN, "dq_matmul_repro.json")))
    K, N = cfg["K"], cfg["N"]
    w_q = np.full((K, N), cfg["code"], np.uint8)
    Wq, scales, zp = mnb.mnb_transpose_dq_weight(w_q, f16([cfg["scale"]]), np.array([cfg["zero_point"]], np.uint8),
                                                 8, blocked=False)
    X = f16(np.random.default_rng(72).standard_normal((1, K)))
    _, Y64, _ = oracle.run(X, Wq, scales, zp, None, None, N, K, 8)
    x = X.view(np.float16).astype(np.float64)
    expect = (cfg["code"] - cfg["zero_point"]) * f16([cfg["scale"]]).view(np.float16).astype(np.float64)[0] * x.sum()
    assert np.allclose(Y64, expect, rtol=1e-12, atol=0)


def test_codes_too_wide_and_bad_shapes_are_rejected():
    w_q = np.full((64, 8), 16, np.uint8)   # 16 does not fit 4 bits
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_transpose_dq_weight(w_q, f16([0.5]), None, 4, blocked=False)
    assert e.value.code == mnb.MNB_ERR_ARG
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_transpose_dq_weight(np.zeros((48, 8), np.uint8), f16([0.5]), None, 4, blocked=False)
    assert e.value.code == mnb.MNB_ERR_UNSUPPORTED
