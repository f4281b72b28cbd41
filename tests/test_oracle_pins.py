"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources of truth used here: numpy's float16 cast (a library routine), golden
fixtures written by hand under tests/golden/, exact rational brute force
(fractions.Fraction), closed forms, and numpy matmul identities.  The negative
controls at the end show that a plausible mistake (swapped nibbles, a dropped
zero point, a transposed operand) makes a pin fail.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from conftest import GOLDEN


def f16(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16val(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------- FP16 format

def test_f16_decode_all_patterns_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_encode_matches_numpy_cast():
    rng = np.random.default_rng(7)
    vals = [0.0, -0.0, 65504.0, 65519.999, 65520.0, -65520.0, 1e9, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -26, 6.1e-5, 2.0 ** -14, np.inf, -np.inf]
    # exact ties between neighbouring FP16 values, normal and subnormal
    for e in range(-24, 16):
        for m in (1024, 1025, 1500, 2046):
            base = m * 2.0 ** (e - 10)
            vals += [base + 0.5 * 2.0 ** (e - 10), -(base + 0.5 * 2.0 ** (e - 10))]
    vals += list(rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000))
    vals = np.array(vals, dtype=np.float64)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f64_to_f16_bits(vals), ref)
    assert oracle.f64_to_f16_bits(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


# ---------------------------------------------------------------- unpacking

def _read_nibble_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "int4_nibble_order.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                b, lo, hi = line.split()
                rows.append((int(b, 16), int(lo), int(hi)))
    return rows


def test_int4_unpack_golden():
    rows = _read_nibble_fixture()
    Wq = np.array([b for b, _, _ in rows], dtype=np.uint8).reshape(1, 1, 16)
    expect = np.array([v for _, lo, hi in rows for v in (lo, hi)], dtype=np.uint8)
    q = oracle.unpack(Wq, 1, 32, 4)
    assert np.array_equal(q[0], expect)


def test_int8_unpack_is_byte_order():
    Wq = np.arange(64, dtype=np.uint8).reshape(2, 1, 32) * 3
    q = oracle.unpack(Wq, 2, 32, 8)
    assert np.array_equal(q, Wq.reshape(2, 32))


def _read_int2_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "int2_code_order.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                parts = line.split()
                rows.append((int(parts[0], 16), [int(v) for v in parts[1:5]], [float(v) for v in parts[5:9]]))
    return rows


def test_int2_unpack_golden():
    rows = _read_int2_fixture()
    Wq = np.array([b for b, _, _ in rows], dtype=np.uint8).reshape(1, 1, 8)
    expect = np.array([c for _, codes, _ in rows for c in codes], dtype=np.uint8)
    assert np.array_equal(oracle.unpack(Wq, 1, 32, 2)[0], expect)


def test_int2_dequant_golden_default_zero_point():
    rows = _read_int2_fixture()
    Wq = np.array([b for b, _, _ in rows], dtype=np.uint8).reshape(1, 1, 8)
    expect = np.array([v for _, _, vals in rows for v in vals]).reshape(1, 32)
    W = oracle.dequant(Wq, f16([[0.25]]), None, 1, 32, 2)
    assert np.array_equal(W, expect)


def test_negative_control_reversed_int2_order_fails_the_golden():
    """Codes read highest bits first would be a plausible mistake: it must not
    pass the golden block."""
    rows = _read_int2_fixture()
    raw = np.array([b for b, _, _ in rows], dtype=np.uint8)
    wrong = np.stack([(raw >> (6 - 2 * i)) & 3 for i in range(4)], axis=1).reshape(-1)
    expect = np.array([c for _, codes, _ in rows for c in codes], dtype=np.uint8)
    assert not np.array_equal(wrong, expect)
    assert np.array_equal(oracle.unpack(raw.reshape(1, 1, 8), 1, 32, 2)[0], expect)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_unpack_roundtrip(bits):
    rng = np.random.default_rng(bits)
    q = rng.integers(0, 1 << bits, size=(5, 96), dtype=np.uint8)
    Wq = oracle.pack(q, bits)
    assert Wq.shape == (5, 3, 32 * bits // 8)
    assert np.array_equal(oracle.unpack(Wq, 5, 96, bits), q)


# ---------------------------------------------------------------- dequant

def test_int4_dequant_golden():
    rows = _read_nibble_fixture()
    Wq = np.array([b for b, _, _ in rows], dtype=np.uint8).reshape(1, 1, 16)
    expect = np.loadtxt(os.path.join(GOLDEN, "int4_dequant_block.txt")).reshape(1, 32)
    scales = f16([[0.5]])
    W = oracle.dequant(Wq, scales, None, 1, 32, 4)
    assert np.array_equal(W, expect)
    W16 = oracle.dequant_f16(Wq, scales, None, 1, 32, 4)
    assert np.array_equal(f16val(W16), expect)


def _codes_numpy(Wq, N, K, bits):
    """Codes decoded with numpy bit operations, independently of the oracle:
    per byte, lowest bits first."""
    raw = Wq.reshape(N, -1).astype(np.int64)
    per = 8 // bits
    codes = np.empty((N, K), dtype=np.int64)
    for i in range(per):
        codes[:, i::per] = (raw >> (bits * i)) & ((1 << bits) - 1)
    return codes


@pytest.mark.parametrize("bits,zp_range", [(2, None), (2, (0, 3)), (4, None), (4, (0, 15)), (8, None),
                                           (8, (120, 136)), (8, (0, 255))])
def test_dequant_exact_vs_rationals(bits, zp_range):
    inp = synth.make_inputs(M=1, K=64, N=6, bits=bits, seed=11, zp_range=zp_range,
                            scale_range=(1e-4, 3.0))
    W = oracle.dequant(inp.Wq, inp.scales, inp.zp, 6, 64, bits)
    codes = _codes_numpy(inp.Wq, 6, 64, bits)
    s = f16val(inp.scales)
    for n in range(6):
        for k in range(64):
            z = (1 << (bits - 1)) if inp.zp is None else int(inp.zp[n, k // 32])
            exact = Fraction(int(codes[n, k]) - z) * Fraction(float(s[n, k // 32]))
            assert Fraction(float(W[n, k])) == exact


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_dequant_f16_is_single_rounding(bits):
    inp = synth.make_inputs(M=1, K=256, N=64, bits=bits, seed=12, zp_range=(0, (1 << bits) - 1),
                            scale_range=(1e-6, 40.0))
    W = oracle.dequant(inp.Wq, inp.scales, inp.zp, 64, 256, bits)
    W16 = oracle.dequant_f16(inp.Wq, inp.scales, inp.zp, 64, 256, bits)
    with np.errstate(over="ignore"):
        assert np.array_equal(W16, W.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------- the product

def test_worked_example_dq_repro_closed_form():
    cfg = json.load(open(os.path.join(GOLDEN, "dq_matmul_repro.json")))
    K, N, bits = cfg["K"], cfg["N"], cfg["bits"]
    q = np.full((N, K), cfg["code"], dtype=np.uint8)
    Wq = oracle.pack(q, bits)
    s16 = f16(np.full((N, K // 32), cfg["scale"]))
    zp = np.full((N, K // 32), cfg["zero_point"], dtype=np.uint8)
    X = f16(np.random.default_rng(3).standard_normal((1, K)))
    Y16, Y64, _ = oracle.run(X, Wq, s16, zp, None, None, N, K, bits)
    sum_x = sum(Fraction(float(v)) for v in f16val(X[0]))
    exact = Fraction(cfg["code"] - cfg["zero_point"]) * Fraction(float(f16val(s16[0, 0]))) * sum_x
    assert np.all(Y64 == float(exact))
    assert np.all(Y16 == np.float64(float(exact)).astype(np.float16).view(np.uint16))


def test_one_hot_rows_recover_dequant_columns():
    inp = synth.make_inputs(M=1, K=64, N=9, bits=4, seed=13, zp_range=(0, 15))
    X = f16(np.eye(64))
    _, Y64, _ = oracle.run(X, inp.Wq, inp.scales, inp.zp, None, None, 9, 64, 4)
    W = oracle.dequant(inp.Wq, inp.scales, inp.zp, 9, 64, 4)
    assert np.array_equal(Y64, W.T)


def _exact_y(inp, round_t=False):
    """Exact rational y for a tiny problem, from numpy-decoded codes."""
    Mt, K, N, bits = inp.batch * inp.M, inp.K, inp.N, inp.bits
    codes = _codes_numpy(inp.Wq, N, K, bits)
    x = [[Fraction(float(v)) for v in row] for row in f16val(inp.X2d)]
    s = f16val(inp.scales)
    w = [[Fraction(int(codes[n, k]) - ((1 << (bits - 1)) if inp.zp is None else int(inp.zp[n, k // 32])))
          * Fraction(float(s[n, k // 32])) for k in range(K)] for n in range(N)]
    y = [[sum(x[m][k] * w[n][k] for k in range(K)) for n in range(N)] for m in range(Mt)]
    if inp.rank:
        A = [[Fraction(float(v)) for v in row] for row in f16val(inp.A)]
        B = [[Fraction(float(v)) for v in row] for row in f16val(inp.B)]
        for m in range(Mt):
            t = [sum(x[m][k] * A[k][r] for k in range(K)) for r in range(inp.rank)]
            for n in range(N):
                y[m][n] += sum(t[r] * B[n][r] for r in range(inp.rank))
    return y


@pytest.mark.parametrize("bits,rank,zp", [(4, 0, None), (4, 32, (0, 15)), (8, 32, (120, 136)), (2, 0, None),
                                         (2, 32, (0, 3))])
def test_brute_force_exact_rationals(bits, rank, zp):
    inp = synth.make_inputs(M=2, K=64, N=5, bits=bits, seed=14, zp_range=zp, rank=rank)
    Y16, Y64, bound = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 5, 64, bits)
    y = _exact_y(inp)
    for m in range(2):
        for n in range(5):
            ex = y[m][n]
            assert abs(Fraction(float(Y64[m, n])) - ex) <= Fraction(1, 10 ** 12) * Fraction(float(bound[m, n]))
            assert Y16[m, n] == np.float64(float(ex)).astype(np.float16).view(np.uint16)


def test_dq_then_matmul_equivalence_transposed_layout():
    """MatMul(X, DequantizeLinear(W[K, N])) equals the N-major MatMulNBits layout."""
    rng = np.random.default_rng(15)
    K, N, bits = 96, 7, 4
    q_kn = rng.integers(0, 16, size=(K, N), dtype=np.uint8)          # DQ weight [K, N]
    zp_bn = rng.integers(0, 16, size=(K // 32, N), dtype=np.uint8)   # per block along K
    s_bn = f16(rng.uniform(0.005, 0.02, size=(K // 32, N)))
    W_kn = (q_kn.astype(np.float64) - np.repeat(zp_bn, 32, axis=0)) * np.repeat(f16val(s_bn), 32, axis=0)
    X = f16(rng.standard_normal((3, K)))
    ref = f16val(X) @ W_kn                                            # numpy matmul, fp64
    Wq = oracle.pack(np.ascontiguousarray(q_kn.T), bits)              # transposed: [N, K/32, 16]
    _, Y64, bound = oracle.run(X, Wq, np.ascontiguousarray(s_bn.T), np.ascontiguousarray(zp_bn.T),
                               None, None, N, K, bits)
    assert np.all(np.abs(Y64 - ref) <= 1e-13 * bound)


def test_codes_equal_zero_point_give_exact_zero_base():
    rng = np.random.default_rng(16)
    N, K = 8, 128
    zp = rng.integers(0, 16, size=(N, K // 32), dtype=np.uint8)
    q = np.repeat(zp, 32, axis=1)
    inp = synth.make_inputs(M=3, K=K, N=N, bits=4, seed=16, rank=32)
    Y16, Y64, _ = oracle.run(inp.X2d, oracle.pack(q, 4), inp.scales, zp, None, None, N, K, 4)
    assert np.all(Y64 == 0.0) and np.all((Y16 & 0x7FFF) == 0)
    # with the adapter the output is exactly the LoRA term
    _, Y64l, bound = oracle.run(inp.X2d, oracle.pack(q, 4), inp.scales, zp, inp.A, inp.B, N, K, 4)
    lora = (f16val(inp.X2d) @ f16val(inp.A)) @ f16val(inp.B).T
    assert np.all(np.abs(Y64l - lora) <= 1e-13 * bound)


def test_constant_offset_closed_form():
    """q - zp == c everywhere  =>  y_n = c * sum_b s[n,b] * sum_{k in b} x_k."""
    rng = np.random.default_rng(17)
    N, K, c = 6, 256, 3
    zp = rng.integers(0, 13, size=(N, K // 32), dtype=np.uint8)
    q = np.repeat(zp + c, 32, axis=1).astype(np.uint8)
    inp = synth.make_inputs(M=4, K=K, N=N, bits=4, seed=17)
    _, Y64, bound = oracle.run(inp.X2d, oracle.pack(q, 4), inp.scales, zp, None, None, N, K, 4)
    xb = f16val(inp.X2d).reshape(4, K // 32, 32).sum(axis=2)          # [M, blocks]
    ref = c * xb @ f16val(inp.scales).T
    assert np.all(np.abs(Y64 - ref) <= 1e-13 * bound)


def test_empty_adapter_is_base_bitwise():
    inp = synth.tiny(M=4, rank=32)
    base = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, 256, 256, 4)
    zero = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, np.zeros((256, 32), np.uint16),
                      np.zeros((256, 32), np.uint16), 256, 256, 4)
    assert np.array_equal(base[0], zero[0]) and np.array_equal(base[1], zero[1])


def test_lora_equals_base_plus_separate_xab():
    inp = synth.tiny(M=4, rank=32)
    _, base, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, 256, 256, 4)
    _, full, bound = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 256, 256, 4)
    xab = (f16val(inp.X2d) @ f16val(inp.A)) @ f16val(inp.B).T
    assert np.all(np.abs(full - (base + xab)) <= 1e-13 * bound)
    T = oracle.lora_down(inp.X2d, inp.A)
    assert np.allclose(T, f16val(inp.X2d) @ f16val(inp.A), rtol=0, atol=1e-12)


def test_partial_adapter_equals_rank16():
    inp = synth.decode_4096(rank=32, partial=True)
    sl = slice(0, 512)   # first 512 output rows keep this quick
    Wq, s, zp, B = inp.Wq[sl], inp.scales[sl], inp.zp[sl], inp.B[sl]
    _, y32, _ = oracle.run(inp.X2d, Wq, s, zp, inp.A, B, 512, 4096, 4)
    _, y16, _ = oracle.run(inp.X2d, Wq, s, zp, np.ascontiguousarray(inp.A[:, :16]),
                           np.ascontiguousarray(B[:, :16]), 512, 4096, 4)
    assert np.array_equal(y32, y16)


def test_rows_are_independent_batch_invariance():
    inp = synth.make_inputs(M=6, K=128, N=16, bits=4, seed=18, batch=2, rank=32)
    full = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 16, 128, 4)
    for b in range(2):
        part = oracle.run(inp.X[b], inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 16, 128, 4)
        assert np.array_equal(part[0], full[0][b * 6:(b + 1) * 6])


def test_exact_arithmetic_case_matches_integer_computation():
    """X in {-1,0,1} (<= 8 nonzeros a row), power-of-two scales, dyadic adapters:
    every intermediate is exact, so the FP16 result is fixed exactly."""
    rng = np.random.default_rng(19)
    M, K, N, r = 3, 128, 12, 32
    x = np.zeros((M, K), dtype=np.int64)
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[m, idx] = rng.choice([-1, 1], 8)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    zp = rng.integers(0, 16, size=(N, K // 32), dtype=np.uint8)
    s_exp = rng.integers(-8, -4, size=(N, K // 32))
    a_int = rng.integers(-3, 4, size=(K, r))
    b_int = rng.integers(-3, 4, size=(N, r))
    scales = f16(np.ldexp(1.0, s_exp))
    A, B = f16(a_int / 16.0), f16(b_int / 16.0)
    _, Y64, _ = oracle.run(f16(x), oracle.pack(q, 4), scales, zp, A, B, N, K, 4)
    Y16, _, _ = oracle.run(f16(x), oracle.pack(q, 4), scales, zp, A, B, N, K, 4)
    for m in range(M):
        for n in range(N):
            base = sum(Fraction(int(x[m, k]) * (int(q[n, k]) - int(zp[n, k // 32])))
                       * Fraction(2) ** int(s_exp[n, k // 32]) for k in range(K))
            t = [sum(int(x[m, k]) * int(a_int[k, j]) for k in range(K)) for j in range(r)]
            lora = Fraction(sum(t[j] * int(b_int[n, j]) for j in range(r)), 256)
            ex = base + lora
            assert Fraction(float(Y64[m, n])) == ex
            assert Y16[m, n] == np.float64(float(ex)).astype(np.float16).view(np.uint16)


def test_bound_is_sum_of_absolute_products():
    inp = synth.tiny(M=1, rank=32)
    _, _, bound = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 256, 256, 4)
    W = oracle.dequant(inp.Wq, inp.scales, inp.zp, 256, 256, 4)
    x = f16val(inp.X2d)
    t = x @ f16val(inp.A)
    ref = np.abs(x[:, None, :] * W[None, :, :]).sum(-1) + np.abs(t[:, None, :] * f16val(inp.B)[None]).sum(-1)
    assert np.allclose(bound, ref, rtol=1e-12, atol=0)


def test_empty_k_gives_zero_output():
    X = np.zeros((2, 0), np.uint16)
    Y16, Y64, _ = oracle.run(X, np.zeros((3, 0, 16), np.uint8), np.zeros((3, 0), np.uint16), None,
                             None, None, 3, 0, 4)
    assert Y16.shape == (2, 3) and np.all(Y16 == 0) and np.all(Y64 == 0)


def test_round_t_matches_fp16_intermediate():
    inp = synth.tiny(M=4, rank=32)
    _, yr, bound = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 256, 256, 4, round_t=True)
    _, base, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, 256, 256, 4)
    t16 = (f16val(inp.X2d) @ f16val(inp.A)).astype(np.float16).astype(np.float64)
    assert np.all(np.abs(yr - (base + t16 @ f16val(inp.B).T)) <= 1e-12 * bound)


# ---------------------------------------------------------------- negative controls

def test_negative_control_swapped_nibbles_fail_the_golden():
    rows = _read_nibble_fixture()
    good = np.array([b for b, _, _ in rows], dtype=np.uint8)
    swapped = ((good & 0x0F) << 4) | (good >> 4)
    expect = np.array([v for _, lo, hi in rows for v in (lo, hi)], dtype=np.uint8)
    q = oracle.unpack(swapped.reshape(1, 1, 16), 1, 32, 4)
    assert not np.array_equal(q[0], expect)


def test_negative_control_dropped_zero_point_fails_closed_form():
    cfg = json.load(open(os.path.join(GOLDEN, "dq_matmul_repro.json")))
    K, N = cfg["K"], cfg["N"]
    Wq = oracle.pack(np.zeros((N, K), np.uint8), 8)
    s16 = f16(np.full((N, K // 32), cfg["scale"]))
    X = f16(np.random.default_rng(3).standard_normal((1, K)))
    _, Y64, _ = oracle.run(X, Wq, s16, None, None, None, N, K, 8)   # zp dropped -> default 128
    sum_x = sum(Fraction(float(v)) for v in f16val(X[0]))
    exact = -3 * Fraction(float(f16val(s16[0, 0]))) * sum_x
    assert not np.all(Y64 == float(exact))


def test_negative_control_untransposed_weight_fails_equivalence():
    rng = np.random.default_rng(15)
    K, N = 64, 64
    q_kn = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = f16(np.full((N, K // 32), 0.01))
    X = f16(rng.standard_normal((2, K)))
    ref = f16val(X) @ ((q_kn.astype(np.float64) - 8) * f16val(s)[0, 0])          # DQ of W[K, N]
    _, Y64, bound = oracle.run(X, oracle.pack(q_kn, 4), s, None, None, None, N, K, 4)  # forgot .T
    assert not np.all(np.abs(Y64 - ref) <= 1e-13 * bound)


# ---------------------------------------------------------------- bias ("[WebGPU] Fuse rank-32 quantized LoRA
# with MatMulNBits", the referenced commit "Support empty packed weights in CPU and WebGPU MatMulNBits",
# Description: the output holds zeros or the broadcast bias)

def _bias_bits(N, seed):
    rng = np.random.default_rng(seed)
    return oracle.f64_to_f16_bits(rng.normal(0.0, 1.0, size=N))


def test_bias_alone_when_every_weight_is_zero():
    # q == zp everywhere: every w is exactly 0, so y[m, n] is exactly bias[n] for every row m
    M, K, N = 3, 64, 40
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=11, zp_range=(0, 15), rank=0)
    q = np.broadcast_to(inp.zp.reshape(N, K // 32, 1), (N, K // 32, 32))
    Wq = oracle.pack(np.ascontiguousarray(q.reshape(N, K)), 4)
    bias = _bias_bits(N, 5)
    Y16, Y64, _ = oracle.run(inp.X2d, Wq, inp.scales, inp.zp, None, None, N, K, 4, bias=bias)
    want = oracle.f16_bits_to_f64(bias)
    assert np.array_equal(Y64, np.broadcast_to(want, (M, N)))
    assert np.array_equal(Y16, np.broadcast_to(bias, (M, N)))


def test_bias_adds_once_after_base_and_adapter():
    inp = synth.make_inputs(M=4, K=128, N=48, bits=4, seed=12, zp_range=(0, 15), rank=32)
    bias = _bias_bits(48, 6)
    _, y0, b0 = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 48, 128, 4)
    y16, y1, b1 = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 48, 128, 4, bias=bias)
    bv = oracle.f16_bits_to_f64(bias)
    assert np.allclose(y1 - y0, np.broadcast_to(bv, y0.shape), rtol=0, atol=1e-12 * (1 + np.abs(y0).max()))
    assert np.allclose(b1 - b0, np.broadcast_to(np.abs(bv), y0.shape), rtol=0, atol=1e-9)
    assert np.array_equal(y16, oracle.f64_to_f16_bits(y1))  # one rounding of the whole sum


def test_no_bias_is_bitwise_the_plain_run():
    inp = synth.make_inputs(M=2, K=64, N=24, bits=8, seed=13, zp_range=(120, 136), rank=32)
    a = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 24, 64, 8)
    b = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, 24, 64, 8, bias=None)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ---------------------------------------------------------------- INT8 adapters

def _qlora_dequant_numpy(q, scales, zp):
    """[rows, nblk, 32] u8 codes -> exact float64 [rows, nblk*32], from numpy
    alone: (q - zp) * scale, zero point 128 when absent."""
    rows, nblk, _ = q.shape
    z = np.full((rows, nblk), 128, np.int64) if zp is None else zp.astype(np.int64)
    s = f16val(scales)
    return ((q.astype(np.int64) - z[:, :, None]) * s[:, :, None]).reshape(rows, nblk * 32)


def _pow2_qlora(K, N, seed, zp=True):
    """INT8 adapters whose dequantized values are exact in FP16: power-of-two
    scales, |q - zp| <= 255 (8 significant bits)."""
    ql = synth.make_qlora(K=K, N=N, seed=seed, zp=zp)
    rng = np.random.default_rng(seed)
    ql.A_scales = f16(np.ldexp(1.0, rng.integers(-14, -10, size=ql.A_scales.shape)))
    ql.B_scales = f16(np.ldexp(1.0, rng.integers(-14, -10, size=ql.B_scales.shape)))
    return ql


@pytest.mark.parametrize("zp", [True, False])
def test_qlora_equals_fp16_adapter_when_dequant_is_exact(zp):
    """With FP16-exact dequantized adapters, the INT8-adapter product equals the
    FP16-adapter product with A = dequant(Aq)^T and B = dequant(Bq), bit for
    bit: the down weight's rows are ranks along K, the up weight's rows are N."""
    K, N, M = 128, 40, 3
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=61, zp_range=(0, 15))
    ql = _pow2_qlora(K, N, 62, zp)
    A = _qlora_dequant_numpy(ql.Aq, ql.A_scales, ql.A_zp)          # [r, K]
    B = _qlora_dequant_numpy(ql.Bq, ql.B_scales, ql.B_zp)          # [N, r]
    A16, B16 = f16(A.T), f16(B)
    assert np.array_equal(f16val(A16), A.T) and np.array_equal(f16val(B16), B)  # exact in FP16
    got = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq, ql.B_scales,
                           ql.B_zp, N, K, 4)
    ref = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, A16, B16, N, K, 4)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_negative_control_untransposed_int8_down_weight_fails():
    """Reading the down weight as [K, r] instead of [r, K] is a plausible
    mistake; it must not reproduce the INT8-adapter product."""
    K, N, M = 32, 24, 2   # K == r, so the wrong reading has the right shape
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=63)
    ql = _pow2_qlora(K, N, 64)
    A = _qlora_dequant_numpy(ql.Aq, ql.A_scales, ql.A_zp)
    B = _qlora_dequant_numpy(ql.Bq, ql.B_scales, ql.B_zp)
    _, got, _ = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                 ql.B_scales, ql.B_zp, N, K, 4)
    _, wrong, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, f16(A), f16(B), N, K, 4)
    _, right, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, f16(A.T), f16(B), N, K, 4)
    assert np.array_equal(got, right) and not np.allclose(got, wrong)


def test_qlora_brute_force_exact_rationals():
    K, N, M = 64, 5, 2
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=65, zp_range=(0, 15))
    ql = synth.make_qlora(K=K, N=N, seed=66)
    Y16, Y64, bound = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                       ql.B_scales, ql.B_zp, N, K, 4)
    base = _exact_y(inp)
    x = [[Fraction(float(v)) for v in row] for row in f16val(inp.X2d)]
    A = [[Fraction(float(v)) for v in row] for row in _qlora_dequant_numpy(ql.Aq, ql.A_scales, ql.A_zp)]
    B = [[Fraction(float(v)) for v in row] for row in _qlora_dequant_numpy(ql.Bq, ql.B_scales, ql.B_zp)]
    for m in range(M):
        t = [sum(x[m][k] * A[r][k] for k in range(K)) for r in range(32)]
        for n in range(N):
            ex = base[m][n] + sum(t[r] * B[n][r] for r in range(32))
            assert abs(Fraction(float(Y64[m, n])) - ex) <= Fraction(1, 10 ** 12) * Fraction(float(bound[m, n]))
            assert Y16[m, n] == np.float64(float(ex)).astype(np.float16).view(np.uint16)


def test_qlora_codes_at_zero_point_is_base_bitwise():
    K, N, M = 96, 33, 3
    inp = synth.make_inputs(M=M, K=K, N=N, bits=8, seed=67, zp_range=(120, 136))
    ql = synth.make_qlora(K=K, N=N, seed=68)
    ql.Aq = np.repeat(ql.A_zp[:, :, None], 32, axis=2)
    ql.Bq = np.repeat(ql.B_zp[:, :, None], 32, axis=2)
    got = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq, ql.B_scales,
                           ql.B_zp, N, K, 8)
    ref = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, N, K, 8)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


# ---------------------------------------------------------------- int8 activations

def _read_act_fixture():
    xs, codes = [], []
    with open(os.path.join(GOLDEN, "int8_activation_blocks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                _, x, c = line.split()
                xs.append(float(x))
                codes.append(int(c))
    return np.array(xs), np.array(codes, dtype=np.int8)


def test_activation_quantization_golden():
    x, codes = _read_act_fixture()
    Xq, Xs = oracle.quantize_x(f16(x.reshape(1, 64)))
    assert np.array_equal(Xq[0], codes)
    # block scales amax / 127 in binary32, computed here with numpy's float32 division
    assert Xs[0, 0] == np.float32(2.0) / np.float32(127.0)
    assert Xs[0, 1] == np.float32(2.0 ** -6)


def test_negative_control_other_roundings_fail_the_activation_golden():
    """Round-half-away-from-zero and truncation are plausible mistakes; both
    disagree with the hand-worked codes."""
    x, codes = _read_act_fixture()
    inv = np.array([63.5] * 32 + [64.0] * 32)
    v = x * inv
    away = np.sign(v) * np.floor(np.abs(v) + 0.5)
    assert not np.array_equal(away.astype(np.int8), codes)
    assert not np.array_equal(np.trunc(v).astype(np.int8), codes)


def test_activation_quantization_error_is_half_a_step():
    X = f16(np.random.default_rng(80).standard_normal((5, 256)) * 3.0)
    Xq, Xs = oracle.quantize_x(X)
    x = f16val(X)
    step = np.repeat(Xs.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(Xq.astype(np.int64)) <= 127)
    assert np.all(np.abs(x - Xq * step) <= 0.5 * step * (1 + 2.0 ** -20))
    # each block's largest magnitude maps to +-127
    amax = np.abs(x).reshape(5, 8, 32).max(axis=2)
    assert np.array_equal(np.abs(Xq).reshape(5, 8, 32).max(axis=2), np.where(amax > 0, 127, 0))


def test_activation_quantization_zero_block_and_power_of_two_scaling():
    rng = np.random.default_rng(81)
    x = rng.standard_normal((1, 64))
    x[0, 32:] = 0.0
    q1, s1 = oracle.quantize_x(f16(x))
    q2, s2 = oracle.quantize_x(f16(x * 4.0))
    assert np.all(q1[0, 32:] == 0) and s1[0, 1] == 0
    assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * 4)


@pytest.mark.parametrize("bits,rank,zp", [(4, 0, (0, 15)), (4, 32, None), (8, 0, (120, 136)), (2, 32, (0, 3))])
def test_q8x_reduces_to_fp16_product_when_x_is_on_the_grid(bits, rank, zp):
    """X whose blocks are integers m in [-127, 127] (with |m| = 127 present)
    times a power of two: quantization is exact (codes m, scale the power of
    two), so the int8-activation product equals the FP16-activation product
    bit for bit (every term and sum is exact in binary64)."""
    M, K, N = 3, 128, 20
    rng = np.random.default_rng(82 + bits + rank)
    m = rng.integers(-127, 128, size=(M, K))
    m[:, ::32] = 127 * rng.choice([-1, 1], size=(M, K // 32))
    c = np.ldexp(1.0, rng.integers(-9, -5, size=(M, K // 32)))
    X = f16(m * np.repeat(c, 32, axis=1))
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=83, zp_range=zp, rank=rank)
    got = oracle.run_q8x(X, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, bits)
    ref = oracle.run(X, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, bits)
    Xq, Xs = oracle.quantize_x(X)
    assert np.array_equal(Xq, m) and np.array_equal(Xs, c.astype(np.float32))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
