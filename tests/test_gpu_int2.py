"""GPU parity of 2-bit weights (four codes per byte, lowest bits first, default
zero point 2) on the dequant step and both routes against the CPU oracle,
through the C ABI.

Dequantization must be bit-exact; outputs must satisfy
|y - y_ref| <= 1e-3 * sum|x w| + 1e-3.
"""
import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, oracle_ref, run_gpu, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


@pytest.mark.parametrize("zp_range,N,K", [(None, 256, 256), ((0, 3), 300, 4096), ((0, 255), 17, 192),
                                          (None, 33, 64)])
@pytest.mark.parametrize("variant", [0, 1])
def test_int2_dequant_bit_exact(env, zp_range, N, K, variant):
    torch, mnb = env
    inp = synth.make_inputs(M=1, K=K, N=N, bits=2, seed=800 + N, zp_range=zp_range, scale_range=(1e-5, 30.0))
    d = upload(inp, torch)
    W16 = torch.empty((N, K), dtype=torch.float16, device="cuda")
    mnb.mnb_dequant(d["Wq"], d["scales"], d["zp"], N, K, 2, W16, variant)
    torch.cuda.synchronize()
    ref = oracle.dequant_f16(inp.Wq, inp.scales, inp.zp, N, K, 2)
    got = bits_of(W16)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} dequantized values differ"


@pytest.mark.parametrize("M,N,K,zp,rank", [
    (1, 4096, 4096, (0, 3), 32),   # decode, staged X, one chunk per row
    (1, 4096, 4096, None, 0),
    (3, 1000, 576, (0, 3), 32),    # ragged N, staged X
    (12, 333, 2048, (0, 3), 32),   # two token tiles, X read from global memory
    (16, 130, 128, None, 0),
    (1, 2048, 14336, (0, 3), 0),   # rows of 3584 bytes: 3-D TMA boxes of 1 KB per row
    (2, 200, 4160, None, 32),      # rows of 1040 bytes: per-row copies, a 16-byte last chunk
])
def test_int2_decode_matches_oracle(env, M, N, K, zp, rank):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=2, seed=810 + M + N, zp_range=zp, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"int2 decode M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K,zp,rank,mode", [
    (64, 256, 256, None, 32, 0),
    (300, 1000, 576, (0, 3), 32, 0),   # ragged N
    (513, 200, 128, None, 0, 0),       # three token tiles, the last one ragged
    (40, 130, 896, (0, 255), 32, 0),
    (5, 256, 4096, (0, 3), 32, "gemm"),  # forced prefill with few tiles: split-K + cluster reduction
])
def test_int2_prefill_matches_oracle(env, M, N, K, zp, rank, mode):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=2, seed=820 + M + N, zp_range=zp, rank=rank)
    m = mnb.MODE_FORCE_GEMM if mode == "gemm" else 0
    if mode == "gemm":
        h = mnb.mnb_create(N, K, 2, 32, 32, m, 0)
        assert mnb.mnb_plan(h, 1, M, rank)["k_splits"] > 1
        mnb.mnb_destroy(h)
    Y, _, route = run_gpu(mnb, torch, inp, mode=m)
    assert route == mnb.ROUTE_GEMM
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"int2 prefill M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 1024])
def test_int2_mlp_up_sampled(env, M):
    """K = 4096, N = 14336 with 2-bit weights on both routes, sampled outputs."""
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=4096, N=14336, bits=2, seed=830 + M, zp_range=(0, 3), rank=32)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == (mnb.ROUTE_GEMV if M == 1 else mnb.ROUTE_GEMM)
    rng = np.random.default_rng(831)
    rows = np.sort(rng.choice(inp.N, 256, replace=False))
    toks = np.sort(rng.choice(M, min(M, 48), replace=False))
    Y64, bound = oracle_ref(inp, rows=rows, tokens=toks)
    got = bits_of(Y).reshape(M, inp.N)[np.ix_(toks, rows)]
    assert_within_tolerance(got, Y64, bound, f"int2 mlp_up M={M}")


@pytest.mark.parametrize("M", [4, 200])
def test_int2_exact_arithmetic_bitwise(env, M):
    """Sparse {-1,0,1} activations, power-of-two scales and dyadic adapters:
    every partial sum is exact in FP32, so both routes match the oracle bit
    for bit -- which also pins the code order of the unpacking."""
    torch, mnb = env
    rng = np.random.default_rng(840 + M)
    K, N = 1024, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=2, seed=840 + M, zp_range=(0, 3), rank=32)
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    inp.A = (rng.integers(-3, 4, size=(K, 32)) / 16.0).astype(np.float16).view(np.uint16)
    inp.B = (rng.integers(-3, 4, size=(N, 32)) / 16.0).astype(np.float16).view(np.uint16)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, 2)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


def test_int2_routes_agree_within_tolerance(env):
    torch, mnb = env
    inp = synth.make_inputs(M=9, K=512, N=384, bits=2, seed=850, zp_range=(0, 3), rank=32)
    d = upload(inp, torch)
    Yv, _, rv = run_gpu(mnb, torch, inp, d=d, mode=mnb.MODE_FORCE_GEMV)
    Ym, _, rm = run_gpu(mnb, torch, inp, d=d, mode=mnb.MODE_FORCE_GEMM)
    assert (rv, rm) == (mnb.ROUTE_GEMV, mnb.ROUTE_GEMM)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Yv), Y64, bound, "int2 forced decode")
    assert_within_tolerance(bits_of(Ym), Y64, bound, "int2 forced prefill")
