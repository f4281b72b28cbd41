"""GPU parity of the prefill (tcgen05 GEMM) route against the CPU oracle,
through the C ABI: |y - y_ref| <= 1e-3 * sum|x w| + 1e-3, bitwise identities
where the arithmetic is exact, and the route chosen from the per-matrix M."""
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


def sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, min(n, k), replace=False))


@pytest.mark.parametrize("M,N,K,bits,zp,rank", [
    (64, 256, 256, 4, None, 32),
    (17, 256, 256, 4, None, 32),       # smallest prefill M: token tile 32
    (300, 1000, 96, 4, (0, 15), 32),   # ragged N (not a multiple of 128), K tail of half a step
    (256, 384, 576, 8, (120, 136), 0),  # INT8 lm_head-like K
    (40, 130, 896, 8, None, 32),
    (513, 200, 160, 4, (0, 255), 0),   # three token tiles, the last one ragged
])
def test_prefill_small_full_oracle(env, M, N, K, bits, zp, rank):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=500 + M + N, zp_range=zp, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMM
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"prefill M={M} N={N} K={K} bits={bits}")


@pytest.mark.parametrize("rank", [32, 0])
def test_prefill_4096_sampled(env, rank):
    torch, mnb = env
    inp = synth.prefill_4096(M=1024, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMM
    rows, toks = sample(inp.N, 384, 1), sample(1024, 96, 2)
    Y64, bound = oracle_ref(inp, rows=rows, tokens=toks)
    got = bits_of(Y).reshape(1024, inp.N)[np.ix_(toks, rows)]
    assert_within_tolerance(got, Y64, bound, f"prefill 4096 rank={rank}")


def test_prefill_batch_of_two_is_one_matrix_bitwise(env):
    """[2, 512, K] and [1, 1024, K] take the prefill route and agree bit for bit."""
    torch, mnb = env
    inp2 = synth.prefill_4096(M=512, batch=2, rank=32)
    d = upload(inp2, torch)
    Y2, _, r2 = run_gpu(mnb, torch, inp2, d=d)
    inp1 = synth.prefill_4096(M=512, batch=2, rank=32)
    inp1.X = inp1.X.reshape(1, 1024, 4096)
    inp1.batch, inp1.M = 1, 1024
    d1 = dict(d, X=d["X"].reshape(1, 1024, 4096))
    Y1, _, r1 = run_gpu(mnb, torch, inp1, d=d1)
    assert r1 == r2 == mnb.ROUTE_GEMM
    assert torch.equal(Y1.reshape(1024, -1), Y2.reshape(1024, -1))


def test_prefill_matches_decode_route_within_tolerance(env):
    torch, mnb = env
    inp = synth.make_inputs(M=48, K=1024, N=512, bits=4, seed=601, zp_range=(0, 15), rank=32)
    Yg, _, rg = run_gpu(mnb, torch, inp, mode=mnb.MODE_FORCE_GEMM)
    Yv, _, rv = run_gpu(mnb, torch, inp, mode=mnb.MODE_FORCE_GEMV)
    assert (rg, rv) == (mnb.ROUTE_GEMM, mnb.ROUTE_GEMV)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Yg), Y64, bound, "forced gemm")
    assert_within_tolerance(bits_of(Yv), Y64, bound, "forced gemv")


@pytest.mark.parametrize("M", [1, 5, 16])
def test_force_gemm_few_tokens(env, M):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=512, N=640, bits=4, seed=602 + M, zp_range=(0, 15), rank=32)
    Y, _, route = run_gpu(mnb, torch, inp, mode=mnb.MODE_FORCE_GEMM)
    assert route == mnb.ROUTE_GEMM
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"force gemm M={M}")


@pytest.mark.parametrize("M", [64, 256, 1024, 4096])
@pytest.mark.parametrize("rank", [32, 0])
def test_mlp_up_prefill_sampled(env, M, rank):
    torch, mnb = env
    inp = synth.mlp_up(M=M, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMM
    rows, toks = sample(inp.N, 256, M), sample(M, 48, M + 1)
    Y64, bound = oracle_ref(inp, rows=rows, tokens=toks)
    got = bits_of(Y).reshape(M, inp.N)[np.ix_(toks, rows)]
    assert_within_tolerance(got, Y64, bound, f"mlp_up prefill M={M} rank={rank}")


def test_prefill_exact_arithmetic_bitwise(env):
    torch, mnb = env
    rng = np.random.default_rng(603)
    M, K, N = 70, 512, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=603, zp_range=(0, 15), rank=32)
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    inp.A = (rng.integers(-3, 4, size=(K, 32)) / 16.0).astype(np.float16).view(np.uint16)
    inp.B = (rng.integers(-3, 4, size=(N, 32)) / 16.0).astype(np.float16).view(np.uint16)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMM
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


def test_prefill_deterministic_and_guarded(env):
    torch, mnb = env
    inp = synth.make_inputs(M=200, K=256, N=260, bits=4, seed=604, rank=32)
    d = upload(inp, torch)
    pad = 8192
    Ybuf = torch.full((200 * 260 + 2 * pad,), 7.0, dtype=torch.float16, device="cuda")
    Y = Ybuf[pad:pad + 200 * 260].view(1, 200, 260)
    run_gpu(mnb, torch, inp, d=d, Y=Y)
    Y2, _, _ = run_gpu(mnb, torch, inp, d=d)
    assert torch.equal(Y, Y2)
    assert torch.all(Ybuf[:pad] == 7.0) and torch.all(Ybuf[pad + 200 * 260:] == 7.0)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, "guarded prefill")


@pytest.mark.parametrize("M", [100, 64])
def test_prefill_adapter_down_on_idle_sms_exact(env, M):
    """A one-wave prefill grid well short of the SM count (80 weight tiles): the LoRA down
    projection runs on the idle SMs, one CTA summing all of K for a group of 64 token rows
    (M=100: a full group and a ragged one).  Exact arithmetic, so T and Y match the oracle
    bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(605 + M)
    K, N = 512, 10240
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    h = mnb.mnb_create(N, K, 4, 32, 32)
    try:
        p = mnb.mnb_plan(h, 1, M, 32, sms)
    finally:
        mnb.mnb_destroy(h)
    assert p["route"] == mnb.ROUTE_GEMM and p["k_splits"] <= 1 and sms - p["grid_x"] >= 8
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=605 + M, zp_range=(0, 15), rank=32)
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    inp.A = (rng.integers(-3, 4, size=(K, 32)) / 16.0).astype(np.float16).view(np.uint16)
    inp.B = (rng.integers(-3, 4, size=(N, 32)) / 16.0).astype(np.float16).view(np.uint16)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMM
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)
