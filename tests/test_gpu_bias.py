"""GPU parity of the optional bias (mnb_run_bias) on both routes against the
CPU oracle, through the C ABI.

The bias is added to every output row before the one FP16 rounding; with
K = 0 the output is the bias broadcast over the rows; a NULL bias is exactly
mnb_run.  Tolerance as everywhere: |y - y_ref| <= 1e-3 * sum|x w| + 1e-3 with
|bias| counted in the sum.
"""
import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, dev, oracle_ref, run_gpu, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


@pytest.mark.parametrize("M,N,K,bits,zp,rank,mode", [
    (1, 4096, 4096, 4, (0, 15), 32, 0),     # decode, adapter, staged X
    (1, 4096, 4096, 4, (0, 15), 0, 0),
    (3, 1000, 576, 8, (120, 136), 32, 0),   # INT8, ragged N
    (16, 333, 544, 4, None, 0, 0),          # decode with the largest M, last 16-row group partial
    (40, 300, 256, 4, (0, 15), 32, "gemv"),  # forced decode route, several token tiles
    (300, 1000, 96, 4, (0, 15), 32, 0),     # prefill, ragged N and K tail
    (256, 384, 576, 8, (120, 136), 0, 0),   # prefill INT8
    (5, 256, 4096, 4, None, 32, "gemm"),    # forced prefill with few tiles: split-K + cluster reduction
])
def test_bias_matches_oracle(env, M, N, K, bits, zp, rank, mode):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=700 + M + N, zp_range=zp, rank=rank)
    bias = synth.make_bias(N, seed=700 + N)
    m = {0: 0, "gemv": mnb.MODE_FORCE_GEMV, "gemm": mnb.MODE_FORCE_GEMM}[mode]
    if mode == "gemm":
        h = mnb.mnb_create(N, K, bits, 32, 32, m, 0)
        assert mnb.mnb_plan(h, 1, M, rank)["k_splits"] > 1
        mnb.mnb_destroy(h)
    Y, _, route = run_gpu(mnb, torch, inp, mode=m, bias=dev(bias, torch))
    if mode == "gemv":
        assert route == mnb.ROUTE_GEMV
    if mode == "gemm":
        assert route == mnb.ROUTE_GEMM
    Y64, bound = oracle_ref(inp, bias=bias)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"bias M={M} N={N} K={K} bits={bits} rank={rank}")


@pytest.mark.parametrize("M", [1, 1024])
def test_bias_4096_sampled(env, M):
    """The 4096 x 4096 layer with an adapter and a bias on both routes, on
    sampled outputs."""
    torch, mnb = env
    inp = synth.prefill_4096(M=M, rank=32)
    bias = synth.make_bias(inp.N, seed=7)
    Y, _, route = run_gpu(mnb, torch, inp, bias=dev(bias, torch))
    assert route == (mnb.ROUTE_GEMV if M == 1 else mnb.ROUTE_GEMM)
    rng = np.random.default_rng(8)
    rows = np.sort(rng.choice(inp.N, 384, replace=False))
    toks = np.sort(rng.choice(M, min(M, 64), replace=False))
    Y64, bound = oracle_ref(inp, rows=rows, tokens=toks, bias=bias)
    got = bits_of(Y).reshape(M, inp.N)[np.ix_(toks, rows)]
    assert_within_tolerance(got, Y64, bound, f"bias 4096 M={M}")


@pytest.mark.parametrize("M,mode", [(2, 0), (600, 0), (5, "gemm")])
def test_null_bias_is_plain_run_bitwise(env, M, mode):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=512, N=640, bits=4, seed=710 + M, zp_range=(0, 15), rank=32)
    m = mnb.MODE_FORCE_GEMM if mode == "gemm" else 0
    d = upload(inp, torch)
    Y0, _, r0 = run_gpu(mnb, torch, inp, d=d, mode=m)
    h = mnb.mnb_create(inp.N, inp.K, 4, 32, 32, m, 0)
    try:
        Y1 = torch.empty_like(Y0)
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run_bias(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, None, Y1, T, 1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0 and mnb.mnb_last_route(h) == r0
    finally:
        mnb.mnb_destroy(h)
    assert torch.equal(Y0, Y1)


def test_zero_bias_is_plain_run_bitwise(env):
    """A bias of +0 changes no output bit: s + 0 = s for every FP32 sum s
    except s = -0, so only outputs that are exactly zero may differ (in sign)."""
    torch, mnb = env
    inp = synth.make_inputs(M=3, K=1024, N=500, bits=4, seed=720, zp_range=(0, 15), rank=32)
    d = upload(inp, torch)
    Y0, _, _ = run_gpu(mnb, torch, inp, d=d)
    Y1, _, _ = run_gpu(mnb, torch, inp, d=d, bias=torch.zeros(inp.N, dtype=torch.float16, device="cuda"))
    nz = Y0 != 0
    assert torch.equal(Y0[nz], Y1[nz])


def test_k0_bias_broadcast_bitwise(env):
    torch, mnb = env
    N, Mt = 77, 5
    bias = synth.make_bias(N, seed=730)
    h = mnb.mnb_create(N, 0, 4)
    try:
        Y = torch.full((Mt, N), 5.0, dtype=torch.float16, device="cuda")
        X = torch.empty((Mt, 0), dtype=torch.float16, device="cuda")
        mnb.mnb_run_bias(h, X, X, X, None, None, None, 0, dev(bias, torch), Y, None, 1, Mt)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)
    Y16, _, _ = oracle.run(np.zeros((Mt, 0), np.uint16), np.zeros((N, 0, 16), np.uint8),
                           np.zeros((N, 0), np.uint16), None, None, None, N, 0, 4, bias=bias)
    assert np.array_equal(bits_of(Y).reshape(Mt, N), Y16)
    assert np.array_equal(Y16, np.broadcast_to(bias, (Mt, N)))


@pytest.mark.parametrize("M", [5, 300])
def test_bias_exact_arithmetic_bitwise(env, M):
    """Sparse {-1,0,1} activations, power-of-two scales, dyadic adapters and
    bias: every partial sum is exact in FP32, so both routes match the oracle
    bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(740 + M)
    K, N = 1024, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=740 + M, zp_range=(0, 15), rank=32)
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    inp.A = (rng.integers(-3, 4, size=(K, 32)) / 16.0).astype(np.float16).view(np.uint16)
    inp.B = (rng.integers(-3, 4, size=(N, 32)) / 16.0).astype(np.float16).view(np.uint16)
    bias = (rng.integers(-64, 65, size=N) / 32.0).astype(np.float16).view(np.uint16)
    Y, _, route = run_gpu(mnb, torch, inp, bias=dev(bias, torch))
    assert route == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, 4, bias=bias)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


def test_misaligned_bias_is_rejected_before_launch(env):
    torch, mnb = env
    inp = synth.make_inputs(M=1, K=256, N=256, bits=4, seed=750)
    d = upload(inp, torch)
    buf = torch.zeros(inp.N + 8, dtype=torch.float16, device="cuda")
    Y = torch.full((1, 1, inp.N), 3.0, dtype=torch.float16, device="cuda")
    h = mnb.mnb_create(inp.N, inp.K, 4)
    try:
        with pytest.raises(mnb.MnbError) as e:
            mnb.mnb_run_bias(h, d["X"], d["Wq"], d["scales"], d["zp"], None, None, 0, buf[1:], Y, None, 1, 1)
        assert e.value.code == mnb.MNB_ERR_ALIGN
    finally:
        mnb.mnb_destroy(h)
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0)


# ------------------------------------------------------------------ empty packed weights

@pytest.mark.parametrize("M", [1, 300])
@pytest.mark.parametrize("with_bias", [False, True])
def test_empty_weight_is_zeros_or_bias_bitwise(env, M, with_bias):
    """Wq NULL with K > 0: the output keeps its logical shape and holds zeros
    or the broadcast bias, on what would be either route."""
    torch, mnb = env
    N, K = 333, 256
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=760 + M)
    bias = synth.make_bias(N, seed=761)
    h = mnb.mnb_create(N, K, 4)
    try:
        Y = torch.full((1, M, N), 5.0, dtype=torch.float16, device="cuda")
        X = dev(inp.X, torch)
        mnb.mnb_run_bias(h, X, None, None, None, None, None, 0, dev(bias, torch) if with_bias else None, Y, None,
                         1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)
    expect = np.broadcast_to(bias, (M, N)) if with_bias else np.zeros((M, N), np.uint16)
    assert np.array_equal(bits_of(Y).reshape(M, N), expect)


@pytest.mark.parametrize("M", [1, 40])
def test_empty_weight_with_adapter_is_adapter_term(env, M):
    """Wq NULL with an adapter: Y = T * B^T + bias, against the oracle with a
    zero base (every code equal to its zero point gives an exactly zero base)."""
    torch, mnb = env
    N, K = 500, 1024
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=770 + M, rank=32)
    bias = synth.make_bias(N, seed=771)
    d = upload(inp, torch)
    h = mnb.mnb_create(N, K, 4)
    try:
        Y = torch.full((1, M, N), 5.0, dtype=torch.float16, device="cuda")
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run_bias(h, d["X"], None, None, None, d["A"], d["B"], 32, dev(bias, torch), Y, T, 1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0 and mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)
    zero_codes = oracle.pack(np.full((N, K), 8, dtype=np.uint8), 4)
    _, Y64, bound = oracle.run(inp.X2d, zero_codes, inp.scales, None, inp.A, inp.B, N, K, 4, bias=bias)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"empty weight + adapter M={M}")
