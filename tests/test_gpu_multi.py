"""GPU parity of the fused multi-projection call (mnb_run_multi): several
projections of one X, empty members giving zeros or their bias.

Each member's output must equal, bit for bit, the single-projection call on
that member (same route, same per-row arithmetic), and the oracle within the
FP16 tolerance.
"""
import numpy as np
import pytest

from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, dev, oracle_ref, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


def members(Ns, K, bits, zp, seed, M, empty=(), with_bias=()):
    """One synthetic problem per member sharing the first member's X."""
    out = []
    for i, N in enumerate(Ns):
        inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=seed + i, zp_range=zp)
        bias = synth.make_bias(N, seed=seed + 50 + i) if i in with_bias else None
        out.append((inp, bias, i in empty))
    x = out[0][0].X
    for inp, _, _ in out:
        inp.X = x
    return out


def run_multi(mnb, torch, mem, K, bits, M, mode=0, flags=0):
    X = dev(mem[0][0].X, torch)
    projs, Ys = [], []
    for inp, bias, empty in mem:
        d = upload(inp, torch)
        Y = torch.full((1, M, inp.N), 9.0, dtype=torch.float16, device="cuda")
        Ys.append(Y)
        projs.append((inp.N, None if empty else d["Wq"], None if empty else d["scales"],
                      None if empty else d["zp"], dev(bias, torch), Y))
    h = mnb.mnb_create(sum(i.N for i, _, _ in mem), K, bits, max_rank=0, mode=mode, flags=flags)
    try:
        mnb.mnb_run_multi(h, X, projs, 1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0
        route = mnb.mnb_last_route(h)
    finally:
        mnb.mnb_destroy(h)
    return Ys, route


def run_single(mnb, torch, inp, bias, K, bits, M, mode=0, flags=0):
    d = upload(inp, torch)
    h = mnb.mnb_create(inp.N, K, bits, max_rank=0, mode=mode, flags=flags)
    try:
        Y = torch.empty((1, M, inp.N), dtype=torch.float16, device="cuda")
        mnb.mnb_run_bias(h, d["X"], d["Wq"], d["scales"], d["zp"], None, None, 0, dev(bias, torch), Y, None, 1, M)
        torch.cuda.synchronize()
        route = mnb.mnb_last_route(h)
    finally:
        mnb.mnb_destroy(h)
    return Y, route


@pytest.mark.parametrize("Ns,K,bits,zp,M", [
    ((4096, 1024, 1024), 4096, 4, (0, 15), 1),   # QKV of a grouped-query layer, decode
    ((4096, 1024, 1024), 4096, 4, (0, 15), 4),
    ((333, 17, 1000), 576, 8, (120, 136), 3),    # ragged members: each starts on its own 16-row group
    ((14336, 14336), 4096, 4, None, 1),          # MLP gate + up: 3-D TMA boxes per member
    ((2048, 512), 1024, 2, (0, 3), 2),           # 2-bit
    ((4096, 1024, 1024), 4096, 4, (0, 15), 300),  # prefill: one tensor-core launch per member
    ((333, 17, 1000), 576, 8, (120, 136), 40),
    ((100, 64, 250), 96, 4, (0, 15), 2),          # K % 64 == 32
    ((100, 64, 250), 160, 8, None, 33),
])
def test_multi_equals_single_calls_bitwise(env, Ns, K, bits, zp, M):
    torch, mnb = env
    mem = members(Ns, K, bits, zp, seed=1000 + sum(Ns) + M, M=M, with_bias={1})
    Ys, route = run_multi(mnb, torch, mem, K, bits, M)
    assert route == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    for (inp, bias, _), Y in zip(mem, Ys):
        Y1, r1 = run_single(mnb, torch, inp, bias, K, bits, M)
        assert r1 == route
        assert torch.equal(Y, Y1), f"member N={inp.N} differs from its single call"


@pytest.mark.parametrize("M", [1, 64])
def test_multi_with_empty_members(env, M):
    """An empty member gets zeros (or its bias) while the others are computed."""
    torch, mnb = env
    Ns, K = (512, 300, 256, 100), 1024
    mem = members(Ns, K, 4, (0, 15), seed=1100 + M, M=M, empty={1, 3}, with_bias={2, 3})
    Ys, route = run_multi(mnb, torch, mem, K, 4, M)
    assert route == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    for (inp, bias, empty), Y in zip(mem, Ys):
        got = bits_of(Y).reshape(M, inp.N)
        if empty:
            expect = np.broadcast_to(bias, (M, inp.N)) if bias is not None else np.zeros((M, inp.N), np.uint16)
            assert np.array_equal(got, expect)
        else:
            Y64, bound = oracle_ref(inp, bias=bias)
            assert_within_tolerance(got, Y64, bound, f"member N={inp.N}")


def test_multi_all_empty_is_fill(env):
    torch, mnb = env
    mem = members((64, 48), 256, 4, None, seed=1200, M=2, empty={0, 1}, with_bias={0})
    Ys, route = run_multi(mnb, torch, mem, 256, 4, 2)
    assert route == mnb.ROUTE_FILL
    assert np.array_equal(bits_of(Ys[0]).reshape(2, 64), np.broadcast_to(mem[0][1], (2, 64)))
    assert torch.all(Ys[1] == 0)


def test_multi_matches_oracle_early_weights(env):
    """With early weights (the member weights stream before X is ready) the
    fused call still matches the oracle."""
    torch, mnb = env
    Ns, K, M = (2048, 512, 512), 2048, 2
    mem = members(Ns, K, 4, (0, 15), seed=1300, M=M, with_bias={0})
    Ys, route = run_multi(mnb, torch, mem, K, 4, M, flags=mnb.FLAG_EARLY_WEIGHTS)
    assert route == mnb.ROUTE_GEMV
    for (inp, bias, _), Y in zip(mem, Ys):
        Y64, bound = oracle_ref(inp, bias=bias)
        assert_within_tolerance(bits_of(Y).reshape(M, inp.N), Y64, bound, f"member N={inp.N}")


# ------------------------------------------------------------------ DQ -> MatMulNBits rewrite

@pytest.mark.parametrize("M", [1, 200])
def test_dq_rewritten_weight_runs_on_both_routes(env, M):
    """A DequantizeLinear weight [K, N] (the tied lm_head shape of the DQ
    fusion page, 576 x 49152, INT8, per-block scales along K) rewritten on the
    host, then run on the GPU, against X * DequantizeLinear(w) in fp64."""
    torch, mnb = env
    K, N = 576, 49152
    rng = np.random.default_rng(1400 + M)
    w_q = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
    w_scale = np.ascontiguousarray(rng.uniform(0.001, 0.01, size=(K // 32, N)).astype(np.float16)).view(np.uint16)
    w_zp = rng.integers(120, 137, size=(K // 32, N), dtype=np.uint8)
    Wq, scales, zp = mnb.mnb_transpose_dq_weight(w_q, w_scale, w_zp, 8)
    X = np.ascontiguousarray(rng.standard_normal((M, K)).astype(np.float16)).view(np.uint16)
    h = mnb.mnb_create(N, K, 8, max_rank=0)
    try:
        Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
        mnb.mnb_run(h, dev(X, torch), dev(Wq, torch), dev(scales, torch), dev(zp, torch), None, None, 0, Y, None, 1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == (mnb.ROUTE_GEMV if M == 1 else mnb.ROUTE_GEMM)
    finally:
        mnb.mnb_destroy(h)
    cols = np.sort(rng.choice(N, 512, replace=False))
    s = np.repeat(w_scale.view(np.float16).astype(np.float64), 32, axis=0)[:, cols]
    z = np.repeat(w_zp.astype(np.float64), 32, axis=0)[:, cols]
    W = (w_q[:, cols].astype(np.float64) - z) * s
    x = X.view(np.float16).astype(np.float64)
    ref, bound = x @ W, np.abs(x) @ np.abs(W)
    got = bits_of(Y).reshape(M, N)[:, cols].view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-3 * bound + 1e-3)
