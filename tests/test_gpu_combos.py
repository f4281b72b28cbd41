"""GPU parity across features: batch invariance of the newer paths (2-bit
weights, int8 activations, INT8 adapters), batched multi-projection calls and
combinations of bias, adapters and bit widths, against the CPU oracle."""
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


def flat(inp):
    """The same rows as one matrix of batch * M rows."""
    f = synth.Inputs(X=inp.X.reshape(1, inp.batch * inp.M, inp.K), Wq=inp.Wq, scales=inp.scales, zp=inp.zp,
                     A=inp.A, B=inp.B, batch=1, M=inp.batch * inp.M, N=inp.N, K=inp.K, bits=inp.bits)
    return f


@pytest.mark.parametrize("bits,M,batch", [(2, 3, 4), (2, 300, 2)])
def test_int2_batch_invariance_bitwise(env, bits, M, batch):
    """[batch, M] equals one matrix of batch*M rows routed the same way."""
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=512, N=640, bits=bits, seed=2000 + M, batch=batch, zp_range=(0, 3), rank=32)
    mode = mnb.MODE_FORCE_GEMV if M <= 16 else mnb.MODE_FORCE_GEMM
    Yb, _, _ = run_gpu(mnb, torch, inp, mode=mode)
    Yf, _, _ = run_gpu(mnb, torch, flat(inp), mode=mode)
    assert torch.equal(Yb.reshape(-1, inp.N), Yf.reshape(-1, inp.N))


def test_q8x_batch_invariance_bitwise(env):
    torch, mnb = env
    inp = synth.make_inputs(M=5, K=1024, N=500, bits=4, seed=2010, batch=3, zp_range=(0, 15), rank=32)
    outs = []
    for x in (inp, flat(inp)):
        d = upload(x, torch)
        h = mnb.mnb_create(x.N, x.K, 4)
        try:
            Y = torch.empty((x.batch, x.M, x.N), dtype=torch.float16, device="cuda")
            T = torch.empty((x.batch * x.M, 32), dtype=torch.float16, device="cuda")
            mnb.mnb_run_q8x(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, None, Y, T, x.batch, x.M)
            torch.cuda.synchronize()
        finally:
            mnb.mnb_destroy(h)
        outs.append(Y.reshape(-1, x.N))
    assert torch.equal(outs[0], outs[1])
    _, Y64, bound = oracle.run_q8x(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, inp.N, inp.K, 4)
    assert_within_tolerance(bits_of(outs[0]), Y64, bound, "q8x batched")


@pytest.mark.parametrize("M,batch,bits", [(2, 4, 4), (256, 2, 2)])
def test_qlora_batched_with_bias(env, M, batch, bits):
    torch, mnb = env
    K, N = 1024, 384
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=2020 + M, batch=batch,
                            zp_range=(0, (1 << bits) - 1))
    ql = synth.make_qlora(K=K, N=N, seed=2021)
    bias = synth.make_bias(N, seed=2022)
    d = upload(inp, torch)
    q = {k: dev(getattr(ql, k), torch) for k in ("Aq", "A_scales", "A_zp", "Bq", "B_scales", "B_zp")}
    h = mnb.mnb_create(N, K, bits)
    try:
        Y = torch.empty((batch, M, N), dtype=torch.float16, device="cuda")
        T = torch.empty((batch * M, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run_qlora(h, d["X"], d["Wq"], d["scales"], d["zp"], q["Aq"], q["A_scales"], q["A_zp"], q["Bq"],
                          q["B_scales"], q["B_zp"], 32, dev(bias, torch), Y, T, batch, M)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    finally:
        mnb.mnb_destroy(h)
    _, Y64, bound = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                     ql.B_scales, ql.B_zp, N, K, bits, bias=bias)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"qlora batched M={M} bits={bits}")


@pytest.mark.parametrize("M,batch", [(3, 2), (100, 3)])
def test_multi_batched_with_biases(env, M, batch):
    """Two projections of a batched X, each with a bias, against the oracle."""
    torch, mnb = env
    K, Ns = 512, (384, 200)
    inps = [synth.make_inputs(M=M, K=K, N=n, bits=4, seed=2030 + i, batch=batch, zp_range=(0, 15))
            for i, n in enumerate(Ns)]
    for x in inps[1:]:
        x.X = inps[0].X
    biases = [synth.make_bias(n, seed=2040 + i) for i, n in enumerate(Ns)]
    X = dev(inps[0].X, torch)
    Ys, projs = [], []
    for x, b in zip(inps, biases):
        d = upload(x, torch)
        Y = torch.empty((batch, M, x.N), dtype=torch.float16, device="cuda")
        Ys.append(Y)
        projs.append((x.N, d["Wq"], d["scales"], d["zp"], dev(b, torch), Y))
    h = mnb.mnb_create(sum(Ns), K, 4, max_rank=0)
    try:
        mnb.mnb_run_multi(h, X, projs, batch, M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == mnb.MNB_OK
    finally:
        mnb.mnb_destroy(h)
    for x, b, Y in zip(inps, biases, Ys):
        Y64, bound = oracle_ref(x, bias=b)
        assert_within_tolerance(bits_of(Y).reshape(-1, x.N), Y64, bound, f"multi batched N={x.N}")
