"""Seeded randomized GPU parity: random combinations of bit width, K, N, M,
batch, zero points, bias, adapter format, int8 activations and route, each
checked against the CPU oracle.  The draw is fixed by the seed, so a failure
names a reproducible case."""
import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, dev, upload

pytestmark = pytest.mark.gpu

N_CASES = 48


def draw(i):
    rng = np.random.default_rng([0xF022, i])
    bits = int(rng.choice([2, 4, 8]))
    unit = 64 if bits == 2 else 32
    K = unit * int(rng.integers(1, 2048 // unit + 1))
    N = int(rng.choice([1, 7, 16, 17, 100, 129, 256, 333, 1000, 1536]))
    M = int(rng.choice([1, 2, 3, 5, 8, 9, 16, 17, 40, 100, 300]))
    batch = int(rng.choice([1, 1, 2, 3]))
    while batch * M * N * K > 60_000_000:  # keep the oracle to about a second
        K = max(unit, (K // 2) // unit * unit)
        if batch * M * N * K > 60_000_000 and batch > 1:
            batch = 1
        elif batch * M * N * K > 60_000_000:
            M = max(1, M // 2)
    zp = bool(rng.integers(0, 2))
    adapter = str(rng.choice(["none", "fp16", "int8"]))
    q8x = bool(rng.integers(0, 4) == 0) and adapter != "int8"
    bias = bool(rng.integers(0, 2))
    mode = int(rng.choice([0, 0, 1, 2]))  # auto, auto, force decode, force prefill
    if q8x:
        mode = 0
    return dict(bits=bits, K=K, N=N, M=M, batch=batch, zp=zp, adapter=adapter, q8x=q8x, bias=bias, mode=mode,
                seed=int(rng.integers(0, 2 ** 31)))


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(env, i):
    torch, mnb = env
    c = draw(i)
    bits, K, N, M, batch = c["bits"], c["K"], c["N"], c["M"], c["batch"]
    zr = (0, (1 << bits) - 1) if c["zp"] else None
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=c["seed"], batch=batch, zp_range=zr,
                            rank=32 if c["adapter"] == "fp16" else 0)
    ql = synth.make_qlora(K=K, N=N, seed=c["seed"]) if c["adapter"] == "int8" else None
    bvec = synth.make_bias(N, seed=c["seed"]) if c["bias"] else None
    d = upload(inp, torch)
    Mt = batch * M
    Y = torch.full((batch, M, N), 7.0, dtype=torch.float16, device="cuda")
    T = torch.empty((Mt, 32), dtype=torch.float16, device="cuda") if c["adapter"] != "none" else None
    h = mnb.mnb_create(N, K, bits, 32, 32, c["mode"], 0)
    try:
        if ql is not None:
            q = {k: dev(getattr(ql, k), torch) for k in ("Aq", "A_scales", "A_zp", "Bq", "B_scales", "B_zp")}
            mnb.mnb_run_qlora(h, d["X"], d["Wq"], d["scales"], d["zp"], q["Aq"], q["A_scales"], q["A_zp"], q["Bq"],
                              q["B_scales"], q["B_zp"], 32, dev(bvec, torch), Y, T, batch, M)
        elif c["q8x"]:
            mnb.mnb_run_q8x(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], inp.rank, dev(bvec, torch),
                            Y, T, batch, M)
        else:
            mnb.mnb_run_bias(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], inp.rank, dev(bvec, torch),
                             Y, T, batch, M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == mnb.MNB_OK
    finally:
        mnb.mnb_destroy(h)
    if ql is not None:
        _, Y64, bound = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                         ql.B_scales, ql.B_zp, N, K, bits, bias=bvec)
    elif c["q8x"]:
        _, Y64, bound = oracle.run_q8x(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, bits, bias=bvec)
    else:
        _, Y64, bound = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, bits, bias=bvec)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"case {i}: {c}")
