"""GPU parity of the int8-activation base (mnb_run_q8x, mnb_quantize_x) against
the CPU oracle, through the C ABI.

The activation codes are integers decided by binary32 arithmetic on both
sides, so codes and scales must match bit for bit; outputs within
|y - y_ref| <= 1e-3 * bound + 1e-3 with bound = sum|xs sw xq (q - zp)| + sum|t B|.
"""
import os

import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, dev, upload

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


def quantize_gpu(mnb, torch, X):
    Mt, K = X.shape
    Xq = torch.empty((Mt, K), dtype=torch.int8, device="cuda")
    Xs = torch.empty((Mt, K // 32), dtype=torch.float32, device="cuda")
    mnb.mnb_quantize_x(dev(X, torch), Mt, K, Xq, Xs)
    torch.cuda.synchronize()
    return Xq.cpu().numpy(), Xs.cpu().numpy()


def test_quantize_x_golden_blocks(env):
    torch, mnb = env
    xs, codes = [], []
    with open(os.path.join(GOLDEN, "int8_activation_blocks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                _, x, c = line.split()
                xs.append(float(x))
                codes.append(int(c))
    X = np.ascontiguousarray(np.array(xs).astype(np.float16).reshape(1, 64)).view(np.uint16)
    Xq, Xs = quantize_gpu(mnb, torch, X)
    assert np.array_equal(Xq[0], np.array(codes, dtype=np.int8))
    assert np.array_equal(Xs, oracle.quantize_x(X)[1])


@pytest.mark.parametrize("Mt,K,scale", [(5, 4096, 1.0), (64, 576, 30.0), (3, 14336, 0.01)])
def test_quantize_x_bit_exact(env, Mt, K, scale):
    torch, mnb = env
    rng = np.random.default_rng(1500 + K)
    x = rng.standard_normal((Mt, K)) * scale
    x[0, :32] = 0.0                    # an all-zero block
    X = np.ascontiguousarray(x.astype(np.float16)).view(np.uint16)
    Xq, Xs = quantize_gpu(mnb, torch, X)
    rq, rs = oracle.quantize_x(X)
    assert np.array_equal(Xq, rq), f"{int((Xq != rq).sum())} codes differ"
    assert np.array_equal(Xs.view(np.uint32), rs.view(np.uint32))


def run_q8x_gpu(mnb, torch, inp, bias=None, d=None):
    d = d or upload(inp, torch)
    Mt = inp.batch * inp.M
    h = mnb.mnb_create(inp.N, inp.K, inp.bits)
    try:
        Y = torch.full((inp.batch, inp.M, inp.N), 7.0, dtype=torch.float16, device="cuda")
        T = torch.empty((Mt, 32), dtype=torch.float16, device="cuda") if inp.rank else None
        mnb.mnb_run_q8x(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"] if inp.rank else None,
                        d["B"] if inp.rank else None, inp.rank, dev(bias, torch), Y, T, inp.batch, inp.M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0
        route = mnb.mnb_last_route(h)
    finally:
        mnb.mnb_destroy(h)
    return Y, route


@pytest.mark.parametrize("M,N,K,bits,zp,rank", [
    (1, 4096, 4096, 4, (0, 15), 32),
    (1, 4096, 4096, 4, None, 0),
    (3, 1000, 576, 8, (120, 136), 0),     # INT8 weights, ragged N
    (8, 333, 896, 8, None, 32),
    (13, 500, 2048, 2, (0, 3), 32),       # two token tiles, 2-bit
    (64, 300, 1024, 4, (0, 15), 0),       # eight token tiles
    (300, 256, 512, 4, None, 32),         # a prefill-size M on the decode kernel
    (1, 4096, 11008, 4, (0, 15), 0),      # a large K (11008 int8 codes per staged token row): two-stage ring
    (3, 300, 96, 4, (0, 15), 32),         # K % 64 == 32: the last 128-byte segment partly past the row
    (9, 130, 160, 8, (120, 136), 0),      # INT8 with K % 64 == 32, two token tiles
])
def test_q8x_matches_oracle(env, M, N, K, bits, zp, rank):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=1600 + M + N, zp_range=zp, rank=rank)
    bias = synth.make_bias(N, seed=1601) if M % 2 else None
    Y, route = run_q8x_gpu(mnb, torch, inp, bias=bias)
    assert route == mnb.ROUTE_GEMV
    _, Y64, bound = oracle.run_q8x(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, bits, bias=bias)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"q8x M={M} N={N} K={K} bits={bits}")


@pytest.mark.parametrize("bits", [4, 8, 2])
def test_q8x_exact_arithmetic_bitwise(env, bits):
    """X on the int8 grid (integers times a power of two per block, |m| = 127
    present) and power-of-two weight scales: every product and sum is exact in
    binary32, so the GPU output equals the oracle's bit for bit."""
    torch, mnb = env
    M, K, N = 9, 512, 300
    rng = np.random.default_rng(1700 + bits)
    m = rng.integers(-6, 7, size=(M, K))
    m[:, ::32] = 127
    c = np.ldexp(1.0, rng.integers(-9, -7, size=(M, K // 32)))
    # |q - zp| <= 136 keeps every block dot within 17 bits and the row sums within binary32's 24
    zp = (120, 136) if bits == 8 else (0, (1 << bits) - 1)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=1701, zp_range=zp)
    inp.X = np.ascontiguousarray((m * np.repeat(c, 32, axis=1)).astype(np.float16)).view(np.uint16).reshape(1, M, K)
    inp.scales = np.ldexp(1.0, rng.integers(-10, -7, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    Y, _ = run_q8x_gpu(mnb, torch, inp)
    Y16, _, _ = oracle.run_q8x(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, N, K, bits)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


def test_q8x_rejects_k_too_large_to_stage(env):
    torch, mnb = env
    K, N = 16384, 64
    h = mnb.mnb_create(N, K, 4)
    try:
        X = torch.zeros((1, K), dtype=torch.float16, device="cuda")
        Wq = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
        S = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
        Y = torch.full((1, N), 5.0, dtype=torch.float16, device="cuda")
        with pytest.raises(mnb.MnbError) as e:
            mnb.mnb_run_q8x(h, X, Wq, S, None, None, None, 0, None, Y, None, 1, 1)
        assert e.value.code == mnb.MNB_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert torch.all(Y == 5.0)
    finally:
        mnb.mnb_destroy(h)


def test_q8x_empty_weight_and_k0(env):
    """The empty-weight and K == 0 rules hold on the int8-activation path too."""
    torch, mnb = env
    bias = synth.make_bias(77, seed=1800)
    h = mnb.mnb_create(77, 64, 4)
    try:
        Y = torch.full((2, 77), 5.0, dtype=torch.float16, device="cuda")
        X = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
        mnb.mnb_run_q8x(h, X, None, None, None, None, None, 0, dev(bias, torch), Y, None, 1, 2)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)
    assert np.array_equal(bits_of(Y).reshape(2, 77), np.broadcast_to(bias, (2, 77)))
