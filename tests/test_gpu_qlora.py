"""GPU parity of INT8 block-32 rank-32 adapters (mnb_run_qlora) on both routes
against the CPU oracle, through the C ABI.

The adapters are 8-bit MatMulNBits weights (down Aq [32, K], up Bq [N, 32]);
the GPU dequantizes them with one FP16 rounding and keeps T in FP16, the
oracle keeps both exact.  Tolerance: |y - y_ref| <= 1e-3 * bound + 1e-3 with
bound = sum|x w| + sum|t b| (+ |bias|).
"""
import numpy as np
import pytest

import oracle
from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, dev, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb.lib()
    return torch, mnb


def run_qlora_gpu(mnb, torch, inp, ql, bias=None, mode=0, d=None):
    d = d or upload(inp, torch)
    q = {k: dev(getattr(ql, k), torch) for k in ("Aq", "A_scales", "A_zp", "Bq", "B_scales", "B_zp")}
    Mt = inp.batch * inp.M
    h = mnb.mnb_create(inp.N, inp.K, inp.bits, 32, 32, mode, 0)
    try:
        Y = torch.full((inp.batch, inp.M, inp.N), 7.0, dtype=torch.float16, device="cuda")
        T = torch.empty((Mt, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run_qlora(h, d["X"], d["Wq"], d["scales"], d["zp"], q["Aq"], q["A_scales"], q["A_zp"], q["Bq"],
                          q["B_scales"], q["B_zp"], 32, None if bias is None else dev(bias, torch), Y, T,
                          inp.batch, inp.M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0
        route = mnb.mnb_last_route(h)
    finally:
        mnb.mnb_destroy(h)
    return Y, T, route


def oracle_qlora(inp, ql, rows=None, tokens=None, bias=None):
    X = inp.X2d if tokens is None else inp.X2d[tokens]
    Wq, S, Z = inp.Wq, inp.scales, inp.zp
    Bq, Bs, Bz = ql.Bq, ql.B_scales, ql.B_zp
    if rows is not None:
        Wq, S = Wq[rows], S[rows]
        Z = None if Z is None else Z[rows]
        Bq, Bs = Bq[rows], Bs[rows]
        Bz = None if Bz is None else Bz[rows]
        bias = None if bias is None else bias[rows]
    _, Y64, bound = oracle.run_qlora(X, Wq, S, Z, ql.Aq, ql.A_scales, ql.A_zp, Bq, Bs, Bz, Wq.shape[0], inp.K,
                                     inp.bits, bias=bias)
    return Y64, bound


@pytest.mark.parametrize("M,N,K,bits,zp,qzp,mode", [
    (1, 4096, 4096, 4, (0, 15), True, 0),     # decode, staged X
    (1, 4096, 4096, 4, None, False, 0),       # default zero points everywhere
    (3, 1000, 576, 8, (120, 136), True, 0),   # INT8 base, ragged N: the last group's scales need tail bytes
    (13, 333, 2048, 4, (0, 15), False, 0),    # two token tiles, X from global memory
    (1, 2048, 4096, 2, (0, 3), True, 0),      # 2-bit base
    (300, 1000, 96, 4, (0, 15), True, 0),     # prefill, ragged N and K tail
    (256, 384, 576, 8, (120, 136), False, 0),
    (5, 256, 4096, 4, None, True, "gemm"),    # forced prefill with few tiles: split-K, LoRA in the last split
])
def test_qlora_matches_oracle(env, M, N, K, bits, zp, qzp, mode):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=900 + M + N, zp_range=zp)
    ql = synth.make_qlora(K=K, N=N, seed=901 + N, zp=qzp)
    m = mnb.MODE_FORCE_GEMM if mode == "gemm" else 0
    Y, T, route = run_qlora_gpu(mnb, torch, inp, ql, mode=m)
    assert route == (mnb.ROUTE_GEMV if (M <= 16 and mode != "gemm") else mnb.ROUTE_GEMM)
    Y64, bound = oracle_qlora(inp, ql)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"qlora M={M} N={N} K={K} bits={bits}")


def test_qlora_T_is_the_fp16_down_projection(env):
    """T_ws holds fp16(X * a) with a = fp16 dequant of Aq: checked against the
    oracle's exact T of the FP16-dequantized down weight (one FP16 rounding
    plus FP32 summation apart)."""
    torch, mnb = env
    M, N, K = 7, 256, 4096
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=910)
    ql = synth.make_qlora(K=K, N=N, seed=911)
    _, T, _ = run_qlora_gpu(mnb, torch, inp, ql)
    a16 = oracle.dequant_f16(ql.Aq, ql.A_scales, ql.A_zp, 32, K, 8)          # [32, K] FP16 bits
    T64 = oracle.lora_down(inp.X2d, np.ascontiguousarray(a16.T))
    got = bits_of(T).view(np.float16).astype(np.float64).reshape(M, 32)
    x = oracle.f16_bits_to_f64(inp.X2d)
    mag = np.abs(x) @ np.abs(oracle.f16_bits_to_f64(a16)).T
    assert np.all(np.abs(got - T64) <= 1e-3 * mag + 1e-6)


@pytest.mark.parametrize("M", [1, 1024])
def test_qlora_4096_sampled_with_bias(env, M):
    torch, mnb = env
    inp = synth.prefill_4096(M=M, rank=0)
    ql = synth.make_qlora(K=4096, N=4096, seed=920)
    bias = synth.make_bias(4096, seed=921)
    Y, _, route = run_qlora_gpu(mnb, torch, inp, ql, bias=bias)
    assert route == (mnb.ROUTE_GEMV if M == 1 else mnb.ROUTE_GEMM)
    rng = np.random.default_rng(922)
    rows = np.sort(rng.choice(inp.N, 384, replace=False))
    toks = np.sort(rng.choice(M, min(M, 64), replace=False))
    Y64, bound = oracle_qlora(inp, ql, rows=rows, tokens=toks, bias=bias)
    got = bits_of(Y).reshape(M, inp.N)[np.ix_(toks, rows)]
    assert_within_tolerance(got, Y64, bound, f"qlora 4096 M={M}")


@pytest.mark.parametrize("M", [1, 5, 300])
def test_qlora_exact_arithmetic_bitwise(env, M):
    """Sparse {-1,0,1} X, power-of-two scales everywhere and adapter codes near
    their zero points: every value and partial sum is exact in FP16/FP32, so
    both routes match the oracle bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(930 + M)
    K, N = 1024, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=930 + M, zp_range=(0, 15))
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    ql = synth.make_qlora(K=K, N=N, seed=931)
    ql.Aq = (ql.A_zp[:, :, None] + rng.integers(-3, 4, size=ql.Aq.shape)).astype(np.uint8)
    ql.Bq = (ql.B_zp[:, :, None] + rng.integers(-3, 4, size=ql.Bq.shape)).astype(np.uint8)
    ql.A_scales = np.full(ql.A_scales.shape, 0x2C00, np.uint16)  # 1/16
    ql.B_scales = np.full(ql.B_scales.shape, 0x2C00, np.uint16)
    Y, T, route = run_qlora_gpu(mnb, torch, inp, ql)
    assert route == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    Y16, _, _ = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                 ql.B_scales, ql.B_zp, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)
    if M == 1:  # the single-token kernel (adapter dequantized in its adapter warp): T exact too
        a16 = oracle.dequant_f16(ql.Aq, ql.A_scales, ql.A_zp, 32, K, 8)
        T64 = oracle.lora_down(inp.X2d, np.ascontiguousarray(a16.T))
        assert np.array_equal(bits_of(T).view(np.float16).astype(np.float64).reshape(M, 32), T64)


@pytest.mark.parametrize("M", [2, 64])
def test_qlora_with_empty_base_weight(env, M):
    """Wq NULL with INT8 adapters: the adapter term alone."""
    torch, mnb = env
    N, K = 500, 1024
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=940 + M)
    ql = synth.make_qlora(K=K, N=N, seed=941)
    q = {k: dev(getattr(ql, k), torch) for k in ("Aq", "A_scales", "A_zp", "Bq", "B_scales", "B_zp")}
    h = mnb.mnb_create(N, K, 4)
    try:
        Y = torch.full((1, M, N), 7.0, dtype=torch.float16, device="cuda")
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run_qlora(h, dev(inp.X, torch), None, None, None, q["Aq"], q["A_scales"], q["A_zp"], q["Bq"],
                          q["B_scales"], q["B_zp"], 32, None, Y, T, 1, M)
        torch.cuda.synchronize()
        assert mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)
    zero = oracle.pack(np.full((N, K), 8, dtype=np.uint8), 4)
    _, Y64, bound = oracle.run_qlora(inp.X2d, zero, inp.scales, None, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                     ql.B_scales, ql.B_zp, N, K, 4)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"qlora empty base M={M}")


def test_qlora_empty_adapter_is_base_bitwise(env):
    torch, mnb = env
    inp = synth.make_inputs(M=3, K=512, N=640, bits=4, seed=950, zp_range=(0, 15))
    d = upload(inp, torch)
    h = mnb.mnb_create(inp.N, inp.K, 4)
    try:
        Y0 = torch.empty((1, 3, 640), dtype=torch.float16, device="cuda")
        Y1 = torch.empty_like(Y0)
        mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], None, None, 0, Y0, None, 1, 3)
        mnb.mnb_run_qlora(h, d["X"], d["Wq"], d["scales"], d["zp"], None, None, None, None, None, None, 32, None,
                          Y1, None, 1, 3)
        torch.cuda.synchronize()
    finally:
        mnb.mnb_destroy(h)
    assert torch.equal(Y0, Y1)


def test_qlora_down_on_idle_sms_exact_bitwise(env):
    """A one-wave prefill grid (80 weight tiles) leaves SMs idle: the INT8 down weight's
    projection runs there, each CTA dequantizing the adapter codes of a K piece while it
    multiplies the one before.  Exact arithmetic: T and Y match the oracle bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(960)
    M, K, N = 100, 1024, 10240
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
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=960, zp_range=(0, 15))
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    ql = synth.make_qlora(K=K, N=N, seed=961)
    ql.Aq = (ql.A_zp[:, :, None] + rng.integers(-3, 4, size=ql.Aq.shape)).astype(np.uint8)
    ql.Bq = (ql.B_zp[:, :, None] + rng.integers(-3, 4, size=ql.Bq.shape)).astype(np.uint8)
    ql.A_scales = np.full(ql.A_scales.shape, 0x2C00, np.uint16)  # 1/16
    ql.B_scales = np.full(ql.B_scales.shape, 0x2C00, np.uint16)
    Y, T, route = run_qlora_gpu(mnb, torch, inp, ql)
    assert route == mnb.ROUTE_GEMM
    Y16, _, _ = oracle.run_qlora(inp.X2d, inp.Wq, inp.scales, inp.zp, ql.Aq, ql.A_scales, ql.A_zp, ql.Bq,
                                 ql.B_scales, ql.B_zp, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)
    a16 = oracle.dequant_f16(ql.Aq, ql.A_scales, ql.A_zp, 32, K, 8)
    T64 = oracle.lora_down(inp.X2d, np.ascontiguousarray(a16.T))
    got = bits_of(T).view(np.float16).astype(np.float64).reshape(M, 32)
    assert np.array_equal(got, T64)
