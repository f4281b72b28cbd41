"""GPU parity of the dequant step, the LoRA down projection and the decode
(GEMV) route against the CPU oracle, through the C ABI.

Dequantization must be bit-exact; outputs must satisfy
|y - y_ref| <= 1e-3 * sum|x w| + 1e-3 (sum over the base and LoRA products).
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


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("bits,zp_range,N,K", [(4, None, 256, 256), (4, (0, 15), 300, 4096), (8, (120, 136), 97, 576),
                                               (8, None, 64, 896), (8, (0, 255), 33, 96), (4, (0, 255), 17, 160)])
@pytest.mark.parametrize("variant", [0, 1])
def test_dequant_bit_exact(env, bits, zp_range, N, K, variant):
    torch, mnb = env
    inp = synth.make_inputs(M=1, K=K, N=N, bits=bits, seed=100 + N, zp_range=zp_range, scale_range=(1e-5, 30.0))
    d = upload(inp, torch)
    W16 = torch.empty((N, K), dtype=torch.float16, device="cuda")
    mnb.mnb_dequant(d["Wq"], d["scales"], d["zp"], N, K, bits, W16, variant)
    torch.cuda.synchronize()
    ref = oracle.dequant_f16(inp.Wq, inp.scales, inp.zp, N, K, bits)
    got = bits_of(W16)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} dequantized values differ"


# ------------------------------------------------------------------ LoRA down

@pytest.mark.parametrize("Mt,K", [(1, 4096), (4, 256), (70, 576), (1024, 4096), (3, 32)])
def test_lora_down_matches_oracle(env, Mt, K):
    torch, mnb = env
    inp = synth.make_inputs(M=Mt, K=K, N=16, bits=4, seed=200 + Mt, rank=32)
    d = upload(inp, torch)
    T = torch.empty((Mt, 32), dtype=torch.float16, device="cuda")
    mnb.mnb_lora_down(d["X"], d["A"], T, Mt, K)
    torch.cuda.synchronize()
    T64 = oracle.lora_down(inp.X2d, inp.A)
    x = np.abs(inp.X2d.view(np.float16).astype(np.float64))
    a = np.abs(inp.A.view(np.float16).astype(np.float64))
    mag = x @ a
    t = bits_of(T).view(np.float16).astype(np.float64)
    # one FP16 rounding of T (2^-11 relative) plus FP32 accumulation
    assert np.all(np.abs(t - T64) <= 2.0 ** -11 * np.abs(T64) + 1e-5 * mag + 1e-7)
    T2 = torch.empty_like(T)
    mnb.mnb_lora_down(d["X"], d["A"], T2, Mt, K)
    torch.cuda.synchronize()
    assert torch.equal(T, T2)


# ------------------------------------------------------------------ decode route

@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("rank", [32, 0])
def test_tiny_config(env, M, rank):
    torch, mnb = env
    inp = synth.tiny(M=M, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"tiny M={M} rank={rank}")


@pytest.mark.parametrize("rank,partial", [(32, False), (0, False), (32, True)])
def test_decode_4096(env, rank, partial):
    torch, mnb = env
    inp = synth.decode_4096(rank=rank, partial=partial)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"decode rank={rank} partial={partial}")


def test_decode_partial_adapter_equals_rank16_on_gpu(env):
    torch, mnb = env
    inp = synth.decode_4096(rank=32, partial=True)
    Y32, _, _ = run_gpu(mnb, torch, inp)
    Y64, bound = oracle_ref(inp)
    inp16 = synth.decode_4096(rank=32, partial=True)
    inp16.A = np.ascontiguousarray(inp.A[:, :16])
    inp16.B = np.ascontiguousarray(inp.B[:, :16])
    Y64_16, _ = oracle_ref(inp16)
    assert np.array_equal(Y64, Y64_16)   # the oracle agrees that the zero columns add nothing
    assert_within_tolerance(bits_of(Y32), Y64_16, bound, "partial vs rank-16")


def test_decode_empty_adapter_is_base_bitwise(env):
    torch, mnb = env
    inp = synth.decode_4096(rank=32)
    d = upload(inp, torch)
    Yb, _, _ = run_gpu(mnb, torch, inp, d=d, rank=0)
    d0 = dict(d, A=torch.zeros_like(d["A"]), B=torch.zeros_like(d["B"]))
    Yz, _, _ = run_gpu(mnb, torch, inp, d=d0)
    assert torch.equal(Yb, Yz)


def test_decode_lora_is_base_plus_separate_xab(env):
    torch, mnb = env
    inp = synth.decode_4096(rank=32)
    Yl, T, _ = run_gpu(mnb, torch, inp)
    Yb, _, _ = run_gpu(mnb, torch, inp, rank=0)
    x = inp.X2d.view(np.float16).astype(np.float64)
    xab = (x @ inp.A.view(np.float16).astype(np.float64)) @ inp.B.view(np.float16).astype(np.float64).T
    _, bound = oracle_ref(inp)
    diff = bits_of(Yl).view(np.float16).astype(np.float64).reshape(xab.shape) - \
        bits_of(Yb).view(np.float16).astype(np.float64).reshape(xab.shape)
    # two FP16 outputs each within tolerance of their exact values
    assert np.all(np.abs(diff - xab) <= 2e-3 * bound + 2e-3)


@pytest.mark.parametrize("K,N", [(576, 49152), (896, 151936)])
def test_lm_head_int8(env, K, N):
    torch, mnb = env
    inp = synth.lm_head(K=K, N=N)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"lm_head K={K} N={N}")


@pytest.mark.parametrize("M,K,N,bits,zp", [
    (1, 2048, 23995, 4, (0, 15)),    # 5 stages per CTA: a ring of three
    (2, 1536, 20007, 8, (120, 136)),  # two K chunks per row (1024 + 512 bytes), ring of three
    (3, 576, 30001, 8, None),        # 13 small stages: a ring of four
    (5, 1024, 20000, 4, None),       # three stages, ring of three
    (1, 4096, 8000, 4, (0, 15)),     # large stages: a ring of two
])
def test_three_ctas_per_sm_rings(env, M, K, N, bits, zp):
    """More than two row groups per SM and a small staged X put three CTAs on
    an SM; the number of stages per CTA and the stage size then pick rings of
    two, three or four stages (slots stepped by a counter).  Every output is
    compared, ragged last groups included."""
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=3300 + M, zp_range=zp)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"three CTAs per SM M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("rank", [32, 0])
def test_mlp_up_decode_sampled_rows(env, M, rank):
    torch, mnb = env
    inp = synth.mlp_up(M=M, rank=rank)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    rows = np.sort(np.random.default_rng(M).choice(inp.N, 768, replace=False))
    Y64, bound = oracle_ref(inp, rows=rows)
    got = bits_of(Y).reshape(inp.batch * inp.M, inp.N)[:, rows]
    assert_within_tolerance(got, Y64, bound, f"mlp_up M={M} rank={rank}")


@pytest.mark.parametrize("M,N,K,bits,zp", [
    (2, 1000, 512, 4, (0, 15)),       # one slot per stage, a ragged last stage
    (6, 2077, 2048, 8, (120, 136)),   # INT8
    (8, 3000, 4096, 4, None),         # K halves per slot, one token tile
    (9, 2100, 4096, 4, (0, 15)),      # two token tiles (the second one token), K quarters per slot
    (16, 1500, 4096, 8, (0, 255)),    # INT8, 16 token rows
    (13, 700, 3072, 4, None),
    (3, 37, 6144, 4, (0, 15)),        # three CTAs, stages of 12 and 13 rows
])
def test_few_token_kernel_matches_oracle(env, M, N, K, bits, zp):
    """2 .. 16 token rows without an adapter run on the kernel with the token rows
    as the MMA's N (its plan: 16-row stages, 8 or 16 token columns); every output
    against the oracle."""
    torch, mnb = env
    h = mnb.mnb_create(N, K, bits)
    try:
        p = mnb.mnb_plan(h, 1, M, 0, torch.cuda.get_device_properties(0).multi_processor_count)
    finally:
        mnb.mnb_destroy(h)
    assert p["k_splits"] == 16 and p["tokens_per_cta"] == (8 if M <= 8 else 16)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=3400 + M, zp_range=zp)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"few tokens M={M} N={N} K={K} bits={bits}")


@pytest.mark.parametrize("M,N,K,bits,zp,partial", [
    (3, 1000, 512, 4, (0, 15), False),
    (8, 2077, 4096, 4, None, True),     # x in registers; ranks 16..31 zero
    (12, 700, 2048, 8, (120, 136), False),
    (16, 1500, 4096, 4, (0, 15), False),
])
def test_few_token_kernel_with_adapter(env, M, N, K, bits, zp, partial):
    """An FP16 rank-32 adapter on the few-token kernel: T from the LoRA down kernel,
    T B^T added by the reducer warp before the one rounding; every output against
    the oracle."""
    torch, mnb = env
    h = mnb.mnb_create(N, K, bits)
    try:
        p = mnb.mnb_plan(h, 1, M, 32, torch.cuda.get_device_properties(0).multi_processor_count)
    finally:
        mnb.mnb_destroy(h)
    assert p["k_splits"] == 16 and p["lora_kernel"] == 1
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=3500 + M, zp_range=zp, rank=32, partial=partial)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"few tokens + adapter M={M} N={N} K={K} bits={bits}")


def test_few_token_exact_arithmetic_bitwise(env):
    """X in {-1,0,1} (<= 8 nonzeros per row), power-of-two scales, 12 token rows, no
    adapter: every product, block sum and partial sum of the few-token kernel is
    exact, so it must match the oracle bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(405)
    M, K, N = 12, 2048, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=405, zp_range=(0, 15))
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    Y, _, route = run_gpu(mnb, torch, inp)
    assert route == mnb.ROUTE_GEMV
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, None, None, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


# ------------------------------------------------------------------ edges

@pytest.mark.parametrize("M,N,K,bits,zp", [(3, 1000, 96, 4, (0, 15)), (5, 17, 160, 8, (0, 255)), (1, 1, 32, 4, None),
                                           (9, 129, 64, 4, None), (16, 333, 544, 8, (120, 136))])
def test_ragged_shapes(env, M, N, K, bits, zp):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=300 + N, zp_range=zp, rank=32)
    Y, _, _ = run_gpu(mnb, torch, inp)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, f"ragged M={M} N={N} K={K}")


def test_force_gemv_many_tokens(env):
    torch, mnb = env
    inp = synth.make_inputs(M=40, K=256, N=300, bits=4, seed=401, zp_range=(0, 15), rank=32)
    Y, _, route = run_gpu(mnb, torch, inp, mode=mnb.MODE_FORCE_GEMV)
    assert route == mnb.ROUTE_GEMV
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, "force gemv M=40")


def test_batch_invariance_bitwise(env):
    torch, mnb = env
    inp = synth.make_inputs(M=3, K=512, N=640, bits=4, seed=402, batch=4, zp_range=(0, 15), rank=32)
    Yb, _, rb = run_gpu(mnb, torch, inp)
    flat = synth.make_inputs(M=3, K=512, N=640, bits=4, seed=402, batch=4, zp_range=(0, 15), rank=32)
    flat.X = flat.X.reshape(1, 12, 512)
    flat.batch, flat.M = 1, 12
    # same rows, one matrix of 12 rows: forced onto the same decode route
    Yf, _, rf = run_gpu(mnb, torch, flat, mode=mnb.MODE_FORCE_GEMV)
    assert rb == rf == mnb.ROUTE_GEMV
    assert torch.equal(Yb.reshape(12, 640), Yf.reshape(12, 640))


def test_deterministic_repeat(env):
    torch, mnb = env
    inp = synth.decode_4096(rank=32)
    d = upload(inp, torch)
    Y1, _, _ = run_gpu(mnb, torch, inp, d=d)
    Y2, _, _ = run_gpu(mnb, torch, inp, d=d)
    assert torch.equal(Y1, Y2)


def test_guard_bands_untouched(env):
    torch, mnb = env
    inp = synth.make_inputs(M=2, K=128, N=1000, bits=4, seed=403, rank=32)
    d = upload(inp, torch)
    pad = 4096
    Ybuf = torch.full((2 * 1000 + 2 * pad,), 7.0, dtype=torch.float16, device="cuda")
    Tbuf = torch.full((2 * 32 + 2 * pad,), 7.0, dtype=torch.float16, device="cuda")
    Y = Ybuf[pad:pad + 2000].view(1, 2, 1000)
    T = Tbuf[pad:pad + 64].view(2, 32)
    run_gpu(mnb, torch, inp, d=d, Y=Y, T=T)
    assert torch.all(Ybuf[:pad] == 7.0) and torch.all(Ybuf[pad + 2000:] == 7.0)
    assert torch.all(Tbuf[:pad] == 7.0) and torch.all(Tbuf[pad + 64:] == 7.0)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, "guarded")


def test_empty_and_k0(env):
    torch, mnb = env
    # M = 0: nothing launched, output untouched
    h = mnb.mnb_create(64, 64, 4)
    Y = torch.full((1, 0, 64), 3.0, dtype=torch.float16, device="cuda")
    mnb.mnb_run(h, Y, Y, Y, None, None, None, 0, Y, None, 1, 0)
    assert mnb.mnb_last_route(h) == mnb.ROUTE_NONE
    mnb.mnb_destroy(h)
    # K = 0: zeros of the logical output shape
    h = mnb.mnb_create(77, 0, 4)
    Y = torch.full((3, 77), 5.0, dtype=torch.float16, device="cuda")
    X = torch.empty((3, 0), dtype=torch.float16, device="cuda")
    mnb.mnb_run(h, X, X, X, None, None, None, 0, Y, None, 1, 3)
    torch.cuda.synchronize()
    assert mnb.mnb_last_route(h) == mnb.ROUTE_FILL
    assert torch.all(Y == 0)
    mnb.mnb_destroy(h)


def test_exact_arithmetic_bitwise(env):
    """X in {-1,0,1} (<= 8 nonzeros per row), power-of-two scales, dyadic adapters:
    every product and partial sum is exact in FP16/FP32, so the GPU must match the
    oracle bit for bit."""
    torch, mnb = env
    rng = np.random.default_rng(404)
    M, K, N = 5, 1024, 300
    x = np.zeros((1, M, K))
    for m in range(M):
        idx = rng.choice(K, 8, replace=False)
        x[0, m, idx] = rng.choice([-1.0, 1.0], 8)
    inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=404, zp_range=(0, 15), rank=32)
    inp.X = x.astype(np.float16).view(np.uint16)
    inp.scales = np.ldexp(1.0, rng.integers(-8, -4, size=(N, K // 32))).astype(np.float16).view(np.uint16)
    inp.A = (rng.integers(-3, 4, size=(K, 32)) / 16.0).astype(np.float16).view(np.uint16)
    inp.B = (rng.integers(-3, 4, size=(N, 32)) / 16.0).astype(np.float16).view(np.uint16)
    Y, _, _ = run_gpu(mnb, torch, inp)
    Y16, _, _ = oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, N, K, 4)
    assert np.array_equal(bits_of(Y).reshape(M, N), Y16)


@pytest.mark.parametrize("M,N,K,rank", [(1, 4096, 4096, 32), (1, 4096, 4096, 0), (3, 1000, 576, 32),
                                        (300, 640, 512, 32)])
def test_early_weights_back_to_back_calls(env, M, N, K, rank):
    """With MNB_FLAG_EARLY_WEIGHTS consecutive calls overlap (each streams its
    weights before the previous call ends); every output must still match."""
    torch, mnb = env
    inps = [synth.make_inputs(M=M, K=K, N=N, bits=4, seed=700 + i, zp_range=(0, 15), rank=rank) for i in range(3)]
    devs = [upload(i, torch) for i in inps]
    h = mnb.mnb_create(N, K, 4, 32, 32, 0, 0, mnb.FLAG_EARLY_WEIGHTS)
    outs = []
    try:
        for rep in range(4):
            for i, d in enumerate(devs):
                Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
                T = torch.empty((M, 32), dtype=torch.float16, device="cuda") if rank else None
                mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"] if rank else None,
                            d["B"] if rank else None, rank, Y, T, 1, M)
                outs.append((i, Y))
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0
    finally:
        mnb.mnb_destroy(h)
    refs = [oracle_ref(i) for i in inps]
    for i, Y in outs:
        assert_within_tolerance(bits_of(Y), refs[i][0], refs[i][1], f"back-to-back call {i}")
    # bitwise equal across repetitions of the same inputs
    for i in range(3):
        same = [Y for j, Y in outs if j == i]
        assert all(torch.equal(same[0], y) for y in same[1:])


def test_bounded_wait_times_out_and_the_context_stays_usable(env):
    """Failure detection without a fault: the kernels' bounded wait, run on a
    barrier nothing completes with a short limit, reports MNB_ERR_DEVICE_TIMEOUT
    through the status word once; the next call works and reports OK."""
    torch, mnb = env
    h = mnb.mnb_create(256, 256, 4)
    try:
        assert mnb.mnb_sync_status(h) == mnb.MNB_OK
        mnb.mnb_check_wait_timeout(2_000_000)          # ~1 ms of waiting
        assert mnb.mnb_sync_status(h) == mnb.MNB_ERR_DEVICE_TIMEOUT
        assert mnb.mnb_sync_status(h) == mnb.MNB_OK    # reported once, then cleared
    finally:
        mnb.mnb_destroy(h)
    inp = synth.tiny(M=1, rank=32)
    Y, _, _ = run_gpu(mnb, torch, inp)                 # run_gpu asserts a clean status
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Y), Y64, bound, "after a timeout check")
