"""CUDA-graph capture of the ABI calls: every call only enqueues work, so it
can be captured; a replay reads the buffers' current contents through the
captured pointers and route.  Adapter on and off are separate captures, and a
captured fill (empty weight) rewrites the output on every replay."""
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


def capture(torch, fn):
    """Capture fn() (ABI calls on the current stream) into a graph."""
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        fn()  # warm: first-use setup stays out of the capture
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("M", [1, 300])
def test_replay_equals_direct_call_bitwise(env, M):
    torch, mnb = env
    inp = synth.make_inputs(M=M, K=1024, N=512, bits=4, seed=2100 + M, zp_range=(0, 15), rank=32)
    d = upload(inp, torch)
    h = mnb.mnb_create(inp.N, inp.K, 4, flags=mnb.FLAG_EARLY_WEIGHTS)
    try:
        Yd = torch.empty((1, M, inp.N), dtype=torch.float16, device="cuda")
        Tg = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, Yd, Tg, 1, M)
        torch.cuda.synchronize()
        Yg = torch.full_like(Yd, 3.0)
        g = capture(torch, lambda: mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, Yg, Tg,
                                               1, M))
        Yg.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == mnb.MNB_OK
        assert mnb.mnb_last_route(h) == (mnb.ROUTE_GEMV if M <= 16 else mnb.ROUTE_GEMM)
    finally:
        mnb.mnb_destroy(h)
    assert torch.equal(Yg, Yd)


def test_adapter_on_and_off_are_separate_captures(env):
    torch, mnb = env
    M = 1
    inp = synth.make_inputs(M=M, K=2048, N=1024, bits=4, seed=2110, zp_range=(0, 15), rank=32)
    d = upload(inp, torch)
    h = mnb.mnb_create(inp.N, inp.K, 4)
    try:
        Yon = torch.empty((1, M, inp.N), dtype=torch.float16, device="cuda")
        Yoff = torch.empty_like(Yon)
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        g_on = capture(torch, lambda: mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32,
                                                  Yon, T, 1, M))
        g_off = capture(torch, lambda: mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], None, None, 0,
                                                   Yoff, None, 1, M))
        for g in (g_off, g_on, g_off):
            g.replay()
        torch.cuda.synchronize()
    finally:
        mnb.mnb_destroy(h)
    Y64, bound = oracle_ref(inp)
    assert_within_tolerance(bits_of(Yon), Y64, bound, "adapter on, replayed")
    base = synth.make_inputs(M=M, K=2048, N=1024, bits=4, seed=2110, zp_range=(0, 15))
    Y64, bound = oracle_ref(base)
    assert_within_tolerance(bits_of(Yoff), Y64, bound, "adapter off, replayed")
    assert not torch.equal(Yon, Yoff)


def test_replay_reads_current_buffer_contents(env):
    """The graph bakes in pointers, not values: new X and new adapter values
    written into the same buffers are picked up by the next replay."""
    torch, mnb = env
    M, K, N = 2, 1024, 384
    a = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=2120, zp_range=(0, 15), rank=32)
    b = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=2121, zp_range=(0, 15), rank=32)
    b.Wq, b.scales, b.zp = a.Wq, a.scales, a.zp  # same weights, new X and adapter
    d = upload(a, torch)
    h = mnb.mnb_create(N, K, 4)
    try:
        Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda")
        g = capture(torch, lambda: mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, Y, T,
                                               1, M))
        g.replay()
        torch.cuda.synchronize()
        Y64, bound = oracle_ref(a)
        assert_within_tolerance(bits_of(Y), Y64, bound, "first contents")
        d["X"].copy_(dev(b.X, torch))
        d["A"].copy_(dev(b.A, torch))
        d["B"].copy_(dev(b.B, torch))
        g.replay()
        torch.cuda.synchronize()
    finally:
        mnb.mnb_destroy(h)
    Y64, bound = oracle_ref(b)
    assert_within_tolerance(bits_of(Y), Y64, bound, "second contents")


@pytest.mark.parametrize("with_bias", [False, True])
def test_captured_fill_rewrites_the_output(env, with_bias):
    """An empty packed weight records a fill: each replay rewrites Y."""
    torch, mnb = env
    N, K, M = 300, 256, 3
    bias = synth.make_bias(N, seed=2130)
    h = mnb.mnb_create(N, K, 4)
    try:
        X = torch.zeros((1, M, K), dtype=torch.float16, device="cuda")
        Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
        bv = dev(bias, torch) if with_bias else None
        g = capture(torch, lambda: mnb.mnb_run_bias(h, X, None, None, None, None, None, 0, bv, Y, None, 1, M))
        for _ in range(2):
            Y.fill_(7.0)
            g.replay()
            torch.cuda.synchronize()
            expect = np.broadcast_to(bias, (M, N)) if with_bias else np.zeros((M, N), np.uint16)
            assert np.array_equal(bits_of(Y).reshape(M, N), expect)
    finally:
        mnb.mnb_destroy(h)


def test_captured_multi_projection(env):
    torch, mnb = env
    M, K, Ns = 1, 1024, (512, 256)
    inps = [synth.make_inputs(M=M, K=K, N=n, bits=4, seed=2140 + i, zp_range=(0, 15)) for i, n in enumerate(Ns)]
    for x in inps[1:]:
        x.X = inps[0].X
    X = dev(inps[0].X, torch)
    ds = [upload(x, torch) for x in inps]
    Ys = [torch.empty((1, M, n), dtype=torch.float16, device="cuda") for n in Ns]
    h = mnb.mnb_create(sum(Ns), K, 4, max_rank=0)
    try:
        g = capture(torch, lambda: mnb.mnb_run_multi(h, X, [(n, dd["Wq"], dd["scales"], dd["zp"], None, Y)
                                                             for n, dd, Y in zip(Ns, ds, Ys)], 1, M))
        for Y in Ys:
            Y.fill_(9.0)
        g.replay()
        torch.cuda.synchronize()
    finally:
        mnb.mnb_destroy(h)
    for x, Y in zip(inps, Ys):
        Y64, bound = oracle_ref(x)
        assert_within_tolerance(bits_of(Y), Y64, bound, f"multi replay N={x.N}")
