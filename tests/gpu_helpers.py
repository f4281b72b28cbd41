"""Shared helpers of the GPU tests: upload seeded inputs, run through the C ABI,
compare with the oracle under the FP16 tolerance |y - y_ref| <= 1e-3 * sum|x w| + 1e-3."""
import numpy as np

import oracle

TOL_REL = 1e-3
TOL_ABS = 1e-3


def dev(a, torch):
    """numpy (uint16 FP16 bits / uint8) -> CUDA tensor; None stays None."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_of(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint16)


def upload(inp, torch):
    return dict(X=dev(inp.X, torch), Wq=dev(inp.Wq, torch), scales=dev(inp.scales, torch), zp=dev(inp.zp, torch),
                A=dev(inp.A, torch), B=dev(inp.B, torch))


def run_gpu(mnb, torch, inp, mode=0, gemv_max_m=0, d=None, Y=None, T=None, rank=None, bias=None):
    """Run one problem through the C ABI; ``bias`` (a CUDA FP16 [N] tensor) goes
    through mnb_run_bias, None through mnb_run."""
    d = d or upload(inp, torch)
    rank = inp.rank if rank is None else rank
    h = mnb.mnb_create(inp.N, inp.K, inp.bits, 32, 32, mode, gemv_max_m)
    try:
        Mt = inp.batch * inp.M
        if Y is None:
            Y = torch.empty((inp.batch, inp.M, inp.N), dtype=torch.float16, device="cuda")
        if T is None and rank:
            T = torch.empty((Mt, rank), dtype=torch.float16, device="cuda")
        AB = (d["A"], d["B"]) if rank else (None, None)
        if bias is None:
            mnb.mnb_run(h, d["X"], d["Wq"], d["scales"], d["zp"], *AB, rank, Y, T, inp.batch, inp.M)
        else:
            mnb.mnb_run_bias(h, d["X"], d["Wq"], d["scales"], d["zp"], *AB, rank, bias, Y, T, inp.batch, inp.M)
        torch.cuda.synchronize()
        assert mnb.mnb_sync_status(h) == 0
        route = mnb.mnb_last_route(h)
    finally:
        mnb.mnb_destroy(h)
    return Y, T, route


def oracle_ref(inp, rows=None, tokens=None, bias=None):
    """Oracle Y64 and bound, optionally on a subset of output rows / token rows;
    ``bias`` is FP16 bits [N] or None."""
    X = inp.X2d if tokens is None else inp.X2d[tokens]
    Wq, S, Z, B = inp.Wq, inp.scales, inp.zp, inp.B
    if rows is not None:
        Wq, S = Wq[rows], S[rows]
        Z = None if Z is None else Z[rows]
        B = None if B is None else B[rows]
        bias = None if bias is None else bias[rows]
    N = Wq.shape[0]
    _, Y64, bound = oracle.run(X, Wq, S, Z, inp.A, B, N, inp.K, inp.bits, bias=bias)
    return Y64, bound


def assert_within_tolerance(y_bits, Y64, bound, what=""):
    y = y_bits.view(np.float16).astype(np.float64).reshape(Y64.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - Y64)
    tol = TOL_REL * bound + TOL_ABS
    ratio = err / tol
    bad = int((ratio > 1).sum())
    assert bad == 0, f"{what}: {bad} of {y.size} outputs outside tolerance (worst err/tol {ratio.max():.3g})"
    return float(ratio.max())
