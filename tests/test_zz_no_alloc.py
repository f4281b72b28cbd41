"""mnb_run_noalloc: the same product for callers that cannot allocate device
memory -- code inside a host runtime that owns every device allocation, or a
loop in which cudaMalloc / cudaFree are not allowed because they can
synchronize the device.  The LoRA scratch T lives in a fixed array inside the
library instead of a caller buffer.

This file is collected last on purpose.  The GPU tests compare the entry point
with mnb_run on the same inputs, under the tolerance the other tests use, on
two calls in a row with different inputs (so stale contents of the shared
array would show), on the decode and the prefill route, up to the array's
limit of 8192 token rows and one row short of it.
"""
import numpy as np
import pytest

from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, oracle_ref, run_gpu, upload
from test_abi_host import run_without_gpu


def check_noalloc_argument_checks():
    """Argument checks with made-up addresses that are never dereferenced (run
    in a child process that sees no GPU)."""
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    h = mnb.mnb_create(64, 64, 4)
    try:
        L = mnb.lib()
        limit = mnb.mnb_noalloc_max_rows()
        assert limit == 8192
        # the checks of mnb_run, in its order, come before the row limit
        assert L.mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, None, 32, 0x4000, 1, 1, None) \
            == mnb.MNB_ERR_ARG
        assert L.mnb_run_noalloc(h, 0x1008, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 1, 1, None) \
            == mnb.MNB_ERR_ALIGN
        assert L.mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 16, 0x4000, 1, 1, None) \
            == mnb.MNB_ERR_UNSUPPORTED
        # no rows: nothing to do, as for mnb_run (no scratch is needed)
        assert L.mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 1, 0, None) \
            == mnb.MNB_OK
        assert mnb.mnb_last_route(h) == mnb.ROUTE_NONE
        assert L.mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 0, 7, None) \
            == mnb.MNB_OK
        # rows beyond the scratch: refused, nothing launched (here: no device is visible either)
        assert L.mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 1, limit + 1,
                                 None) in (mnb.MNB_ERR_UNSUPPORTED, mnb.MNB_ERR_NO_DEVICE)
    finally:
        mnb.mnb_destroy(h)
    h0 = mnb.mnb_create(64, 64, 4, max_rank=0)
    try:  # an adapter on a handle without one is an argument error, not a size error
        assert mnb.lib().mnb_run_noalloc(h0, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 1,
                                         limit + 1, None) == mnb.MNB_ERR_ARG
    finally:
        mnb.mnb_destroy(h0)


def test_noalloc_argument_checks_without_a_device():
    from block_quantized_matmul_matmulnbits_gb300 import build as mnb_build
    mnb_build.build()
    run_without_gpu(check_noalloc_argument_checks)


@pytest.mark.gpu
@pytest.mark.parametrize("batch,M,N,K", [(1, 1, 4096, 4096), (1, 300, 1000, 512), (2, 4096, 256, 256),
                                         (1, 8191, 256, 256)])
def test_noalloc_matches_mnb_run_twice(batch, M, N, K):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    Mt = batch * M
    for call in range(2):  # two calls in a row, different inputs each time
        inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=900 + 17 * call + Mt, zp_range=(0, 15), rank=32,
                                batch=batch)
        d = upload(inp, torch)
        Y_ref, _, route = run_gpu(mnb, torch, inp, d=d)
        h = mnb.mnb_create(N, K, 4)
        try:
            Y = torch.empty((batch, M, N), dtype=torch.float16, device="cuda")
            mnb.mnb_run_noalloc(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, Y, batch, M)
            torch.cuda.synchronize()
            assert mnb.mnb_sync_status(h) == 0
            assert mnb.mnb_last_route(h) == route
        finally:
            mnb.mnb_destroy(h)
        rng = np.random.default_rng(call)
        rows = np.arange(N) if N <= 1024 else np.sort(rng.choice(N, 1024, replace=False))
        # token rows: all of a small call; else a sample that includes the last row of the scratch
        tokens = np.arange(Mt) if Mt <= 512 else np.unique(np.concatenate(
            [rng.choice(Mt, 96, replace=False), [0, Mt - 1]]))
        Y64, bound = oracle_ref(inp, rows=rows, tokens=tokens)
        ref = bits_of(Y_ref).reshape(Mt, N)[np.ix_(tokens, rows)]
        got = bits_of(Y).reshape(Mt, N)[np.ix_(tokens, rows)]
        assert_within_tolerance(ref, Y64, bound, "mnb_run")
        assert_within_tolerance(got, Y64, bound, "mnb_run_noalloc")
        diff = np.abs(got.view(np.float16).astype(np.float64) - ref.view(np.float16).astype(np.float64))
        assert np.all(diff <= 1e-3 * bound + 1e-3)
