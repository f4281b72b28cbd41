"""mnb_run_noalloc: the same product for callers that cannot allocate device
memory (the LoRA scratch T lives in a fixed array inside the library).

This file is collected last on purpose.  The GPU test compares the entry point
with mnb_run on the same inputs, under the tolerance the other tests use, on
two calls in a row with different inputs (so stale contents of the shared
array would show), for both the decode and the prefill route.
"""
import numpy as np
import pytest

from block_quantized_matmul_matmulnbits_gb300 import synth

from gpu_helpers import assert_within_tolerance, bits_of, oracle_ref, run_gpu, upload


def test_noalloc_rejects_rows_beyond_its_scratch_without_a_device():
    from block_quantized_matmul_matmulnbits_gb300 import build as mnb_build
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    mnb_build.build()
    h = mnb.mnb_create(64, 64, 4)
    try:
        limit = mnb.mnb_noalloc_max_rows()
        assert limit == 8192
        rc = mnb.lib().mnb_run_noalloc(h, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 1, limit + 1,
                                       None)
        assert rc == mnb.MNB_ERR_UNSUPPORTED
    finally:
        mnb.mnb_destroy(h)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (300, 1000, 512)])
def test_noalloc_matches_mnb_run_twice(M, N, K):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_matmulnbits_gb300 import mnb
    for call in range(2):  # two calls in a row, different inputs each time
        inp = synth.make_inputs(M=M, K=K, N=N, bits=4, seed=900 + 17 * call + M, zp_range=(0, 15), rank=32)
        d = upload(inp, torch)
        Y_ref, _, route = run_gpu(mnb, torch, inp, d=d)
        h = mnb.mnb_create(N, K, 4)
        try:
            Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
            mnb.mnb_run_noalloc(h, d["X"], d["Wq"], d["scales"], d["zp"], d["A"], d["B"], 32, Y, 1, M)
            torch.cuda.synchronize()
            assert mnb.mnb_sync_status(h) == 0
            assert mnb.mnb_last_route(h) == route
        finally:
            mnb.mnb_destroy(h)
        rows = np.arange(N) if N <= 1024 else np.sort(np.random.default_rng(call).choice(N, 1024, replace=False))
        Y64, bound = oracle_ref(inp, rows=rows)
        ref = bits_of(Y_ref).reshape(M, N)[:, rows]
        got = bits_of(Y).reshape(M, N)[:, rows]
        assert_within_tolerance(ref, Y64, bound, "mnb_run")
        assert_within_tolerance(got, Y64, bound, "mnb_run_noalloc")
        diff = np.abs(got.view(np.float16).astype(np.float64) - ref.view(np.float16).astype(np.float64))
        assert np.all(diff <= 1e-3 * bound + 1e-3)
