"""Host-side checks of libmnb.so that need no GPU: the library loads, exports
every entry point include/mnb.h declares, validates its arguments and makes
the dispatch decision from the per-matrix row count.  No compute call here.

The argument checks pass made-up device addresses (0x1000, ...) that are never
dereferenced because the call is rejected first.  They run in a child process
that sees no GPU (CUDA_VISIBLE_DEVICES=""), so on a machine with a GPU a
regression in the checks returns MNB_ERR_NO_DEVICE instead of launching a
kernel on those addresses."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from conftest import ROOT

from block_quantized_matmul_matmulnbits_gb300 import build as mnb_build
from block_quantized_matmul_matmulnbits_gb300 import mnb


@pytest.fixture(scope="module", autouse=True)
def built():
    mnb_build.build()
    yield


def run_without_gpu(fn):
    """Run the module-level function `fn` of this file in a child process in
    which no GPU is visible; its assertion failures fail the calling test."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    here = os.path.dirname(os.path.abspath(__file__))
    mod = os.path.splitext(os.path.basename(fn.__code__.co_filename))[0]
    code = (f"import sys; sys.path[:0] = [{here!r}, {ROOT!r}]; import {mod} as m; m.{fn.__name__}(); "
            "print('child ok')")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-4000:] + r.stderr[-4000:]


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mnb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mnb_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_what_the_binding_wraps():
    assert declared_symbols() == sorted(mnb.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(mnb.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = mnb.status_str(code)
        assert s.startswith("MNB_")
    assert "UNKNOWN" in mnb.status_str(-99)


@pytest.mark.parametrize("kw,code", [
    (dict(N=-1, K=64), mnb.MNB_ERR_ARG),
    (dict(N=64, K=-32), mnb.MNB_ERR_ARG),
    (dict(N=64, K=48), mnb.MNB_ERR_UNSUPPORTED),
    (dict(N=64, K=96, bits=2), mnb.MNB_ERR_UNSUPPORTED),   # 2-bit rows must be whole 16-byte units
    (dict(N=64, K=64, bits=3), mnb.MNB_ERR_UNSUPPORTED),
    (dict(N=64, K=64, block_size=64), mnb.MNB_ERR_UNSUPPORTED),
    (dict(N=64, K=64, max_rank=16), mnb.MNB_ERR_UNSUPPORTED),
    (dict(N=64, K=64, mode=7), mnb.MNB_ERR_ARG),
])
def test_create_rejects_bad_descriptors(kw, code):
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_create(**kw)
    assert e.value.code == code


def test_create_accepts_valid_descriptors_and_empty_shapes():
    for kw in (dict(N=4096, K=4096), dict(N=49152, K=576, bits=8, max_rank=0), dict(N=0, K=0), dict(N=5, K=0),
               dict(N=4096, K=4096, bits=2), dict(N=64, K=0, bits=2)):
        h = mnb.mnb_create(**kw)
        mnb.mnb_destroy(h)
    mnb.mnb_destroy(None)


def test_route_follows_per_matrix_rows_not_batch():
    h = mnb.mnb_create(4096, 4096, 4)
    try:
        for M, route in ((1, mnb.ROUTE_GEMV), (16, mnb.ROUTE_GEMV), (17, mnb.ROUTE_GEMM), (1024, mnb.ROUTE_GEMM)):
            assert mnb.mnb_plan(h, 1, M, 0, 152)["route"] == route
        # batch never changes the route: 64 one-row matrices stay on the decode path,
        # 2 x 512 stays on the prefill path
        assert mnb.mnb_plan(h, 64, 1, 0, 152)["route"] == mnb.ROUTE_GEMV
        assert mnb.mnb_plan(h, 2, 512, 0, 152)["route"] == mnb.ROUTE_GEMM
        assert mnb.mnb_plan(h, 0, 5, 0, 152)["route"] == mnb.ROUTE_NONE
        assert mnb.mnb_plan(h, 3, 0, 0, 152)["route"] == mnb.ROUTE_NONE
        # one token row: the adapter runs inside the single-token decode kernel (one launch);
        # more token rows: the LoRA down kernel first
        assert mnb.mnb_plan(h, 1, 1, 32, 152)["lora_kernel"] == 0
        assert mnb.mnb_plan(h, 1, 2, 32, 152)["lora_kernel"] == 1
        assert mnb.mnb_plan(h, 1, 1, 0, 152)["lora_kernel"] == 0
    finally:
        mnb.mnb_destroy(h)


def test_forced_modes_and_threshold():
    g = mnb.mnb_create(4096, 4096, 4, mode=mnb.MODE_FORCE_GEMV)
    m = mnb.mnb_create(4096, 4096, 4, mode=mnb.MODE_FORCE_GEMM)
    t = mnb.mnb_create(4096, 4096, 4, gemv_max_m=64)
    try:
        assert mnb.mnb_plan(g, 1, 1024, 0, 152)["route"] == mnb.ROUTE_GEMV
        assert mnb.mnb_plan(m, 1, 1, 0, 152)["route"] == mnb.ROUTE_GEMM
        assert mnb.mnb_plan(t, 1, 64, 0, 152)["route"] == mnb.ROUTE_GEMV
        assert mnb.mnb_plan(t, 1, 65, 0, 152)["route"] == mnb.ROUTE_GEMM
    finally:
        for h in (g, m, t):
            mnb.mnb_destroy(h)


def test_k_zero_is_a_fill():
    h = mnb.mnb_create(100, 0, 4)
    try:
        assert mnb.mnb_plan(h, 1, 3, 0, 152)["route"] == mnb.ROUTE_FILL
    finally:
        mnb.mnb_destroy(h)


def test_gemv_plan_balances_rows_over_sms():
    # the general multi-token decode kernel (here: two token rows with an FP16 adapter;
    # INT2 weights at K = 4096, where INT4 / INT8 run on the few-token kernel)
    for N, K, bits in ((4096, 4096, 2), (14336, 4096, 2), (49152, 576, 8), (151936, 896, 8), (1000, 96, 4)):
        h = mnb.mnb_create(N, K, bits)
        try:
            p = mnb.mnb_plan(h, 1, 2, 32, 152)
            R, C, G = p["rows_per_cta"], p["grid_x"], -(-N // 16)
            # whole 16-row groups dealt out evenly: the largest share is ceil(G / C) groups
            assert C <= G and R == 16 * -(-G // C)
            # two or three CTAs per SM (three for one token tile with X staged)
            assert C <= 3 * 152
            # no other CTA count gives the busiest SM fewer groups
            cost = lambda c: -(-c // 152) * -(-G // c)
            assert all(cost(C) <= cost(c) for c in range(1, min(G, 3 * 152) + 1))
            assert p["block_threads"] == 288 and p["k_splits"] % 64 == 0 and 64 <= p["k_splits"] <= 1024
            assert p["tokens_per_cta"] == 8 and p["lora_kernel"] == 1
        finally:
            mnb.mnb_destroy(h)


def test_few_token_plan_splits_rows_evenly():
    # 2 .. 16 token rows without an adapter, K a multiple of 512 up to 7680: the kernel
    # with the token rows as the MMA's N, rows split evenly over one CTA per SM, one
    # launch for up to 16 tokens; other shapes keep the general multi-token kernel
    # (N, K, bits, most token rows on the kernel): x of 16 token rows and K = 4608
    # leave no room for two stage slots, nor x of 8 token rows and INT8 rows of 7 KB;
    # K % 512 != 0 or K > 7680 are outside the kernel's copies
    for N, K, bits, mt_max in ((4096, 4096, 4, 16), (14336, 4096, 4, 16), (14336, 4096, 8, 16), (49152, 576, 8, 0),
                               (4096, 4608, 4, 8), (4096, 7168, 4, 8), (4096, 6144, 8, 8), (4096, 7168, 8, 0),
                               (1000, 96, 4, 0), (4096, 7680, 4, 0), (4096, 8192, 4, 0)):
        h = mnb.mnb_create(N, K, bits)
        try:
            for M in (2, 5, 8, 9, 16):
                # an FP16 adapter keeps the kernel (the LoRA down kernel runs first)
                assert mnb.mnb_plan(h, 1, M, 32, 152)["k_splits"] == mnb.mnb_plan(h, 1, M, 0, 152)["k_splits"]
                p = mnb.mnb_plan(h, 1, M, 0, 152)
                assert p["route"] == mnb.ROUTE_GEMV and p["lora_kernel"] == 0
                if M <= mt_max:
                    C = min(152, -(-N // 16))
                    assert p["grid_x"] == C and p["grid_y"] == 1 and p["rows_per_cta"] == -(-N // C)
                    assert p["tokens_per_cta"] == (8 if M <= 8 else 16) and p["k_splits"] == 16
                else:
                    assert p["k_splits"] % 64 == 0  # general kernel: K bytes per stage
            # more than 16 token rows in one matrix: the prefill route (auto mode)
            assert mnb.mnb_plan(h, 1, 17, 0, 152)["route"] == mnb.ROUTE_GEMM
        finally:
            mnb.mnb_destroy(h)


def test_single_token_plan_splits_rows_evenly():
    # one token row: rows split evenly over one CTA per SM (any row count, not 16-row
    # groups), the same grid with an adapter (one more warp), stages of 16..128 rows
    for N, K, bits in ((4096, 4096, 4), (14336, 4096, 4), (49152, 576, 8), (151936, 896, 8), (1000, 96, 4),
                       (256, 256, 4), (5, 64, 8)):
        h = mnb.mnb_create(N, K, bits)
        try:
            for rank in (0, 32):
                p = mnb.mnb_plan(h, 1, 1, rank, 152)
                C = min(152, max(1, -(-N // 16)))
                if rank and -(-(-(-N // C)) // 16) * 16 > 256:
                    # more than 256 rows a CTA: the adapter's buffers would not fit, so the
                    # multi-token kernel runs behind the LoRA down kernel
                    assert p["tokens_per_cta"] == 8 and p["lora_kernel"] == 1
                    continue
                R, SR = p["rows_per_cta"], p["k_splits"]
                assert p["route"] == mnb.ROUTE_GEMV and p["tokens_per_cta"] == 1 and p["lora_kernel"] == 0
                assert p["grid_y"] == 1 and p["block_threads"] == (320 if rank else 288)
                assert p["grid_x"] == C and R == -(-N // C)
                assert SR in (16, 32, 64, 128)
                # shares differ by at most one row
                shares = [(c + 1) * N // C - c * N // C for c in range(C)]
                assert max(shares) - min(shares) <= 1 and sum(shares) == N
        finally:
            mnb.mnb_destroy(h)
    # the headline decode shape: 4096 rows over 152 CTAs, 26 or 27 rows each, in one stage
    h = mnb.mnb_create(4096, 4096, 4)
    try:
        p = mnb.mnb_plan(h, 1, 1, 32, 152)
        assert p["grid_x"] == 152 and p["rows_per_cta"] == 27 and p["k_splits"] == 32
    finally:
        mnb.mnb_destroy(h)
    # INT2, or the int8-activation entry point, keep the multi-token decode kernel
    h = mnb.mnb_create(4096, 4096, 2)
    try:
        assert mnb.mnb_plan(h, 1, 1, 0, 152)["tokens_per_cta"] == 8
    finally:
        mnb.mnb_destroy(h)


def check_run_validation_needs_no_device():
    h = mnb.mnb_create(64, 64, 4)
    try:
        def rc(**kw):
            args = dict(X=0x1000, Wq=0x2000, scales=0x3000, zp=None, A=None, B=None, rank=0, Y=0x4000,
                        T_ws=None, batch=1, M=1)
            args.update(kw)
            return mnb.lib().mnb_run(h, args["X"], args["Wq"], args["scales"], args["zp"], args["A"], args["B"],
                                     args["rank"], args["Y"], args["T_ws"], args["batch"], args["M"], None)
        assert rc(X=None) == mnb.MNB_ERR_ARG
        assert rc(Y=None) == mnb.MNB_ERR_ARG
        assert rc(scales=None) == mnb.MNB_ERR_ARG
        # an empty packed weight (Wq NULL) needs X only for the adapter term
        assert rc(Wq=None, scales=None, X=None, rank=32, A=0x5000, B=0x6000, T_ws=0x7000) == mnb.MNB_ERR_ARG
        assert rc(Wq=None, scales=None, X=0x1004) == mnb.MNB_ERR_ALIGN
        assert rc(batch=-1) == mnb.MNB_ERR_ARG
        assert rc(rank=16) == mnb.MNB_ERR_UNSUPPORTED
        assert rc(rank=32, A=0x5000, B=None) == mnb.MNB_ERR_ARG
        assert rc(rank=32, A=0x5000, B=0x6000, T_ws=None) == mnb.MNB_ERR_ARG
        assert rc(X=0x1008) == mnb.MNB_ERR_ALIGN
        assert rc(zp=0x7001) == mnb.MNB_ERR_ALIGN
        assert rc(M=0) == mnb.MNB_OK and mnb.mnb_last_route(h) == mnb.ROUTE_NONE
        assert rc(batch=0) == mnb.MNB_OK
    finally:
        mnb.mnb_destroy(h)
    h0 = mnb.mnb_create(64, 64, 4, max_rank=0)
    try:
        assert mnb.lib().mnb_run(h0, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 32, 0x4000, 0x7000, 1, 1,
                                 None) == mnb.MNB_ERR_ARG
    finally:
        mnb.mnb_destroy(h0)


def check_qlora_validation_needs_no_device():
    h = mnb.mnb_create(64, 64, 4)
    try:
        def rc(**kw):
            args = dict(X=0x1000, Wq=0x2000, scales=0x3000, zp=None, Aq=0x5000, As=0x6000, Az=None, Bq=0x7000,
                        Bs=0x8000, Bz=None, rank=32, bias=None, Y=0x4000, T_ws=0x9000, batch=1, M=1)
            args.update(kw)
            return mnb.lib().mnb_run_qlora(h, args["X"], args["Wq"], args["scales"], args["zp"], args["Aq"],
                                           args["As"], args["Az"], args["Bq"], args["Bs"], args["Bz"], args["rank"],
                                           args["bias"], args["Y"], args["T_ws"], args["batch"], args["M"], None)
        assert rc(As=None) == mnb.MNB_ERR_ARG          # an INT8 weight needs its scales
        assert rc(Bs=None) == mnb.MNB_ERR_ARG
        assert rc(Bq=None) == mnb.MNB_ERR_ARG          # half an adapter
        assert rc(T_ws=None) == mnb.MNB_ERR_ARG
        assert rc(rank=16) == mnb.MNB_ERR_UNSUPPORTED
        assert rc(Az=0x6008) == mnb.MNB_ERR_ALIGN
        assert rc(Bs=0x8002) == mnb.MNB_ERR_ALIGN
        assert rc(M=0) == mnb.MNB_OK and mnb.mnb_last_route(h) == mnb.ROUTE_NONE
    finally:
        mnb.mnb_destroy(h)


def check_multi_projection_validation_needs_no_device():
    h = mnb.mnb_create(96, 64, 4)
    try:
        def rc(projs, M=1, X=0x1000):
            arr = (mnb.MnbProjection * len(projs))(*[mnb.MnbProjection(*p) for p in projs])
            return mnb.lib().mnb_run_multi(h, X, arr, len(projs), 1, M, None)
        ok = (64, 0x2000, 0x3000, None, None, 0x4000)
        ok2 = (32, 0x5000, 0x6000, None, None, 0x7000)
        assert rc([ok]) == mnb.MNB_ERR_ARG                          # 64 != desc N 96
        assert rc([ok, ok2, ok2]) == mnb.MNB_ERR_ARG                # 128 != 96
        assert rc([ok] * 5) == mnb.MNB_ERR_UNSUPPORTED              # at most four members
        assert mnb.lib().mnb_run_multi(h, 0x1000, (mnb.MnbProjection * 1)(), 0, 1, 1, None) == mnb.MNB_ERR_UNSUPPORTED
        assert rc([ok, (32, 0x5000, 0x6000, 0x8000, None, 0x7000)]) == mnb.MNB_ERR_UNSUPPORTED  # zp for some only
        assert rc([ok, (32, 0x5000, None, None, None, 0x7000)]) == mnb.MNB_ERR_ARG  # weight without scales
        assert rc([ok, (32, 0x5000, 0x6000, None, None, None)]) == mnb.MNB_ERR_ARG  # no output
        assert rc([ok, (32, 0x5008, 0x6000, None, None, 0x7000)]) == mnb.MNB_ERR_ALIGN
        assert rc([ok, ok2], X=0x1002) == mnb.MNB_ERR_ALIGN
        assert rc([ok, ok2], M=0) == mnb.MNB_OK and mnb.mnb_last_route(h) == mnb.ROUTE_NONE
        # an empty member needs neither weight nor scales
        assert rc([ok, (32, None, None, None, None, 0x7000)], M=0) == mnb.MNB_OK
    finally:
        mnb.mnb_destroy(h)


def check_dequant_and_lora_down_validation_needs_no_device():
    L = mnb.lib()
    assert L.mnb_check_wait_timeout(10, None) == mnb.MNB_ERR_ARG
    assert L.mnb_check_wait_timeout(5_000_000_000, None) == mnb.MNB_ERR_ARG
    assert L.mnb_quantize_x(0x1000, 4, 48, 0x2000, 0x3000, None) == mnb.MNB_ERR_UNSUPPORTED
    assert L.mnb_quantize_x(0x1000, 0, 64, 0x2000, 0x3000, None) == mnb.MNB_OK
    assert L.mnb_quantize_x(0x1000, 4, 64, None, 0x3000, None) == mnb.MNB_ERR_ARG
    assert L.mnb_quantize_x(0x1000, 4, 64, 0x2004, 0x3000, None) == mnb.MNB_ERR_ALIGN
    assert L.mnb_dequant(0x1000, 0x2000, None, 4, 48, 4, 32, 0x3000, 0, None) == mnb.MNB_ERR_UNSUPPORTED
    assert L.mnb_dequant(0x1000, 0x2000, None, 4, 96, 2, 32, 0x3000, 0, None) == mnb.MNB_ERR_UNSUPPORTED
    assert L.mnb_dequant(0x1000, 0x2000, None, 0, 128, 2, 32, 0x3000, 1, None) == mnb.MNB_OK
    assert L.mnb_dequant(0x1000, 0x2000, None, 4, 64, 4, 32, 0x3000, 2, None) == mnb.MNB_ERR_ARG
    assert L.mnb_dequant(0x1000, 0x2000, None, 0, 64, 4, 32, 0x3000, 0, None) == mnb.MNB_OK
    assert L.mnb_dequant(0x1004, 0x2000, None, 4, 64, 4, 32, 0x3000, 0, None) == mnb.MNB_ERR_ALIGN
    assert L.mnb_lora_down(0x1000, 0x2000, 0x3000, 4, 64, 16, None) == mnb.MNB_ERR_UNSUPPORTED
    assert L.mnb_lora_down(0x1000, 0x2000, 0x3000, 0, 64, 32, None) == mnb.MNB_OK


def test_gemm_plan_splits_k_only_when_tiles_are_few():
    # 4096 x 4096 at M = 1: 32 tiles of 128 weight rows -> 4 CTAs (one cluster) per tile
    h = mnb.mnb_create(4096, 4096, 4, mode=mnb.MODE_FORCE_GEMM)
    try:
        p = mnb.mnb_plan(h, 1, 1, 0, 152)
        assert p["route"] == mnb.ROUTE_GEMM and p["k_splits"] == 4 and p["grid_x"] == 128
        assert p["tokens_per_cta"] == 16
        # prefill M = 1024: 128 tiles, persistent CTAs, no split
        p = mnb.mnb_plan(h, 1, 1024, 0, 152)
        assert p["k_splits"] == 1 and p["grid_x"] == 128 and p["tokens_per_cta"] == 256
        # many tiles: one CTA per SM walks over them
        p = mnb.mnb_plan(h, 1, 4096, 0, 152)
        assert p["k_splits"] == 1 and p["grid_x"] == 152
    finally:
        mnb.mnb_destroy(h)
    # never more CTAs per tile than K steps, never more than a portable cluster
    h = mnb.mnb_create(256, 128, 4, mode=mnb.MODE_FORCE_GEMM)
    try:
        p = mnb.mnb_plan(h, 1, 1, 0, 152)
        assert p["k_splits"] == 2 and p["grid_x"] == 4
    finally:
        mnb.mnb_destroy(h)
    h = mnb.mnb_create(128, 4096, 4, mode=mnb.MODE_FORCE_GEMM)
    try:
        assert mnb.mnb_plan(h, 1, 1, 0, 152)["k_splits"] == 8
    finally:
        mnb.mnb_destroy(h)


def test_run_validation_needs_no_device():
    run_without_gpu(check_run_validation_needs_no_device)


def test_qlora_validation_needs_no_device():
    run_without_gpu(check_qlora_validation_needs_no_device)


def test_multi_projection_validation_needs_no_device():
    run_without_gpu(check_multi_projection_validation_needs_no_device)


def test_dequant_and_lora_down_validation_needs_no_device():
    run_without_gpu(check_dequant_and_lora_down_validation_needs_no_device)
