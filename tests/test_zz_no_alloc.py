"""gqa_decode_attn_noalloc: the entry point for callers that cannot let the
library allocate device memory (a process whose memory is all handed to its
own pool at start-up, or a loop that cannot take the synchronisation a
cudaFree brings).  Its partial results live in a fixed array inside the
library instead of a cudaMalloc'd workspace.

The GPU test calls it through the C ABI on several problems in a row, so the
fixed array is used by each call after the previous one left its contents
there, and checks every output against the double-precision oracle within
the tolerance the parity tests use.  The sequence covers the CUDA-core path
at D = 64, 128 and 256, and a call on a small grid right after a call on a
large one: the second call reads fewer partial slots than the first wrote,
so reading a stale slot would show.  This file is named so that pytest
collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import grouped_query_kv_gb300 as g
import oracle
from grouped_query_kv_gb300 import workloads as wl

from helpers import assert_close, bits


@pytest.fixture(scope="module")
def lib():
    from grouped_query_kv_gb300 import build
    build.build()
    oracle.build()
    h = g.lib()
    assert h.kvattn_set_tuning(0, 0) == 0
    yield h
    assert h.kvattn_set_tuning(0, 0) == 0


def _call(fn, x, w, lens, out, stream):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return fn(P(x["q"]), P(x["k_cache"]), P(x["v_cache"]), P(lens), P(out),
              w.B, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale),
              ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_on_calls_in_a_row(lib):
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    cases = [
        # (workload, forced grid: 0 = one CTA per SM)
        # one long sequence: every CTA gets a piece of it
        (wl.Workload("noalloc_a", B=1, Hq=16, Hkv=2, D=128, Lmax=3000, scale=0.088,
                     lens=(3000,)), 0),
        # ragged multi-query batch with wide heads
        (wl.Workload("noalloc_b", B=6, Hq=16, Hkv=1, D=256, Lmax=2048, scale=1 / 16,
                     lens=(2048, 1, 900, 1500, 64, 2047)), 0),
        # D = 64 (the CUDA-core kernel's own head size), grouped heads
        (wl.Workload("noalloc_c", B=3, Hq=8, Hkv=2, D=64, Lmax=4000, scale=0.125,
                     lens=(4000, 17, 2500)), 0),
        # a large forced grid (many split pieces, slots up to 2 x 400) ...
        (wl.Workload("noalloc_d", B=2, Hq=8, Hkv=1, D=128, Lmax=6000, scale=0.088,
                     lens=(6000, 5999)), 400),
        # ... then a small one on a problem of its own: it reads only the
        # first slots, which the previous call also wrote
        (wl.Workload("noalloc_e", B=4, Hq=4, Hkv=4, D=64, Lmax=900, scale=0.125,
                     lens=(900, 3, 450, 77)), 6),
    ]
    try:
        for seed, (w, ctas) in enumerate(cases):
            assert lib.kvattn_set_tuning(0, ctas) == 0
            x = wl.make_inputs(w, seed=40 + seed, device=dev)
            lens = x["attn_lens"]
            got = torch.full((w.B, w.Hq, w.D), float("nan"), device=dev)
            assert _call(lib.gqa_decode_attn_noalloc, x, w, lens, got, stream) == 0, \
                lib.kvattn_last_error()
            assert lib.kvattn_check_device_error(ctypes.c_void_p(stream.cuda_stream)) == 0
            lens_np = lens.cpu().numpy()
            ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]),
                                    lens_np, w.scale)
            assert_close(got, ref, bits(x["v_cache"]), lens_np)
    finally:
        assert lib.kvattn_set_tuning(0, 0) == 0


def test_noalloc_rejects_a_grid_whose_partials_do_not_fit(lib):
    # a forced grid of 2000 CTAs needs 2*2000*8*(256+2)*4 bytes > 4 MiB; the
    # check comes before any device work, so this runs without a GPU
    assert lib.kvattn_set_tuning(0, 2000) == 0
    try:
        fake = ctypes.c_void_p(0x10000)
        rc = lib.gqa_decode_attn_noalloc(fake, fake, fake, fake, fake, 4, 64, 8, 256,
                                         1024, 0.0625, None)
        assert rc == g.KVATTN_ERR_UNSUPPORTED
        assert b"scratch" in lib.kvattn_last_error()
    finally:
        assert lib.kvattn_set_tuning(0, 0) == 0
