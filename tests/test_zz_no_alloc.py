"""gqa_decode_attn_noalloc: the entry point for callers that cannot let the
library allocate device memory (a process whose memory is all handed to its
own pool at start-up, or a loop that cannot take the synchronisation a
cudaFree brings).  Its partial results live in a fixed array inside the
library instead of a cudaMalloc'd workspace.

The GPU test calls it through the C ABI twice in a row, on two different
problems that both split sequences across CTAs (so the fixed array is used,
and the second call runs on whatever the first left in it), and checks each
result against the regular gqa_decode_attn within the tolerance the parity
tests use.  This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import grouped_query_kv_gb300 as g
from grouped_query_kv_gb300 import workloads as wl

from helpers import ATOL, VREL


def _call(fn, x, w, lens, out, stream):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return fn(P(x["q"]), P(x["k_cache"]), P(x["v_cache"]), P(lens), P(out),
              w.B, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale),
              ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row():
    from grouped_query_kv_gb300 import build
    build.build()
    lib = g.lib()
    assert lib.kvattn_set_tuning(0, 0) == 0
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    cases = [
        # one long sequence: every CTA gets a piece of it
        wl.Workload("noalloc_a", B=1, Hq=16, Hkv=2, D=128, Lmax=3000, scale=0.088,
                    lens=(3000,)),
        # ragged multi-query batch with wide heads
        wl.Workload("noalloc_b", B=6, Hq=16, Hkv=1, D=256, Lmax=2048, scale=1 / 16,
                    lens=(2048, 1, 900, 1500, 64, 2047)),
    ]
    for seed, w in enumerate(cases):
        x = wl.make_inputs(w, seed=40 + seed, device=dev)
        lens = x["attn_lens"]
        got = torch.full((w.B, w.Hq, w.D), float("nan"), device=dev)
        want = torch.empty((w.B, w.Hq, w.D), device=dev)
        assert _call(lib.gqa_decode_attn_noalloc, x, w, lens, got, stream) == 0, \
            lib.kvattn_last_error()
        assert _call(lib.gqa_decode_attn, x, w, lens, want, stream) == 0, \
            lib.kvattn_last_error()
        assert lib.kvattn_check_device_error(ctypes.c_void_p(stream.cuda_stream)) == 0
        vmax = max(float(x["v_cache"][b, :, :int(n)].abs().max())
                   for b, n in enumerate(lens.tolist()))
        err = float((got - want).abs().max())
        assert torch.isfinite(got).all()
        assert err <= min(ATOL, VREL * vmax), (w.name, err)


def test_noalloc_rejects_a_grid_whose_partials_do_not_fit():
    # a forced grid of 2000 CTAs needs 2*2000*8*(256+2)*4 bytes > 4 MiB; the
    # check comes before any device work, so this runs without a GPU
    lib = g.lib()
    assert lib.kvattn_set_tuning(0, 2000) == 0
    try:
        fake = ctypes.c_void_p(0x10000)
        rc = lib.gqa_decode_attn_noalloc(fake, fake, fake, fake, fake, 4, 64, 8, 256,
                                         1024, 0.0625, None)
        assert rc == g.KVATTN_ERR_UNSUPPORTED
        assert b"scratch" in lib.kvattn_last_error()
    finally:
        assert lib.kvattn_set_tuning(0, 0) == 0
