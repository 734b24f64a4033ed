"""Failure detection on the GPU without a fault: every wait inside the
tensor-core split-KV kernel is bounded, and a kernel that gives up reports
KVATTN_ERR_TIMEOUT through the sticky device error word instead of hanging.

kvattn_set_wait_limit shortens the pipeline waits (the softmax threads'
waits for scores and for finished P.V products, the MMA thread's polling
while nothing is ready) to a single poll, so the call is sure to give up
before its first K/V tile has arrived.  Waits for copies and MMAs already
issued keep their full limit, so the CTA returns only after all of them have
finished and its tensor memory is freed.  The test then checks that the
error is reported once and cleared, and that the next normal call on the
same stream -- same workspace, same device -- matches the oracle."""
import numpy as np
import pytest
import torch

import grouped_query_kv_gb300 as g
import oracle
from grouped_query_kv_gb300 import workloads as wl

from helpers import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from grouped_query_kv_gb300 import build
    build.build()
    oracle.build()
    g.set_tuning(0, 0)
    g.set_wait_limit(0)
    yield
    g.set_wait_limit(0)
    g.set_tuning(0, 0)


def _expect_timeout():
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_TIMEOUT
    g.check_device_error()  # the word was cleared by the first check


# (the 32-head pass runs its softmax in two groups of warps, the others in one)
@pytest.mark.parametrize("D,Hq,Hkv,ctas", [(128, 16, 2, 0), (256, 48, 1, 0), (128, 64, 8, 37),
                                           (128, 32, 1, 0), (128, 32, 1, 37)])
def test_a_wait_that_runs_out_reports_a_timeout_and_the_next_call_is_clean(D, Hq, Hkv, ctas):
    dev = torch.device("cuda")
    lens = (700, 5, 300, 129)
    w = wl.Workload("timeout", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=700,
                    scale=1.0 / np.sqrt(D), lens=lens)
    x = wl.make_inputs(w, seed=D + Hq, device=dev)
    g.check_device_error()  # start from a clean word
    g.set_tuning(2, ctas)   # the tensor-core kernel; ctas > 0 forces split segments
    try:
        g.set_wait_limit(1)
        out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
        _expect_timeout()
        # the fused step gives up the same way (its append may or may not run)
        g.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"].clone(),
                          x["v_cache"].clone(), x["append_pos"], w.scale)
        _expect_timeout()
        g.set_wait_limit(0)
        out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
        g.check_device_error()
    finally:
        g.set_wait_limit(0)
        g.set_tuning(0, 0)
    lens_np = x["attn_lens"].cpu().numpy()
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]), lens_np, w.scale)
    assert_close(out, ref, bits(x["v_cache"]), lens_np)


def test_a_timed_out_call_inside_a_chain_leaves_later_calls_correct():
    # several calls queued back to back on one stream, the middle one made to
    # give up: the calls after it run on the same workspace and must be exact
    dev = torch.device("cuda")
    w = wl.WORKLOADS["palm8b_mqa"]
    x = wl.make_inputs(w, seed=5, device=dev)
    g.check_device_error()
    outs = []
    try:
        for k in range(5):
            g.set_wait_limit(1 if k == 2 else 0)
            outs.append(g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"],
                                          w.scale))
    finally:
        g.set_wait_limit(0)
    _expect_timeout()
    lens_np = x["attn_lens"].cpu().numpy()
    sel = [0, 17, 63]
    ref = oracle.gqa_decode(bits(x["q"])[sel], bits(x["k_cache"])[sel], bits(x["v_cache"])[sel],
                            lens_np[sel], w.scale)
    for k in (3, 4):
        assert_close(outs[k][sel], ref, bits(x["v_cache"])[sel], lens_np[sel])


@pytest.mark.parametrize("D,Hq,Hkv,T", [(128, 64, 8, 4), (256, 48, 1, 2)])
def test_several_token_pass_that_times_out_reports_it_and_the_next_call_is_clean(D, Hq, Hkv, T):
    # passes of 32 and 48 (token, head) columns: softmax in two groups of warps
    dev = torch.device("cuda")
    lens = (600, T, 129, 300)
    gen = torch.Generator(device="cpu").manual_seed(T + D)
    q = torch.randn((len(lens), T, Hq, D), generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn((len(lens), Hkv, 600, D), generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn((len(lens), Hkv, 600, D), generator=gen).to(torch.bfloat16).to(dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(D)
    g.check_device_error()
    try:
        g.set_wait_limit(1)
        g.gqa_decode_attn_multi(q, k, v, lens_t, scale)
        _expect_timeout()
        g.set_wait_limit(0)
        out = g.gqa_decode_attn_multi(q, k, v, lens_t, scale)
        g.check_device_error()
    finally:
        g.set_wait_limit(0)
    lens_np = np.array(lens, np.int32)
    ref = oracle.gqa_decode_multi(bits(q), bits(k), bits(v), lens_np, scale)
    B = len(lens)
    assert_close(out.reshape(B * T, Hq, D), ref.reshape(B * T, Hq, D), bits(v), lens_np)


def test_wait_limit_knob_round_trips():
    g.set_wait_limit(123)
    g.set_wait_limit(0)
