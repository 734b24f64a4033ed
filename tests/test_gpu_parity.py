"""GPU parity: the CUDA path through the C ABI against the double oracle on
the same seeded inputs.  kv_append must be bit-exact (the whole caches are
compared, so every row it must not touch is checked too); attention must be
within max|err| <= 2e-3 and <= 1e-2 * max|V|."""
import numpy as np
import pytest
import torch

import grouped_query_kv_gb300 as g
import oracle
from grouped_query_kv_gb300 import workloads as wl

from helpers import assert_close, bits, oracle_threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from grouped_query_kv_gb300 import build
    build.build()
    oracle.build()
    g.set_tuning(0, 0)
    yield
    g.set_tuning(0, 0)


def run_step(w, seed=0, lens=None, sample_b=None):
    """kv_append then gqa_decode_attn on the GPU (whole batch), compared with
    the oracle on every sequence, or on the sequences listed in sample_b."""
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=seed, device=dev, lens=lens)
    bsel = list(range(w.B)) if sample_b is None else sorted(int(b) for b in sample_b)
    idx = torch.tensor(bsel, device=dev)
    k_ref = bits(x["k_cache"].index_select(0, idx))
    v_ref = bits(x["v_cache"].index_select(0, idx))
    pos = x["append_pos"].cpu().numpy()[bsel]
    oracle.kv_append(k_ref, v_ref, bits(x["k_new"])[bsel], bits(x["v_new"])[bsel], pos)
    g.kv_append(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], x["append_pos"])
    out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
    g.check_device_error()
    assert np.array_equal(bits(x["k_cache"].index_select(0, idx)), k_ref), "kv_append: K differs"
    assert np.array_equal(bits(x["v_cache"].index_select(0, idx)), v_ref), "kv_append: V differs"
    lens_np = x["attn_lens"].cpu().numpy()[bsel]
    ref = oracle.gqa_decode(bits(x["q"])[bsel], k_ref, v_ref, lens_np, w.scale,
                            nthreads=oracle_threads())
    return assert_close(out.index_select(0, idx), ref, v_ref, lens_np)


def test_tiny_mqa_append_then_attend():
    run_step(wl.WORKLOADS["tiny_mqa"])


@pytest.mark.parametrize("name", ["palm8b_mqa", "llama70b_gqa_ragged", "palm540b_long_mqa"])
def test_full_size_configs_every_output(name):
    run_step(wl.WORKLOADS[name])


@pytest.mark.parametrize("name", [n for n in wl.CONFIG_ORDER if n.startswith("sweep")])
def test_sweep_points(name):
    w = wl.WORKLOADS[name]
    if w.B * w.Hkv * w.Lmax * w.D * 2 * 2 > (1 << 30):
        rng = np.random.default_rng(1)
        run_step(w, sample_b=rng.choice(w.B, 8, replace=False))
    else:
        run_step(w)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 3), (12, 4), (20, 4), (16, 2), (48, 1), (64, 8)])
def test_head_shapes_and_ragged_edges(D, Hq, Hkv):
    # lengths around tile boundaries (64 / 128 positions), 1, and Lmax
    Lmax = 300
    lens = [1, 63, 64, 65, 127, 128, 129, 300, 255, 2][: 10]
    w = wl.Workload("edge", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax,
                    scale=1.0 / np.sqrt(D), lens=tuple(lens))
    run_step(w, seed=D + Hq)


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 17, 152, 1000])
def test_split_pieces_combine_for_any_grid(ctas):
    # forcing the persistent grid size moves the cuts between CTAs, so
    # segments get split into 1..many pieces and merged by the combine
    w = wl.Workload("split", B=5, Hq=16, Hkv=2, D=128, Lmax=2000, scale=0.09,
                    lens=(2000, 1, 700, 1333, 129))
    g.set_tuning(0, ctas)
    try:
        run_step(w, seed=ctas)
    finally:
        g.set_tuning(0, 0)


def test_empty_sequences_give_zero_rows():
    dev = torch.device("cuda")
    w = wl.Workload("empty", B=3, Hq=8, Hkv=2, D=128, Lmax=256, scale=0.1, lens=(5, 5, 5))
    x = wl.make_inputs(w, seed=3, device=dev)
    lens = torch.tensor([0, 17, 0], dtype=torch.int32, device=dev)
    out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], lens, w.scale)
    g.check_device_error()
    o = out.cpu()
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]),
                            lens.cpu().numpy(), w.scale)
    assert_close(out, ref, bits(x["v_cache"]), [0, 17, 0])


def test_out_of_range_lengths_are_flagged_not_faulted():
    dev = torch.device("cuda")
    w = wl.Workload("bad", B=3, Hq=4, Hkv=1, D=64, Lmax=64, scale=0.1, lens=(5, 5, 5))
    x = wl.make_inputs(w, seed=4, device=dev)
    bad = torch.tensor([10, 65, -3], dtype=torch.int32, device=dev)
    out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], bad, w.scale)
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_DEVICE_BOUNDS
    o = out.cpu()
    assert torch.all(o[1] == 0) and torch.all(o[2] == 0)
    g.check_device_error()  # the word was cleared
    # append past the end: skipped, flagged, cache untouched
    before = bits(x["k_cache"])
    g.kv_append(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"],
                torch.tensor([64, 0, 63], dtype=torch.int32, device=dev))
    with pytest.raises(g.KvAttnError):
        g.check_device_error()
    after = bits(x["k_cache"])
    assert np.array_equal(after[0], before[0])
    assert np.array_equal(after[1, :, 0], bits(x["k_new"])[1])
    assert np.array_equal(after[2, :, 63], bits(x["k_new"])[2])


def test_side_stream_and_repeatability():
    dev = torch.device("cuda")
    w = wl.Workload("rep", B=4, Hq=32, Hkv=4, D=128, Lmax=1024, scale=0.088,
                    lens=(1024, 77, 512, 900))
    x = wl.make_inputs(w, seed=5, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
        b = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
    s.synchronize()
    g.check_device_error(s)
    assert torch.equal(a, b)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (4, 1), (12, 1), (16, 2), (96, 1), (128, 2)])
def test_each_path_on_each_head_shape(path, D, Hq, Hkv):
    # path 1 = CUDA-core kernel, 2 = tensor-core kernel, forced for any G
    lens = (700, 1, 129, 256, 1000, 383)
    w = wl.Workload("forced", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=1000,
                    scale=1.0 / np.sqrt(D), lens=lens)
    g.set_tuning(path, 0)
    try:
        assert g.get_plan(w.B, Hq, Hkv, D, w.Lmax, num_sms=152)["path"] == path
        run_step(w, seed=7 * path + D + Hq)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("path", [1, 2])
def test_non_finite_padding_is_never_used(path):
    # rows at and past each length hold NaN keys and infinite values; padding
    # is not part of the attention ("The Basics of Transformer Inference",
    # item "Using ragged HBM reads and Paged Attention"), so none of it may leak
    dev = torch.device("cuda")
    w = wl.Workload("nanpad", B=4, Hq=16, Hkv=2, D=128, Lmax=600, scale=0.088,
                    lens=(600, 5, 130, 257))
    x = wl.make_inputs(w, seed=11, device=dev)
    for b, n in enumerate(w.lens):
        x["k_cache"][b, :, n:] = float("nan")
        x["v_cache"][b, :, n:] = float("inf")
    g.set_tuning(path, 0)
    try:
        out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
        g.check_device_error()
    finally:
        g.set_tuning(0, 0)
    lens_np = x["attn_lens"].cpu().numpy()
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]), lens_np,
                            w.scale)
    assert_close(out, ref, bits(x["v_cache"]), lens_np)


@pytest.mark.parametrize("ctas", [15, 16, 17, 40])
def test_combine_rows_by_segment_and_by_record(ctas):
    # 16 segments: with more CTAs than segments the combine locates each
    # segment's pieces from the lengths (before waiting on the split-KV
    # kernel), otherwise it reads the CTAs' records; both must merge alike,
    # with ragged and one-tile sequences among the split ones
    w = wl.Workload("rows", B=16, Hq=8, Hkv=1, D=128, Lmax=3000, scale=0.1,
                    lens=(3000, 1, 2, 2999, 128, 129, 1500, 257, 3000, 64, 700, 2048, 5, 1000,
                          2500, 1777))
    g.set_tuning(2, ctas)
    try:
        run_step(w, seed=ctas)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("ctas", [1, 3, 152, 600])
def test_tensor_core_split_pieces(ctas):
    w = wl.Workload("tcsplit", B=3, Hq=48, Hkv=1, D=256, Lmax=5000, scale=1 / 16,
                    lens=(5000, 130, 2047), k_scale=0.5)
    g.set_tuning(2, ctas)
    try:
        run_step(w, seed=ctas + 1)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("ctas", [1, 2, 5, 152])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 2), (256, 96, 2)])
def test_tensor_core_many_short_pieces_with_padding(ctas, D, Hq, Hkv):
    # runs of one- to three-tile segments, most ending in a partial tile, with
    # non-finite padding: consecutive pieces alternate between the two output
    # buffers, and a partial tile's padded V rows are cleared while the next
    # tile is already in flight (D = 256 with 48 heads per pass has a single
    # probability stage and clears them at once)
    dev = torch.device("cuda")
    lens = (1, 129, 300, 128, 2, 257, 5, 383, 64, 256, 1, 200, 130, 17, 384, 255)
    w = wl.Workload("short", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=384,
                    scale=1.0 / np.sqrt(D), lens=lens)
    x = wl.make_inputs(w, seed=ctas + D, device=dev)
    for b, n in enumerate(lens):
        x["k_cache"][b, :, n:] = float("nan")
        x["v_cache"][b, :, n:] = float("inf")
    g.set_tuning(2, ctas)
    try:
        out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
        g.check_device_error()
    finally:
        g.set_tuning(0, 0)
    lens_np = x["attn_lens"].cpu().numpy()
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]), lens_np,
                            w.scale, nthreads=oracle_threads())
    assert_close(out, ref, bits(x["v_cache"]), lens_np)


def test_split_merges_across_changing_shapes():
    # calls of different shapes and split structures, queued on one stream
    # with no synchronisation in between, twice over: no state that one call
    # leaves on the device (workspace, split records) may leak into the next
    dev = torch.device("cuda")
    shapes = [
        wl.Workload("m16", B=3, Hq=16, Hkv=1, D=128, Lmax=3000, scale=0.088,
                    lens=(3000, 700, 129)),
        wl.Workload("m48", B=2, Hq=96, Hkv=2, D=256, Lmax=2500, scale=1 / 16,
                    lens=(2500, 1300), k_scale=0.5),
        wl.Workload("m8", B=6, Hq=32, Hkv=4, D=128, Lmax=1500, scale=0.088,
                    lens=(1500, 1, 640, 1499, 300, 1024)),
    ]
    inputs = [wl.make_inputs(w, seed=40 + i, device=dev) for i, w in enumerate(shapes)]
    outs = []
    for _ in range(2):
        for w, x in zip(shapes, inputs):
            outs.append(g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"],
                                          w.scale))
    g.check_device_error()
    for r in range(2):
        for i, (w, x) in enumerate(zip(shapes, inputs)):
            lens_np = x["attn_lens"].cpu().numpy()
            ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]), lens_np,
                                    w.scale, nthreads=oracle_threads())
            assert_close(outs[r * len(shapes) + i], ref, bits(x["v_cache"]), lens_np)


@pytest.mark.parametrize("name,calls", [("palm8b_mqa", 400), ("palm540b_long_mqa", 150),
                                        ("llama70b_gqa_ragged", 150)])
def test_many_back_to_back_calls_are_stable(name, calls):
    # hundreds of launches with no host synchronisation in between: a race in
    # the pipeline's barrier phases shows up as a changed result or a device
    # error word (the kernel's waits are bounded)
    w = wl.WORKLOADS[name]
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=21, device=dev)
    lens = x["attn_lens"]
    first = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], lens, w.scale)
    outs = [torch.empty_like(first) for _ in range(4)]
    for i in range(calls):
        g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], lens, w.scale, out=outs[i % 4])
        if i % 4 == 3:
            torch.cuda.synchronize()
            for o in outs:
                assert torch.equal(o, first), "result changed between identical calls"
    g.check_device_error()


def run_fused_step(w, seed=0, lens=None, sample_b=None):
    """gqa_decode_step (append fused into the attention kernel) vs the oracle's
    append followed by its attention over one more position."""
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=seed, device=dev, lens=lens)
    bsel = list(range(w.B)) if sample_b is None else sorted(int(b) for b in sample_b)
    idx = torch.tensor(bsel, device=dev)
    k_ref = bits(x["k_cache"].index_select(0, idx))
    v_ref = bits(x["v_cache"].index_select(0, idx))
    pos = x["append_pos"].cpu().numpy()[bsel]
    oracle.kv_append(k_ref, v_ref, bits(x["k_new"])[bsel], bits(x["v_new"])[bsel], pos)
    out = g.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                            x["append_pos"], w.scale)
    g.check_device_error()
    assert np.array_equal(bits(x["k_cache"].index_select(0, idx)), k_ref), "fused append: K differs"
    assert np.array_equal(bits(x["v_cache"].index_select(0, idx)), v_ref), "fused append: V differs"
    lens_np = x["attn_lens"].cpu().numpy()[bsel]
    ref = oracle.gqa_decode(bits(x["q"])[bsel], k_ref, v_ref, lens_np, w.scale,
                            nthreads=oracle_threads())
    return assert_close(out.index_select(0, idx), ref, v_ref, lens_np)


@pytest.mark.parametrize("name", ["tiny_mqa", "palm8b_mqa", "llama70b_gqa_ragged",
                                  "palm540b_long_mqa", "sweep_hkv8_b64", "sweep_hkv32_b8"])
def test_fused_step_on_the_configs(name):
    run_fused_step(wl.WORKLOADS[name])


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 2), (256, 48, 1), (64, 4, 1), (128, 96, 1)])
def test_fused_step_edges_and_paths(path, D, Hq, Hkv):
    if path == 2 and D == 64:
        pytest.skip("tensor-core path needs D in {128, 256}")
    # lengths after the append: 1 (append into an empty cache), tile edges, Lmax
    lens = (1, 127, 128, 129, 300, 64, 65, 2)
    w = wl.Workload("fused", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=300,
                    scale=1.0 / np.sqrt(D), lens=lens)
    g.set_tuning(path, 0)
    try:
        run_fused_step(w, seed=3 * path + D)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_fused_step_with_split_pieces(ctas):
    w = wl.Workload("fsplit", B=4, Hq=32, Hkv=4, D=128, Lmax=3000, scale=0.088,
                    lens=(3000, 1, 1700, 250))
    g.set_tuning(0, ctas)
    try:
        run_fused_step(w, seed=ctas)
    finally:
        g.set_tuning(0, 0)


def test_fused_step_flags_rows_outside_the_cache():
    dev = torch.device("cuda")
    w = wl.Workload("fbad", B=3, Hq=16, Hkv=2, D=128, Lmax=64, scale=0.1, lens=(5, 5, 5))
    x = wl.make_inputs(w, seed=9, device=dev)
    before = bits(x["k_cache"])
    pos = torch.tensor([64, 3, -1], dtype=torch.int32, device=dev)
    out = g.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], pos,
                            w.scale)
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_DEVICE_BOUNDS
    after = bits(x["k_cache"])
    assert np.array_equal(after[0], before[0]) and np.array_equal(after[2], before[2])
    assert np.array_equal(after[1, :, 3], bits(x["k_new"])[1])
    o = out.cpu()
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    ref = oracle.gqa_decode(bits(x["q"])[1:2], after[1:2], bits(x["v_cache"])[1:2],
                            np.array([4], np.int32), w.scale)
    assert_close(out[1:2], ref, bits(x["v_cache"])[1:2], [4])


# ------------------------------------------------------- local (window) layers
# "The Basics of Transformer Inference", item on mixing in local attention
# layers: the query attends only the last `window` positions.

def _window_case(w, seed, window, nan_pad=True):
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=seed, device=dev)
    if nan_pad:
        for b, n in enumerate(x["attn_lens"].tolist()):
            x["k_cache"][b, :, n:] = float("nan")
            x["v_cache"][b, :, n:] = float("inf")
    out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale,
                            window=window)
    g.check_device_error()
    lens_np = x["attn_lens"].cpu().numpy()
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]), lens_np,
                            w.scale, nthreads=oracle_threads(), window=window)
    assert_close(out, ref, bits(x["v_cache"]), lens_np)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 2), (256, 48, 1), (128, 8, 8)])
@pytest.mark.parametrize("window", [1, 5, 127, 128, 129, 300, 5000])
def test_local_window_attention(path, D, Hq, Hkv, window):
    lens = (700, 1, 129, 256, 1000, 383, 128, 4)
    w = wl.Workload("win", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Lmax=1000,
                    scale=1.0 / np.sqrt(D), lens=lens)
    g.set_tuning(path, 0)
    try:
        _window_case(w, seed=window + D + path, window=window)
    finally:
        g.set_tuning(0, 0)


def test_local_window_on_the_cuda_core_path_at_d64():
    w = wl.Workload("win64", B=4, Hq=8, Hkv=2, D=64, Lmax=600, scale=0.125,
                    lens=(600, 77, 1, 300))
    for window in (1, 63, 64, 65, 200):
        _window_case(w, seed=window, window=window)


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_local_window_with_split_pieces(ctas):
    w = wl.Workload("winsplit", B=3, Hq=48, Hkv=1, D=256, Lmax=5000, scale=1 / 16,
                    lens=(5000, 130, 2047), k_scale=0.5)
    g.set_tuning(2, ctas)
    try:
        _window_case(w, seed=ctas, window=1500)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("window", [1, 100, 2000])
def test_local_window_fused_step(window):
    dev = torch.device("cuda")
    w = wl.Workload("winstep", B=5, Hq=32, Hkv=4, D=128, Lmax=1500, scale=0.088,
                    lens=(1500, 1, 640, 129, 1000))
    x = wl.make_inputs(w, seed=window, device=dev)
    k_ref, v_ref = bits(x["k_cache"]), bits(x["v_cache"])
    oracle.kv_append(k_ref, v_ref, bits(x["k_new"]), bits(x["v_new"]),
                     x["append_pos"].cpu().numpy())
    out = g.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                            x["append_pos"], w.scale, window=window)
    g.check_device_error()
    assert np.array_equal(bits(x["k_cache"]), k_ref)
    assert np.array_equal(bits(x["v_cache"]), v_ref)
    lens_np = x["attn_lens"].cpu().numpy()
    ref = oracle.gqa_decode(bits(x["q"]), k_ref, v_ref, lens_np, w.scale,
                            nthreads=oracle_threads(), window=window)
    assert_close(out, ref, v_ref, lens_np)


def test_local_window_workload_every_output():
    w = wl.WORKLOADS["local_gqa_w4096"]
    _window_case(w, seed=0, window=w.window, nan_pad=False)


def test_local_window_must_be_positive():
    dev = torch.device("cuda")
    w = wl.WORKLOADS["tiny_mqa"]
    x = wl.make_inputs(w, seed=0, device=dev)
    with pytest.raises(g.KvAttnError):
        g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale, window=0)


# --------------------------------------------- several new tokens (speculative)
# "The Basics of Transformer Inference", speculative sampling: T drafted
# tokens scored in one pass; token t attends the prefix and the new tokens up
# to itself.

def _multi_case(B, T, Hq, Hkv, D, Lmax, lens, seed, nan_pad=True, window=None):
    dev = torch.device("cuda")
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn((B, T, Hq, D), generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn((B, Hkv, Lmax, D), generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn((B, Hkv, Lmax, D), generator=gen).to(torch.bfloat16).to(dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    if nan_pad:
        for b, n in enumerate(lens):
            k[b, :, n:] = float("nan")
            v[b, :, n:] = float("inf")
    scale = 1.0 / np.sqrt(D)
    out = g.gqa_decode_attn_multi(q, k, v, lens_t, scale, window=window)
    g.check_device_error()
    lens_np = np.array(lens, np.int32)
    ref = oracle.gqa_decode_multi(bits(q), bits(k), bits(v), lens_np, scale,
                                  nthreads=oracle_threads(), window=window)
    assert_close(out.reshape(B * T, Hq, D), ref.reshape(B * T, Hq, D), bits(v), lens_np)


@pytest.mark.parametrize("D,Hq,Hkv,T", [(128, 64, 8, 1), (128, 64, 8, 2), (128, 64, 8, 4),
                                        (128, 64, 8, 8), (128, 16, 16, 2), (128, 16, 16, 8),
                                        (128, 4, 4, 64), (256, 16, 1, 2), (256, 16, 1, 3),
                                        (256, 8, 8, 5)])
def test_new_tokens_attend_causally(D, Hq, Hkv, T):
    lens = (700, T, 129, 256, 1000, 383, max(1, T - 1), 128)
    _multi_case(len(lens), T, Hq, Hkv, D, 1000, lens, seed=T * 7 + D + Hq)


# G x T rows beyond one pass: the heads split over several passes, each pass
# re-reading the K/V head ("Efficiently Scaling Transformer Inference", §3:
# 48 query heads sharing one K/V head; PaLM-8B's 16 heads of 256)
@pytest.mark.parametrize("D,Hq,Hkv,T", [(256, 16, 1, 5), (256, 16, 1, 8), (256, 48, 1, 2),
                                        (256, 48, 1, 4), (256, 48, 1, 8), (256, 96, 2, 3),
                                        (128, 64, 4, 5), (128, 16, 1, 9), (128, 32, 1, 64),
                                        (256, 13, 1, 7), (256, 4, 1, 48), (256, 4, 1, 64)])
def test_new_tokens_over_several_head_passes(D, Hq, Hkv, T):
    G = Hq // Hkv
    cols = 64  # (token, head) columns one pass holds, at D = 128 and 256
    passes = -(-G // (cols // T))
    assert G * T > cols or T == cols  # the shapes need several passes (or a full one)
    plan_hpg = -(-G // passes)
    assert plan_hpg * T <= cols
    lens = (600, T, 129, 257, max(1, T - 1), 383)
    _multi_case(len(lens), T, Hq, Hkv, D, 600, lens, seed=T * 5 + D + Hq)


@pytest.mark.parametrize("ctas", [1, 19, 152, 500])
def test_new_tokens_over_head_passes_with_split_pieces(ctas):
    # the PaLM-540B head shape, 4 drafted tokens: 3 passes of 16 heads, each
    # sequence's passes cut into pieces by the forced grid
    g.set_tuning(0, ctas)
    try:
        _multi_case(2, 4, 48, 1, 256, 3000, (3000, 1291), seed=ctas + 3)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_new_tokens_with_split_pieces(ctas):
    g.set_tuning(0, ctas)
    try:
        _multi_case(3, 4, 32, 4, 128, 3000, (3000, 130, 2047), seed=ctas)
    finally:
        g.set_tuning(0, 0)


# Several drafted tokens on a local layer: token t attends the `window`
# positions that end at its own.
@pytest.mark.parametrize("D,Hq,Hkv,T", [(128, 64, 8, 2), (128, 16, 16, 8), (256, 16, 1, 3),
                                        (256, 16, 1, 8), (256, 48, 1, 2), (128, 4, 4, 64)])
@pytest.mark.parametrize("window", [1, 7, 127, 128, 129, 500, 5000])
def test_new_tokens_with_a_local_window(D, Hq, Hkv, T, window):
    lens = (700, T, 129, 256, 1000, 383, max(1, T - 1), 128)
    _multi_case(len(lens), T, Hq, Hkv, D, 1000, lens, seed=T * 11 + D + Hq + window,
                window=window)


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_new_tokens_with_a_local_window_and_split_pieces(ctas):
    g.set_tuning(0, ctas)
    try:
        _multi_case(3, 4, 48, 1, 256, 3000, (3000, 130, 2047), seed=ctas + 5, window=1500)
    finally:
        g.set_tuning(0, 0)


def test_new_tokens_reject_what_one_pass_cannot_hold():
    # more tokens than one pass has rows, or a head width without the
    # tensor-core kernel
    dev = torch.device("cuda")
    for (B, T, Hq, Hkv, D) in [(1, 65, 16, 1, 256), (1, 65, 8, 1, 128), (1, 2, 4, 1, 64)]:
        q = torch.zeros((B, T, Hq, D), dtype=torch.bfloat16, device=dev)
        k = torch.zeros((B, Hkv, 256, D), dtype=torch.bfloat16, device=dev)
        lens = torch.full((B,), 100, dtype=torch.int32, device=dev)
        with pytest.raises(g.KvAttnError):
            g.gqa_decode_attn_multi(q, k, k, lens, 0.1)


@pytest.mark.parametrize("name,nsel", [("llama70b_spec4", 8), ("palm8b_spec4", 8),
                                       ("palm540b_spec4", 2)])
def test_drafted_token_workloads_at_full_size_sampled(name, nsel):
    # the benchmark's drafted-token shapes as it runs them; a seeded sample
    # of sequences checked against the oracle, every token and head of each
    w = wl.WORKLOADS[name]
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=0, device=dev)
    out = g.gqa_decode_attn_multi(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale)
    g.check_device_error()
    rng = np.random.default_rng(11)
    sel = sorted(rng.choice(w.B, nsel, replace=False).tolist())
    lens = x["attn_lens"].cpu().numpy()[sel]
    k = bits(x["k_cache"][sel])
    v = bits(x["v_cache"][sel])
    ref = oracle.gqa_decode_multi(bits(x["q"][sel]), k, v, lens, w.scale,
                                  nthreads=oracle_threads())
    n = len(sel)
    assert_close(out[sel].reshape(n * w.T, w.Hq, w.D), ref.reshape(n * w.T, w.Hq, w.D), v, lens)


@pytest.mark.parametrize("T", [1, 3, 8])
def test_appending_several_tokens_is_bit_exact(T):
    # T single-row appends in the oracle, one call on the GPU; then the same
    # tokens scored together
    dev = torch.device("cuda")
    B, Hq, Hkv, D, Lmax = 4, 32, 4, 128, 600
    before = np.array([0, 37, 590 - T, 300], np.int32)
    gen = torch.Generator(device="cpu").manual_seed(T)
    k = torch.randn((B, Hkv, Lmax, D), generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn((B, Hkv, Lmax, D), generator=gen).to(torch.bfloat16).to(dev)
    kn = torch.randn((B, T, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    vn = torch.randn((B, T, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    q = torch.randn((B, T, Hq, D), generator=gen).to(torch.bfloat16).to(dev)
    k_ref, v_ref = bits(k), bits(v)
    for t in range(T):
        oracle.kv_append(k_ref, v_ref, np.ascontiguousarray(bits(kn)[:, t]),
                         np.ascontiguousarray(bits(vn)[:, t]), before + t)
    g.kv_append_multi(k, v, kn, vn, torch.tensor(before, device=dev))
    g.check_device_error()
    assert np.array_equal(bits(k), k_ref) and np.array_equal(bits(v), v_ref)
    lens = before + T
    out = g.gqa_decode_attn_multi(q, k, v, torch.tensor(lens, device=dev), 0.088)
    ref = oracle.gqa_decode_multi(bits(q), k_ref, v_ref, lens, 0.088, nthreads=oracle_threads())
    assert_close(out.reshape(B * T, Hq, D), ref.reshape(B * T, Hq, D), v_ref, lens)


def test_appending_rows_that_do_not_fit_is_flagged_and_skipped():
    dev = torch.device("cuda")
    B, T, Hkv, D, Lmax = 2, 4, 2, 128, 64
    k = torch.zeros((B, Hkv, Lmax, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    kn = torch.ones((B, T, Hkv, D), dtype=torch.bfloat16, device=dev)
    before = torch.tensor([10, Lmax - T + 1], dtype=torch.int32, device=dev)
    g.kv_append_multi(k, v, kn, kn, before)
    with pytest.raises(g.KvAttnError):
        g.check_device_error()
    assert torch.all(k[1] == 0) and torch.all(k[0, :, 10:14] == 1)


def test_graph_captured_before_the_workspace_grows_stays_valid():
    # a call that needs a larger workspace retires the old buffer instead of
    # freeing it, so a graph captured with the old one still replays
    dev = torch.device("cuda")
    w = wl.Workload("grow", B=6, Hq=16, Hkv=2, D=128, Lmax=1500, scale=0.1,
                    lens=(1500, 3, 700, 1200, 129, 64))
    x = wl.make_inputs(w, seed=21, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    try:
        g.set_tuning(0, 7)
        with torch.cuda.stream(s):
            g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale,
                              out=out, stream=s)
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale,
                              out=out, stream=s)
        g.set_tuning(0, 3000)  # needs a much larger workspace on the same stream
        with torch.cuda.stream(s):
            g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["attn_lens"], w.scale,
                              out=torch.empty_like(out), stream=s)
        s.synchronize()
        out.zero_()
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
    finally:
        g.set_tuning(0, 0)
    g.check_device_error()
    ref = oracle.gqa_decode(bits(x["q"]), bits(x["k_cache"]), bits(x["v_cache"]),
                            x["attn_lens"].cpu().numpy(), w.scale)
    assert_close(out, ref, bits(x["v_cache"]), list(w.lens))
