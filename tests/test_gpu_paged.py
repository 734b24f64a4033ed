"""GPU parity for the paged KV cache: the pools and block table that
workloads.make_paged builds, read through the C ABI, against the oracle's
gather-through-the-table decode ("Machine Learning Engineering and AI
Systems at Scale", section "The key and value cache": fixed-size blocks and
a per-sequence block table).  Appends must be bit-exact; attention within
max|err| <= 2e-3 and <= 1e-2 * max|V|.  Every pool row that no attended
position maps to holds NaN, and table entries of unused blocks are -1, so a
kernel that read either would fail the comparison."""
import dataclasses

import numpy as np
import pytest
import torch

import grouped_query_kv_gb300 as g
import oracle
from grouped_query_kv_gb300 import workloads as wl

from helpers import assert_close, bits, oracle_threads

pytestmark = pytest.mark.gpu

NAN = 0x7FC0


@pytest.fixture(scope="module", autouse=True)
def _built():
    from grouped_query_kv_gb300 import build
    build.build()
    oracle.build()
    g.set_tuning(0, 0)
    yield
    g.set_tuning(0, 0)


def _case(B, Hq, Hkv, D, Lmax, bs, lens, seed, T=1, spare=5):
    w = wl.Workload("paged", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, scale=1.0 / np.sqrt(D),
                    lens=tuple(lens), T=T, block_size=bs)
    x = wl.make_inputs(w, seed=seed, device=torch.device("cuda"))
    pg = wl.make_paged(w, x, seed=seed, spare_blocks=spare, fill_unused=NAN)
    return w, x, pg


def _oracle_paged(w, x, pg, lens=None, window=None):
    lens = x["attn_lens"].cpu().numpy() if lens is None else np.asarray(lens)
    table = pg["block_table"].cpu().numpy()
    k = oracle.gather_paged(bits(pg["k_pool"]), table, lens, w.block_size)
    v = oracle.gather_paged(bits(pg["v_pool"]), table, lens, w.block_size)
    q = bits(x["q"])
    if w.T > 1:
        ref = oracle.gqa_decode_multi(q, k, v, lens, w.scale, nthreads=oracle_threads(),
                                      window=window)
    else:
        ref = oracle.gqa_decode(q, k, v, lens, w.scale, nthreads=oracle_threads(),
                                window=window)
    return ref, v, lens


def _attend(w, x, pg):
    out = g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], pg["block_table"],
                                  x["attn_lens"], w.scale)
    g.check_device_error()
    ref, v, lens = _oracle_paged(w, x, pg)
    return assert_close(out, ref, v, list(lens))


# lengths around block and tile edges for each block size
def _edge_lens(bs, Lmax):
    ls = {1, 2, bs - 1, bs, bs + 1, 127, 128, 129, 255, 256, 257, 3 * bs + 5, Lmax - 1, Lmax}
    return sorted(n for n in ls if 1 <= n <= Lmax)


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256, 1024])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 64, 8), (128, 8, 8), (256, 16, 1), (256, 48, 1)])
def test_paged_attention_matches_oracle(bs, D, Hq, Hkv):
    Lmax = 1100
    lens = _edge_lens(bs, Lmax)
    w, x, pg = _case(len(lens), Hq, Hkv, D, Lmax, bs, lens, seed=bs + D + Hq)
    _attend(w, x, pg)


@pytest.mark.parametrize("bs", [16, 128])
@pytest.mark.parametrize("ctas", [1, 3, 17, 152, 600])
def test_paged_split_pieces_merge(bs, ctas):
    g.set_tuning(0, ctas)
    try:
        w, x, pg = _case(4, 32, 4, 128, 3000, bs, (3000, 1, 1709, 130), seed=ctas + bs)
        _attend(w, x, pg)
    finally:
        g.set_tuning(0, 0)


def test_paged_empty_sequences_give_zero_rows():
    w, x, pg = _case(3, 16, 2, 128, 512, 16, (40, 40, 40), seed=11)
    lens = torch.tensor([0, 33, 0], dtype=torch.int32, device="cuda")
    out = g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], pg["block_table"], lens,
                                  w.scale)
    g.check_device_error()
    o = out.cpu()
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    ref, v, ls = _oracle_paged(w, x, pg, lens=[0, 33, 0])
    assert_close(out, ref, v, list(ls))


@pytest.mark.parametrize("bs", [16, 64, 256])
@pytest.mark.parametrize("T", [2, 4, 8])
def test_paged_new_tokens_attend_causally(bs, T):
    # G * T query rows per pass: 8 * T <= 64
    lens = sorted({T, T + 1, bs - 1 if bs > T else T, bs + 3, 129, 700, 1000})
    w, x, pg = _case(len(lens), 8, 1, 128, 1000, bs, lens, seed=T * 31 + bs, T=T)
    _attend(w, x, pg)


def test_shared_prefix_blocks_are_read_by_every_sequence():
    # sequences 1 and 2 point at sequence 0's first three blocks (a shared
    # prompt) and continue in blocks of their own
    dev = torch.device("cuda")
    w, x, pg = _case(3, 32, 4, 128, 256, 32, (200, 200, 200), seed=5)
    table = pg["block_table"].clone()
    table[1, :3] = table[0, :3]
    table[2, :3] = table[0, :3]
    pg = dict(pg, block_table=table.contiguous())
    lens = torch.tensor([200, 150, 97], dtype=torch.int32, device=dev)
    out = g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], pg["block_table"], lens,
                                  w.scale)
    g.check_device_error()
    ref, v, ls = _oracle_paged(w, x, pg, lens=[200, 150, 97])
    assert_close(out, ref, v, list(ls))


@pytest.mark.parametrize("bs", [16, 128])
@pytest.mark.parametrize("T", [1, 3])
def test_paged_append_is_bit_exact(bs, T):
    dev = torch.device("cuda")
    B, Hkv, D, Lmax = 4, 4, 128, 600
    before = np.array([0, 37, 590 - T, 300], np.int32)
    w = wl.Workload("pa", B=B, Hq=Hkv, Hkv=Hkv, D=D, Lmax=Lmax, scale=0.1,
                    lens=tuple(int(n) + T for n in before), block_size=bs)
    x = wl.make_inputs(w, seed=bs + T, device=dev)
    pg = wl.make_paged(w, x, seed=bs, spare_blocks=3, fill_unused=NAN)
    gen = torch.Generator(device="cpu").manual_seed(T)
    kn = torch.randn((B, T, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    vn = torch.randn((B, T, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
    k_ref, v_ref = bits(pg["k_pool"]), bits(pg["v_pool"])
    table = pg["block_table"].cpu().numpy()
    for b in range(B):
        for t in range(T):
            j = int(before[b]) + t
            k_ref[table[b, j // bs], :, j % bs] = bits(kn)[b, t]
            v_ref[table[b, j // bs], :, j % bs] = bits(vn)[b, t]
    pos = torch.tensor(before, device=dev)
    if T == 1:
        g.kv_append_paged(pg["k_pool"], pg["v_pool"], kn[:, 0].contiguous(),
                          vn[:, 0].contiguous(), pg["block_table"], pos)
    else:
        g.kv_append_paged(pg["k_pool"], pg["v_pool"], kn, vn, pg["block_table"], pos)
    g.check_device_error()
    assert np.array_equal(bits(pg["k_pool"]), k_ref)
    assert np.array_equal(bits(pg["v_pool"]), v_ref)


@pytest.mark.parametrize("bs", [16, 32, 128, 512])
def test_paged_fused_step_is_append_then_attend(bs):
    dev = torch.device("cuda")
    lens = (1, 16, 17, 128, 129, 500, 1024)   # attended, after the append
    w, x, pg = _case(len(lens), 32, 4, 128, 1024, bs, lens, seed=bs)
    k_ref, v_ref = bits(pg["k_pool"]), bits(pg["v_pool"])
    table = pg["block_table"].cpu().numpy()
    pos = x["append_pos"].cpu().numpy()
    for b in range(w.B):
        j = int(pos[b])
        k_ref[table[b, j // bs], :, j % bs] = bits(x["k_new"])[b]
        v_ref[table[b, j // bs], :, j % bs] = bits(x["v_new"])[b]
    out = g.gqa_decode_step_paged(x["q"], x["k_new"], x["v_new"], pg["k_pool"], pg["v_pool"],
                                  pg["block_table"], x["append_pos"], w.scale)
    g.check_device_error()
    assert np.array_equal(bits(pg["k_pool"]), k_ref)
    assert np.array_equal(bits(pg["v_pool"]), v_ref)
    _attend(w, x, pg)  # the pools now hold the new rows: attention alone agrees too
    ref, v, ls = _oracle_paged(w, x, pg)
    assert_close(out, ref, v, list(ls))


def test_bad_table_entries_are_flagged_not_faulted():
    dev = torch.device("cuda")
    w, x, pg = _case(2, 16, 2, 128, 256, 16, (100, 100), seed=9)
    table = pg["block_table"].clone()
    nblk = pg["k_pool"].shape[0]
    table[0, 2] = nblk + 5      # past the pool
    table[1, 0] = -2            # negative
    before_k = bits(pg["k_pool"])
    out = g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], table.contiguous(),
                                  x["attn_lens"], w.scale)
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_DEVICE_BOUNDS
    assert torch.all(torch.isfinite(out))
    # an append whose block is outside the pool is skipped
    bad = torch.tensor([[nblk] * table.shape[1]] * 2, dtype=torch.int32, device=dev)
    g.kv_append_paged(pg["k_pool"], pg["v_pool"], x["k_new"], x["v_new"], bad,
                      torch.tensor([5, 6], dtype=torch.int32, device=dev))
    with pytest.raises(g.KvAttnError):
        g.check_device_error()
    assert np.array_equal(bits(pg["k_pool"]), before_k)
    g.check_device_error()  # cleared


def test_paged_rejects_bad_sizes():
    dev = torch.device("cuda")
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device=dev)
    lens = torch.ones((1,), dtype=torch.int32, device=dev)
    for bs in (8, 24):  # below 16, not a power of two
        pool = torch.zeros((4, 1, bs, 128), dtype=torch.bfloat16, device=dev)
        table = torch.zeros((1, 4), dtype=torch.int32, device=dev)
        with pytest.raises(g.KvAttnError):
            g.gqa_decode_attn_paged(q, pool, pool, table, lens, 0.1)
    q64 = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device=dev)
    pool = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(g.KvAttnError) as ei:  # D = 64 has no tensor-core kernel
        g.gqa_decode_attn_paged(q64, pool, pool, torch.zeros((1, 4), dtype=torch.int32,
                                                             device=dev), lens, 0.1)
    assert ei.value.status == g.KVATTN_ERR_UNSUPPORTED


def test_llama70b_paged_workload_sampled():
    # the benchmark's paged workload at full size; four sequences checked
    w = wl.WORKLOADS["llama70b_paged16"]
    dev = torch.device("cuda")
    x = wl.make_inputs(w, seed=0, device=dev)
    pg = wl.make_paged(w, x, seed=0)
    del x["k_cache"], x["v_cache"]
    out = g.gqa_decode_step_paged(x["q"], x["k_new"], x["v_new"], pg["k_pool"], pg["v_pool"],
                                  pg["block_table"], x["append_pos"], w.scale)
    g.check_device_error()
    rng = np.random.default_rng(3)
    sel = sorted(rng.choice(w.B, 8, replace=False).tolist())
    lens = x["attn_lens"].cpu().numpy()[sel]
    table = pg["block_table"].cpu().numpy()[sel]
    k = oracle.gather_paged(bits(pg["k_pool"]), table, lens, w.block_size)
    v = oracle.gather_paged(bits(pg["v_pool"]), table, lens, w.block_size)
    ref = oracle.gqa_decode(bits(x["q"])[sel], k, v, lens, w.scale, nthreads=oracle_threads())
    assert_close(out[sel], ref, v, list(lens))


# ------------------------------------------------ local window over a paged cache
# "The Basics of Transformer Inference", the items on local attention layers
# and on ragged reads with Paged Attention: a local layer's queries attend
# their last `window` positions through the block table.

def _table_without_early_blocks(pg, lens, bs, span):
    """The block table with every block that lies wholly more than 127
    positions before a sequence's window span set to -1: the kernel may read
    at most 127 positions before the span, so reading one of these blocks
    would raise the device bounds error."""
    tab = pg["block_table"].cpu().numpy().copy()
    for b, n in enumerate(lens):
        lo = int(n) - span - 127
        for kb in range(tab.shape[1]):
            if (kb + 1) * bs - 1 < lo:
                tab[b, kb] = -1
    return torch.from_numpy(tab).to(pg["block_table"].device).contiguous()


def _attend_window(w, x, pg, window):
    lens = x["attn_lens"].cpu().numpy()
    table = _table_without_early_blocks(pg, lens, w.block_size, window + w.T - 1)
    out = g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], table, x["attn_lens"],
                                  w.scale, window=window)
    g.check_device_error()
    ref, v, ls = _oracle_paged(w, x, pg, window=window)
    if w.T > 1:
        B, T, Hq, D = out.shape
        return assert_close(out.reshape(B * T, Hq, D), ref.reshape(B * T, Hq, D), v, list(ls))
    return assert_close(out, ref, v, list(ls))


@pytest.mark.parametrize("bs", [16, 64, 128, 512])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 64, 8), (256, 16, 1), (256, 48, 1)])
@pytest.mark.parametrize("window", [1, 5, 127, 128, 129, 300, 5000])
def test_paged_local_window_matches_oracle(bs, D, Hq, Hkv, window):
    Lmax = 1100
    lens = _edge_lens(bs, Lmax)
    w, x, pg = _case(len(lens), Hq, Hkv, D, Lmax, bs, lens, seed=bs + D + Hq + window)
    _attend_window(w, x, pg, window)


@pytest.mark.parametrize("bs", [16, 128])
@pytest.mark.parametrize("ctas", [1, 3, 17, 152, 600])
def test_paged_local_window_split_pieces_merge(bs, ctas):
    g.set_tuning(0, ctas)
    try:
        w, x, pg = _case(4, 32, 4, 128, 3000, bs, (3000, 1, 1709, 130), seed=ctas + bs + 1)
        _attend_window(w, x, pg, 1500)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("bs", [16, 256])
@pytest.mark.parametrize("T,window", [(2, 1), (2, 200), (4, 5), (4, 129), (8, 64)])
def test_paged_new_tokens_with_a_local_window(bs, T, window):
    lens = sorted({T, T + 1, bs + 3, 129, 700, 1000})
    w, x, pg = _case(len(lens), 8, 1, 128, 1000, bs, lens, seed=T * 37 + bs + window, T=T)
    _attend_window(w, x, pg, window)


@pytest.mark.parametrize("ctas", [1, 19, 152])
def test_paged_new_tokens_window_over_head_passes(ctas):
    # the PaLM-540B head shape (48 heads on one K/V head, D = 256), 3 drafted
    # tokens: 3 passes of 16 heads, each with its tile-aligned window span
    g.set_tuning(0, ctas)
    try:
        w, x, pg = _case(2, 48, 1, 256, 3000, 64, (3000, 1291), seed=ctas + 7, T=3)
        _attend_window(w, x, pg, 700)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("bs", [16, 128])
@pytest.mark.parametrize("window", [1, 100, 2000])
def test_paged_local_window_fused_step(bs, window):
    lens = (1, 16, 17, 128, 129, 500, 1024)   # attended, after the append
    w, x, pg = _case(len(lens), 32, 4, 128, 1024, bs, lens, seed=bs + window)
    k_ref, v_ref = bits(pg["k_pool"]), bits(pg["v_pool"])
    table = pg["block_table"].cpu().numpy()
    pos = x["append_pos"].cpu().numpy()
    for b in range(w.B):
        j = int(pos[b])
        k_ref[table[b, j // bs], :, j % bs] = bits(x["k_new"])[b]
        v_ref[table[b, j // bs], :, j % bs] = bits(x["v_new"])[b]
    early = _table_without_early_blocks(pg, x["attn_lens"].cpu().numpy(), bs, window)
    out = g.gqa_decode_step_paged(x["q"], x["k_new"], x["v_new"], pg["k_pool"], pg["v_pool"],
                                  early, x["append_pos"], w.scale, window=window)
    g.check_device_error()
    assert np.array_equal(bits(pg["k_pool"]), k_ref)
    assert np.array_equal(bits(pg["v_pool"]), v_ref)
    ref, v, ls = _oracle_paged(w, x, pg, window=window)
    assert_close(out, ref, v, list(ls))


def test_paged_local_window_must_be_positive():
    w, x, pg = _case(2, 16, 2, 128, 256, 16, (100, 30), seed=12)
    with pytest.raises(g.KvAttnError):
        g.gqa_decode_attn_paged(x["q"], pg["k_pool"], pg["v_pool"], pg["block_table"],
                                x["attn_lens"], w.scale, window=0)
