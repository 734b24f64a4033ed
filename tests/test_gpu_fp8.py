"""GPU parity for the 8-bit KV cache ("The Basics of Transformer Inference",
item "Quantization"; "Machine Learning Engineering and AI Systems at Scale",
section "Quantization": FP8 E4M3 codes with one fp32 scale per row).  The
quantizer and the append must be bit-exact against the oracle (the same
binary32 divisions and the same rounding); the attention over the codes
must be within max|err| <= 2e-3 and <= 1e-2 * max|V| of the oracle's double
attention over the dequantized cache."""
import numpy as np
import pytest
import torch

import grouped_query_kv_gb300 as g
import oracle
from grouped_query_kv_gb300 import workloads as wl

from helpers import ATOL, VREL, bits, oracle_threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from grouped_query_kv_gb300 import build
    build.build()
    oracle.build()
    g.set_tuning(0, 0)
    yield
    g.set_tuning(0, 0)


def _rows(n, D, seed):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn((n, D), generator=gen) * torch.exp(torch.empty((n, 1)).uniform_(-8, 8, generator=gen))
    x[0] = 0.0                                  # an all-zero row
    x[1, : D // 2] = 0.0
    x[2] = x[2] * 1e-30                         # subnormal-range codes
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_quantizer_is_bit_exact(D):
    x = _rows(517, D, D)
    codes, scales = g.kv_quantize_fp8(x.cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.quantize_fp8(bits(x))
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def test_fp8_append_is_bit_exact():
    dev = torch.device("cuda")
    B, Hkv, D, Lmax = 5, 4, 128, 300
    gen = torch.Generator().manual_seed(3)
    kc = torch.randint(0, 256, (B, Hkv, Lmax, D), generator=gen, dtype=torch.uint8)
    vc = torch.randint(0, 256, (B, Hkv, Lmax, D), generator=gen, dtype=torch.uint8)
    ks = torch.randn((B, Hkv, Lmax), generator=gen)
    vs = torch.randn((B, Hkv, Lmax), generator=gen)
    kn = torch.randn((B, Hkv, D), generator=gen).to(torch.bfloat16)
    vn = (torch.randn((B, Hkv, D), generator=gen) * 100).to(torch.bfloat16)
    pos = torch.tensor([0, 299, 17, 128, 5], dtype=torch.int32)
    refs = [a.numpy().copy() for a in (kc, vc, ks, vs)]
    oracle.kv_append_fp8(*refs, bits(kn), bits(vn), pos.numpy())
    dk, dv, dks, dvs = kc.to(dev), vc.to(dev), ks.to(dev), vs.to(dev)
    g.kv_append_fp8(dk, dv, dks, dvs, kn.to(dev), vn.to(dev), pos.to(dev))
    g.check_device_error()
    assert np.array_equal(dk.cpu().numpy(), refs[0])
    assert np.array_equal(dv.cpu().numpy(), refs[1])
    assert np.array_equal(dks.cpu().numpy().view(np.uint32), refs[2].view(np.uint32))
    assert np.array_equal(dvs.cpu().numpy().view(np.uint32), refs[3].view(np.uint32))
    bad = torch.tensor([0, 300, -1, 0, 0], dtype=torch.int32, device=dev)
    g.kv_append_fp8(dk, dv, dks, dvs, kn.to(dev), vn.to(dev), bad)
    with pytest.raises(g.KvAttnError):
        g.check_device_error()


def _fp8_case(B, Hq, Hkv, Lmax, lens, seed, v_mul=1.0, k_mul=1.0, poison=True, D=128):
    """bf16 draws quantized on the GPU (the quantizer is bit-exact), rows
    past each length poisoned with NaN codes and scales."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(seed)
    q = torch.randn((B, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Lmax, D), generator=gen, device=dev)
    v = torch.randn((B, Hkv, Lmax, D), generator=gen, device=dev)
    if k_mul == "rows":  # magnitudes varying row by row
        k = k * torch.exp(torch.empty((B, Hkv, Lmax, 1), device=dev).uniform_(-5, 2, generator=gen))
        v = v * torch.exp(torch.empty((B, Hkv, Lmax, 1), device=dev).uniform_(-3, 0.5, generator=gen))
    else:
        k, v = k * k_mul, v * v_mul
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    kc, ks = g.kv_quantize_fp8(k)
    vc, vs = g.kv_quantize_fp8(v)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    if poison:
        for b, n in enumerate(lens):
            kc[b, :, n:] = 0x7F
            vc[b, :, n:] = 0x7F
            ks[b, :, n:] = float("nan")
            vs[b, :, n:] = float("inf")
    return q, kc, vc, ks, vs, lens_t


def _check(q, kc, vc, ks, vs, lens, scale, sel=None):
    out = g.gqa_decode_attn_fp8(q, kc, vc, ks, vs, lens, scale)
    g.check_device_error()
    bsel = list(range(q.shape[0])) if sel is None else list(sel)
    idx = torch.tensor(bsel, device=q.device)
    qb = bits(q.index_select(0, idx))
    kc_h, vc_h = kc.index_select(0, idx).cpu().numpy(), vc.index_select(0, idx).cpu().numpy()
    ks_h, vs_h = ks.index_select(0, idx).cpu().numpy(), vs.index_select(0, idx).cpu().numpy()
    ln = lens.cpu().numpy()[bsel]
    ref = oracle.gqa_decode_fp8(qb, kc_h, vc_h, ks_h, vs_h, ln, scale, nthreads=oracle_threads())
    o = out.index_select(0, idx).cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o))
    vmax = 0.0
    for i, n in enumerate(ln):
        if n > 0:
            vmax = max(vmax, float(np.abs(oracle.dequantize_fp8(vc_h[i, :, :n], vs_h[i, :, :n])).max()))
    err = float(np.abs(o - ref).max())
    bound = min(ATOL, VREL * vmax) if vmax > 0 else ATOL
    assert err <= bound, "max|err| %.3g > bound %.3g" % (err, bound)
    return out


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 8), (128, 32, 4), (128, 64, 8), (128, 16, 1),
                                      (128, 48, 1), (128, 64, 1), (128, 24, 2), (256, 8, 8),
                                      (256, 16, 1), (256, 32, 2), (256, 48, 1), (256, 96, 2),
                                      (256, 24, 3)])
def test_fp8_attention_matches_oracle(D, Hq, Hkv):
    lens = [1, 2, 63, 127, 128, 129, 255, 256, 300, 511, 600]
    q, kc, vc, ks, vs, lt = _fp8_case(len(lens), Hq, Hkv, 600, lens, seed=Hq + Hkv + D, D=D)
    _check(q, kc, vc, ks, vs, lt, 1.0 / np.sqrt(D))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("ctas", [1, 3, 17, 152, 500])
def test_fp8_split_pieces_merge(ctas, D):
    g.set_tuning(0, ctas)
    try:
        q, kc, vc, ks, vs, lt = _fp8_case(4, 32, 4, 3000, [3000, 1, 1709, 130], seed=ctas, D=D)
        _check(q, kc, vc, ks, vs, lt, 0.09)
    finally:
        g.set_tuning(0, 0)


@pytest.mark.parametrize("D", [128, 256])
def test_fp8_scales_across_magnitudes(D):
    # key rows spread over e^-5 .. e^2 and value rows over e^-3 .. e^0.5: the
    # per-row scales carry them (the weights enter as three E4M3 parts, so
    # their error is relative to |V|, about 2^-12; values of order one keep
    # it inside the absolute bound)
    q, kc, vc, ks, vs, lt = _fp8_case(3, 16, 2, 400, [400, 250, 77], seed=9, k_mul="rows", D=D)
    _check(q, kc, vc, ks, vs, lt, 1.0 / np.sqrt(D / 128))


def test_fp8_empty_sequences_and_bad_lengths():
    q, kc, vc, ks, vs, lt = _fp8_case(3, 8, 2, 256, [5, 17, 5], seed=4)
    lens = torch.tensor([0, 17, 0], dtype=torch.int32, device="cuda")
    out = _check(q, kc, vc, ks, vs, lens, 0.1)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    bad = torch.tensor([10, 257, -3], dtype=torch.int32, device="cuda")
    out = g.gqa_decode_attn_fp8(q, kc, vc, ks, vs, bad, 0.1)
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)


def test_fp8_rejects_other_head_dims():
    dev = torch.device("cuda")
    for D in (64,):
        q = torch.zeros((1, 8, D), dtype=torch.bfloat16, device=dev)
        c = torch.zeros((1, 1, 64, D), dtype=torch.uint8, device=dev)
        s = torch.ones((1, 1, 64), dtype=torch.float32, device=dev)
        with pytest.raises(g.KvAttnError) as ei:
            g.gqa_decode_attn_fp8(q, c, c, s, s, torch.ones(1, dtype=torch.int32, device=dev), 0.1)
        assert ei.value.status == g.KVATTN_ERR_UNSUPPORTED


def test_llama70b_fp8_workload_sampled():
    w = wl.WORKLOADS["llama70b_gqa_ragged"]
    lens = wl.attn_lens(w, 0).tolist()
    q, kc, vc, ks, vs, lt = _fp8_case(w.B, w.Hq, w.Hkv, w.Lmax, lens, seed=0, poison=False)
    rng = np.random.default_rng(2)
    _check(q, kc, vc, ks, vs, lt, w.scale, sel=sorted(rng.choice(w.B, 8, replace=False).tolist()))


@pytest.mark.parametrize("name,nsel", [("palm8b_mqa", 8), ("palm540b_long_mqa", 8)])
def test_palm_fp8_workloads_sampled(name, nsel):
    # the pages' multi-query shapes at D = 256 over an 8-bit cache, with the
    # workloads' own lengths and key scaling; sampled sequences against the
    # oracle
    w = wl.WORKLOADS[name]
    lens = wl.attn_lens(w, 0).tolist()
    q, kc, vc, ks, vs, lt = _fp8_case(w.B, w.Hq, w.Hkv, w.Lmax, lens, seed=1, poison=False,
                                      k_mul=w.k_scale, D=w.D)
    rng = np.random.default_rng(3)
    _check(q, kc, vc, ks, vs, lt, w.scale, sel=sorted(rng.choice(w.B, nsel, replace=False).tolist()))


def _step_check(D, Hq, Hkv, Lmax, cached, seed, scale):
    """gqa_decode_step_fp8 against the oracle's kv_append_fp8 followed by its
    attention over one more position: the codes and scales bit for bit (the
    whole caches, so rows the step must not touch are checked too; rows past
    each sequence's new row stay NaN-poisoned), the output within the bound."""
    dev = torch.device("cuda")
    B = len(cached)
    q, kc, vc, ks, vs, pos = _fp8_case(B, Hq, Hkv, Lmax, cached, seed=seed, D=D)
    gen = torch.Generator(device=dev).manual_seed(seed + 1)
    kn = (torch.randn((B, Hkv, D), generator=gen, device=dev) * 3).to(torch.bfloat16)
    vn = torch.randn((B, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
    refs = [a.cpu().numpy().copy() for a in (kc, vc, ks, vs)]
    oracle.kv_append_fp8(*refs, bits(kn), bits(vn), np.asarray(cached, dtype=np.int32))
    out = g.gqa_decode_step_fp8(q, kn, vn, kc, vc, ks, vs, pos, scale)
    g.check_device_error()
    assert np.array_equal(kc.cpu().numpy(), refs[0]), "fused append: K codes differ"
    assert np.array_equal(vc.cpu().numpy(), refs[1]), "fused append: V codes differ"
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), refs[2].view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), refs[3].view(np.uint32))
    lens = np.asarray(cached, dtype=np.int32) + 1
    ref = oracle.gqa_decode_fp8(bits(q), refs[0], refs[1], refs[2], refs[3], lens, scale,
                                nthreads=oracle_threads())
    o = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o))
    vmax = max(float(np.abs(oracle.dequantize_fp8(refs[1][b, :, :n], refs[3][b, :, :n])).max())
               for b, n in enumerate(lens))
    err = float(np.abs(o - ref).max())
    assert err <= min(ATOL, VREL * vmax), "max|err| %.3g" % err


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 1), (128, 32, 4), (128, 64, 8), (256, 16, 1),
                                      (256, 48, 1), (256, 32, 2)])
def test_fp8_fused_step_matches_append_then_attend(D, Hq, Hkv):
    # cached lengths on every tile edge (the new row opens a tile, ends one,
    # or lands inside the shifted last tile), up to Lmax - 1
    cached = [0, 1, 126, 127, 128, 129, 255, 299]
    _step_check(D, Hq, Hkv, 300, cached, seed=D + Hq, scale=1.0 / np.sqrt(D))


@pytest.mark.parametrize("ctas", [1, 3, 152, 500])
def test_fp8_fused_step_split_grids(ctas):
    g.set_tuning(0, ctas)
    try:
        _step_check(256, 16, 1, 2500, [2499, 0, 1300, 700], seed=ctas, scale=1.0 / 16)
    finally:
        g.set_tuning(0, 0)


def test_fp8_fused_step_full_cache_is_flagged():
    # seq_lens[b] = Lmax: no room for the new row -- no append, a zero row,
    # KVATTN_ERR_DEVICE_BOUNDS; the other sequences are served
    dev = torch.device("cuda")
    q, kc, vc, ks, vs, pos = _fp8_case(3, 16, 1, 256, [5, 5, 5], seed=8, poison=False)
    kn = torch.randn((3, 1, 128), device=dev).to(torch.bfloat16)
    bad = torch.tensor([4, 256, 17], dtype=torch.int32, device=dev)
    before = kc.clone()
    out = g.gqa_decode_step_fp8(q, kn, kn, kc, vc, ks, vs, bad, 0.1)
    with pytest.raises(g.KvAttnError) as ei:
        g.check_device_error()
    assert ei.value.status == g.KVATTN_ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0)
    assert torch.equal(kc[1], before[1])
    assert not torch.equal(kc[0, :, 4], before[0, :, 4])  # the in-range rows were written


def test_quantizer_on_rows_near_e4m3_ties():
    # rows whose exact quotients x / scale lie within one binary32 rounding
    # of an E4M3 midpoint (test_oracle_fp8.py builds them): the GPU must
    # divide in binary32 exactly as the oracle does
    import test_oracle_fp8 as t8
    r = t8._near_tie_rows()
    rows = np.zeros((r.shape[0], 64), dtype=np.uint16)
    rows[:, :2] = r
    x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = g.kv_quantize_fp8(x)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.quantize_fp8(rows)
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
