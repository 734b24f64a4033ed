"""Pins for the oracle's 8-bit KV cache ("The Basics of Transformer
Inference", item "Quantization"; "Machine Learning Engineering and AI
Systems at Scale", section "Quantization": FP8 E4M3).  The E4M3 codec is
checked against torch's float8_e4m3fn (a library routine) and against an
exhaustive nearest-value search; the quantizer by its properties; the
decode over the 8-bit cache against torch's attention on the dequantized
values and against the bf16 decode when every scale is 1.  CPU only."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _bits(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _unbits(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _torch_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


FINITE = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)


def test_every_code_decodes_like_torch():
    d = oracle.e4m3_decode(FINITE)
    assert np.array_equal(d, _torch_e4m3(FINITE))
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert oracle.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9


def _grid():
    vals = np.sort(np.unique(oracle.e4m3_decode(FINITE)))
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [vals, mids]
    for m in mids.astype(np.float32):
        pts.append(np.array([np.nextafter(m, np.float32(-1e9)), np.nextafter(m, np.float32(1e9))]))
    rng = np.random.default_rng(5)
    pts.append(rng.uniform(-448, 448, 20000))
    pts.append(rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 8, 20000))
    x = np.concatenate(pts).astype(np.float32)
    return x[np.abs(x) <= 448]


def test_encoding_matches_torch_on_values_ties_and_neighbours():
    x = _grid()
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encoding_is_the_nearest_value_ties_to_even():
    # exhaustive search over the finite values, independent of torch
    vals = oracle.e4m3_decode(FINITE)
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.uniform(-448, 448, 3000),
                        rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 6, 3000)]) \
        .astype(np.float32)
    x = x[np.abs(x) <= 448]
    codes = oracle.e4m3_encode(x)
    for xi, c in zip(x.astype(np.float64), codes):
        dist = np.abs(vals - xi)
        best = FINITE[dist == dist.min()]
        if len(best) > 1:                      # a tie: the even mantissa wins
            best = best[(best & 1) == 0]
            best = best[best >> 7 == (1 if xi < 0 else 0)] if len(best) > 1 else best
        assert c in best, (xi, c, best)


def test_encoding_saturates_and_keeps_the_sign_of_zero():
    x = np.array([449.0, 470.0, 1e30, np.inf, -449.0, -np.inf, 0.0, -0.0], np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x00, 0x80]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_quantized_rows_reproduce_their_values():
    rng = np.random.default_rng(7)
    rows = _bits(rng.standard_normal((64, 128)) * np.exp(rng.uniform(-6, 6, (64, 1))))
    codes, scales = oracle.quantize_fp8(rows)
    x = _unbits(rows)
    deq = oracle.dequantize_fp8(codes, scales)
    amax = np.abs(x).max(axis=1)
    # the largest element lands on +-448 exactly; scales are amax / 448
    for r in range(64):
        i = int(np.argmax(np.abs(x[r])))
        assert codes[r, i] & 0x7F == 0x7E
        assert abs(scales[r] * 448 / amax[r] - 1) < 1e-6
    # every element within half a unit in the last place of its binade
    # (relative 2^-4) in the normal range, 2^-10 * scale below it
    y = np.abs(x) / scales[:, None]
    err = np.abs(deq - x) / scales[:, None]
    normal = y >= 2.0 ** -6
    assert np.all(err[normal] <= y[normal] * 2.0 ** -4 * (1 + 1e-6) + 1e-12)
    assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))


def _near_tie_rows():
    """Rows [amax, x] of bf16 values chosen so that x / (amax / 448) is,
    exactly, an E4M3 midpoint (1.3125 times a power of two: 448 x / amax =
    21 / 16 * 2^e with x = 3 amax 2^e / 1024), while amax / 448 is not a
    binary32 value: the binary32 scale is off by one rounding, the exact
    quotient x / scale sits within a binary32 ulp of the midpoint, and the
    quotient rounded to binary32 may land on the midpoint itself.  Whether
    the code then comes out even (a tie) or from the exact side is what tells
    a binary32 division from a double one."""
    rows = []
    for amax in range(1, 86, 2):
        if amax % 7 == 0:
            continue
        for e in range(-6, 3):
            x = 3.0 * amax * 2.0 ** e / 1024
            if x >= amax:
                continue
            rows.append([amax, x])
    r = np.asarray(rows, dtype=np.float64)
    bits = _bits(r)
    assert np.array_equal(_unbits(bits), r), "the constructed values are bf16-exact"
    return bits


def _e4m3_nearest_exact(q):
    """Fractions -> E4M3 codes by exhaustive nearest search, ties to even
    (exact rational comparison)."""
    from fractions import Fraction
    table = [(Fraction(float(v)), int(c)) for c, v in zip(FINITE, oracle.e4m3_decode(FINITE))
             if v >= 0]
    out = []
    for v in q:
        a = abs(v)
        best = min(table, key=lambda t: (abs(t[0] - a), t[1] & 1))
        out.append(best[1] | (0x80 if v < 0 else 0))
    return np.asarray(out, dtype=np.uint8)


def test_quantizer_divides_in_binary32():
    # The reading: scale = absmax / 448 and code = E4M3(x / scale), both
    # divisions IEEE binary32.  torch's float32 division and its
    # float8_e4m3fn conversion restate that rule with library routines; the
    # codes and scales must match them bit for bit, on rows where dividing
    # in double (or exactly) instead gives other codes.
    from fractions import Fraction
    rows = _near_tie_rows()
    codes, scales = oracle.quantize_fp8(rows)
    x = torch.from_numpy(_unbits(rows)).to(torch.float32)
    s32 = x.abs().amax(dim=1, keepdim=True) / 448.0
    want_codes = (x / s32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales.view(np.uint32), s32[:, 0].numpy().view(np.uint32))
    assert np.array_equal(codes, want_codes)
    # the pin has teeth: the exact quotients round to other codes on some rows
    exact = []
    for r, s in zip(_unbits(rows), s32[:, 0].numpy()):
        exact.append(_e4m3_nearest_exact([Fraction(float(v)) / Fraction(float(s)) for v in r]))
    exact = np.asarray(exact)
    assert (exact != want_codes).any(axis=1).sum() >= 5


def test_zero_row_has_scale_one():
    codes, scales = oracle.quantize_fp8(np.zeros((2, 64), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 1.0)


def _case(rng, B, Hq, Hkv, D, L, lens):
    q = _bits(rng.standard_normal((B, Hq, D)))
    k = _bits(rng.standard_normal((B, Hkv, L, D)))
    v = _bits(rng.standard_normal((B, Hkv, L, D)))
    kc, ks = oracle.quantize_fp8(k)
    vc, vs = oracle.quantize_fp8(v)
    return q, kc, ks, vc, vs, np.array(lens, np.int32)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (16, 1)])
def test_fp8_decode_is_attention_over_the_dequantized_cache(Hq, Hkv):
    rng = np.random.default_rng(Hq + Hkv)
    B, D, L = 3, 32, 40
    q, kc, ks, vc, vs, lens = _case(rng, B, Hq, Hkv, D, L, [40, 9, 1])
    out = oracle.gqa_decode_fp8(q, kc, vc, ks, vs, lens, 0.2)
    kd, vd = oracle.dequantize_fp8(kc, ks), oracle.dequantize_fp8(vc, vs)
    for b in range(B):
        n = int(lens[b])
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(_unbits(q[b:b + 1]))[:, :, None, :],
            torch.from_numpy(kd[b:b + 1, :, :n]), torch.from_numpy(vd[b:b + 1, :, :n]),
            scale=0.2, enable_gqa=True)[0, :, 0].numpy()
        assert np.allclose(out[b], ref, rtol=1e-12, atol=1e-13)
    # length one returns the dequantized V[0]
    G = Hq // Hkv
    assert np.array_equal(out[2], vd[2, np.arange(Hq) // G, 0])


def test_fp8_decode_with_unit_scales_equals_the_bf16_decode():
    # every E4M3 value is exactly a bf16 value, so a cache of codes with
    # scales 1 is the bf16 cache holding those values
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, L = 2, 8, 2, 16, 24
    q = _bits(rng.standard_normal((B, Hq, D)))
    kc = rng.choice(FINITE, size=(B, Hkv, L, D)).astype(np.uint8)
    vc = rng.choice(FINITE, size=(B, Hkv, L, D)).astype(np.uint8)
    ones = np.ones((B, Hkv, L), np.float32)
    lens = np.array([24, 5], np.int32)
    out8 = oracle.gqa_decode_fp8(q, kc, vc, ones, ones, lens, 0.01)
    kb = _bits(oracle.e4m3_decode(kc))
    vb = _bits(oracle.e4m3_decode(vc))
    assert np.array_equal(_unbits(kb), oracle.e4m3_decode(kc))
    assert np.array_equal(out8, oracle.gqa_decode(q, kb, vb, lens, 0.01))


def test_fp8_rows_past_the_length_are_never_read():
    rng = np.random.default_rng(12)
    q, kc, ks, vc, vs, lens = _case(rng, 2, 4, 1, 16, 20, [7, 20])
    out = oracle.gqa_decode_fp8(q, kc, vc, ks, vs, lens, 0.3)
    kc2, vc2, ks2, vs2 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    kc2[0, :, 7:] = 0x7F
    vc2[0, :, 7:] = 0x7F
    ks2[0, :, 7:] = np.nan
    vs2[0, :, 7:] = np.inf
    assert np.array_equal(oracle.gqa_decode_fp8(q, kc2, vc2, ks2, vs2, lens, 0.3), out)


def test_fp8_append_writes_the_quantized_row_and_nothing_else():
    rng = np.random.default_rng(13)
    B, Hkv, D, L = 3, 2, 32, 10
    kc = rng.integers(0, 256, (B, Hkv, L, D)).astype(np.uint8)
    vc = rng.integers(0, 256, (B, Hkv, L, D)).astype(np.uint8)
    ks = rng.standard_normal((B, Hkv, L)).astype(np.float32)
    vs = rng.standard_normal((B, Hkv, L)).astype(np.float32)
    kn = _bits(rng.standard_normal((B, Hkv, D)))
    vn = _bits(rng.standard_normal((B, Hkv, D)))
    pos = np.array([0, 9, 4], np.int32)
    ref = [a.copy() for a in (kc, vc, ks, vs)]
    qk, sk = oracle.quantize_fp8(kn)
    qv, sv = oracle.quantize_fp8(vn)
    for b in range(B):
        ref[0][b, :, pos[b]] = qk[b]
        ref[1][b, :, pos[b]] = qv[b]
        ref[2][b, :, pos[b]] = sk[b]
        ref[3][b, :, pos[b]] = sv[b]
    oracle.kv_append_fp8(kc, vc, ks, vs, kn, vn, pos)
    for got, want in zip((kc, vc, ks, vs), ref):
        assert np.array_equal(got, want)
    with pytest.raises(ValueError):
        oracle.kv_append_fp8(kc, vc, ks, vs, kn, vn, np.array([0, 10, 0], np.int32))


# ------------------------------------------------------------------ mutants

def _fp8_pins_pass(orc) -> bool:
    try:
        if not np.array_equal(orc.e4m3_decode(FINITE), _torch_e4m3(FINITE)):
            return False
        x = _grid()
        if not np.array_equal(orc.e4m3_encode(x),
                              torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()):
            return False
        tie_rows = _near_tie_rows()
        tc, ts = orc.quantize_fp8(tie_rows)
        xt = torch.from_numpy(_unbits(tie_rows)).to(torch.float32)
        st = xt.abs().amax(dim=1, keepdim=True) / 448.0
        if not np.array_equal(tc, (xt / st).to(torch.float8_e4m3fn).view(torch.uint8).numpy()):
            return False
        rng = np.random.default_rng(21)
        rows = _bits(rng.standard_normal((8, 64)))
        codes, scales = orc.quantize_fp8(rows)
        amax = np.abs(_unbits(rows)).max(axis=1)
        if not np.allclose(scales * 448 / amax, 1, rtol=1e-6):
            return False
        q, kc, ks, vc, vs, lens = _case(rng, 2, 4, 2, 16, 12, [12, 3])
        out = orc.gqa_decode_fp8(q, kc, vc, ks, vs, lens, 0.25)
        kd, vd = orc.dequantize_fp8(kc, ks), orc.dequantize_fp8(vc, vs)
        kd0, vd0 = oracle.dequantize_fp8(kc, ks), oracle.dequantize_fp8(vc, vs)
        for b in range(2):
            n = int(lens[b])
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(_unbits(q[b:b + 1]))[:, :, None, :],
                torch.from_numpy(kd0[b:b + 1, :, :n]), torch.from_numpy(vd0[b:b + 1, :, :n]),
                scale=0.25, enable_gqa=True)[0, :, 0].numpy()
            if not np.allclose(out[b], ref, rtol=1e-12, atol=1e-13):
                return False
    except (ValueError, AssertionError):
        return False
    return True


MUTANTS = {
    "exponent bias off by one": ("        v = ldexp(1.0 + m / 8.0, e - 7);", "        v = ldexp(1.0 + m / 8.0, e - 8);"),
    "subnormal step wrong": ("        v = ldexp((double)m, -9);", "        v = ldexp((double)m, -10);"),
    "mantissa truncated": ("    double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);",
                           "    double m = floor((a / ldexp(1.0, e) - 1.0) * 8.0);"),
    "scale maps absmax to 240": ("amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 240.0f : 1.0f"),
    "K read with the V scales": ("oracle_cache_at(k_cache, q8->k, q8->k_scale, row0, j, D, d)",
                                 "oracle_cache_at(k_cache, q8->k, q8->v_scale, row0, j, D, d)"),
    "scale of the previous row": ("* (double)scales[row0 + j];", "* (double)scales[row0 + (j > 0 ? j - 1 : 0)];"),
    "quotient divided in double": ("        codes[d] = oracle_e4m3_from_float(x);\n",
                                   "        codes[d] = oracle_e4m3_from_double(oracle_bf16_to_double(row[d]) / (double)s);\n"),
    "quotient by the reciprocal": ("        volatile float x = (float)oracle_bf16_to_double(row[d]) / s;",
                                   "        volatile float x = (float)oracle_bf16_to_double(row[d]) * (1.0f / s);"),
}


def test_unmodified_fp8_oracle_passes():
    assert _fp8_pins_pass(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_fp8_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, name
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    assert not _fp8_pins_pass(oracle.Oracle(so)), name
