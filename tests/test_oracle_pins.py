"""Pins for the CPU oracle: every check here is independent of the oracle's
own code (closed forms, a library routine, an explicit brute-force formula,
invariants of the mathematics).  Marked `not gpu`; runs in seconds.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit

import oracle


def bits(x):
    """bf16 bits of a float tensor/array (round to nearest even via torch)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def unbits(b):
    """bf16 bits -> float64 through torch's own conversion (a library path)."""
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def rand_case(rng, B, Hq, Hkv, D, Lmax, lens=None, kmul=1.0):
    q = bits(rng.standard_normal((B, Hq, D)))
    k = bits(kmul * rng.standard_normal((B, Hkv, Lmax, D)))
    v = bits(rng.standard_normal((B, Hkv, Lmax, D)))
    if lens is None:
        lens = rng.integers(1, Lmax + 1, size=B)
    return q, k, v, np.asarray(lens, dtype=np.int32)


# --------------------------------------------------------------- bf16 decode

def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    # drop NaN patterns (exponent all ones, mantissa non-zero)
    pats = pats[~(((pats & 0x7F80) == 0x7F80) & ((pats & 0x007F) != 0))]
    special = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4000, 0xC000, 0x0001,
                        0x007F, 0x0080, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80],
                       dtype=np.uint16)
    pats = np.concatenate([pats, special])
    ref = unbits(pats)
    got = np.array([oracle.bf16_to_double(int(p)) for p in pats])
    assert np.array_equal(got, ref)
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133  # smallest subnormal


# --------------------------------------------------------------- closed forms

def test_length_one_returns_first_value_row_exactly():
    rng = np.random.default_rng(2)
    q, k, v, _ = rand_case(rng, 3, 8, 2, 64, 16)
    lens = np.ones(3, dtype=np.int32)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.125)
    G = 4
    for b in range(3):
        for h in range(8):
            assert np.array_equal(out[b, h], unbits(v[b, h // G, 0]))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D, L = 2, 6, 3, 32, 40
    q, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    k[:] = k[:, :, :1, :]           # every position carries the same key
    lens = np.array([40, 17], dtype=np.int32)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.3)
    vf = unbits(v)
    for b in range(B):
        for h in range(Hq):
            want = vf[b, h // 2, :lens[b]].mean(axis=0)
            np.testing.assert_allclose(out[b, h], want, rtol=0, atol=1e-14)


def test_one_dominant_logit_returns_that_value_row():
    # s_{j*} exceeds every other score by >= 800, so exp(-800) underflows to
    # zero in double and the softmax is exactly one-hot.
    B, Hq, Hkv, D, L = 1, 2, 1, 16, 12
    rng = np.random.default_rng(4)
    q = np.zeros((B, Hq, D), np.float32)
    q[0, :, 0] = 1.0
    k = np.zeros((B, Hkv, L, D), np.float32)
    jstar = 7
    k[0, 0, jstar, 0] = 1024.0
    v = rng.standard_normal((B, Hkv, L, D))
    out = oracle.gqa_decode(bits(q), bits(k), bits(v), np.array([L], np.int32),
                            scale=1.0)
    for h in range(Hq):
        assert np.array_equal(out[0, h], unbits(bits(v))[0, 0, jstar])


@pytest.mark.parametrize("which", ["scale", "query"])
def test_zero_logits_give_mean_of_values(which):
    rng = np.random.default_rng(5)
    q, k, v, lens = rand_case(rng, 2, 4, 1, 64, 30)
    scale = 0.125
    if which == "scale":
        scale = 0.0
    else:
        q[:] = 0
    out = oracle.gqa_decode(q, k, v, lens, scale=scale)
    vf = unbits(v)
    for b in range(2):
        want = vf[b, 0, :lens[b]].mean(axis=0)
        for h in range(4):
            np.testing.assert_allclose(out[b, h], want, rtol=0, atol=1e-14)


def test_two_positions_follow_the_logistic_closed_form():
    # softmax over two scores is (sigma(s0 - s1), sigma(s1 - s0)), with sigma
    # the logistic function (scipy's expit).
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, L = 2, 4, 2, 16, 5
    q, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.full(B, 2, np.int32)
    scale = 0.37
    out = oracle.gqa_decode(q, k, v, lens, scale=scale)
    qf, kf, vf = unbits(q), unbits(k), unbits(v)
    for b in range(B):
        for h in range(Hq):
            kvh = h // 2
            s0 = scale * float(np.dot(qf[b, h], kf[b, kvh, 0]))
            s1 = scale * float(np.dot(qf[b, h], kf[b, kvh, 1]))
            want = expit(s0 - s1) * vf[b, kvh, 0] + expit(s1 - s0) * vf[b, kvh, 1]
            np.testing.assert_allclose(out[b, h], want, rtol=1e-13, atol=1e-14)


def test_empty_sequence_gives_zero_row():
    rng = np.random.default_rng(7)
    q, k, v, _ = rand_case(rng, 3, 4, 2, 16, 8)
    lens = np.array([0, 5, 0], np.int32)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.25)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.any(out[1] != 0)


# --------------------------------------------------- library special case

@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax", [
    (2, 4, 1, 64, 37),      # MQA
    (3, 8, 2, 32, 50),      # GQA, group 4
    (2, 6, 6, 16, 21),      # MHA
    (1, 48, 1, 256, 9),     # PaLM-540B head shape
    (2, 64, 8, 128, 19),    # Llama-2-70B head shape
])
def test_matches_torch_sdpa_in_float64(B, Hq, Hkv, D, Lmax):
    rng = np.random.default_rng(B * 1000 + Hq * 10 + D)
    q, k, v, lens = rand_case(rng, B, Hq, Hkv, D, Lmax)
    lens[0] = Lmax
    scale = 1.0 / math.sqrt(D)
    out = oracle.gqa_decode(q, k, v, lens, scale=scale)
    qt = torch.from_numpy(unbits(q))
    kt = torch.from_numpy(unbits(k))
    vt = torch.from_numpy(unbits(v))
    for b in range(B):
        L = int(lens[b])
        ref = F.scaled_dot_product_attention(
            qt[b:b + 1, :, None, :], kt[b:b + 1, :, :L], vt[b:b + 1, :, :L],
            scale=scale, enable_gqa=(Hq != Hkv))
        np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=1e-12,
                                   atol=1e-13)


# ------------------------------------------------------------- brute force

def test_brute_force_explicit_weights_tiny():
    # p_j = 1 / sum_i exp(s_i - s_j): a different arrangement of the softmax,
    # summed exactly with math.fsum, on every row of a tiny case.
    rng = np.random.default_rng(8)
    for trial in range(6):
        B = int(rng.integers(1, 4)); Hkv = int(rng.integers(1, 3))
        G = int(rng.integers(1, 3)); Hq = Hkv * G
        D = int(rng.integers(1, 9)); Lmax = int(rng.integers(1, 9))
        q, k, v, lens = rand_case(rng, B, Hq, Hkv, D, Lmax)
        scale = float(rng.uniform(0.05, 1.5))
        out = oracle.gqa_decode(q, k, v, lens, scale=scale)
        qf, kf, vf = unbits(q), unbits(k), unbits(v)
        for b in range(B):
            for h in range(Hq):
                kvh = h // G
                L = int(lens[b])
                s = [scale * math.fsum(qf[b, h, d] * kf[b, kvh, j, d] for d in range(D))
                     for j in range(L)]
                p = [1.0 / math.fsum(math.exp(s[i] - s[j]) for i in range(L))
                     for j in range(L)]
                for d in range(D):
                    want = math.fsum(p[j] * vf[b, kvh, j, d] for j in range(L))
                    assert abs(out[b, h, d] - want) <= 1e-13 * max(1.0, abs(want))


# --------------------------------------------------------------- invariants

def test_joint_permutation_of_positions_leaves_output_unchanged():
    rng = np.random.default_rng(9)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 64, 33)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.125)
    k2, v2 = k.copy(), v.copy()
    for b in range(3):
        L = int(lens[b])
        perm = rng.permutation(L)
        k2[b, :, :L] = k[b][:, perm]
        v2[b, :, :L] = v[b][:, perm]
    out2 = oracle.gqa_decode(q, k2, v2, lens, scale=0.125)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)


def test_gqa_equals_mha_with_each_kv_head_repeated_over_its_group():
    # pins the contiguous grouping kvh = h // G (not h % Hkv)
    rng = np.random.default_rng(10)
    B, Hq, Hkv, D, L = 2, 12, 3, 32, 25
    q, k, v, lens = rand_case(rng, B, Hq, Hkv, D, L)
    k[:, 1] = bits(3.0 * unbits(k[:, 1]) + 1.0)   # make the KV heads unlike
    out = oracle.gqa_decode(q, k, v, lens, scale=0.2)
    G = Hq // Hkv
    k_rep = np.repeat(k, G, axis=1)
    v_rep = np.repeat(v, G, axis=1)
    out_mha = oracle.gqa_decode(q, k_rep, v_rep, lens, scale=0.2)
    assert np.array_equal(out, out_mha)
    # and the interleaved mapping would differ
    k_tile = np.tile(k, (1, G, 1, 1))
    v_tile = np.tile(v, (1, G, 1, 1))
    out_wrong = oracle.gqa_decode(q, k_tile, v_tile, lens, scale=0.2)
    assert not np.allclose(out_wrong, out)


def test_batch_rows_are_independent():
    rng = np.random.default_rng(11)
    q, k, v, lens = rand_case(rng, 4, 4, 2, 16, 20)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.25)
    q2, k2, v2, lens2 = q.copy(), k.copy(), v.copy(), lens.copy()
    q2[2] = bits(rng.standard_normal(q2[2].shape))
    k2[2] = bits(rng.standard_normal(k2[2].shape))
    v2[2] = bits(rng.standard_normal(v2[2].shape))
    lens2[2] = 1 + (lens[2] % 20)
    out2 = oracle.gqa_decode(q2, k2, v2, lens2, scale=0.25)
    for b in (0, 1, 3):
        assert np.array_equal(out[b], out2[b])


def test_rows_past_the_length_are_never_read():
    rng = np.random.default_rng(12)
    q, k, v, lens = rand_case(rng, 3, 4, 1, 32, 24)
    lens = np.array([5, 24, 1], np.int32)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.2)
    k2, v2 = k.copy(), v.copy()
    for b in range(3):
        k2[b, :, lens[b]:] = 0x7FC0   # NaN
        v2[b, :, lens[b]:] = 0x7F80   # +inf
    out2 = oracle.gqa_decode(q, k2, v2, lens, scale=0.2)
    assert np.array_equal(out, out2)


def test_values_enter_linearly():
    # scaling V by 2 (exact in bf16) doubles the output; shifting every value
    # row by a constant vector t (small integers, exact in bf16) shifts it by t
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D, L = 2, 4, 2, 16, 30
    q, k, _, lens = rand_case(rng, B, Hq, Hkv, D, L)
    vi = rng.integers(-8, 9, size=(B, Hkv, L, D)).astype(np.float32)
    t = rng.integers(-16, 17, size=D).astype(np.float32)
    base = oracle.gqa_decode(q, k, bits(vi), lens, scale=0.3)
    doubled = oracle.gqa_decode(q, k, bits(2 * vi), lens, scale=0.3)
    shifted = oracle.gqa_decode(q, k, bits(vi + t), lens, scale=0.3)
    np.testing.assert_allclose(doubled, 2 * base, rtol=1e-14, atol=1e-13)
    np.testing.assert_allclose(shifted, base + t, rtol=0, atol=1e-12)


def test_output_is_a_convex_combination_of_value_rows():
    rng = np.random.default_rng(14)
    q, k, v, lens = rand_case(rng, 3, 8, 4, 64, 40, kmul=4.0)
    out = oracle.gqa_decode(q, k, v, lens, scale=0.5)
    vf = unbits(v)
    for b in range(3):
        for h in range(8):
            rows = vf[b, h // 2, :lens[b]]
            assert np.all(out[b, h] <= rows.max(axis=0) + 1e-12)
            assert np.all(out[b, h] >= rows.min(axis=0) - 1e-12)


# ----------------------------------------------------- bookkeeping / errors

def test_pairs_threads_and_full_agree_bitwise():
    rng = np.random.default_rng(15)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 32, 40)
    full = oracle.gqa_decode(q, k, v, lens, scale=0.2)
    mt = oracle.gqa_decode(q, k, v, lens, scale=0.2, nthreads=4)
    assert np.array_equal(full, mt)
    pairs = np.array([[0, 3], [2, 7], [1, 0]])
    part = oracle.gqa_decode(q, k, v, lens, scale=0.2, pairs=pairs, nthreads=2)
    for b, h in pairs:
        assert np.array_equal(part[b, h], full[b, h])


def test_bad_arguments_are_rejected():
    rng = np.random.default_rng(16)
    q, k, v, lens = rand_case(rng, 2, 6, 4, 16, 8)   # 6 % 4 != 0
    with pytest.raises(ValueError):
        oracle.gqa_decode(q, k, v, lens, scale=1.0)
    q, k, v, lens = rand_case(rng, 2, 4, 2, 16, 8)
    lens[1] = 9                                        # > Lmax
    with pytest.raises(ValueError):
        oracle.gqa_decode(q, k, v, lens, scale=1.0)
    lens[1] = -1
    with pytest.raises(ValueError):
        oracle.gqa_decode(q, k, v, lens, scale=1.0)


# ---------------------------------------------------------------- kv append

def test_kv_append_matches_index_assignment_and_touches_nothing_else():
    rng = np.random.default_rng(17)
    B, Hkv, L, D = 3, 2, 10, 16
    k = bits(rng.standard_normal((B, Hkv, L, D)))
    v = bits(rng.standard_normal((B, Hkv, L, D)))
    kn = bits(rng.standard_normal((B, Hkv, D)))
    vn = bits(rng.standard_normal((B, Hkv, D)))
    pos = np.array([0, 9, 4], np.int32)
    k_ref, v_ref = k.copy(), v.copy()
    k_ref[np.arange(B), :, pos] = kn          # numpy fancy indexing
    v_ref[np.arange(B), :, pos] = vn
    oracle.kv_append(k, v, kn, vn, pos)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


@pytest.mark.parametrize("bad", [-1, 10])
def test_kv_append_rejects_rows_outside_the_cache(bad):
    rng = np.random.default_rng(18)
    k = bits(rng.standard_normal((2, 1, 10, 8)))
    v = k.copy()
    kn = bits(rng.standard_normal((2, 1, 8)))
    before = k.copy()
    with pytest.raises(ValueError):
        oracle.kv_append(k, v, kn, kn, np.array([3, bad], np.int32))
    assert np.array_equal(k, before)


# ------------------------------------------------------- local (window) layers
# "The Basics of Transformer Inference", item on mixing in local attention
# layers: a local layer attends only the last W positions.

def test_window_covering_the_sequence_is_the_full_attention():
    rng = np.random.default_rng(60)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 16, 40, lens=[40, 13, 1])
    full = oracle.gqa_decode(q, k, v, lens, 0.25)
    for W in (40, 41, 1000):
        assert np.array_equal(oracle.gqa_decode(q, k, v, lens, 0.25, window=W), full)


def test_window_of_one_returns_the_last_value_row_exactly():
    rng = np.random.default_rng(61)
    q, k, v, lens = rand_case(rng, 2, 4, 1, 8, 30, lens=[30, 7])
    out = oracle.gqa_decode(q, k, v, lens, 0.5, window=1)
    for b in range(2):
        assert np.array_equal(out[b], unbits(v[b, 0, lens[b] - 1])[None].repeat(4, 0))


@pytest.mark.parametrize("W", [2, 7, 16, 29])
def test_window_equals_full_attention_on_the_window_rows(W):
    # the same rows copied to the front of a fresh cache, attended in full
    rng = np.random.default_rng(62 + W)
    q, k, v, lens = rand_case(rng, 3, 6, 3, 8, 32, lens=[32, 20, 9])
    out = oracle.gqa_decode(q, k, v, lens, 0.3, window=W)
    for b in range(3):
        n = int(lens[b]); j0 = max(0, n - W)
        ks = np.zeros_like(k[b:b + 1]); vs = np.zeros_like(v[b:b + 1])
        ks[:, :, :n - j0] = k[b:b + 1, :, j0:n]
        vs[:, :, :n - j0] = v[b:b + 1, :, j0:n]
        ref = oracle.gqa_decode(q[b:b + 1], ks, vs, np.array([n - j0], np.int32), 0.3)
        assert np.array_equal(out[b:b + 1], ref)


def test_window_matches_torch_sdpa_with_a_band_mask():
    rng = np.random.default_rng(63)
    B, Hq, Hkv, D, L, W = 2, 8, 2, 16, 48, 10
    q, k, v, lens = rand_case(rng, B, Hq, Hkv, D, L, lens=[48, 25])
    out = oracle.gqa_decode(q, k, v, lens, 0.2, window=W)
    for b in range(B):
        n = int(lens[b])
        mask = torch.zeros(1, 1, 1, n, dtype=torch.bool)
        mask[..., max(0, n - W):] = True
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(unbits(q[b:b + 1]))[:, :, None, :],
            torch.from_numpy(unbits(k[b:b + 1, :, :n])),
            torch.from_numpy(unbits(v[b:b + 1, :, :n])),
            attn_mask=mask, scale=0.2, enable_gqa=True)[0, :, 0].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def test_window_must_be_positive():
    rng = np.random.default_rng(64)
    q, k, v, lens = rand_case(rng, 1, 2, 1, 8, 8, lens=[5])
    with pytest.raises(ValueError):
        oracle.gqa_decode(q, k, v, lens, 0.5, window=0)


# ----------------------------------------------- several new tokens (speculative)
# "The Basics of Transformer Inference", speculative sampling: the T drafted
# tokens are scored in one pass; token t sits at position len - T + t and
# attends the prefix and the new tokens up to itself.

def test_one_new_token_is_the_single_token_decode():
    rng = np.random.default_rng(70)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 16, 40, lens=[40, 13, 1])
    out = oracle.gqa_decode_multi(q[:, None], k, v, lens, 0.25)
    assert np.array_equal(out[:, 0], oracle.gqa_decode(q, k, v, lens, 0.25))


@pytest.mark.parametrize("T", [2, 4, 8])
def test_each_new_token_equals_a_single_decode_over_its_prefix(T):
    rng = np.random.default_rng(71 + T)
    B, Hq, Hkv, D, L = 3, 6, 3, 8, 32
    q = bits(rng.standard_normal((B, T, Hq, D)))
    _, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.array([32, 20, T], np.int32)
    out = oracle.gqa_decode_multi(q, k, v, lens, 0.3)
    for t in range(T):
        ref = oracle.gqa_decode(np.ascontiguousarray(q[:, t]), k, v, lens - (T - 1 - t), 0.3)
        assert np.array_equal(out[:, t], ref)


def test_new_tokens_match_torch_sdpa_with_a_causal_block_mask():
    rng = np.random.default_rng(72)
    B, T, Hq, Hkv, D, L = 2, 4, 8, 2, 16, 30
    q = bits(rng.standard_normal((B, T, Hq, D)))
    _, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.array([30, 9], np.int32)
    out = oracle.gqa_decode_multi(q, k, v, lens, 0.2)
    for b in range(B):
        n = int(lens[b])
        # queries [Hq, T, D] against n positions; token t sees positions < n - T + 1 + t
        mask = torch.zeros(1, 1, T, n, dtype=torch.bool)
        for t in range(T):
            mask[..., t, :n - T + 1 + t] = True
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(unbits(q[b:b + 1])).permute(0, 2, 1, 3),
            torch.from_numpy(unbits(k[b:b + 1, :, :n])),
            torch.from_numpy(unbits(v[b:b + 1, :, :n])),
            attn_mask=mask, scale=0.2, enable_gqa=True)[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def test_new_tokens_before_the_start_of_the_sequence_get_zero_rows():
    rng = np.random.default_rng(73)
    T = 5
    q = bits(rng.standard_normal((1, T, 2, 8)))
    _, k, v, _ = rand_case(rng, 1, 2, 1, 8, 10)
    out = oracle.gqa_decode_multi(q, k, v, np.array([3], np.int32), 0.5)
    assert np.all(out[0, :2] == 0.0)                 # len - T + 1 + t <= 0
    assert np.array_equal(out[0, 2], unbits(v[0, 0, 0])[None].repeat(2, 0))  # sees one row


# Several new tokens on a local layer: each token keeps its own window, the
# last W positions up to and including itself.

def test_new_tokens_with_a_window_covering_the_sequence_are_the_full_pass():
    rng = np.random.default_rng(74)
    B, T, Hq, Hkv, D, L = 3, 4, 6, 3, 8, 32
    q = bits(rng.standard_normal((B, T, Hq, D)))
    _, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.array([32, 11, 2], np.int32)
    full = oracle.gqa_decode_multi(q, k, v, lens, 0.3)
    for W in (32, 33, 10 ** 6):
        assert np.array_equal(oracle.gqa_decode_multi(q, k, v, lens, 0.3, window=W), full)


def test_window_of_one_gives_each_new_token_its_own_value_row():
    rng = np.random.default_rng(75)
    B, T, Hq, Hkv, D, L = 2, 3, 4, 2, 8, 20
    q = bits(rng.standard_normal((B, T, Hq, D)))
    _, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.array([20, 5], np.int32)
    out = oracle.gqa_decode_multi(q, k, v, lens, 0.5, window=1)
    for b in range(B):
        for t in range(T):
            pos = int(lens[b]) - T + t
            for h in range(Hq):
                assert np.array_equal(out[b, t, h], unbits(v[b, h // 2, pos]))


@pytest.mark.parametrize("W", [1, 3, 9, 17])
def test_new_tokens_with_a_window_match_torch_sdpa_with_a_band_mask(W):
    rng = np.random.default_rng(76 + W)
    B, T, Hq, Hkv, D, L = 3, 5, 8, 2, 16, 40
    q = bits(rng.standard_normal((B, T, Hq, D)))
    _, k, v, _ = rand_case(rng, B, Hq, Hkv, D, L)
    lens = np.array([40, 13, 4], np.int32)
    out = oracle.gqa_decode_multi(q, k, v, lens, 0.2, window=W)
    for b in range(B):
        n = int(lens[b])
        # token t (end e = n - T + 1 + t) sees positions [e - W, e)
        mask = torch.zeros(1, 1, T, n, dtype=torch.bool)
        for t in range(T):
            e = n - T + 1 + t
            if e > 0:
                mask[..., t, max(0, e - W):e] = True
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(unbits(q[b:b + 1])).permute(0, 2, 1, 3),
            torch.from_numpy(unbits(k[b:b + 1, :, :n])),
            torch.from_numpy(unbits(v[b:b + 1, :, :n])),
            attn_mask=mask, scale=0.2, enable_gqa=True)[0].permute(1, 0, 2).numpy()
        for t in range(T):
            if n - T + 1 + t > 0:   # SDPA gives NaN for an all-masked row
                np.testing.assert_allclose(out[b, t], ref[t], rtol=1e-12, atol=1e-13)
            else:
                assert np.all(out[b, t] == 0.0)


# --------------------------------------------------------------- paged KV cache
# "Machine Learning Engineering and AI Systems at Scale", "The key and value
# cache" (PagedAttention):
# fixed-size blocks of positions and a per-sequence block table mapping
# logical positions to physical blocks; shared prefixes share blocks.

def _pool_from_contiguous(k, bs):
    """[B, Hkv, L, D] -> pool [B*L/bs, Hkv, bs, D] with the identity table,
    by numpy reshapes (a library routine, independent of the oracle)."""
    B, Hkv, L, D = k.shape
    pool = k.reshape(B, Hkv, L // bs, bs, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, bs, D)
    table = np.arange(B * (L // bs), dtype=np.int32).reshape(B, L // bs)
    return np.ascontiguousarray(pool), table


def test_paged_with_the_identity_table_is_the_contiguous_cache():
    rng = np.random.default_rng(80)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 16, 64, lens=[64, 17, 1])
    kp, table = _pool_from_contiguous(k, 16)
    vp, _ = _pool_from_contiguous(v, 16)
    out = oracle.gqa_decode_paged(q, kp, vp, table, lens, 16, 0.25)
    assert np.array_equal(out, oracle.gqa_decode(q, k, v, lens, 0.25))


def test_paged_result_does_not_depend_on_where_blocks_live():
    rng = np.random.default_rng(81)
    q, k, v, lens = rand_case(rng, 2, 4, 1, 8, 48, lens=[48, 30])
    kp, table = _pool_from_contiguous(k, 8)
    vp, _ = _pool_from_contiguous(v, 8)
    perm = rng.permutation(kp.shape[0])            # physical block i moves to perm[i]
    kq, vq = np.empty_like(kp), np.empty_like(vp)
    kq[perm], vq[perm] = kp, vp
    out = oracle.gqa_decode_paged(q, kq, vq, perm[table].astype(np.int32), lens, 8, 0.5)
    assert np.array_equal(out, oracle.gqa_decode_paged(q, kp, vp, table, lens, 8, 0.5))


def test_sequences_sharing_prefix_blocks_match_private_copies():
    rng = np.random.default_rng(82)
    bs, Hkv, D = 8, 2, 16
    shared = rng.integers(0, 2 ** 15, size=(3, Hkv, bs, D)).astype(np.uint16) & 0x3FFF
    own = rng.integers(0, 2 ** 15, size=(2, Hkv, bs, D)).astype(np.uint16) & 0x3FFF
    pool = np.concatenate([shared, own])
    table = np.array([[0, 1, 2, 3], [0, 1, 2, 4]], np.int32)   # 3 prefix blocks shared
    lens = np.array([29, 32], np.int32)
    q = bits(rng.standard_normal((2, 4, D)))
    out = oracle.gqa_decode_paged(q, pool, pool, table, lens, bs, 0.3)
    # the same sequences with private copies of the prefix
    priv = np.concatenate([shared, own[:1], shared, own[1:]])
    table2 = np.array([[0, 1, 2, 3], [4, 5, 6, 7]], np.int32)
    assert np.array_equal(out, oracle.gqa_decode_paged(q, priv, priv, table2, lens, bs, 0.3))


def test_paged_window_is_the_contiguous_window():
    rng = np.random.default_rng(84)
    q, k, v, lens = rand_case(rng, 3, 8, 2, 16, 64, lens=[64, 37, 3])
    kp, table = _pool_from_contiguous(k, 16)
    vp, _ = _pool_from_contiguous(v, 16)
    for W in (1, 20, 64):
        out = oracle.gqa_decode_paged(q, kp, vp, table, lens, 16, 0.25, window=W)
        assert np.array_equal(out, oracle.gqa_decode(q, k, v, lens, 0.25, window=W))
    qm = bits(rng.standard_normal((3, 4, 8, 16)))
    out = oracle.gqa_decode_paged(qm, kp, vp, table, lens, 16, 0.25, window=6)
    assert np.array_equal(out, oracle.gqa_decode_multi(qm, k, v, lens, 0.25, window=6))


def test_paged_rejects_tables_outside_the_pool():
    rng = np.random.default_rng(83)
    pool = np.zeros((2, 1, 8, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.gather_paged(pool, np.array([[0, 5]], np.int32), np.array([12]), 8)
