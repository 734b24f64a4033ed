"""Plant plausible mistakes in a copy of the oracle's C source, compile each
copy, and check that the independent pins reject it.  This is evidence that
the pins can tell a wrong oracle from a right one (CPU only)."""
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
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def pins_pass(orc) -> bool:
    """A compact battery of the independent pins; False on the first miss."""
    rng = np.random.default_rng(99)
    B, Hq, Hkv, D, L = 3, 8, 2, 32, 24
    q = _bits(rng.standard_normal((B, Hq, D)))
    k = _bits(rng.standard_normal((B, Hkv, L, D)))
    v = _bits(rng.standard_normal((B, Hkv, L, D)))
    lens = np.array([24, 7, 1], np.int32)
    scale = 1.0 / math.sqrt(D)
    try:
        out = orc.gqa_decode(q, k, v, lens, scale=scale)
    except ValueError:
        return False
    # library special case
    for b in range(B):
        n = int(lens[b])
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(_unbits(q[b:b + 1]))[:, :, None, :],
            torch.from_numpy(_unbits(k[b:b + 1, :, :n])),
            torch.from_numpy(_unbits(v[b:b + 1, :, :n])),
            scale=scale, enable_gqa=True)[0, :, 0].numpy()
        if not np.allclose(out[b], ref, rtol=1e-12, atol=1e-13):
            return False
    # length one returns V[0]
    if not np.array_equal(out[2], _unbits(v[2, np.arange(Hq) // 4, 0])):
        return False
    # rows past the length are never read
    k2, v2 = k.copy(), v.copy()
    k2[1, :, 7:] = 0x7FC0
    v2[1, :, 7:] = 0x7F80
    if not np.array_equal(orc.gqa_decode(q, k2, v2, lens, scale=scale), out):
        return False
    # append: exactly one row per (b, kvh) changes, to the new values
    kc, vc = k.copy(), v.copy()
    kn = _bits(rng.standard_normal((B, Hkv, D)))
    vn = _bits(rng.standard_normal((B, Hkv, D)))
    pos = np.array([3, 0, 23], np.int32)
    kr, vr = kc.copy(), vc.copy()
    kr[np.arange(B), :, pos] = kn
    vr[np.arange(B), :, pos] = vn
    try:
        orc.kv_append(kc, vc, kn, vn, pos)
    except ValueError:
        return False
    if not (np.array_equal(kc, kr) and np.array_equal(vc, vr)):
        return False
    # a window of W positions: the full attention over a cache that holds
    # only those W rows (checked with torch's attention on the rows)
    for W in (1, 5, 23):
        try:
            ow = orc.gqa_decode(q, k, v, lens, scale=scale, window=W)
        except ValueError:
            return False
        for b in range(B):
            n = int(lens[b])
            j0 = max(0, n - W)
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(_unbits(q[b:b + 1]))[:, :, None, :],
                torch.from_numpy(_unbits(k[b:b + 1, :, j0:n])),
                torch.from_numpy(_unbits(v[b:b + 1, :, j0:n])),
                scale=scale, enable_gqa=True)[0, :, 0].numpy()
            if not np.allclose(ow[b], ref, rtol=1e-12, atol=1e-13):
                return False
    # T new tokens: token t is a single-token decode over len - T + 1 + t
    # positions (torch's attention on those rows)
    T = 3
    qm = _bits(rng.standard_normal((B, T, Hq, D)))
    lm = np.array([24, 7, 3], np.int32)
    try:
        om = orc.gqa_decode_multi(qm, k, v, lm, scale=scale)
    except ValueError:
        return False
    for b in range(B):
        for t in range(T):
            n = int(lm[b]) - T + 1 + t
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(_unbits(qm[b:b + 1, t]))[:, :, None, :],
                torch.from_numpy(_unbits(k[b:b + 1, :, :n])),
                torch.from_numpy(_unbits(v[b:b + 1, :, :n])),
                scale=scale, enable_gqa=True)[0, :, 0].numpy()
            if not np.allclose(om[b, t], ref, rtol=1e-12, atol=1e-13):
                return False
    # T new tokens on a local layer: token t attends the W positions that
    # end at its own (torch's attention on those rows)
    for W in (3, 6):
        try:
            ow = orc.gqa_decode_multi(qm, k, v, lm, scale=scale, window=W)
        except ValueError:
            return False
        for b in range(B):
            for t in range(T):
                n = int(lm[b]) - T + 1 + t
                j0 = max(0, n - W)
                ref = F.scaled_dot_product_attention(
                    torch.from_numpy(_unbits(qm[b:b + 1, t]))[:, :, None, :],
                    torch.from_numpy(_unbits(k[b:b + 1, :, j0:n])),
                    torch.from_numpy(_unbits(v[b:b + 1, :, j0:n])),
                    scale=scale, enable_gqa=True)[0, :, 0].numpy()
                if not np.allclose(ow[b, t], ref, rtol=1e-12, atol=1e-13):
                    return False
    return True


MUTANTS = {
    "interleaved head mapping": ("const int64_t kvh = h / G;",
                                 "const int64_t kvh = h % Hkv;"),
    "dropped scale": ("s_buf[j - j0] = scale * dot;", "s_buf[j - j0] = dot;"),
    "normaliser without max shift": ("denom += exp(s_buf[j] - m);",
                                     "denom += exp(s_buf[j]);"),
    "flipped sign in weights": ("double p = exp(s_buf[j] - m) / denom;",
                                "double p = exp(m - s_buf[j]) / denom;"),
    "keys and values swapped": (
        "oracle_cache_at(v_cache, q8->v, q8->v_scale, row0, j0 + j, D, d)",
        "oracle_cache_at(k_cache, q8->k, q8->k_scale, row0, j0 + j, D, d)"),
    "wrong query row": ("const uint16_t *qh = q + ((b * T + t) * Hq + h) * D;",
                        "const uint16_t *qh = q + ((b * T + t) * Hq + kvh) * D;"),
    "reads one row past the length": (
        "int64_t len = seq_lens[b] - (T - 1 - t);",
        "int64_t len = seq_lens[b] - (T - 1 - t) + (seq_lens[b] < Lmax);"),
    "new tokens see one position too few": ("int64_t len = seq_lens[b] - (T - 1 - t);",
                                            "int64_t len = seq_lens[b] - (T - t);"),
    "new tokens see the whole run": ("int64_t len = seq_lens[b] - (T - 1 - t);",
                                     "int64_t len = seq_lens[b] - 0 * t;"),
    "new tokens' queries reversed": (
        "const uint16_t *qh = q + ((b * T + t) * Hq + h) * D;",
        "const uint16_t *qh = q + ((b * T + (T - 1 - t)) * Hq + h) * D;"),
    "append one row late": ("int64_t pos = seq_lens[b];",
                            "int64_t pos = seq_lens[b] + (seq_lens[b] + 1 < Lmax);"),
    "append swaps k and v": ("v_cache[dst] = v_new[src];",
                             "v_cache[dst] = k_new[src];"),
    "window one position short": ("const int64_t j0 = len > window ? len - window : 0;",
                                  "const int64_t j0 = len > window ? len - window + 1 : 0;"),
    "window one position long": ("const int64_t j0 = len > window ? len - window : 0;",
                                 "const int64_t j0 = len > window ? len - window - 1 : 0;"),
    "new tokens share the last token's window": (
        "const int64_t j0 = len > window ? len - window : 0;",
        "const int64_t j0 = len > window ? seq_lens[b] - window : 0;"),
    "window values not shifted": ("oracle_cache_at(v_cache, q8->v, q8->v_scale, row0, j0 + j, D, d)",
                                  "oracle_cache_at(v_cache, q8->v, q8->v_scale, row0, j, D, d)"),
}


def test_unmodified_oracle_passes_the_battery():
    assert pins_pass(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    assert not pins_pass(oracle.Oracle(so)), name


# ------------------------------------------------------- paged cache gather
# The paged oracle is a plain gather through the block table followed by the
# contiguous decode; mistakes are planted in copies of the gather.

def _paged_pins_pass(orc) -> bool:
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, bs, nb = 3, 4, 2, 16, 8, 4
    L = bs * nb
    q = _bits(rng.standard_normal((B, Hq, D)))
    k = _bits(rng.standard_normal((B, Hkv, L, D)))
    v = _bits(rng.standard_normal((B, Hkv, L, D)))
    lens = np.array([32, 19, 9], np.int32)
    # identity table over a pool made by numpy reshapes
    kp = np.ascontiguousarray(k.reshape(B, Hkv, nb, bs, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, bs, D))
    vp = np.ascontiguousarray(v.reshape(B, Hkv, nb, bs, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, bs, D))
    table = np.arange(B * nb, dtype=np.int32).reshape(B, nb)
    try:
        out = orc.gqa_decode_paged(q, kp, vp, table, lens, bs, 0.25)
    except (ValueError, IndexError):
        return False
    if not np.array_equal(out, orc.gqa_decode(q, k, v, lens, 0.25)):
        return False
    # blocks moved around the pool
    perm = rng.permutation(B * nb)
    kq, vq = np.empty_like(kp), np.empty_like(vp)
    kq[perm], vq[perm] = kp, vp
    try:
        out2 = orc.gqa_decode_paged(q, kq, vq, perm[table].astype(np.int32), lens, bs, 0.25)
    except (ValueError, IndexError):
        return False
    return np.array_equal(out2, out)


class _PagedMutant(oracle.Oracle):
    def __init__(self, kind):
        super().__init__()
        self.kind = kind

    def gather_paged(self, pool, block_table, seq_lens, block_size):
        nblk, Hkv, bs, D = pool.shape
        table = np.asarray(block_table)
        B, maxb = table.shape
        out = np.zeros((B, Hkv, maxb * bs, D), dtype=pool.dtype)
        for b in range(B):
            for p in range(int(seq_lens[b])):
                if self.kind == "row_and_block_swapped":
                    blk, r = int(table[b, p % maxb]), p // maxb
                    r = min(r, bs - 1)
                elif self.kind == "block_table_of_sequence_zero":
                    blk, r = int(table[0, p // bs]), p % bs
                elif self.kind == "table_read_one_block_late":
                    blk, r = int(table[b, min(p // bs + 1, maxb - 1)]), p % bs
                else:  # "row_within_block_ignored"
                    blk, r = int(table[b, p // bs]), 0
                out[b, :, p] = pool[blk, :, r]
        return out


def test_unmodified_paged_oracle_passes():
    assert _paged_pins_pass(oracle.Oracle())


@pytest.mark.parametrize("kind", ["row_and_block_swapped", "block_table_of_sequence_zero",
                                  "table_read_one_block_late", "row_within_block_ignored"])
def test_planted_paged_mistake_is_caught(kind):
    assert not _paged_pins_pass(_PagedMutant(kind)), kind
