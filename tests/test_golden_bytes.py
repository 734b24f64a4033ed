"""Byte counts the pages print for KV caches pin the accounting that the
benchmark's roofline uses (tests/golden/kv_bytes.tsv, one cited row each)."""
import os

import pytest

from grouped_query_kv_gb300 import accounting

HERE = os.path.dirname(os.path.abspath(__file__))


def _rows():
    rows = []
    with open(os.path.join(HERE, "golden", "kv_bytes.tsv")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, layers, kvh, hd, eb, batch, tokens, want, tol, cite = \
                line.rstrip("\n").split("\t")
            rows.append((name, int(layers), int(kvh), int(hd), int(eb),
                         int(batch), int(tokens), int(want), float(tol), cite))
    return rows


@pytest.mark.parametrize("row", _rows(), ids=lambda r: r[0])
def test_kv_cache_bytes_match_the_pages(row):
    name, layers, kvh, hd, eb, batch, tokens, want, tol, cite = row
    got = accounting.kv_cache_bytes(layers, kvh, hd, eb, batch, tokens)
    if tol == 0:
        assert got == want, cite
    else:
        assert abs(got - want) <= tol * want, (got, want, cite)


def test_kv_bytes_read_counts_only_the_non_padding_part():
    # one decode call over two sequences of 8 and 34 cached tokens, one K/V
    # head of width 64, bf16: (8 + 34) positions * 64 * 2 (K and V) * 2 bytes
    assert accounting.kv_bytes_read([8, 34], 1, 64) == 42 * 64 * 4
    # the per-token figure for one layer equals the read per position
    assert accounting.kv_bytes_read([1], 8, 128) == \
        accounting.kv_bytes_per_token(1, 8, 128, 2)
    assert accounting.attn_flops([10], Hq=16, D=256) == 4 * 16 * 256 * 10
