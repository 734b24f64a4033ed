"""Byte and FLOP accounting for the decode-attention roofline.

The algorithmic unit of work is one cached position of one K/V head: its key
row and value row are read once (2 * D elements) and every one of the G query
heads sharing that K/V head spends 2 * D multiply-adds on it (q . k and p * v),
i.e. 4 * D * G FLOPs.  Padding beyond a sequence's length is not counted,
matching "The Basics of Transformer Inference", the item "Using ragged HBM
reads and Paged Attention" (only the non-padding part of the cache needs to be
read).
"""
from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                       elem_bytes: int) -> int:
    """Cache bytes one token adds: keys and values, for every layer and K/V
    head ("Machine Learning Engineering and AI Systems at Scale", section
    "The key and value cache": two, times layers, K/V heads, head dimension
    and bytes per element)."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, elem_bytes: int,
                   batch: int, tokens: int) -> int:
    """Whole-cache bytes for `batch` sequences of `tokens` cached tokens."""
    return kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes) * batch * tokens


def attended_positions(attn_lens, window=None) -> int:
    """Positions attended over the batch: each sequence's length, capped at
    the window for a local attention layer ("The Basics of Transformer
    Inference", item on mixing in local attention layers)."""
    if window is None:
        return int(sum(int(x) for x in attn_lens))
    return int(sum(min(int(x), int(window)) for x in attn_lens))


def kv_bytes_read(attn_lens, Hkv: int, D: int, elem_bytes: int = 2, window=None) -> int:
    """Algorithmic K+V bytes one decode-attention call reads (one layer)."""
    return attended_positions(attn_lens, window) * Hkv * D * 2 * elem_bytes


def kv_bytes_read_fp8(attn_lens, Hkv: int, D: int, window=None) -> int:
    """The same for an 8-bit cache: one byte per element plus one fp32
    scale per cached row, for K and for V."""
    return attended_positions(attn_lens, window) * Hkv * 2 * (D + 4)


def attn_flops(attn_lens, Hq: int, D: int, window=None) -> int:
    """Algorithmic FLOPs of one call: 2*D for q.k plus 2*D for p*v per query
    head and position."""
    return 4 * Hq * D * attended_positions(attn_lens, window)
