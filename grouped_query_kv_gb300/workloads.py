"""Seeded synthetic decode workloads.

This module only draws inputs (random numbers and lengths); it holds none of
the attention arithmetic, so that the CUDA library and the CPU oracle can be
fed the same tensors without sharing any of the method's code.

The shapes follow the workloads the pages discuss: PaLM-8B / PaLM-540B
multi-query attention ("Efficiently Scaling Transformer Inference",
section 3 "Attention Layer Partitioning" and section 5 "Experiments": 48
query heads of width 256 sharing one K/V head) and Llama-2-70B grouped-query
attention ("Tensor Parallelism: Splitting Operations Across GPUs", section
"The GQA ceiling: a worked memory audit": 64 query heads, 8 K/V heads, head
width 128).  No page uses a dataset; the values are N(0,1) draws rounded to
bf16, which stand in for projected activations.

Length convention.  ``attn_lens[b]`` is the number of cached positions the
attention reads after this step's new token has been appended; the append
writes row ``attn_lens[b] - 1`` (the number of tokens cached before it).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Lmax: int
    scale: float
    # attention lengths: a fixed list, a single value for every sequence, or
    # None with `ragged=True` for uniform draws in [1, Lmax]
    lens: Optional[tuple] = None
    ragged: bool = False
    k_scale: float = 1.0
    # a local (sliding-window) attention layer: attend the last `window`
    # positions only; None is the full attention
    window: Optional[int] = None
    # new tokens (queries) per sequence scored in one pass, causal among
    # themselves (speculative sampling); their K/V rows are already cached
    T: int = 1
    # a paged cache: positions grouped in blocks of `block_size` in a shared
    # pool, reached through a per-sequence block table; None: contiguous
    block_size: Optional[int] = None
    # "fp8": an 8-bit cache (E4M3 codes, one fp32 scale per row); "bf16" else
    kv_dtype: str = "bf16"
    note: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


def _sweep() -> List[Workload]:
    out = []
    for hkv in (32, 8, 1):
        for b in (1, 8, 64, 256):
            out.append(Workload(
                name=f"sweep_hkv{hkv}_b{b}", B=b, Hq=32, Hkv=hkv, D=128,
                Lmax=4096, scale=1.0 / math.sqrt(128), lens=(4096,),
                note="MHA vs GQA vs MQA sweep at D=128, Hq=32, length 4096"))
    return out


WORKLOADS = {w.name: w for w in [
    Workload("tiny_mqa", B=2, Hq=4, Hkv=1, D=64, Lmax=64, scale=1.0 / 8.0,
             lens=(8, 34),
             note="tiny MQA: cached lengths [7, 33], one append then one "
                  "attention over [8, 34]"),
    Workload("palm8b_mqa", B=64, Hq=16, Hkv=1, D=256, Lmax=2048,
             scale=1.0 / 16.0, lens=(2048,),
             note="PaLM-8B-shaped MQA decode, every sequence at length 2048"),
    Workload("llama70b_gqa_ragged", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), ragged=True,
             note="Llama-70B-shaped GQA decode, lengths uniform in [1, 8192]"),
    Workload("palm540b_long_mqa", B=8, Hq=48, Hkv=1, D=256, Lmax=32768,
             scale=1.0 / 16.0, lens=(32768,), k_scale=0.5,
             note="PaLM-540B-shaped long-context MQA decode, k scaled by 0.5"),
    Workload("llama70b_spec4", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), ragged=True, T=4,
             note="Llama-70B-shaped GQA scoring 4 drafted tokens per sequence in "
                  "one pass (speculative sampling), lengths uniform in [4, 8192]"),
    Workload("palm540b_spec4", B=8, Hq=48, Hkv=1, D=256, Lmax=32768,
             scale=1.0 / 16.0, lens=(32768,), k_scale=0.5, T=4,
             note="PaLM-540B-shaped MQA scoring 4 drafted tokens per sequence in one "
                  "pass: 48 heads x 4 tokens = 192 query rows per K/V head, three passes "
                  "of 16 heads"),
    Workload("palm8b_spec4", B=64, Hq=16, Hkv=1, D=256, Lmax=2048,
             scale=1.0 / 16.0, lens=(2048,), T=4,
             note="PaLM-8B-shaped MQA scoring 4 drafted tokens per sequence: 16 heads "
                  "x 4 tokens = 64 query rows per K/V head, one pass"),
    Workload("local_gqa_w4096", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), lens=(8192,), window=4096,
             note="Llama-70B-shaped GQA decode through a local attention layer: "
                  "8192-token caches, the last 4096 positions attended"),
    Workload("llama70b_paged16", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), ragged=True, block_size=16,
             note="Llama-70B-shaped GQA decode over a paged cache: 16-position "
                  "blocks scattered through one pool, lengths uniform in [1, 8192]"),
    Workload("llama70b_fp8", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), ragged=True, kv_dtype="fp8",
             note="Llama-70B-shaped GQA decode over an 8-bit (E4M3 + per-row scale) "
                  "cache, lengths uniform in [1, 8192]"),
    Workload("palm8b_fp8", B=64, Hq=16, Hkv=1, D=256, Lmax=2048,
             scale=1.0 / 16.0, lens=(2048,), kv_dtype="fp8",
             note="the PaLM-8B-shaped MQA decode over an 8-bit (E4M3 + per-row scale) cache"),
    Workload("palm540b_fp8", B=8, Hq=48, Hkv=1, D=256, Lmax=32768,
             scale=1.0 / 16.0, lens=(32768,), k_scale=0.5, kv_dtype="fp8",
             note="the PaLM-540B-shaped long-context MQA decode over an 8-bit cache"),
    Workload("llama70b_paged64", B=32, Hq=64, Hkv=8, D=128, Lmax=8192,
             scale=1.0 / math.sqrt(128), ragged=True, block_size=64,
             note="the same over 64-position blocks"),
] + _sweep()}

# the five configurations in the order the benchmark suite lists them
CONFIG_ORDER = ["tiny_mqa", "palm8b_mqa", "llama70b_gqa_ragged",
                "palm540b_long_mqa"] + [w.name for w in _sweep()]


def attn_lens(w: Workload, seed: int = 0) -> torch.Tensor:
    """int32 [B] attention lengths (drawn on the CPU so they never depend on
    the device the values are drawn on)."""
    if w.ragged:
        g = torch.Generator().manual_seed(seed + 7919)
        return torch.randint(w.T, w.Lmax + 1, (w.B,), generator=g,
                             dtype=torch.int64).to(torch.int32)
    if len(w.lens) == 1:
        return torch.full((w.B,), w.lens[0], dtype=torch.int32)
    assert len(w.lens) == w.B
    return torch.tensor(w.lens, dtype=torch.int32)


def _normal_bf16(shape, gen, device, mul=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if mul != 1.0:
        x.mul_(mul)
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, seed: int = 0, device="cpu", lens=None):
    """Draw one decode step's inputs.

    Returns a dict of tensors on `device`:
      q        bf16 [B, Hq, D], or [B, T, Hq, D] for T new tokens
      k_cache  bf16 [B, Hkv, Lmax, D]   (every row drawn, padding included)
      v_cache  bf16 [B, Hkv, Lmax, D]
      k_new    bf16 [B, Hkv, D]         this step's new token
      v_new    bf16 [B, Hkv, D]
      append_pos int32 [B]              row the append writes (= attn_lens-1)
      attn_lens  int32 [B]              positions the attention reads
    """
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    al = attn_lens(w, seed) if lens is None else torch.as_tensor(lens, dtype=torch.int32)
    assert al.shape == (w.B,)
    assert int(al.min()) >= 1 and int(al.max()) <= w.Lmax
    q = _normal_bf16((w.B, w.Hq, w.D) if w.T == 1 else (w.B, w.T, w.Hq, w.D), gen, device)
    k_cache = _normal_bf16((w.B, w.Hkv, w.Lmax, w.D), gen, device, w.k_scale)
    v_cache = _normal_bf16((w.B, w.Hkv, w.Lmax, w.D), gen, device)
    k_new = _normal_bf16((w.B, w.Hkv, w.D), gen, device, w.k_scale)
    v_new = _normal_bf16((w.B, w.Hkv, w.D), gen, device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new,
                v_new=v_new, append_pos=(al - 1).to(device),
                attn_lens=al.to(device))


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bits (copied to the host)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def make_paged(w: Workload, x: dict, seed: int = 0, spare_blocks: int = 0,
               fill_unused=None):
    """A paged copy of make_inputs' caches: each sequence's first
    ceil(attn_lens[b] / block_size) blocks of positions are moved to blocks
    of one pool in a seeded random order (the way an allocator hands out
    free blocks), and the block table records where each went.

    Returns dict(k_pool, v_pool: bf16 [num_blocks, Hkv, block_size, D],
    block_table: int32 [B, ceil(Lmax / block_size)]).  Table entries of
    blocks a sequence does not use are -1; `spare_blocks` unused blocks are
    added to the pool, and fill_unused (a bf16 bit pattern, e.g. 0x7FC0 for
    NaN) overwrites every pool row no sequence position maps to.  A plain
    copy: no attention arithmetic."""
    bs = w.block_size
    assert bs and bs & (bs - 1) == 0
    k, v = x["k_cache"], x["v_cache"]
    dev = k.device
    B, Hkv, L, D = k.shape
    maxb = (L + bs - 1) // bs
    if maxb * bs != L:  # pad the positions to whole blocks
        pad = maxb * bs - L
        k = torch.cat([k, k.new_zeros((B, Hkv, pad, D))], dim=2)
        v = torch.cat([v, v.new_zeros((B, Hkv, pad, D))], dim=2)
    lens = x["attn_lens"].cpu().to(torch.int64)
    nb = (lens + bs - 1) // bs
    used = torch.arange(maxb)[None, :] < nb[:, None]            # [B, maxb]
    n_used = int(used.sum())
    total = n_used + spare_blocks
    g = torch.Generator().manual_seed(seed + 104729)
    phys = torch.randperm(total, generator=g)[:n_used]
    table = torch.full((B, maxb), -1, dtype=torch.int32)
    table[used] = phys.to(torch.int32)
    kb = k.view(B, Hkv, maxb, bs, D).transpose(1, 2)            # [B, maxb, Hkv, bs, D]
    vb = v.view(B, Hkv, maxb, bs, D).transpose(1, 2)
    used_d = used.to(dev)
    k_pool = torch.zeros((total, Hkv, bs, D), dtype=k.dtype, device=dev)
    v_pool = torch.zeros((total, Hkv, bs, D), dtype=v.dtype, device=dev)
    phys_d = phys.to(dev)
    k_pool[phys_d] = kb[used_d]
    v_pool[phys_d] = vb[used_d]
    if fill_unused is not None:
        pat = torch.tensor([fill_unused], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        mask = torch.ones((total, bs), dtype=torch.bool)
        mask[phys] = False                                      # blocks in use...
        last = (lens - 1).clamp(min=0)                          # ...but rows past the length
        for b in range(B):
            n = int(lens[b])
            if n > 0:
                r = n - int(last[b]) // bs * bs
                mask[int(table[b, int(last[b]) // bs]), r:] = True
        m = mask.to(dev)[:, None, :].expand(total, Hkv, bs)
        k_pool[m] = pat.to(dev)
        v_pool[m] = pat.to(dev)
    return dict(k_pool=k_pool, v_pool=v_pool, block_table=table.to(dev))
