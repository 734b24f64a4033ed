"""grouped_query_kv_gb300 -- Python binding of libkvattn (GB300 decode
attention over a grouped-query / multi-query KV cache).

The binding only marshals arguments: it checks dtypes, shapes, devices and
contiguity of torch tensors, and passes raw device pointers and the current
CUDA stream to the C ABI declared in ``include/kvattn.h``.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and importing the entry points fails loudly if the compiled
library is missing (build it with ``python -m grouped_query_kv_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "kv_append", "kv_append_multi", "kv_append_paged", "gqa_decode_attn", "gqa_decode_step",
    "gqa_decode_attn_multi", "gqa_decode_attn_paged", "gqa_decode_step_paged",
    "kv_quantize_fp8", "kv_append_fp8", "gqa_decode_attn_fp8", "gqa_decode_step_fp8",
    "check_device_error", "get_plan",
    "set_tuning", "set_wait_limit", "set_kernel_events", "release", "KvAttnError", "library_path", "lib",
    "KVATTN_OK", "KVATTN_ERR_INVALID_ARG", "KVATTN_ERR_UNSUPPORTED",
    "KVATTN_ERR_CUDA", "KVATTN_ERR_OOM", "KVATTN_ERR_DEVICE_BOUNDS",
    "KVATTN_ERR_TIMEOUT", "EXPORTED_SYMBOLS",
]

KVATTN_OK = 0
KVATTN_ERR_INVALID_ARG = 1
KVATTN_ERR_UNSUPPORTED = 2
KVATTN_ERR_CUDA = 3
KVATTN_ERR_OOM = 4
KVATTN_ERR_DEVICE_BOUNDS = 5
KVATTN_ERR_TIMEOUT = 6

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkvattn.so")
_lock = threading.Lock()
_lib = None


class KvAttnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__("%s (%d): %s" % (_status_name(status), status, detail))


class kvattn_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("tile_positions", ctypes.c_int),
                ("heads_per_cta", ctypes.c_int), ("head_groups", ctypes.c_int),
                ("stages", ctypes.c_int), ("threads", ctypes.c_int),
                ("num_ctas", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("workspace_bytes", ctypes.c_int64)]


# name -> (restype, argtypes); mirrors include/kvattn.h
_VP = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "kv_append": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "kv_append_multi": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "gqa_decode_attn": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                             ctypes.c_float, _VP]),
    "gqa_decode_step": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                             ctypes.c_float, _VP]),
    "gqa_decode_attn_multi": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                                   ctypes.c_float, _VP]),
    "gqa_decode_attn_window": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                                    ctypes.c_float, _I, _VP]),
    "gqa_decode_step_window": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                                    ctypes.c_float, _I, _VP]),
    "gqa_decode_attn_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _VP]),
    "kv_append_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "kv_quantize_fp8": (_I, [_VP, _VP, _VP, ctypes.c_longlong, _I, _VP]),
    "kv_append_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "gqa_decode_attn_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                                 ctypes.c_float, _VP]),
    "gqa_decode_step_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I,
                                 _I, ctypes.c_float, _VP]),
    "gqa_decode_attn_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I,
                                   _I, ctypes.c_float, _VP]),
    "gqa_decode_step_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I,
                                   _I, _I, _I, ctypes.c_float, _VP]),
    "gqa_decode_attn_multi_window": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                                          ctypes.c_float, _I, _VP]),
    "gqa_decode_attn_paged_window": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                                          _I, _I, ctypes.c_float, _I, _VP]),
    "gqa_decode_step_paged_window": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I,
                                          _I, _I, _I, _I, ctypes.c_float, _I, _VP]),
    "kvattn_status_string": (ctypes.c_char_p, [_I]),
    "kvattn_last_error": (ctypes.c_char_p, []),
    "kvattn_check_device_error": (_I, [_VP]),
    "kvattn_release": (None, []),
    "kvattn_set_tuning": (_I, [_I, _I]),
    "kvattn_set_wait_limit": (_I, [ctypes.c_uint]),
    "kvattn_set_kernel_events": (_I, [_VP, _VP]),
    "kvattn_get_plan": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(kvattn_plan)]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    h = _lib
    if h is not None:  # per-call fast path: no lock once loaded
        return h
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    "libkvattn.so is not built (%s); run "
                    "`python -m grouped_query_kv_gb300.build`" % _LIB_PATH)
            h = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _status_name(status: int) -> str:
    try:
        return lib().kvattn_status_string(status).decode()
    except Exception:  # library not loadable: still give a readable error
        return "status"


def _check(status: int):
    if status != KVATTN_OK:
        raise KvAttnError(status, lib().kvattn_last_error().decode())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream  # a plain int: ctypes converts it for the c_void_p argument


def _ptr(t):
    return t.data_ptr()


def _need(t, name, dtype, shape=None):
    # the checks run on every call of a decode loop, so they use the cheapest
    # torch attributes (is_cuda, dtype identity, torch.Size == tuple)
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (got %s)" % (name, t.device))
    if t.dtype is not dtype:
        raise TypeError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and t.shape != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))


def kv_append(k_cache, v_cache, k_new, v_new, seq_lens, stream=None):
    """Write the new token's K/V rows into row seq_lens[b] of the caches.

    k_cache, v_cache: bf16 [B, Hkv, Lmax, D] (in place); k_new, v_new: bf16
    [B, Hkv, D]; seq_lens: int32 [B], tokens cached before this one (not
    modified).
    """
    import torch
    _need(k_cache, "k_cache", torch.bfloat16)
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [B, Hkv, Lmax, D]")
    B, Hkv, Lmax, D = k_cache.shape
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D))
    _need(k_new, "k_new", torch.bfloat16, (B, Hkv, D))
    _need(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _check(lib().kv_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                           _ptr(seq_lens), B, Hkv, D, Lmax, _stream_ptr(stream)))


def kv_append_multi(k_cache, v_cache, k_new, v_new, seq_lens, stream=None):
    """Write T new tokens' K/V rows: token t into row seq_lens[b] + t.

    k_cache, v_cache: bf16 [B, Hkv, Lmax, D] (in place); k_new, v_new: bf16
    [B, T, Hkv, D]; seq_lens: int32 [B], tokens cached before them (not
    modified).
    """
    import torch
    _need(k_cache, "k_cache", torch.bfloat16)
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [B, Hkv, Lmax, D]")
    B, Hkv, Lmax, D = k_cache.shape
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D))
    _need(k_new, "k_new", torch.bfloat16)
    if k_new.dim() != 4 or k_new.shape[0] != B or k_new.shape[2:] != (Hkv, D):
        raise ValueError("k_new must be [B, T, Hkv, D]")
    T = k_new.shape[1]
    _need(v_new, "v_new", torch.bfloat16, (B, T, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _check(lib().kv_append_multi(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                 _ptr(seq_lens), B, T, Hkv, D, Lmax, _stream_ptr(stream)))


def gqa_decode_attn(q, k_cache, v_cache, seq_lens, scale, out=None, stream=None,
                    window=None):
    """out[b,h] = softmax(scale * q[b,h] . K[b,h//G]^T) . V[b,h//G] over the
    first seq_lens[b] cached positions (only the last `window` of them for a
    local attention layer).

    q: bf16 [B, Hq, D]; caches: bf16 [B, Hkv, Lmax, D]; seq_lens: int32 [B];
    out: optional fp32 [B, Hq, D] (allocated if None); window: None (all
    positions) or an int >= 1.  Returns out.
    """
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    _need(k_cache, "k_cache", torch.bfloat16)
    if k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("k_cache must be [B, Hkv, Lmax, D] matching q")
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    if window is None:
        _check(lib().gqa_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                     _ptr(out), B, Hq, Hkv, D, Lmax, float(scale),
                                     _stream_ptr(stream)))
    else:
        _check(lib().gqa_decode_attn_window(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, Lmax,
                                            float(scale), int(window), _stream_ptr(stream)))
    return out


def gqa_decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out=None,
                    stream=None, window=None):
    """One fused decode step: write k_new/v_new into row seq_lens[b] of the
    caches, then attend over positions [0, seq_lens[b] + 1) (only the last
    `window` of them for a local attention layer).

    q: bf16 [B, Hq, D]; k_new, v_new: bf16 [B, Hkv, D]; caches: bf16
    [B, Hkv, Lmax, D] (modified in place); seq_lens: int32 [B], tokens cached
    before this step (not modified); out: optional fp32 [B, Hq, D].
    """
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    _need(k_cache, "k_cache", torch.bfloat16)
    if k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("k_cache must be [B, Hkv, Lmax, D] matching q")
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D))
    _need(k_new, "k_new", torch.bfloat16, (B, Hkv, D))
    _need(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    if window is None:
        _check(lib().gqa_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D,
                                     Lmax, float(scale), _stream_ptr(stream)))
    else:
        _check(lib().gqa_decode_step_window(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(seq_lens), _ptr(out), B, Hq,
                                            Hkv, D, Lmax, float(scale), int(window),
                                            _stream_ptr(stream)))
    return out


def gqa_decode_attn_multi(q, k_cache, v_cache, seq_lens, scale, out=None, stream=None,
                          window=None):
    """Attention for T new tokens per sequence, causal among themselves: token
    t of sequence b attends positions [0, e) with e = seq_lens[b] - T + 1 + t
    (only [e - window, e) for a local attention layer).

    q: bf16 [B, T, Hq, D]; caches: bf16 [B, Hkv, Lmax, D] already holding the
    new tokens' rows; seq_lens: int32 [B], tokens in the cache including the
    new ones; out: optional fp32 [B, T, Hq, D]; window: None (all positions)
    or an int >= 1.  Returns out.
    """
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, T, Hq, D]")
    B, T, Hq, D = q.shape
    _need(k_cache, "k_cache", torch.bfloat16)
    if k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("k_cache must be [B, Hkv, Lmax, D] matching q")
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, T, Hq, D))
    if window is None:
        _check(lib().gqa_decode_attn_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(seq_lens), _ptr(out), B, T, Hq, Hkv, D, Lmax,
                                           float(scale), _stream_ptr(stream)))
    else:
        _check(lib().gqa_decode_attn_multi_window(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                  _ptr(seq_lens), _ptr(out), B, T, Hq, Hkv, D,
                                                  Lmax, float(scale), int(window),
                                                  _stream_ptr(stream)))
    return out


def _pool_shape(k_pool, block_table, name="k_pool"):
    """(num_blocks, Hkv, block_size, D, B, max_blocks) of a paged cache."""
    import torch
    _need(k_pool, name, torch.bfloat16)
    if k_pool.dim() != 4:
        raise ValueError("%s must be [num_blocks, Hkv, block_size, D]" % name)
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B, max_blocks]")
    return tuple(k_pool.shape) + tuple(block_table.shape)


def kv_append_paged(k_pool, v_pool, k_new, v_new, block_table, seq_lens, stream=None):
    """Write new K/V rows into a paged pool: token t of sequence b goes to
    position seq_lens[b] + t, i.e. row (seq_lens[b] + t) % block_size of block
    block_table[b, (seq_lens[b] + t) // block_size].

    k_pool, v_pool: bf16 [num_blocks, Hkv, block_size, D] (in place);
    k_new, v_new: bf16 [B, Hkv, D] (one token) or [B, T, Hkv, D];
    block_table: int32 [B, max_blocks]; seq_lens: int32 [B], tokens cached
    before the new ones (not modified).
    """
    import torch
    nblk, Hkv, bs, D, B, maxb = _pool_shape(k_pool, block_table)
    _need(v_pool, "v_pool", torch.bfloat16, (nblk, Hkv, bs, D))
    _need(k_new, "k_new", torch.bfloat16)
    if k_new.dim() == 3:
        T = 1
    elif k_new.dim() == 4:
        T = k_new.shape[1]
    else:
        raise ValueError("k_new must be [B, Hkv, D] or [B, T, Hkv, D]")
    if k_new.shape[0] != B or tuple(k_new.shape[-2:]) != (Hkv, D):
        raise ValueError("k_new must be [B, (T,) Hkv, D] matching the pool")
    _need(v_new, "v_new", torch.bfloat16, tuple(k_new.shape))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _check(lib().kv_append_paged(_ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                                 _ptr(block_table), _ptr(seq_lens), B, T, Hkv, D, nblk, bs,
                                 maxb, _stream_ptr(stream)))


def gqa_decode_attn_paged(q, k_pool, v_pool, block_table, seq_lens, scale, out=None,
                          stream=None, window=None):
    """gqa_decode_attn (q [B, Hq, D]) or gqa_decode_attn_multi (q [B, T, Hq, D])
    over a paged cache: position j of sequence b is row j % block_size of
    block block_table[b, j // block_size] of the pools.

    k_pool, v_pool: bf16 [num_blocks, Hkv, block_size, D]; block_table: int32
    [B, max_blocks]; seq_lens: int32 [B]; out: optional fp32 shaped like q;
    window: None (all positions) or an int >= 1, each query's local window.
    Returns out.
    """
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() not in (3, 4):
        raise ValueError("q must be [B, Hq, D] or [B, T, Hq, D]")
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    T = 1 if q.dim() == 3 else q.shape[1]
    nblk, Hkv, bs, Dp, Bt, maxb = _pool_shape(k_pool, block_table)
    if Dp != D or Bt != B:
        raise ValueError("k_pool / block_table do not match q")
    _need(v_pool, "v_pool", torch.bfloat16, (nblk, Hkv, bs, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty(tuple(q.shape), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, tuple(q.shape))
    if window is None:
        _check(lib().gqa_decode_attn_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                           _ptr(block_table), _ptr(seq_lens), _ptr(out), B, T,
                                           Hq, Hkv, D, nblk, bs, maxb, float(scale),
                                           _stream_ptr(stream)))
    else:
        _check(lib().gqa_decode_attn_paged_window(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                  _ptr(block_table), _ptr(seq_lens), _ptr(out),
                                                  B, T, Hq, Hkv, D, nblk, bs, maxb,
                                                  float(scale), int(window),
                                                  _stream_ptr(stream)))
    return out


def gqa_decode_step_paged(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, scale,
                          out=None, stream=None, window=None):
    """gqa_decode_step over a paged cache: the new token's rows go to position
    seq_lens[b] through the block table, then attention over [0, seq_lens[b] + 1)
    (only its last `window` positions for a local attention layer).

    q: bf16 [B, Hq, D]; k_new, v_new: bf16 [B, Hkv, D]; pools and table as
    for gqa_decode_attn_paged; seq_lens: tokens cached before this step.
    """
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    nblk, Hkv, bs, Dp, Bt, maxb = _pool_shape(k_pool, block_table)
    if Dp != D or Bt != B:
        raise ValueError("k_pool / block_table do not match q")
    _need(v_pool, "v_pool", torch.bfloat16, (nblk, Hkv, bs, D))
    _need(k_new, "k_new", torch.bfloat16, (B, Hkv, D))
    _need(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    if window is None:
        _check(lib().gqa_decode_step_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                                           _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                                           _ptr(out), B, Hq, Hkv, D, nblk, bs, maxb,
                                           float(scale), _stream_ptr(stream)))
    else:
        _check(lib().gqa_decode_step_paged_window(_ptr(q), _ptr(k_new), _ptr(v_new),
                                                  _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                                  _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D,
                                                  nblk, bs, maxb, float(scale), int(window),
                                                  _stream_ptr(stream)))
    return out


def kv_quantize_fp8(src, codes=None, scales=None, stream=None):
    """Quantize bf16 rows [..., D] into E4M3 codes (uint8 [..., D]) and one
    fp32 scale per row ([...]): scale = absmax / 448, code = E4M3(x / scale).
    Returns (codes, scales)."""
    import torch
    _need(src, "src", torch.bfloat16)
    D = src.shape[-1]
    rows = src.numel() // D if D else 0
    if codes is None:
        codes = torch.empty(tuple(src.shape), dtype=torch.uint8, device=src.device)
    if scales is None:
        scales = torch.empty(tuple(src.shape[:-1]), dtype=torch.float32, device=src.device)
    _need(codes, "codes", torch.uint8, tuple(src.shape))
    _need(scales, "scales", torch.float32, tuple(src.shape[:-1]))
    _check(lib().kv_quantize_fp8(_ptr(src), _ptr(codes), _ptr(scales), rows, D,
                                 _stream_ptr(stream)))
    return codes, scales


def kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, seq_lens, stream=None):
    """Quantize the new token's K/V rows into position seq_lens[b] of an
    8-bit cache (codes uint8 [B, Hkv, Lmax, D], scales fp32 [B, Hkv, Lmax];
    k_new, v_new bf16 [B, Hkv, D])."""
    import torch
    _need(k_codes, "k_codes", torch.uint8)
    if k_codes.dim() != 4:
        raise ValueError("k_codes must be [B, Hkv, Lmax, D]")
    B, Hkv, Lmax, D = k_codes.shape
    _need(v_codes, "v_codes", torch.uint8, (B, Hkv, Lmax, D))
    _need(k_scale, "k_scale", torch.float32, (B, Hkv, Lmax))
    _need(v_scale, "v_scale", torch.float32, (B, Hkv, Lmax))
    _need(k_new, "k_new", torch.bfloat16, (B, Hkv, D))
    _need(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _check(lib().kv_append_fp8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                               _ptr(k_new), _ptr(v_new), _ptr(seq_lens), B, Hkv, D, Lmax,
                               _stream_ptr(stream)))


def gqa_decode_attn_fp8(q, k_codes, v_codes, k_scale, v_scale, seq_lens, scale, out=None,
                        stream=None):
    """gqa_decode_attn over an 8-bit cache: K = E4M3(k_codes) * k_scale per
    row, V likewise.  q bf16 [B, Hq, D]; codes uint8 [B, Hkv, Lmax, D];
    scales fp32 [B, Hkv, Lmax]; seq_lens int32 [B]; out optional fp32
    [B, Hq, D].  Returns out."""
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    _need(k_codes, "k_codes", torch.uint8)
    if k_codes.dim() != 4 or k_codes.shape[0] != B or k_codes.shape[3] != D:
        raise ValueError("k_codes must be [B, Hkv, Lmax, D] matching q")
    Hkv, Lmax = k_codes.shape[1], k_codes.shape[2]
    _need(v_codes, "v_codes", torch.uint8, (B, Hkv, Lmax, D))
    _need(k_scale, "k_scale", torch.float32, (B, Hkv, Lmax))
    _need(v_scale, "v_scale", torch.float32, (B, Hkv, Lmax))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    _check(lib().gqa_decode_attn_fp8(_ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D,
                                     Lmax, float(scale), _stream_ptr(stream)))
    return out


def gqa_decode_step_fp8(q, k_new, v_new, k_codes, v_codes, k_scale, v_scale, seq_lens, scale,
                        out=None, stream=None):
    """kv_append_fp8 then gqa_decode_attn_fp8 over seq_lens[b] + 1 positions,
    in one pass (the attention kernel writes the quantized rows first).
    q bf16 [B, Hq, D]; k_new, v_new bf16 [B, Hkv, D]; codes uint8
    [B, Hkv, Lmax, D] and scales fp32 [B, Hkv, Lmax], updated in place;
    seq_lens int32 [B] (tokens cached before this step, not modified);
    out optional fp32 [B, Hq, D].  Returns out."""
    import torch
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    _need(k_codes, "k_codes", torch.uint8)
    if k_codes.dim() != 4 or k_codes.shape[0] != B or k_codes.shape[3] != D:
        raise ValueError("k_codes must be [B, Hkv, Lmax, D] matching q")
    Hkv, Lmax = k_codes.shape[1], k_codes.shape[2]
    _need(v_codes, "v_codes", torch.uint8, (B, Hkv, Lmax, D))
    _need(k_scale, "k_scale", torch.float32, (B, Hkv, Lmax))
    _need(v_scale, "v_scale", torch.float32, (B, Hkv, Lmax))
    _need(k_new, "k_new", torch.bfloat16, (B, Hkv, D))
    _need(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    _check(lib().gqa_decode_step_fp8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_codes),
                                     _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                     _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, Lmax,
                                     float(scale), _stream_ptr(stream)))
    return out


def check_device_error(stream=None):
    """Synchronise the stream and raise KvAttnError if the device flagged one."""
    _check(lib().kvattn_check_device_error(_stream_ptr(stream)))


def get_plan(B, Hq, Hkv, D, Lmax, num_sms=0) -> dict:
    p = kvattn_plan()
    _check(lib().kvattn_get_plan(B, Hq, Hkv, D, Lmax, num_sms, ctypes.byref(p)))
    return {name: getattr(p, name) for name, _ in kvattn_plan._fields_}


def set_tuning(force_path: int = 0, num_ctas: int = 0):
    _check(lib().kvattn_set_tuning(force_path, num_ctas))


def set_wait_limit(polls: int = 0):
    """Test knob: polls before the tensor-core kernel's pipeline waits give
    up (0 restores the default); see kvattn_set_wait_limit."""
    _check(lib().kvattn_set_wait_limit(int(polls)))


def set_kernel_events(before=None, after=None):
    """Measurement hook: record these torch.cuda.Event objects just before
    and just after the split-KV kernel of every later attention call (None,
    None stops).  The events must have been created (recorded once) first."""
    if (before is None) != (after is None):
        raise ValueError("give both events or neither")
    b = before.cuda_event if before is not None else None
    a = after.cuda_event if after is not None else None
    if before is not None and (not b or not a):
        raise ValueError("record each event once before handing it over (torch creates it lazily)")
    _check(lib().kvattn_set_kernel_events(b, a))


def release():
    lib().kvattn_release()
