"""CPU oracle for decode attention over a grouped-query KV cache.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product library
never imports this package, and this package imports nothing from the
product.  The arithmetic lives in ``kvattn_oracle.c`` (plain C, double
precision); this module only compiles it with gcc and marshals numpy arrays.

What is computed and which passages it follows is documented at the top of
``kvattn_oracle.c``.  Every function here is pinned by ``tests/test_oracle_*``
(closed forms, a library special case, brute force and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvattn_oracle.c")
_LIB = os.path.join(_HERE, "libkvattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (a second or so). Returns the .so path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add, every product rounds to double
    # before the sum, as written in the source.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_kv_append.restype = ctypes.c_int
    lib.oracle_kv_append.argtypes = [u16p, u16p, u16p, u16p, i32p,
                                     i64, i64, i64, i64]
    lib.oracle_gqa_decode.restype = ctypes.c_int
    lib.oracle_gqa_decode.argtypes = [u16p, u16p, u16p, i32p, f64p,
                                      i64, i64, i64, i64, i64,
                                      ctypes.c_double, ctypes.c_int]
    lib.oracle_gqa_decode_window.restype = ctypes.c_int
    lib.oracle_gqa_decode_window.argtypes = [u16p, u16p, u16p, i32p, f64p,
                                             i64, i64, i64, i64, i64,
                                             ctypes.c_double, i64, ctypes.c_int]
    lib.oracle_gqa_decode_multi.restype = ctypes.c_int
    lib.oracle_gqa_decode_multi.argtypes = [u16p, u16p, u16p, i32p, f64p,
                                            i64, i64, i64, i64, i64, i64,
                                            ctypes.c_double, ctypes.c_int]
    lib.oracle_gqa_decode_pairs.restype = ctypes.c_int
    lib.oracle_gqa_decode_pairs.argtypes = [u16p, u16p, u16p, i32p, f64p,
                                            i64, i64, i64, i64, i64,
                                            ctypes.c_double, i64p, i64,
                                            ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def compile_variant(src_text: str, out_dir: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    src = os.path.join(out_dir, "variant.c")
    so = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                    "-ffp-contract=off", "-fno-fast-math", "-o", so, src,
                    "-lm", "-lpthread"], check=True)
    return so


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, path=None):
        self._path = path

    @property
    def lib(self):
        if self._path is None:
            return _load()
        if not hasattr(self, "_lib"):
            self._lib = _bind(self._path)
        return self._lib

    def bf16_to_double(self, bits: int) -> float:
        """Exact widening of one bf16 bit pattern."""
        return self.lib.oracle_bf16_to_double(int(bits) & 0xFFFF)

    def kv_append(self, k_cache, v_cache, k_new, v_new, seq_lens):
        """Copy each sequence's new K/V rows into row seq_lens[b], in place.

        k_cache, v_cache: uint16 [B, Hkv, Lmax, D] (bf16 bits), in place.
        k_new, v_new:     uint16 [B, Hkv, D].
        seq_lens:         int32 [B], tokens cached before the new one.
        """
        B, Hkv, Lmax, D = k_cache.shape
        if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("caches must be C-contiguous")
        if k_cache.dtype != np.uint16 or v_cache.dtype != np.uint16:
            raise TypeError("caches must be uint16 bf16 bits")
        if v_cache.shape != k_cache.shape:
            raise ValueError("shape mismatch")
        kn, kn_p = _u16(k_new)
        vn, vn_p = _u16(v_new)
        sl, sl_p = _i32(seq_lens)
        if kn.shape != (B, Hkv, D) or vn.shape != (B, Hkv, D) or sl.shape != (B,):
            raise ValueError("shape mismatch")
        rc = self.lib.oracle_kv_append(
            k_cache.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
            v_cache.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
            kn_p, vn_p, sl_p, B, Hkv, D, Lmax)
        if rc != 0:
            raise ValueError("oracle_kv_append: seq_lens out of [0, Lmax)")

    def gqa_decode(self, q, k_cache, v_cache, seq_lens, scale, nthreads=1,
                   pairs=None, window=None):
        """softmax(scale * q . K^T) . V per query head, in double.

        q:        uint16 [B, Hq, D] (bf16 bits)
        k_cache:  uint16 [B, Hkv, Lmax, D];  v_cache the same shape
        seq_lens: int32 [B], positions [0, seq_lens[b]) take part
        pairs:    optional int64 [n, 2] list of (b, h) rows to compute; the
                  other rows of the returned array are left at zero.
        window:   optional W >= 1: only positions [max(0, len - W), len)
                  take part (a local attention layer); not with pairs.
        Returns float64 [B, Hq, D].
        """
        qa, q_p = _u16(q)
        ka, k_p = _u16(k_cache)
        va, v_p = _u16(v_cache)
        sl, sl_p = _i32(seq_lens)
        B, Hq, D = qa.shape
        Bk, Hkv, Lmax, Dk = ka.shape
        if Bk != B or Dk != D or va.shape != ka.shape or sl.shape != (B,):
            raise ValueError("shape mismatch")
        out = np.zeros((B, Hq, D), dtype=np.float64)
        out_p = out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
        if window is not None:
            if pairs is not None:
                raise ValueError("window and pairs together are not supported")
            rc = self.lib.oracle_gqa_decode_window(q_p, k_p, v_p, sl_p, out_p, B, Hq,
                                                   Hkv, D, Lmax, float(scale),
                                                   int(window), int(nthreads))
        elif pairs is None:
            rc = self.lib.oracle_gqa_decode(q_p, k_p, v_p, sl_p, out_p, B, Hq,
                                            Hkv, D, Lmax, float(scale),
                                            int(nthreads))
        else:
            pa = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
            rc = self.lib.oracle_gqa_decode_pairs(
                q_p, k_p, v_p, sl_p, out_p, B, Hq, Hkv, D, Lmax, float(scale),
                pa.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), pa.shape[0],
                int(nthreads))
        if rc != 0:
            raise ValueError("oracle_gqa_decode: bad arguments (rc=%d)" % rc)
        return out


    def gqa_decode_multi(self, q, k_cache, v_cache, seq_lens, scale, nthreads=1):
        """T new tokens per sequence, causal among themselves.

        q:        uint16 [B, T, Hq, D] (bf16 bits); token t of sequence b sits
                  at position seq_lens[b] - T + t and attends positions
                  [0, seq_lens[b] - T + 1 + t) (a zero row when that is empty)
        k_cache:  uint16 [B, Hkv, Lmax, D];  v_cache the same shape
        Returns float64 [B, T, Hq, D].
        """
        qa, q_p = _u16(q)
        ka, k_p = _u16(k_cache)
        va, v_p = _u16(v_cache)
        sl, sl_p = _i32(seq_lens)
        B, T, Hq, D = qa.shape
        Bk, Hkv, Lmax, Dk = ka.shape
        if Bk != B or Dk != D or va.shape != ka.shape or sl.shape != (B,):
            raise ValueError("shape mismatch")
        out = np.zeros((B, T, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_gqa_decode_multi(
            q_p, k_p, v_p, sl_p, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            B, T, Hq, Hkv, D, Lmax, float(scale), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_gqa_decode_multi: bad arguments (rc=%d)" % rc)
        return out


    def gather_paged(self, pool, block_table, seq_lens, block_size):
        """The contiguous cache [B, Hkv, Lmax, D] a paged cache stands for
        ("Machine Learning Engineering and AI Systems at Scale", section "The
        key and value cache": fixed-size blocks and a per-sequence block
        table that maps logical positions to physical blocks).  Position p of
        sequence b lives in row p % block_size of physical block
        block_table[b, p // block_size]; pool is [num_blocks, Hkv,
        block_size, D].  Rows past a sequence's length are left zero.
        A plain copy -- no arithmetic."""
        pool = np.ascontiguousarray(pool)
        table = np.asarray(block_table)
        lens = np.asarray(seq_lens)
        nblk, Hkv, bs, D = pool.shape
        if bs != block_size:
            raise ValueError("block_size mismatch")
        B, maxb = table.shape
        out = np.zeros((B, Hkv, maxb * bs, D), dtype=pool.dtype)
        for b in range(B):
            n = int(lens[b])
            if n < 0 or n > maxb * bs:
                raise ValueError("length outside the block table")
            for p in range(n):
                blk = int(table[b, p // bs])
                if blk < 0 or blk >= nblk:
                    raise ValueError("block index outside the pool")
                out[b, :, p] = pool[blk, :, p % bs]
        return out

    def gqa_decode_paged(self, q, k_pool, v_pool, block_table, seq_lens, block_size, scale,
                         nthreads=1):
        """Decode attention over a paged cache: the same softmax(scale q K^T) V
        over the positions the block table maps, i.e. gqa_decode on the
        gathered contiguous cache."""
        k = self.gather_paged(k_pool, block_table, seq_lens, block_size)
        v = self.gather_paged(v_pool, block_table, seq_lens, block_size)
        return self.gqa_decode(q, k, v, seq_lens, scale, nthreads=nthreads)


_default = Oracle()
bf16_to_double = _default.bf16_to_double
kv_append = _default.kv_append
gqa_decode = _default.gqa_decode
gqa_decode_multi = _default.gqa_decode_multi
gather_paged = _default.gather_paged
gqa_decode_paged = _default.gqa_decode_paged


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as its uint16 bit pattern")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
