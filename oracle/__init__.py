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
    lib.oracle_gqa_decode_multi_window.restype = ctypes.c_int
    lib.oracle_gqa_decode_multi_window.argtypes = [u16p, u16p, u16p, i32p, f64p,
                                                   i64, i64, i64, i64, i64, i64,
                                                   ctypes.c_double, i64, ctypes.c_int]
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_e4m3_encode_n.restype = None
    lib.oracle_e4m3_encode_n.argtypes = [f32p, u8p, i64]
    lib.oracle_e4m3_decode_n.restype = None
    lib.oracle_e4m3_decode_n.argtypes = [u8p, f64p, i64]
    lib.oracle_quantize_fp8.restype = None
    lib.oracle_quantize_fp8.argtypes = [u16p, u8p, f32p, i64, i64]
    lib.oracle_kv_append_fp8.restype = ctypes.c_int
    lib.oracle_kv_append_fp8.argtypes = [u8p, u8p, f32p, f32p, u16p, u16p, i32p,
                                         i64, i64, i64, i64]
    lib.oracle_gqa_decode_fp8.restype = ctypes.c_int
    lib.oracle_gqa_decode_fp8.argtypes = [u16p, u8p, u8p, f32p, f32p, i32p, f64p,
                                          i64, i64, i64, i64, i64, ctypes.c_double,
                                          ctypes.c_int]
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


    def gqa_decode_multi(self, q, k_cache, v_cache, seq_lens, scale, nthreads=1,
                         window=None):
        """T new tokens per sequence, causal among themselves.

        q:        uint16 [B, T, Hq, D] (bf16 bits); token t of sequence b sits
                  at position seq_lens[b] - T + t and attends positions
                  [0, e) with e = seq_lens[b] - T + 1 + t (a zero row when
                  that is empty)
        k_cache:  uint16 [B, Hkv, Lmax, D];  v_cache the same shape
        window:   optional W >= 1: token t attends only [max(0, e - W), e)
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
        out_p = out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
        if window is None:
            rc = self.lib.oracle_gqa_decode_multi(q_p, k_p, v_p, sl_p, out_p, B, T, Hq, Hkv,
                                                  D, Lmax, float(scale), int(nthreads))
        else:
            rc = self.lib.oracle_gqa_decode_multi_window(q_p, k_p, v_p, sl_p, out_p, B, T,
                                                         Hq, Hkv, D, Lmax, float(scale),
                                                         int(window), int(nthreads))
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
                         nthreads=1, window=None):
        """Decode attention over a paged cache: the same softmax(scale q K^T) V
        over the positions the block table maps, i.e. gqa_decode (q [B, Hq,
        D]) or gqa_decode_multi (q [B, T, Hq, D]) on the gathered contiguous
        cache, with the same optional local window."""
        k = self.gather_paged(k_pool, block_table, seq_lens, block_size)
        v = self.gather_paged(v_pool, block_table, seq_lens, block_size)
        if np.asarray(q).ndim == 4:
            return self.gqa_decode_multi(q, k, v, seq_lens, scale, nthreads=nthreads,
                                         window=window)
        return self.gqa_decode(q, k, v, seq_lens, scale, nthreads=nthreads, window=window)


    # ------------------------------------------------------------ 8-bit cache
    # ("The Basics of Transformer Inference", item "Quantization"; "Machine
    # Learning Engineering and AI Systems at Scale", section "Quantization":
    # FP8 E4M3; the rule itself is the reading in kvattn_oracle.c's header)

    def e4m3_encode(self, x):
        """float32 values -> E4M3 codes (nearest, ties to even, saturating)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.oracle_e4m3_encode_n(x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                      x.size)
        return out

    def e4m3_decode(self, codes):
        """E4M3 codes -> float64 values (exact)."""
        c, c_p = _u8(codes)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.oracle_e4m3_decode_n(c_p, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                      c.size)
        return out

    def quantize_fp8(self, rows):
        """bf16 bits [..., D] -> (codes uint8 [..., D], scales float32 [...]):
        one scale per row of D values."""
        r, r_p = _u16(rows)
        D = r.shape[-1]
        n = r.size // D if D else 0
        codes = np.empty(r.shape, dtype=np.uint8)
        scales = np.empty(r.shape[:-1], dtype=np.float32)
        self.lib.oracle_quantize_fp8(r_p, codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                     scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, D)
        return codes, scales

    def dequantize_fp8(self, codes, scales):
        """codes [..., D] and scales [...] -> float64 values, code * scale."""
        return self.e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]

    def kv_append_fp8(self, k_codes, v_codes, k_scale, v_scale, k_new, v_new, seq_lens):
        """Quantize each sequence's new K/V rows into position seq_lens[b] of
        an 8-bit cache, in place (codes uint8 [B, Hkv, Lmax, D], scales
        float32 [B, Hkv, Lmax]; k_new, v_new bf16 bits [B, Hkv, D])."""
        B, Hkv, Lmax, D = k_codes.shape
        for a, dt in ((k_codes, np.uint8), (v_codes, np.uint8), (k_scale, np.float32),
                      (v_scale, np.float32)):
            if a.dtype != dt or not a.flags.c_contiguous:
                raise TypeError("8-bit cache arrays must be contiguous uint8 / float32")
        if v_codes.shape != k_codes.shape or k_scale.shape != (B, Hkv, Lmax) or \
                v_scale.shape != (B, Hkv, Lmax):
            raise ValueError("shape mismatch")
        kn, kn_p = _u16(k_new)
        vn, vn_p = _u16(v_new)
        sl, sl_p = _i32(seq_lens)
        if kn.shape != (B, Hkv, D) or vn.shape != (B, Hkv, D) or sl.shape != (B,):
            raise ValueError("shape mismatch")
        u8 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))  # noqa: E731
        f32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))  # noqa: E731
        rc = self.lib.oracle_kv_append_fp8(u8(k_codes), u8(v_codes), f32(k_scale), f32(v_scale),
                                           kn_p, vn_p, sl_p, B, Hkv, D, Lmax)
        if rc != 0:
            raise ValueError("oracle_kv_append_fp8: length outside [0, Lmax)")

    def gqa_decode_fp8(self, q, k_codes, v_codes, k_scale, v_scale, seq_lens, scale,
                       nthreads=1):
        """gqa_decode over an 8-bit cache: K = e4m3(code) * k_scale per row,
        V likewise, in double.  q bf16 bits [B, Hq, D]; codes uint8
        [B, Hkv, Lmax, D]; scales float32 [B, Hkv, Lmax].  Returns float64
        [B, Hq, D]."""
        qq, q_p = _u16(q)
        kc, kc_p = _u8(k_codes)
        vc, vc_p = _u8(v_codes)
        ks, ks_p = _f32(k_scale)
        vs, vs_p = _f32(v_scale)
        sl, sl_p = _i32(seq_lens)
        B, Hq, D = qq.shape
        Hkv, Lmax = kc.shape[1], kc.shape[2]
        if kc.shape != (B, Hkv, Lmax, D) or vc.shape != kc.shape or \
                ks.shape != (B, Hkv, Lmax) or vs.shape != ks.shape or sl.shape != (B,):
            raise ValueError("shape mismatch")
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_gqa_decode_fp8(q_p, kc_p, vc_p, ks_p, vs_p, sl_p,
                                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                            B, Hq, Hkv, D, Lmax, float(scale), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_gqa_decode_fp8: bad arguments (heads or lengths)")
        return out


_default = Oracle()
bf16_to_double = _default.bf16_to_double
kv_append = _default.kv_append
gqa_decode = _default.gqa_decode
gqa_decode_multi = _default.gqa_decode_multi
gather_paged = _default.gather_paged
e4m3_encode = _default.e4m3_encode
e4m3_decode = _default.e4m3_decode
quantize_fp8 = _default.quantize_fp8
dequantize_fp8 = _default.dequantize_fp8
kv_append_fp8 = _default.kv_append_fp8
gqa_decode_fp8 = _default.gqa_decode_fp8
gqa_decode_paged = _default.gqa_decode_paged


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("E4M3 codes must be uint8")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _f32(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError("scales must be float32")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as its uint16 bit pattern")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
