"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package imports nothing from the product.  The arithmetic lives in ``pa_oracle.c``
(plain C, IEEE double); this module only marshals numpy arrays through ctypes.

Every array argument is a numpy array; 16-bit floating-point tensors (q, caches,
new rows) are passed as their raw ``uint16`` bit patterns, so both fp16 and bf16
take the same route and the oracle decodes them itself from the format
definitions.

Layouts (row-major):
  q            [num_seqs, q_len, num_q_heads, head_dim]
  k/v cache    [num_blocks, num_kv_heads, block_size, head_dim]
  k/v new      [n_tokens, num_kv_heads, head_dim]
  block_tables [num_seqs, max_blocks_per_seq] int32
  context_lens [num_seqs] int32 (they already count this step's new tokens)
"""
from __future__ import annotations

import ctypes
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

DTYPES = {"fp16": 0, "bf16": 1}

_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_u16p = ctypes.POINTER(ctypes.c_uint16)
_c_f64p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctype)


def _run_rows(run, n: int, threads: int) -> list:
    """run(lo, hi) over [0, n), in slices over a thread pool when threads > 1 (the
    C calls release the interpreter lock); returns the status codes."""
    if threads <= 1 or n < 2:
        return [run(0, n)]
    bounds = np.linspace(0, n, min(n, threads * 4) + 1).astype(int)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a
    if a.dtype in (np.int16, np.float16):
        return a.view(np.uint16)
    raise TypeError(f"expected 16-bit pattern array, got {a.dtype}")


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return DTYPES[dtype]


class Oracle:
    """ctypes wrapper around one compiled copy of ``pa_oracle.c``."""

    def __init__(self, path: str = _build.LIBRARY):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.orc_fp16_to_double.restype = ctypes.c_double
        lib.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_decode_bits.restype = None
        lib.orc_decode_bits.argtypes = [_c_f64p, _c_u16p, ctypes.c_int64, ctypes.c_int]
        lib.orc_slot_mapping.restype = ctypes.c_int
        lib.orc_slot_mapping.argtypes = [_c_i64p, _c_i32p, _c_i32p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int]
        lib.orc_append_kv.restype = None
        lib.orc_append_kv.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _c_u8p = ctypes.POINTER(ctypes.c_uint8)
        _c_f32p = ctypes.POINTER(ctypes.c_float)
        lib.orc_decode_e4m3.restype = None
        lib.orc_decode_e4m3.argtypes = [_c_f64p, _c_u8p, ctypes.c_int64]
        lib.orc_encode_e4m3.restype = None
        lib.orc_encode_e4m3.argtypes = [_c_u8p, _c_f32p, ctypes.c_int64]
        lib.orc_append_kv_fp8.restype = None
        lib.orc_append_kv_fp8.argtypes = [_c_u8p, _c_u8p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _c_f32p, _c_f32p]
        lib.orc_decode_fp8.restype = ctypes.c_int
        lib.orc_decode_fp8.argtypes = [_c_f64p, _c_i64p, ctypes.c_int64, _c_u16p, _c_u8p, _c_u8p,
                                       _c_f32p, _c_f32p, _c_i32p, _c_i32p, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        self._u8p, self._f32p = _c_u8p, _c_f32p
        lib.orc_copy_blocks.restype = ctypes.c_int
        lib.orc_copy_blocks.argtypes = [_c_u16p, _c_u16p, _c_i32p, _c_i32p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_decode.restype = ctypes.c_int
        lib.orc_decode.argtypes = [_c_f64p, _c_i64p, ctypes.c_int64, _c_u16p, _c_u16p, _c_u16p,
                                   _c_i32p, _c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int]
        lib.orc_decode_partitions.restype = ctypes.c_int
        lib.orc_decode_partitions.argtypes = [_c_f64p, _c_f64p, _c_f64p, _c_u16p, _c_u16p,
                                              _c_u16p, _c_i32p, _c_i32p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_combine.restype = None
        lib.orc_combine.argtypes = [_c_f64p, _c_f64p, _c_f64p, _c_f64p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int64, ctypes.c_int]
        self.lib = lib

    # -- element decoding -------------------------------------------------------
    def decode_bits(self, bits: np.ndarray, dtype) -> np.ndarray:
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.orc_decode_bits(_ptr(out, _c_f64p), _ptr(b, _c_u16p), b.size, _dtype_code(dtype))
        return out

    # -- slot mapping -----------------------------------------------------------
    def slot_mapping(self, block_tables: np.ndarray, context_lens: np.ndarray,
                     block_size: int, q_len: int = 1) -> np.ndarray:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        n = cl.shape[0]
        out = np.empty(n * q_len, dtype=np.int64)
        rc = self.lib.orc_slot_mapping(_ptr(out, _c_i64p), _ptr(bt, _c_i32p), _ptr(cl, _c_i32p),
                                       n, bt.shape[1], block_size, q_len)
        if rc != 0:
            raise ValueError("a new token's position lies beyond the block table")
        return out

    # -- append (in place) ------------------------------------------------------
    def append_kv(self, k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                  v_new: np.ndarray, slot_mapping: np.ndarray) -> None:
        for a in (k_cache, v_cache):
            if not (a.flags.c_contiguous and a.dtype in (np.uint16, np.int16, np.float16)):
                raise TypeError("caches must be contiguous 16-bit arrays (modified in place)")
        kc, vc = k_cache.view(np.uint16), v_cache.view(np.uint16)
        kn, vn = _u16(k_new), _u16(v_new)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        _, h_kv, block_size, head_dim = kc.shape
        self.lib.orc_append_kv(_ptr(kc, _c_u16p), _ptr(vc, _c_u16p), _ptr(kn, _c_u16p),
                               _ptr(vn, _c_u16p), _ptr(sm, _c_i64p), sm.shape[0], h_kv,
                               head_dim, block_size)

    # -- FP8 (e4m3) -------------------------------------------------------------
    def decode_e4m3(self, codes: np.ndarray) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.orc_decode_e4m3(_ptr(out, _c_f64p), _ptr(c, self._u8p), c.size)
        return out

    def encode_e4m3(self, x: np.ndarray) -> np.ndarray:
        f = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(f.shape, dtype=np.uint8)
        self.lib.orc_encode_e4m3(_ptr(out, self._u8p), _ptr(f, self._f32p), f.size)
        return out

    def append_kv_fp8(self, k_cache: np.ndarray, v_cache: np.ndarray, k_new, v_new,
                      slot_mapping, new_dtype, k_scale, v_scale) -> None:
        """Quantising append into uint8 e4m3 caches [P, H, B, D] (in place)."""
        for a in (k_cache, v_cache):
            if not (a.flags.c_contiguous and a.dtype == np.uint8):
                raise TypeError("FP8 caches must be contiguous uint8 arrays (modified in place)")
        kn, vn = _u16(k_new), _u16(v_new)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        _, h_kv, block_size, head_dim = k_cache.shape
        self.lib.orc_append_kv_fp8(_ptr(k_cache, self._u8p), _ptr(v_cache, self._u8p),
                                   _ptr(kn, _c_u16p), _ptr(vn, _c_u16p), _ptr(sm, _c_i64p),
                                   sm.shape[0], h_kv, head_dim, block_size,
                                   _dtype_code(new_dtype), _ptr(ks, self._f32p),
                                   _ptr(vs, self._f32p))

    def decode_fp8(self, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                   scale: float, dtype, q_len: int = 1, rows=None, threads: int = 1) -> np.ndarray:
        """fp64 attention over e4m3 caches (value = code * per-KV-head scale).
        ``threads`` > 1 splits the rows over a thread pool (each row is computed on
        its own, so the result does not depend on the split)."""
        qb = _u16(q)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        _, h_kv, block_size, head_dim = kc.shape
        h_q = qb.size // (num_seqs * q_len * head_dim)
        rows_arr = (np.arange(num_seqs * q_len * h_q, dtype=np.int64) if rows is None
                    else np.ascontiguousarray(rows, dtype=np.int64))
        out = np.empty((rows_arr.shape[0], head_dim), dtype=np.float64)

        def run(lo: int, hi: int) -> int:
            sub = rows_arr[lo:hi]
            return self.lib.orc_decode_fp8(_ptr(out[lo:hi], _c_f64p), _ptr(sub, _c_i64p), hi - lo,
                                           _ptr(qb, _c_u16p), _ptr(kc, self._u8p),
                                           _ptr(vc, self._u8p), _ptr(ks, self._f32p),
                                           _ptr(vs, self._f32p), _ptr(bt, _c_i32p),
                                           _ptr(cl, _c_i32p), num_seqs, h_q, h_kv, head_dim,
                                           block_size, float(scale), bt.shape[1], q_len,
                                           _dtype_code(dtype))

        rcs = _run_rows(run, rows_arr.shape[0], threads)
        if any(rc != 0 for rc in rcs):
            raise ValueError(f"oracle fp8 decode failed: {rcs}")
        return out.reshape(qb.shape) if rows is None else out

    # -- copy-on-write block copy (in place) ------------------------------------
    def copy_blocks(self, k_cache: np.ndarray, v_cache: np.ndarray, src, dst) -> int:
        kc, vc = k_cache.view(np.uint16), v_cache.view(np.uint16)
        s = np.ascontiguousarray(src, dtype=np.int32)
        d = np.ascontiguousarray(dst, dtype=np.int32)
        num_blocks, h_kv, block_size, head_dim = kc.shape
        return self.lib.orc_copy_blocks(_ptr(kc, _c_u16p), _ptr(vc, _c_u16p), _ptr(s, _c_i32p),
                                        _ptr(d, _c_i32p), s.shape[0], h_kv, head_dim, block_size,
                                        num_blocks)

    # -- attention --------------------------------------------------------------
    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
               dtype, q_len: int = 1, rows=None, threads: int = 1) -> np.ndarray:
        """fp64 attention output.

        ``q`` is [num_seqs, q_len, num_q_heads, head_dim] (or [num_seqs, num_q_heads,
        head_dim] when q_len == 1).  Without ``rows`` the result has q's shape; with
        ``rows`` (flat output-row indices r = (seq*q_len + u)*num_q_heads + head) it
        is [len(rows), head_dim].
        """
        qb = _u16(q)
        kc, vc = _u16(k_cache), _u16(v_cache)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        _, h_kv, block_size, head_dim = kc.shape
        h_q = qb.size // (num_seqs * q_len * head_dim)
        if rows is None:
            rows_arr = np.arange(num_seqs * q_len * h_q, dtype=np.int64)
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows_arr.shape[0], head_dim), dtype=np.float64)

        def run(lo: int, hi: int) -> int:
            sub = rows_arr[lo:hi]
            o = out[lo:hi]
            return self.lib.orc_decode(_ptr(o, _c_f64p), _ptr(sub, _c_i64p), hi - lo,
                                       _ptr(qb, _c_u16p), _ptr(kc, _c_u16p), _ptr(vc, _c_u16p),
                                       _ptr(bt, _c_i32p), _ptr(cl, _c_i32p), num_seqs, h_q, h_kv,
                                       head_dim, block_size, float(scale), bt.shape[1], q_len,
                                       _dtype_code(dtype))

        rcs = _run_rows(run, rows_arr.shape[0], threads)
        if any(rc != 0 for rc in rcs):
            raise ValueError(f"oracle decode failed: {rcs}")
        if rows is None:
            return out.reshape(qb.shape)
        return out

    def decode_partitions(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                          dtype, num_splits: int, q_len: int = 1):
        """Per-partition (m, l, acc), natural-log domain, fp64.

        m, l: [num_seqs, num_splits, q_len*num_q_heads]; acc: same + [head_dim].
        """
        qb = _u16(q)
        kc, vc = _u16(k_cache), _u16(v_cache)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        _, h_kv, block_size, head_dim = kc.shape
        h_q = qb.size // (num_seqs * q_len * head_dim)
        rps = q_len * h_q
        m = np.empty((num_seqs, num_splits, rps), dtype=np.float64)
        l = np.empty_like(m)
        acc = np.empty((num_seqs, num_splits, rps, head_dim), dtype=np.float64)
        rc = self.lib.orc_decode_partitions(_ptr(m, _c_f64p), _ptr(l, _c_f64p), _ptr(acc, _c_f64p),
                                            _ptr(qb, _c_u16p), _ptr(kc, _c_u16p), _ptr(vc, _c_u16p),
                                            _ptr(bt, _c_i32p), _ptr(cl, _c_i32p), num_seqs, h_q,
                                            h_kv, head_dim, block_size, float(scale), bt.shape[1],
                                            q_len, _dtype_code(dtype), num_splits)
        if rc != 0:
            raise ValueError(f"oracle partitions failed: {rc}")
        return m, l, acc

    def combine(self, m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        acc = np.ascontiguousarray(acc, dtype=np.float64)
        num_seqs, num_splits, rps, head_dim = acc.shape
        out = np.empty((num_seqs, rps, head_dim), dtype=np.float64)
        self.lib.orc_combine(_ptr(out, _c_f64p), _ptr(m, _c_f64p), _ptr(l, _c_f64p),
                             _ptr(acc, _c_f64p), num_seqs, num_splits, rps, head_dim)
        return out


_lock = threading.Lock()
_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            if _build.needs_build():
                _build.build()
            _default = Oracle()
        return _default


def load(path: str) -> Oracle:
    """Load another compiled copy (e.g. a deliberately altered one in a test)."""
    return Oracle(os.path.abspath(path))
