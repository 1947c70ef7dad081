"""Python binding of libpagedattn.so (paged decode attention for GB300, sm_103a).

Argument marshalling only: every function below checks shapes and dtypes, takes
raw device pointers and the current CUDA stream from PyTorch tensors, and calls
the C function of the same name.  All arithmetic runs in the library's CUDA
kernels; there is no fallback.  If the library has not been built the first call
raises ``RuntimeError``.

Layouts match ``include/pagedattn.h``:
  k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim]  fp16 | bf16
  q, out            [num_seqs, q_len, num_q_heads, head_dim]
  k_new, v_new      [n_tokens, num_kv_heads, head_dim]
  block_tables      int32 [num_seqs, max_blocks_per_seq]
  context_lens      int32 [num_seqs]       (count this step's new tokens)
  slot_mapping      int64 [n_tokens]
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

LIBRARY = _build.LIBRARY

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_DEVICE_CHECK = -4
PA_ERR_DEVICE_TIMEOUT = -5

PA_FP16, PA_BF16 = 0, 1
_DTYPE = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16}

_c_int, _c_float, _c_size, _c_vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes): mirrors include/pagedattn.h
_SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_c_int]),
    "pa_version": (_c_int, []),
    "pa_slot_mapping": (_c_int, [_c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int, _c_vp]),
    "pa_append_kv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int,
                              _c_int, _c_int, _c_vp]),
    "pa_decode": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int,
                           _c_int, _c_int, _c_float, _c_vp, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode_partial": (_c_int, [_c_vp, _c_size, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_vp]),
    "pa_decode_combine": (_c_int, [_c_vp, _c_vp, _c_size, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_vp]),
    "pa_device_error": (_c_int, [_c_vp, _c_int]),
    "pa_selftest_wait_timeout": (_c_int, [_c_vp]),
    "pa_copy_blocks": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int,
                                _c_int, _c_int, _c_vp]),
    "pa_append_kv_fp8": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_vp, _c_vp, _c_vp]),
    "pa_decode_fp8": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                               _c_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                               _c_int, _c_int, _c_int, _c_int, _c_vp, _c_size, _c_vp]),
    "pa_append_decode": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_vp, _c_size, _c_vp]),
    "pa_decode_cascade": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_vp, _c_size, _c_vp]),
    "pa_decode_split_noalloc": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_vp]),
}

NOALLOC_SCRATCH_BYTES = 8 << 20   # PA_NOALLOC_SCRATCH_BYTES

_lock = threading.Lock()
_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Load the library (once).  Raises RuntimeError when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_20_gb300."
                                   "_build.build() (or __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _cuda(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _elt(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _DTYPE:
        raise TypeError(f"{name} must be float16 or bfloat16, got {t.dtype}")
    return _DTYPE[t.dtype]


def _cache_dims(k_cache: torch.Tensor):
    if k_cache.dim() != 4:
        raise ValueError("caches must be [num_blocks, num_kv_heads, block_size, head_dim]")
    return tuple(int(x) for x in k_cache.shape)


# ---------------------------------------------------------------------------- API
def pa_slot_mapping(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int,
                    q_len: int = 1, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Slots of each sequence's last q_len positions -> int64 [num_seqs * q_len]."""
    n, maxb = (int(x) for x in block_tables.shape)
    if out is None:
        out = torch.empty(n * q_len, dtype=torch.int64, device=block_tables.device)
    _check("pa_slot_mapping", load().pa_slot_mapping(
        _cuda(out, "out", torch.int64), _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), n, maxb, block_size, q_len,
        _stream(stream)))
    return out


def pa_append_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                 v_new: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Copy rows k_new[t], v_new[t] into slot slot_mapping[t] of the caches."""
    num_blocks, h_kv, block_size, head_dim = _cache_dims(k_cache)
    dt = _elt(k_cache, "k_cache")
    for t, nm in ((v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        if t.dtype != k_cache.dtype:
            raise TypeError(f"{nm} must have the cache dtype {k_cache.dtype}")
    n_tokens = int(slot_mapping.shape[0])
    if k_new.shape != (n_tokens, h_kv, head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [n_tokens, num_kv_heads, head_dim]")
    _check("pa_append_kv", load().pa_append_kv(
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"), _cuda(k_new, "k_new"),
        _cuda(v_new, "v_new"), _cuda(slot_mapping, "slot_mapping", torch.int64), n_tokens, h_kv,
        head_dim, block_size, num_blocks, dt, _stream(stream)))


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor,
                   dst_blocks: torch.Tensor, stream=None) -> None:
    """Copy whole blocks src_blocks[i] -> dst_blocks[i] in both caches (copy-on-write)."""
    num_blocks, h_kv, block_size, head_dim = _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("v_cache must match k_cache")
    n = int(src_blocks.shape[0])
    if int(dst_blocks.shape[0]) != n:
        raise ValueError("src_blocks and dst_blocks must have the same length")
    _check("pa_copy_blocks", load().pa_copy_blocks(
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(src_blocks, "src_blocks", torch.int32), _cuda(dst_blocks, "dst_blocks", torch.int32),
        n, h_kv, head_dim, block_size, num_blocks, _elt(k_cache, "k_cache"), _stream(stream)))


_FP8_CACHE = (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


def _fp8_cache(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _FP8_CACHE:
        raise TypeError(f"{name} must hold e4m3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    return _cuda(t, name)


def pa_append_kv_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                     v_new: torch.Tensor, slot_mapping: torch.Tensor, k_scale: torch.Tensor,
                     v_scale: torch.Tensor, stream=None) -> None:
    """Quantise 16-bit rows k_new[t], v_new[t] into slot slot_mapping[t] of FP8 caches."""
    num_blocks, h_kv, block_size, head_dim = _cache_dims(k_cache)
    n_tokens = int(slot_mapping.shape[0])
    if k_new.shape != (n_tokens, h_kv, head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [n_tokens, num_kv_heads, head_dim]")
    _check("pa_append_kv_fp8", load().pa_append_kv_fp8(
        _fp8_cache(k_cache, "k_cache"), _fp8_cache(v_cache, "v_cache"), _cuda(k_new, "k_new"),
        _cuda(v_new, "v_new"), _cuda(slot_mapping, "slot_mapping", torch.int64), n_tokens, h_kv,
        head_dim, block_size, num_blocks, _elt(k_new, "k_new"),
        _cuda(k_scale, "k_scale", torch.float32), _cuda(v_scale, "v_scale", torch.float32),
        _stream(stream)))


def pa_decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                  q_len: int = 1, num_splits: int = 1, workspace: torch.Tensor | None = None,
                  k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Attention over FP8 caches; with k_new/v_new the new rows are appended first
    (quantised, same launch).  num_splits > 1 uses the split-KV pair."""
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    kn = vn = None
    if k_new is not None or v_new is not None:
        if k_new is None or v_new is None or k_new.shape != (num_seqs * q_len, h_kv, head_dim) \
                or v_new.shape != k_new.shape or k_new.dtype != q.dtype:
            raise ValueError("k_new/v_new must both be [num_seqs * q_len, num_kv_heads, head_dim]"
                             " of q's dtype")
        kn, vn = _cuda(k_new, "k_new"), _cuda(v_new, "v_new")
    ws_ptr, ws_bytes = None, 0
    if num_splits > 1:
        if workspace is None:
            nbytes = pa_decode_workspace_size(num_seqs, h_q, q_len, head_dim, num_splits)
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        ws_ptr, ws_bytes = _cuda(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check("pa_decode_fp8", load().pa_decode_fp8(
        _cuda(out, "out"), _cuda(q, "q"), kn, vn, _fp8_cache(k_cache, "k_cache"),
        _fp8_cache(v_cache, "v_cache"), _cuda(k_scale, "k_scale", torch.float32),
        _cuda(v_scale, "v_scale", torch.float32), _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), maxb, num_blocks, q_len, _elt(q, "q"), num_splits, ws_ptr,
        ws_bytes, _stream(stream)))
    return out


def _decode_dims(q, k_cache, block_tables, context_lens, q_len):
    num_blocks, h_kv, block_size, head_dim = _cache_dims(k_cache)
    num_seqs = int(context_lens.shape[0])
    if q.dim() == 3:  # [num_seqs, num_q_heads, head_dim] with q_len == 1
        q_len_t, h_q = 1, int(q.shape[1])
    else:
        q_len_t, h_q = int(q.shape[1]), int(q.shape[2])
    if q_len_t != q_len or int(q.shape[0]) != num_seqs or int(q.shape[-1]) != head_dim:
        raise ValueError("q must be [num_seqs, q_len, num_q_heads, head_dim]")
    if block_tables.dim() != 2 or int(block_tables.shape[0]) != num_seqs:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    return num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, int(block_tables.shape[1])


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
              q_len: int = 1, stream=None) -> torch.Tensor:
    """Single-pass paged attention; writes and returns ``out`` (shape of q)."""
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out must match q; q must have the cache dtype")
    _check("pa_decode", load().pa_decode(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), _stream(stream), maxb, num_blocks, q_len,
        _elt(k_cache, "k_cache")))
    return out


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, q_len: int, head_dim: int,
                             num_splits: int) -> int:
    """Bytes of the split-KV workspace for these sizes (0 for invalid ones)."""
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, q_len, head_dim, num_splits))


def workspace_views(workspace: torch.Tensor, num_seqs: int, num_q_heads: int, q_len: int,
                    head_dim: int, num_splits: int):
    """fp32 views (acc, m, l) of a split-KV workspace, per the header's layout."""
    rows = q_len * num_q_heads
    n = num_seqs * num_splits * rows
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    acc_b, m_b = align(n * head_dim * 4), align(n * 4)
    raw = workspace.view(torch.uint8)
    acc = raw[:n * head_dim * 4].view(torch.float32).view(num_seqs, num_splits, rows, head_dim)
    m = raw[acc_b:acc_b + n * 4].view(torch.float32).view(num_seqs, num_splits, rows)
    l = raw[acc_b + m_b:acc_b + m_b + n * 4].view(torch.float32).view(num_seqs, num_splits, rows)
    return acc, m, l


def pa_decode_partial(workspace: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, num_splits: int,
                      q_len: int = 1, stream=None) -> torch.Tensor:
    """Split-KV pass: each of num_splits partitions of every sequence's blocks writes
    its (m, l, unnormalised acc) into the workspace; returns the workspace."""
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    nbytes = workspace.numel() * workspace.element_size()
    _check("pa_decode_partial", load().pa_decode_partial(
        _cuda(workspace, "workspace"), nbytes, _cuda(q, "q"), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache"), _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), num_splits, maxb, num_blocks, q_len, _elt(k_cache, "k_cache"),
        _stream(stream)))
    return workspace


def pa_decode_combine(out: torch.Tensor, workspace: torch.Tensor, num_splits: int,
                      stream=None) -> torch.Tensor:
    """out: [num_seqs, q_len, num_q_heads, head_dim] (or 3-D with q_len 1)."""
    if out.dim() == 3:
        num_seqs, q_len, h_q, head_dim = int(out.shape[0]), 1, int(out.shape[1]), int(out.shape[2])
    else:
        num_seqs, q_len, h_q, head_dim = (int(x) for x in out.shape)
    nbytes = workspace.numel() * workspace.element_size()
    _check("pa_decode_combine", load().pa_decode_combine(
        _cuda(out, "out"), _cuda(workspace, "workspace"), nbytes, num_seqs, h_q, head_dim, q_len,
        num_splits, _elt(out, "out"), _stream(stream)))
    return out


def pa_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (sets PA_ERR_DEVICE_TIMEOUT after ~2 s)."""
    _check("pa_selftest_wait_timeout", load().pa_selftest_wait_timeout(_stream(stream)))


def pa_device_error(stream=None, clear: bool = True) -> int:
    """Synchronise the stream; return the device error status (PA_OK == 0)."""
    return int(load().pa_device_error(_stream(stream), 1 if clear else 0))


def pa_append_decode(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor,
                     v_new: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                     q_len: int = 1, num_splits: int = 1, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Fused step: slot mapping + append of k_new/v_new + attention (one launch)."""
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out must match q; q must have the cache dtype")
    if k_new.shape != (num_seqs * q_len, h_kv, head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_seqs * q_len, num_kv_heads, head_dim]")
    for t, nm in ((k_new, "k_new"), (v_new, "v_new"), (v_cache, "v_cache")):
        if t.dtype != k_cache.dtype:
            raise TypeError(f"{nm} must have the cache dtype {k_cache.dtype}")
    ws_ptr, ws_bytes = None, 0
    if num_splits > 1:
        if workspace is None:
            nbytes = pa_decode_workspace_size(num_seqs, h_q, q_len, head_dim, num_splits)
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        ws_ptr, ws_bytes = _cuda(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check("pa_append_decode", load().pa_append_decode(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_new, "k_new"), _cuda(v_new, "v_new"),
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), maxb, num_blocks, q_len, _elt(k_cache, "k_cache"), num_splits,
        ws_ptr, ws_bytes, _stream(stream)))
    return out


def pa_decode_cascade(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, prefix_blocks: int,
                      q_len: int = 1, tail_splits: int = 1, k_new: torch.Tensor | None = None,
                      v_new: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Attention of a batch sharing its first ``prefix_blocks`` blocks (block-table row
    0): one pass over the shared prefix for all rows, one over each sequence's own
    blocks (with the append of k_new/v_new when given), then the combine."""
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out must match q; q must have the cache dtype")
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new, or neither")
    if k_new is not None:
        if k_new.shape != (num_seqs * q_len, h_kv, head_dim) or v_new.shape != k_new.shape:
            raise ValueError("k_new/v_new must be [num_seqs * q_len, num_kv_heads, head_dim]")
        for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
            if t.dtype != k_cache.dtype:
                raise TypeError(f"{nm} must have the cache dtype {k_cache.dtype}")
    if workspace is None:
        nbytes = pa_decode_workspace_size(num_seqs, h_q, q_len, head_dim, 1 + tail_splits)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("pa_decode_cascade", load().pa_decode_cascade(
        _cuda(out, "out"), _cuda(q, "q"),
        None if k_new is None else _cuda(k_new, "k_new"),
        None if v_new is None else _cuda(v_new, "v_new"),
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), maxb, num_blocks, q_len, _elt(k_cache, "k_cache"),
        int(prefix_blocks), int(tail_splits), _cuda(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, q_len: int = 1,
                      num_splits: int = 1, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None,
                      slot_mapping: torch.Tensor | None = None, stream=None,
                      fused: bool = False) -> torch.Tensor:
    """One decode step: slot mapping, KV append, then attention.

    fused=False runs pa_slot_mapping -> pa_append_kv -> pa_decode (num_splits == 1)
    or pa_decode_partial + pa_decode_combine (num_splits > 1) on one stream;
    fused=True runs the same step as pa_append_decode (one launch, two with splits).
    Optional ``out``, ``workspace`` and ``slot_mapping`` buffers are reused when
    given (no allocation on the hot path).
    """
    if fused:
        if out is None:
            out = torch.empty_like(q)
        return pa_append_decode(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                context_lens, scale, q_len, num_splits, workspace, stream)
    block_size = int(k_cache.shape[2])
    slot_mapping = pa_slot_mapping(block_tables, context_lens, block_size, q_len,
                                   out=slot_mapping, stream=stream)
    pa_append_kv(k_cache, v_cache, k_new, v_new, slot_mapping, stream=stream)
    if out is None:
        out = torch.empty_like(q)
    if num_splits <= 1:
        return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, q_len,
                         stream=stream)
    if workspace is None:
        num_seqs, h_q, head_dim = int(q.shape[0]), int(q.shape[-2]), int(q.shape[-1])
        nbytes = pa_decode_workspace_size(num_seqs, h_q, q_len, head_dim, num_splits)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    pa_decode_partial(workspace, q, k_cache, v_cache, block_tables, context_lens, scale,
                      num_splits, q_len, stream=stream)
    return pa_decode_combine(out, workspace, num_splits, stream=stream)


def pa_decode_split_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, scale: float, num_splits: int,
                            q_len: int = 1, stream=None) -> torch.Tensor:
    """Split-KV attention whose workspace is the library's fixed device array.

    For callers that may not allocate device memory at this point; no tensor is
    allocated here either.  Raises PagedAttnError (PA_ERR_INVALID_ARG) when the
    workspace this call needs exceeds NOALLOC_SCRATCH_BYTES.  Calls that can run
    concurrently on one GPU share the array and must be ordered by the caller.
    """
    num_blocks, h_kv, block_size, head_dim, num_seqs, h_q, maxb = _decode_dims(
        q, k_cache, block_tables, context_lens, q_len)
    if out.shape != q.shape or out.dtype != q.dtype or q.dtype != k_cache.dtype:
        raise ValueError("out must match q; q must have the cache dtype")
    _check("pa_decode_split_noalloc", load().pa_decode_split_noalloc(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(block_tables, "block_tables", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), num_seqs, h_q, h_kv, head_dim,
        block_size, float(scale), num_splits, maxb, num_blocks, q_len, _elt(k_cache, "k_cache"),
        _stream(stream)))
    return out
