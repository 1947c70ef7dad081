"""The allocation-free split-KV entry point (pa_decode_split_noalloc), on a GPU.

Its workspace is a fixed device array inside the library, for callers that
cannot allocate device memory where they run attention.  It must give what the
caller-workspace pair pa_decode_partial + pa_decode_combine gives, call after
call (the array keeps the previous call's contents), and refuse sizes beyond the
array.  This file sorts last so that a run stopping at its first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests import _tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    return pa


def _inputs(name, **over):
    w = workloads.make(name, **over)
    d = {k: getattr(w, k).to(DEV) for k in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                            "block_tables", "context_lens")}
    return w, d


def _noalloc_via_abi(pa, w, d, out, num_splits):
    """Call the C entry point directly through ctypes (the C ABI)."""
    c = w.cfg
    lib = pa.load()
    return lib.pa_decode_split_noalloc(
        out.data_ptr(), d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_tables"].data_ptr(), d["context_lens"].data_ptr(), c.num_seqs, c.num_q_heads,
        c.num_kv_heads, c.head_dim, c.block_size, ctypes.c_float(w.scale), num_splits,
        w.max_blocks_per_seq, w.num_blocks, c.q_len, 0 if c.dtype == "fp16" else 1,
        torch.cuda.current_stream().cuda_stream)


def _with_workspace(pa, w, d, num_splits):
    c = w.cfg
    nbytes = pa.pa_decode_workspace_size(c.num_seqs, c.num_q_heads, c.q_len, c.head_dim,
                                         num_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])
    pa.pa_decode_partial(ws, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                         d["context_lens"], w.scale, num_splits, c.q_len)
    pa.pa_decode_combine(out, ws, num_splits)
    return out


def test_noalloc_matches_workspace_pair_two_calls_in_a_row(pa):
    cases = [
        ("long_split", {"num_seqs": 2, "lens": ("fixed", (20000, 7000))}, 16),
        ("prefix_verify", {"num_seqs": 3}, 5),
    ]
    for name, over, splits in cases:
        w, d = _inputs(name, **over)
        c = w.cfg
        slots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], c.block_size, c.q_len)
        pa.pa_append_kv(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], slots)
        want = _with_workspace(pa, w, d, splits)
        for call in range(2):
            out = torch.full_like(d["q"], float("nan"))
            assert _noalloc_via_abi(pa, w, d, out, splits) == pa.PA_OK
            torch.cuda.synchronize()
            got = out.cpu().double().numpy()
            _tol.check(got, want.cpu().double().numpy(), c.dtype, f"{name} call {call}")
            assert torch.equal(out, want)
        # the Python binding of the same entry point
        out = torch.full_like(d["q"], float("nan"))
        pa.pa_decode_split_noalloc(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                   d["context_lens"], w.scale, splits, q_len=c.q_len)
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert pa.pa_device_error() == pa.PA_OK


def test_noalloc_refuses_sizes_beyond_its_array(pa):
    w, d = _inputs("llama7b_mha", num_seqs=32)
    c = w.cfg
    need = pa.pa_decode_workspace_size(c.num_seqs, c.num_q_heads, c.q_len, c.head_dim, 64)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(d["q"])
    assert _noalloc_via_abi(pa, w, d, out, 64) == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0          # nothing was launched
    # the binding raises the library's status and leaves out untouched
    with pytest.raises(pa.PagedAttnError) as exc:
        pa.pa_decode_split_noalloc(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                   d["context_lens"], w.scale, 64, q_len=c.q_len)
    assert exc.value.status == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0
