"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
function declared in include/*.h, and rejects bad arguments before any launch."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_20_gb300 import _build
    import paged_kv_cache_20_gb300 as pa
    if _build.needs_build():
        _build.build()
    return pa.load()


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_api():
    names = _declared()
    for want in ("pa_append_kv", "pa_decode", "pa_decode_partial", "pa_decode_combine",
                 "pa_decode_workspace_size", "pa_slot_mapping", "pa_status_string",
                 "pa_device_error", "pa_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_only_api_symbols_exported(lib):
    # hidden visibility: nothing else from the library's own code leaks out
    import subprocess
    from paged_kv_cache_20_gb300 import _build
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIBRARY], capture_output=True,
                         text=True).stdout
    ours = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in ours if s.startswith("pa_")}
    assert ours == set(_declared())


def test_status_strings(lib):
    import paged_kv_cache_20_gb300 as pa
    for code, name in ((0, "PA_OK"), (-1, "PA_ERR_INVALID_ARG"), (-2, "PA_ERR_UNSUPPORTED"),
                       (-3, "PA_ERR_CUDA"), (-4, "PA_ERR_DEVICE_CHECK"),
                       (-5, "PA_ERR_DEVICE_TIMEOUT")):
        assert pa.status_string(code) == name
    assert pa.status_string(7) == "PA_UNKNOWN_STATUS"
    assert lib.pa_version() == 100


def test_workspace_size_layout(lib):
    import paged_kv_cache_20_gb300 as pa
    n, h, ql, d, s = 4, 32, 1, 128, 16
    rows = n * s * ql * h
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert pa.pa_decode_workspace_size(n, h, ql, d, s) == al(rows * d * 4) + 2 * al(rows * 4)
    assert pa.pa_decode_workspace_size(0, h, ql, d, s) == 0
    assert pa.pa_decode_workspace_size(n, h, ql, d, 0) == 0


FAKE = 0x10000  # 16-byte-aligned non-null address; every call below returns before using it


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, n=2, hq=8, hkv=2, d=128, bs=16,
             scale=0.1, stream=None, maxb=4, nblocks=8, qlen=1, dtype=0)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["n"], a["hq"],
                         a["hkv"], a["d"], a["bs"], a["scale"], a["stream"], a["maxb"],
                         a["nblocks"], a["qlen"], a["dtype"])


@pytest.mark.parametrize("kw,status", [
    ({"out": None}, -1), ({"q": None}, -1), ({"k": None}, -1), ({"bt": None}, -1),
    ({"n": 0}, -1), ({"hq": 6, "hkv": 4}, -1), ({"hkv": 0}, -1), ({"qlen": 0}, -1),
    ({"maxb": 0}, -1), ({"nblocks": -1}, -1), ({"q": FAKE + 2}, -1), ({"out": FAKE + 8}, -1),
    ({"scale": float("nan")}, -1), ({"d": 96}, -2), ({"d": 256}, -2), ({"bs": 24}, -2), ({"bs": 4}, -2),
    ({"qlen": 4097}, -2), ({"dtype": 5}, -2), ({"nblocks": 1 << 30, "hkv": 4, "hq": 4}, -1),
])
def test_decode_rejects_bad_arguments(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_partial_and_combine_reject_bad_arguments(lib):
    ws_ok = lib.pa_decode_workspace_size(2, 8, 1, 128, 4)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 0.1]
    # workspace too small, zero splits, misaligned workspace
    assert lib.pa_decode_partial(FAKE, ws_ok - 1, *args, 4, 4, 8, 1, 0, None) == -1
    assert lib.pa_decode_partial(FAKE, ws_ok, *args, 0, 4, 8, 1, 0, None) == -1
    assert lib.pa_decode_partial(FAKE + 16, ws_ok, *args, 4, 4, 8, 1, 0, None) == -1
    assert lib.pa_decode_combine(FAKE, FAKE, ws_ok - 1, 2, 8, 128, 1, 4, 0, None) == -1
    assert lib.pa_decode_combine(FAKE, FAKE, ws_ok, 2, 8, 128, 1, 0, 0, None) == -1
    assert lib.pa_decode_combine(FAKE, FAKE, ws_ok, 2, 8, 96, 1, 4, 0, None) == -2
    assert lib.pa_decode_combine(None, FAKE, ws_ok, 2, 8, 128, 1, 4, 0, None) == -1


def test_append_and_slot_mapping_reject_bad_arguments(lib):
    assert lib.pa_append_kv(None, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_append_kv(FAKE, FAKE, FAKE + 4, FAKE, FAKE, 4, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 80, 16, 8, 0, None) == -2
    assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 24, 8, 0, None) == -2
    for bs in (8, 16, 32):  # the block sizes the kernels take (nothing to append: no launch)
        assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, bs, 8, 0, None) == 0
    assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 3, None) == -2
    assert lib.pa_append_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, 0, None) == 0
    assert lib.pa_slot_mapping(None, FAKE, FAKE, 2, 4, 16, 1, None) == -1
    assert lib.pa_slot_mapping(FAKE, FAKE, FAKE, 0, 4, 16, 1, None) == -1
    assert lib.pa_slot_mapping(FAKE, FAKE, FAKE, 2, 4, 16, 0, None) == -1
    assert lib.pa_slot_mapping(FAKE, FAKE, FAKE, 2, 4, 24, 1, None) == -2


def test_product_and_oracle_share_nothing():
    """The CUDA package never imports the oracle and the oracle never imports the
    package; neither reads the other's sources."""
    pkg = os.path.join(ROOT, "paged_kv_cache_20_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h")):
            assert "oracle" not in open(path).read().lower(), path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*")):
        if path.endswith((".py", ".c")):
            src = open(path).read()
            assert "paged_kv_cache_20_gb300" not in src and "pagedattn" not in src, path


def test_append_decode_rejects_bad_arguments(lib):
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 0.1, 4, 8, 1, 0]
    ok_ws = lib.pa_decode_workspace_size(2, 8, 1, 128, 4)
    call = lambda args, splits, ws, wsb: lib.pa_append_decode(*args, splits, ws, wsb, None)  # noqa: E731
    bad_knew = list(base); bad_knew[2] = None
    assert call(bad_knew, 1, None, 0) == -1
    mis = list(base); mis[3] = FAKE + 8
    assert call(mis, 1, None, 0) == -1
    assert call(base, 0, None, 0) == -1                 # no splits
    assert call(base, 4, None, 0) == -1                 # splits need a workspace
    assert call(base, 4, FAKE, ok_ws - 1) == -1         # too small
    d96 = list(base); d96[11] = 96
    assert call(d96, 1, None, 0) == -2


def test_copy_blocks_rejects_bad_arguments(lib):
    assert lib.pa_copy_blocks(None, FAKE, FAKE, FAKE, 2, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, -1, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_copy_blocks(FAKE + 4, FAKE, FAKE, FAKE, 2, 2, 128, 16, 8, 0, None) == -1
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, 2, 2, 100, 16, 8, 0, None) == -2
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, 0, None) == 0


def test_cascade_rejects_bad_arguments(lib):
    # out, q, k_new, v_new, k, v, tables, lens, n, hq, hkv, d, bs, scale, maxb, nblocks, qlen, dtype
    base = [FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 0.1, 4, 8, 1, 0]
    ws_ok = lib.pa_decode_workspace_size(2, 8, 1, 128, 3)
    call = lambda args, prefix, tail, ws, wsb: lib.pa_decode_cascade(  # noqa: E731
        *args, prefix, tail, ws, wsb, None)
    assert call(base, 0, 2, FAKE, ws_ok) == -1          # no prefix
    assert call(base, 5, 2, FAKE, ws_ok) == -1          # prefix longer than the table
    assert call(base, 2, 0, FAKE, ws_ok) == -1          # no tail partition
    assert call(base, 2, 2, None, ws_ok) == -1          # workspace required
    assert call(base, 2, 2, FAKE + 16, ws_ok) == -1     # 256-byte alignment
    assert call(base, 2, 2, FAKE, ws_ok - 1) == -1      # 1 + tail_splits partitions
    one_new = list(base); one_new[2] = FAKE
    assert call(one_new, 2, 2, FAKE, ws_ok) == -1       # k_new without v_new
    d96 = list(base); d96[11] = 96
    assert call(d96, 2, 2, FAKE, ws_ok) == -2


def test_fp8_query_length_limit(lib):
    # an FP8 cache takes the same q_len range as a 16-bit one, 1..4096
    args = [FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 0.1, 4,
            8]
    assert lib.pa_decode_fp8(*args, 4097, 0, 1, None, 0, None) == -2
    assert lib.pa_decode_fp8(*args, 0, 0, 1, None, 0, None) == -1
