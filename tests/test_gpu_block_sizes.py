"""Pools of 8- and 32-token blocks through the C ABI vs the fp64 oracle (needs a
GPU).

The kernels walk a sequence in 16-token tiles: a 32-token block is read as two
tiles (two 16-row boxes of the cache's tensor map), a tile of an 8-token pool
spans two blocks (two 8-row boxes).  The append and slot mapping follow the
block size directly.  "LLM 推理优化全景实战" §2.3: block_size is a parameter of
the pool.  Every element is compared; append bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import _tol
from tests.oracle_pins import Paged
from tests.test_gpu_parity import (DEV, _dev, _f64, _gpu_decode, _logical_case, _to_dev, _u16,
                                   gpu_step, oracle_step)
from tests.test_gpu_prefill import gpu_cascade
from tests.test_gpu_fp8 import gpu_step as gpu_step8, oracle_step as oracle_step8

pytestmark = pytest.mark.gpu

SIZES = [8, 32]


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    assert pa.pa_device_error() == 0
    return pa


CASES = [
    ("tiny", {}),                                                           # head_dim 64
    ("llama7b_mha", {"num_seqs": 3}),                                       # 1 row
    ("gqa", {"num_seqs": 5}),                                               # 4 rows
    ("gqa", {"num_seqs": 4, "num_q_heads": 16, "num_kv_heads": 8}),         # 2 rows
    ("prefix_verify", {"num_seqs": 4}),                                     # 16 rows, causal
    ("chunked_prefill", {"num_seqs": 2, "q_len": 100, "lens": ("fixed", (100, 357))}),
]


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("bs", SIZES)
def test_block_size_every_element(pa, orc, bs, case, fused, splits):
    name, over = CASES[case]
    w = workloads.make(name, block_size=bs, **over)
    out, d = gpu_step(pa, w, num_splits=splits, fused=fused)
    ref, kc, vc, slots = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    gslots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], bs, w.cfg.q_len)
    assert np.array_equal(gslots.cpu().numpy(), slots)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"block {bs} {name} {over} splits {splits}")


EDGE_LENS = [0, 1, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 257]


@pytest.mark.parametrize("q_len", [1, 2, 20])
@pytest.mark.parametrize("bs", SIZES)
def test_block_size_edge_lengths(pa, orc, bs, q_len):
    """Contexts ending anywhere inside a block or a tile, empty ones included; with
    8-token blocks a context ending in the first half of a tile leaves the second
    block unread."""
    q, K, V = _logical_case(71, EDGE_LENS, 8, 2, 128, "bf16", q_len=q_len, qscale=2.0)
    pc = Paged(orc, K, V, bs, "bf16", perm_seed=9)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(128)))
    ref = pc.decode(orc, q, scale, q_len=q_len)
    for S in (1, 3):
        _tol.check(_gpu_decode(pa, pc, q, scale, q_len, num_splits=S), ref, "bf16",
                   f"block {bs} edges q_len {q_len} splits {S}")


@pytest.mark.parametrize("bs", SIZES)
def test_block_size_paging_is_bit_invariant(pa, orc, bs):
    """Any physical order of the same logical blocks gives bit-identical outputs."""
    q, K, V = _logical_case(72, [5, 40, 333], 8, 4, 128, "fp16")
    outs = [_gpu_decode(pa, Paged(orc, K, V, bs, "fp16", perm_seed=s), q, 0.0884, 1)
            for s in (1, 2, 3)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_32_token_blocks_partition_statistics(pa, orc):
    """Split-KV partials over 32-token blocks cut each sequence at whole blocks, as
    the oracle's partitions do: the per-partition statistics agree."""
    lens = [40, 300, 700, 33]
    q_len, S = 3, 3
    q, K, V = _logical_case(73, lens, 8, 2, 128, "bf16", q_len=q_len)
    pc = Paged(orc, K, V, 32, "bf16", perm_seed=10)
    m, l, acc = orc.decode_partitions(q, pc.k, pc.v, pc.tables, pc.lens, 0.0884, "bf16", S,
                                      q_len=q_len)
    nbytes = pa.pa_decode_workspace_size(4, 8, q_len, 128, S)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=DEV)
    pa.pa_decode_partial(ws, _to_dev(q, "bf16"), _to_dev(pc.k, "bf16"), _to_dev(pc.v, "bf16"),
                         torch.from_numpy(pc.tables).to(DEV), torch.from_numpy(pc.lens).to(DEV),
                         0.0884, S, q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    g_acc, g_m, g_l = (t.double().cpu().numpy() for t in pa.workspace_views(ws, 4, 8, q_len, 128, S))
    empty = l == 0
    assert np.array_equal(g_l == 0, empty)
    ok = ~empty
    _tol.check(g_acc[ok] / g_l[ok][:, None], acc[ok] / l[ok][:, None], "bf16", "partitions")


@pytest.mark.parametrize("bs", SIZES)
def test_block_size_cascade(pa, orc, bs):
    """The shared prefix (1024 tokens: 128 blocks of 8 or 32 of 32) once for all query
    rows, then the tails, then the merge."""
    w = workloads.make("prefix_verify", num_seqs=6, block_size=bs)
    out, d = gpu_cascade(pa, w)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"cascade block {bs}")


@pytest.mark.parametrize("q_len", [1, 40])
@pytest.mark.parametrize("bs", SIZES)
def test_block_size_fp8_cache(pa, orc, bs, q_len):
    w = workloads.make("gqa_fp8", num_seqs=4, q_len=q_len, block_size=bs,
                       lens=("fixed", (q_len, 77, 300, 1000)))
    out, d = gpu_step8(pa, w)
    ref, kc, vc = oracle_step8(orc, w)
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(d["v_cache"].cpu().numpy(), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"fp8 block {bs} q_len {q_len}")


@pytest.mark.parametrize("bs", SIZES)
def test_block_size_full_size_gqa(pa, orc, bs):
    """The full GQA workload (64 sequences) over 8- and 32-token blocks, fused."""
    w = workloads.make("gqa", block_size=bs)
    out, d = gpu_step(pa, w, fused=True)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"gqa block {bs}")


@pytest.mark.parametrize("bs", SIZES)
def test_block_size_copy_blocks(pa, orc, bs):
    w = workloads.make("gqa", num_seqs=3, block_size=bs)
    d = _dev(w)
    P = w.k_cache.shape[0]
    rng = np.random.default_rng(bs)
    perm = rng.permutation(P).astype(np.int32)
    src, dst = perm[:5], perm[5:10]
    pa.pa_copy_blocks(d["k_cache"], d["v_cache"], torch.from_numpy(src).to(DEV),
                      torch.from_numpy(dst).to(DEV))
    torch.cuda.synchronize()
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    orc.copy_blocks(kc, vc, src, dst)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
