"""CUDA library vs the fp64 oracle, through the C ABI (needs a GPU).

Append and slot mapping are compared bit for bit; attention within the tolerance
of tests/_tol.py.  Every output element is compared, at small sizes and at the
full workload sizes (in the launch configuration bench.py times), plus properties
that hold at any size.
"""
import os

import numpy as np
import pytest
import torch

import workloads
from tests import _tol
from tests.oracle_pins import Paged, _bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    assert pa.pa_device_error() == 0
    return pa


DEV = "cuda:0"


def _dev(w):
    return {k: getattr(w, k).to(DEV) for k in
            ("q", "k_new", "v_new", "k_cache", "v_cache", "block_tables", "context_lens")}


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def gpu_step(pa, w, num_splits=None, fused=False):
    d = _dev(w)
    s = w.cfg.num_splits if num_splits is None else num_splits
    out = pa.paged_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                               d["block_tables"], d["context_lens"], w.scale, q_len=w.cfg.q_len,
                               num_splits=s, fused=fused)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    return out, d


THREADS = os.cpu_count() or 1


def oracle_step(orc, w, rows=None, threads=THREADS):
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    slots = orc.slot_mapping(w.block_tables.numpy(), w.context_lens.numpy(), w.cfg.block_size,
                             w.cfg.q_len)
    orc.append_kv(kc, vc, w.bits("k_new"), w.bits("v_new"), slots)
    out = orc.decode(w.bits("q"), kc, vc, w.block_tables.numpy(), w.context_lens.numpy(),
                     w.scale, w.cfg.dtype, q_len=w.cfg.q_len, rows=rows, threads=threads)
    return out, kc, vc, slots


SMALL = [
    ("tiny", {}),
    ("llama7b_mha", {"num_seqs": 3}),
    ("gqa", {"num_seqs": 5}),
    ("long_split", {"num_seqs": 1, "lens": ("fixed", (4100,))}),
    ("prefix_verify", {"num_seqs": 4}),
]


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("name,over", SMALL, ids=[s[0] for s in SMALL])
def test_small_configs_every_element(pa, orc, name, over, fused):
    w = workloads.make(name, **over)
    out, d = gpu_step(pa, w, fused=fused)
    ref, kc, vc, slots = oracle_step(orc, w)
    # append is bit-exact over the whole pool (NaN-poisoned slots included)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, name)


# gqa-96: 768 units of 4 rows, more than one wave of 3-warp CTAs, so the
# swapped-operand path launches its 4-warp form (the 64-sequence gqa takes the
# 3-warp form).
FULL = [("llama7b_mha", {}), ("gqa", {}), ("long_split", {}), ("prefix_verify", {}),
        ("gqa", {"num_seqs": 96, "pool_blocks": None})]

# The separate and fused runs of one workload are adjacent in the parametrised
# order (the workload varies slowest), so one cached oracle result serves both.
_LAST_FULL = {}


def full_oracle(orc, key, w):
    """The oracle's whole step (every output row, the appended pools and slots) for
    ``w``, computed once per key on all host cores."""
    if _LAST_FULL.get("key") != key:
        _LAST_FULL.clear()
        _LAST_FULL.update(key=key, res=oracle_step(orc, w))
    return _LAST_FULL["res"]


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("name,over", FULL, ids=["llama7b_mha", "gqa", "long_split",
                                                 "prefix_verify", "gqa-96"])
def test_full_size_every_element(pa, orc, name, over, fused):
    """Full-size workloads in the launch configuration bench.py times (fused), every
    output element against the oracle."""
    w = workloads.make(name, **over)
    out, d = gpu_step(pa, w, fused=fused)
    ref, kc, vc, slots = full_oracle(orc, (name, repr(over)), w)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{name} {over}")
    # slot mapping and the appended rows, bit for bit
    gslots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], w.cfg.block_size,
                               w.cfg.q_len)
    assert np.array_equal(gslots.cpu().numpy(), slots)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)


def _logical_case(seed, lens, h_q, h_kv, d, dtype, q_len=1, qscale=1.0):
    rng = np.random.default_rng(seed)
    K = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    V = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    q = _bits(qscale * rng.standard_normal((len(lens), q_len, h_q, d)), dtype)
    return q, K, V


def _to_dev(arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
    return t.view(torch.float16 if dtype == "fp16" else torch.bfloat16).to(DEV)


def _gpu_decode(pa, pc, q, scale, q_len, num_splits=1, lens=None):
    qd = _to_dev(q, pc.dtype)
    kd, vd = _to_dev(pc.k, pc.dtype), _to_dev(pc.v, pc.dtype)
    bt = torch.from_numpy(pc.tables).to(DEV)
    cl = torch.from_numpy(pc.lens if lens is None else np.asarray(lens, np.int32)).to(DEV)
    out = torch.empty_like(qd)
    if num_splits == 1:
        pa.pa_decode(out, qd, kd, vd, bt, cl, scale, q_len)
    else:
        nbytes = pa.pa_decode_workspace_size(q.shape[0], q.shape[2], q_len, q.shape[3], num_splits)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        pa.pa_decode_partial(ws, qd, kd, vd, bt, cl, scale, num_splits, q_len)
        pa.pa_decode_combine(out, ws, num_splits)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    return _f64(out)


EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 100, 257]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h_q,h_kv,q_len", [(4, 4, 1), (8, 4, 1), (12, 4, 1), (16, 4, 1),
                                            (8, 8, 2), (8, 2, 4), (32, 4, 4), (6, 2, 3),
                                            # 5..8 rows per KV head, causal ones included
                                            (8, 4, 3), (16, 2, 1), (10, 2, 1), (4, 2, 4),
                                            (7, 1, 1)])
def test_edge_lengths_groups_and_query_counts(pa, orc, dtype, d, h_q, h_kv, q_len):
    lens = EDGE_LENS
    q, K, V = _logical_case(3, lens, h_q, h_kv, d, dtype, q_len=q_len, qscale=2.0)
    pc = Paged(orc, K, V, 16, dtype, perm_seed=5)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    ref = pc.decode(orc, q, scale, q_len=q_len)
    got = _gpu_decode(pa, pc, q, scale, q_len)
    _tol.check(got, ref, dtype, f"{dtype} d{d} {h_q}/{h_kv} q_len{q_len}")
    for S in (2, 3, 16, 40):
        got_s = _gpu_decode(pa, pc, q, scale, q_len, num_splits=S)
        _tol.check(got_s, ref, dtype, f"split {S}")


def test_context_one_returns_v_exactly(pa, orc):
    for dtype in ("fp16", "bf16"):
        q, K, V = _logical_case(4, [1, 1, 1], 8, 2, 128, dtype, qscale=5.0)
        pc = Paged(orc, K, V, 16, dtype, perm_seed=1)
        got = _gpu_decode(pa, pc, q, 0.1, 1)
        for i in range(3):
            want = np.repeat(orc.decode_bits(V[i][0], dtype), 4, axis=0)
            assert np.array_equal(got[i, 0], want)


def test_identical_value_rows(pa, orc):
    rng = np.random.default_rng(6)
    L = 300
    row = _bits(rng.standard_normal((1, 2, 128)), "bf16")
    V = [np.repeat(row, L, axis=0)]
    K = [_bits(rng.standard_normal((L, 2, 128)), "bf16")]
    q = _bits(2 * rng.standard_normal((1, 1, 8, 128)), "bf16")
    pc = Paged(orc, K, V, 16, "bf16", perm_seed=2)
    got = _gpu_decode(pa, pc, q, 0.09, 1)
    want = np.repeat(orc.decode_bits(row[0], "bf16"), 4, axis=0)
    assert np.abs(got[0, 0] - want).max() <= 2e-3


def test_paging_permutation_is_bit_invariant(pa, orc):
    lens = [70, 511, 1000, 33]
    for h_q, h_kv in ((8, 8), (32, 8)):
        q, K, V = _logical_case(7, lens, h_q, h_kv, 128, "fp16")
        outs = []
        for seed in (None, 11, 12):
            pc = Paged(orc, K, V, 16, "fp16", perm_seed=seed)
            outs.append(_gpu_decode(pa, pc, q, 0.0884, 1))
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_stress_rescale_peaked_scores(pa, orc):
    # large q makes each row's softmax nearly one-hot and the running max move often
    lens = [40, 333, 900]
    q, K, V = _logical_case(8, lens, 8, 2, 128, "fp16", qscale=8.0)
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=3)
    ref = pc.decode(orc, q, 0.0884)
    _tol.check(_gpu_decode(pa, pc, q, 0.0884, 1), ref, "fp16", "peaked")
    # increasing scores along the sequence: every block raises the max
    L = 400
    rng = np.random.default_rng(9)
    k = rng.standard_normal((L, 1, 128)) * 0.1
    k[:, 0, 0] = np.linspace(-4, 4, L)
    qv = np.zeros((1, 1, 1, 128))
    qv[..., 0] = 3.0
    qb = _bits(qv, "fp16")
    pc2 = Paged(orc, [_bits(k, "fp16")], [_bits(rng.standard_normal((L, 1, 128)), "fp16")], 16,
                "fp16", perm_seed=4)
    _tol.check(_gpu_decode(pa, pc2, qb, 1.0, 1), pc2.decode(orc, qb, 1.0), "fp16", "rising")


def test_partial_statistics_match_oracle_partitions(pa, orc):
    lens = [1, 40, 700, 0]
    q_len, S = 2, 5
    q, K, V = _logical_case(10, lens, 8, 2, 128, "bf16", q_len=q_len)
    pc = Paged(orc, K, V, 16, "bf16", perm_seed=6)
    m, l, acc = orc.decode_partitions(q, pc.k, pc.v, pc.tables, pc.lens, 0.0884, "bf16", S,
                                      q_len=q_len)
    qd = _to_dev(q, "bf16")
    nbytes = pa.pa_decode_workspace_size(4, 8, q_len, 128, S)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=DEV)   # garbage-filled
    pa.pa_decode_partial(ws, qd, _to_dev(pc.k, "bf16"), _to_dev(pc.v, "bf16"),
                         torch.from_numpy(pc.tables).to(DEV), torch.from_numpy(pc.lens).to(DEV),
                         0.0884, S, q_len)
    g_acc, g_m, g_l = (t.double().cpu().numpy() for t in pa.workspace_views(ws, 4, 8, q_len, 128, S))
    empty = l == 0
    assert np.array_equal(g_l == 0, empty)
    assert np.all(np.isneginf(g_m[empty])) and np.all(g_acc[empty] == 0)
    ok = ~empty
    # normalised partition output and log-sum-exp (natural units) per partition
    norm_g = g_acc[ok] / g_l[ok][:, None]
    norm_o = acc[ok] / l[ok][:, None]
    _tol.check(norm_g, norm_o, "bf16", "partition output")
    lse_g = g_m[ok] * np.log(2.0) + np.log(g_l[ok])
    lse_o = m[ok] + np.log(l[ok])
    assert np.abs(lse_g - lse_o).max() < 1e-4


# 7 partitions: one warp per row; 12 and 33 (more than 8, few rows): one dimension
# per lane, and 33 also takes the second group of 32 partitions
@pytest.mark.parametrize("S,D", [(7, 64), (12, 64), (12, 128), (33, 128)])
def test_combine_alone_on_oracle_partials(pa, orc, S, D):
    lens = [3, 64, 500, 0, 17]
    q_len = 1
    q, K, V = _logical_case(12, lens, 4, 4, D, "fp16", q_len=q_len, qscale=2.0)
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=8)
    m, l, acc = orc.decode_partitions(q, pc.k, pc.v, pc.tables, pc.lens, 0.125, "fp16", S)
    want = orc.combine(m, l, acc).reshape(5, 1, 4, D)
    nbytes = pa.pa_decode_workspace_size(5, 4, 1, D, S)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    g_acc, g_m, g_l = pa.workspace_views(ws, 5, 4, 1, D, S)
    g_acc.copy_(torch.from_numpy(acc).float())
    g_m.copy_(torch.from_numpy(m / np.log(2.0)).float())   # base-2 units
    g_l.copy_(torch.from_numpy(l).float())
    out = torch.empty((5, 1, 4, D), dtype=torch.float16, device=DEV)
    pa.pa_decode_combine(out, ws, S)
    torch.cuda.synchronize()
    _tol.check(_f64(out), want, "fp16", f"combine of {S} partitions")


def test_bad_block_id_is_reported_not_faulted(pa, orc):
    q, K, V = _logical_case(13, [40, 40], 4, 4, 128, "fp16")
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=9)
    pc.tables[1, 1] = pc.k.shape[0] + 5          # beyond the pool
    qd = _to_dev(q, "fp16")
    out = torch.empty_like(qd)
    pa.pa_decode(out, qd, _to_dev(pc.k, "fp16"), _to_dev(pc.v, "fp16"),
                 torch.from_numpy(pc.tables).to(DEV), torch.from_numpy(pc.lens).to(DEV), 0.1, 1)
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    assert pa.pa_device_error() == 0                         # cleared
    got = _f64(out)
    assert np.isfinite(got).all()
    ref = pc.decode(orc, q, 0.1)
    _tol.check(got[0], ref[0], "fp16", "unaffected sequence")


def test_append_skips_negative_and_reports_out_of_pool_slots(pa):
    P, H, D = 6, 2, 128
    kc = torch.zeros((P, H, 16, D), dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = torch.randn((3, H, D), dtype=torch.float16, device=DEV)
    vn = torch.randn((3, H, D), dtype=torch.float16, device=DEV)
    slots = torch.tensor([5, -1, P * 16 + 3], dtype=torch.int64, device=DEV)
    pa.pa_append_kv(kc, vc, kn, vn, slots)
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    assert torch.equal(kc[0, :, 5], kn[0]) and torch.equal(vc[0, :, 5], vn[0])
    kc[0, :, 5] = 0
    vc[0, :, 5] = 0
    assert int(kc.abs().sum()) == 0 and int(vc.abs().sum()) == 0


def test_device_wait_times_out_and_reports(pa):
    """A device-side wait that nothing satisfies gives up after its limit, reports
    PA_ERR_DEVICE_TIMEOUT, and leaves the context usable."""
    import time
    assert pa.pa_device_error() == 0
    t0 = time.time()
    pa.pa_selftest_wait_timeout()
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_TIMEOUT
    assert 1.0 < time.time() - t0 < 30.0
    assert pa.pa_device_error() == 0                 # cleared
    x = torch.ones(1024, device=DEV)
    assert float(x.sum()) == 1024.0                  # context still works


@pytest.mark.parametrize("h_q,h_kv,q_len,dtype", [(32, 1, 1, "bf16"), (32, 1, 2, "fp16"),
                                                  (16, 16, 16, "fp16"), (64, 8, 4, "bf16")])
def test_many_rows_per_kv_head(pa, orc, h_q, h_kv, q_len, dtype):
    """MQA and long verify windows: 16-64 query rows per KV head (several row groups)."""
    lens = [1, 15, 16, 40, 129, 700]
    q, K, V = _logical_case(20, lens, h_q, h_kv, 128, dtype, q_len=q_len, qscale=1.5)
    pc = Paged(orc, K, V, 16, dtype, perm_seed=21)
    ref = pc.decode(orc, q, 0.0884, q_len=q_len)
    _tol.check(_gpu_decode(pa, pc, q, 0.0884, q_len), ref, dtype, "single pass")
    _tol.check(_gpu_decode(pa, pc, q, 0.0884, q_len, num_splits=5), ref, dtype, "split 5")


def test_many_sequences_without_length_ranking(pa, orc):
    """More sequences than the in-kernel longest-first ranking handles (300 > 256)."""
    rng = np.random.default_rng(22)
    lens = [int(x) for x in rng.integers(0, 90, size=300)]
    q, K, V = _logical_case(23, lens, 8, 2, 64, "bf16")
    pc = Paged(orc, K, V, 16, "bf16", perm_seed=24)
    _tol.check(_gpu_decode(pa, pc, q, 0.125, 1), pc.decode(orc, q, 0.125), "bf16", "300 seqs")


def test_wide_block_table_and_short_table(pa, orc):
    q, K, V = _logical_case(25, [20, 50], 4, 4, 128, "fp16")
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=26)
    ref = pc.decode(orc, q, 0.1)
    # extra table columns (never read) pointing at the NaN-poisoned padding block
    wide = np.concatenate([pc.tables, np.full((2, 5), pc.tables[0, -1], np.int32)], axis=1)
    pc.tables = wide
    _tol.check(_gpu_decode(pa, pc, q, 0.1, 1), ref, "fp16", "wide table")
    # a context longer than its table: reported, the rest still finite
    pc.tables = np.ascontiguousarray(wide[:, :2])
    got = _gpu_decode_unchecked(pa, pc, q, 0.1, lens=[20, 50])
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    assert np.isfinite(got).all()


def _gpu_decode_unchecked(pa, pc, q, scale, lens):
    qd = _to_dev(q, pc.dtype)
    out = torch.empty_like(qd)
    pa.pa_decode(out, qd, _to_dev(pc.k, pc.dtype), _to_dev(pc.v, pc.dtype),
                 torch.from_numpy(pc.tables).to(DEV),
                 torch.from_numpy(np.asarray(lens, np.int32)).to(DEV), scale, 1)
    torch.cuda.synchronize()
    return _f64(out)


@pytest.mark.parametrize("q_len,splits", [(1, 1), (4, 1), (4, 3), (16, 1), (2, 40)])
def test_fused_append_decode_edges(pa, orc, q_len, splits):
    """Fused step on edge lengths, including sequences shorter than q_len and new
    tokens that straddle a block boundary or a split boundary."""
    cfg = workloads.config("gqa", num_seqs=9, q_len=q_len,
                           lens=("fixed", (0, 1, 3, 15, 16, 17, 33, 100, 257)), spare_blocks=3)
    w = workloads.make(cfg)
    out, d = gpu_step(pa, w, num_splits=splits, fused=True)
    ref, kc, vc, slots = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"fused q_len {q_len} splits {splits}")


@pytest.mark.parametrize("name,q_len", [("llama7b_mha", 2), ("gqa", 4), ("prefix_verify", 4),
                                        ("gqa", 16)])
def test_fused_append_by_the_ctas_that_read_the_new_tiles(pa, orc, name, q_len):
    """In the fused step only the CTAs whose warps read a tile holding a new position
    write the new rows.  Few sequences launch as 2-8-CTA clusters, and lengths of
    1-41 tiles with offsets inside and across tiles put those tiles on every warp
    and CTA of a cluster (the walk's start also rotates with the KV head): the
    whole pool must still match the oracle's append bit for bit."""
    lens = tuple(16 * t + o for t, o in zip(range(1, 42, 4), (1, 15, 16, 3, 8, 0, 12, 5, 16, 9, 2)))
    cfg = workloads.config(name, num_seqs=len(lens), q_len=q_len, lens=("fixed", lens),
                           spare_blocks=3, shared_prefix=0)
    w = workloads.make(cfg)
    out, d = gpu_step(pa, w, num_splits=1, fused=True)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{name} q_len {q_len}")


def test_copy_blocks_bit_exact_and_cow_decode(pa, orc):
    """Copy-on-write: copies are bit-exact against the oracle on the whole pool, bad
    pairs are skipped and reported, and a sequence redirected to its private copy
    attends exactly as before."""
    w = workloads.make("gqa", num_seqs=6)
    d = _dev(w)
    P = w.num_blocks
    rng = np.random.default_rng(30)
    src = rng.choice(P, size=20, replace=False).astype(np.int32)
    dst = np.setdiff1d(np.arange(P), src)[:20].astype(np.int32)
    src_b = np.concatenate([src, [P + 3]]).astype(np.int32)    # one bad pair
    dst_b = np.concatenate([dst, [0]]).astype(np.int32)
    pa.pa_copy_blocks(d["k_cache"], d["v_cache"], torch.from_numpy(src_b).to(DEV),
                      torch.from_numpy(dst_b).to(DEV))
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    assert orc.copy_blocks(kc, vc, src_b, dst_b) == 1
    assert np.array_equal(_u16(d["k_cache"]), kc) and np.array_equal(_u16(d["v_cache"]), vc)
    # redirect sequence 0's last block to a fresh copy: attention unchanged (bit-exact)
    out_a, _ = gpu_step(pa, w, fused=True)
    d2 = _dev(w)
    last = int((int(w.context_lens[0]) - 1) // 16)
    old_blk = int(w.block_tables[0, last])
    spare = int(np.setdiff1d(np.arange(P), w.block_tables.numpy().ravel())[0])
    pa.pa_copy_blocks(d2["k_cache"], d2["v_cache"], torch.tensor([old_blk], dtype=torch.int32,
                      device=DEV), torch.tensor([spare], dtype=torch.int32, device=DEV))
    d2["block_tables"][0, last] = spare
    out_b = pa.pa_append_decode(torch.empty_like(d2["q"]), d2["q"], d2["k_new"], d2["v_new"],
                                d2["k_cache"], d2["v_cache"], d2["block_tables"],
                                d2["context_lens"], w.scale, w.cfg.q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(out_a, out_b)
