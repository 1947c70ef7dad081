"""Many query rows per sequence (chunked prefill) and cascade shared-prefix attention,
CUDA library vs the fp64 oracle through the C ABI (needs a GPU).

Both reach the same attention as pa_decode -- softmax(scale q K^T) V over each
row's causal window -- so each is compared with the oracle's plain definition:
every element, at small sizes and at the full workload sizes, and the appended
cache bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import _tol
from tests.oracle_pins import Paged
from tests.test_gpu_parity import (DEV, THREADS, _dev, _f64, _gpu_decode, _logical_case,
                                   _to_dev, _u16, full_oracle, gpu_step, oracle_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    assert pa.pa_device_error() == 0
    return pa


# ------------------------------------------------------------------- chunked prefill
PREFILL_SMALL = [
    ("chunked_prefill", {"num_seqs": 2, "q_len": 100, "lens": ("fixed", (100, 357))}),
    ("llama7b_mha", {"num_seqs": 2, "q_len": 40, "lens": ("fixed", (40, 700))}),
    ("tiny", {"q_len": 17, "lens": ("fixed", (17, 33, 60))}),
    ("gqa", {"num_seqs": 3, "q_len": 64, "lens": ("fixed", (64, 65, 1000))}),
]


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("name,over", PREFILL_SMALL, ids=[c[0] for c in PREFILL_SMALL])
def test_chunked_prefill_every_element(pa, orc, name, over, fused, splits):
    w = workloads.make(name, **over)
    out, d = gpu_step(pa, w, num_splits=splits, fused=fused)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{name} q_len {w.cfg.q_len}")


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_chunked_prefill_full_size_every_element(pa, orc, fused):
    """The full chunked-prefill workload in the launch configuration bench.py times,
    every output element (the oracle runs once for both launch forms)."""
    w = workloads.make("chunked_prefill")
    out, d = gpu_step(pa, w, fused=fused)
    ref, kc, vc, _ = full_oracle(orc, ("chunked_prefill", ""), w)
    _tol.check(_f64(out), ref, w.cfg.dtype, "chunked_prefill")
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)


PREFILL_LENS = [0, 1, 15, 16, 17, 33, 100, 257]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h_q,h_kv,q_len", [(8, 8, 17), (8, 2, 33), (12, 4, 64)])
def test_prefill_edge_lengths(pa, orc, dtype, d, h_q, h_kv, q_len):
    # contexts shorter than q_len: the first rows see nothing (zeros), later ones a
    # prefix of the context
    q, K, V = _logical_case(21, PREFILL_LENS, h_q, h_kv, d, dtype, q_len=q_len, qscale=2.0)
    pc = Paged(orc, K, V, 16, dtype, perm_seed=9)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    ref = pc.decode(orc, q, scale, q_len=q_len)
    _tol.check(_gpu_decode(pa, pc, q, scale, q_len), ref, dtype, f"{dtype} d{d} q_len {q_len}")
    for S in (2, 7):
        _tol.check(_gpu_decode(pa, pc, q, scale, q_len, num_splits=S), ref, dtype, f"split {S}")


def test_prefill_paging_permutation_is_bit_invariant(pa, orc):
    lens = [64, 511, 1000]
    q, K, V = _logical_case(22, lens, 32, 8, 128, "bf16", q_len=40)
    outs = [_gpu_decode(pa, Paged(orc, K, V, 16, "bf16", perm_seed=s), q, 0.0884, 40)
            for s in (None, 13, 14)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_prefill_peaked_scores(pa, orc):
    lens = [300, 900]
    q, K, V = _logical_case(23, lens, 8, 2, 128, "fp16", q_len=48, qscale=8.0)
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=15)
    _tol.check(_gpu_decode(pa, pc, q, 0.0884, 48), pc.decode(orc, q, 0.0884, q_len=48), "fp16",
               "peaked prefill")


# -------------------------------------------------------------------------- cascade
def gpu_cascade(pa, w, tail_splits=1, fused=True):
    d = _dev(w)
    P = w.cfg.shared_prefix // w.cfg.block_size
    out = torch.empty_like(d["q"])
    if fused:
        pa.pa_decode_cascade(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, P, q_len=w.cfg.q_len,
                             tail_splits=tail_splits, k_new=d["k_new"], v_new=d["v_new"])
    else:
        slots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], w.cfg.block_size, w.cfg.q_len)
        pa.pa_append_kv(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], slots)
        pa.pa_decode_cascade(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, P, q_len=w.cfg.q_len,
                             tail_splits=tail_splits)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    return out, d


CASCADE_SMALL = [
    ("prefix_verify", {"num_seqs": 4}),
    ("prefix_verify", {"num_seqs": 3, "q_len": 40, "lens": ("prefix", 1024, 64, 300)}),
    ("prefix_verify", {"num_seqs": 5, "q_len": 1, "num_q_heads": 8, "num_kv_heads": 8,
                       "head_dim": 64, "dtype": "bf16", "shared_prefix": 48,
                       "lens": ("prefix", 48, 1, 100)}),
]


@pytest.mark.parametrize("tail_splits", [1, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("case", range(len(CASCADE_SMALL)))
def test_cascade_every_element(pa, orc, case, fused, tail_splits):
    name, over = CASCADE_SMALL[case]
    w = workloads.make(name, **over)
    out, d = gpu_cascade(pa, w, tail_splits=tail_splits, fused=fused)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"cascade {case}")


def test_cascade_full_size_every_element(pa, orc):
    """prefix_verify at full size, in the launch configuration bench.py times."""
    w = workloads.make("prefix_verify")
    out, d = gpu_cascade(pa, w)
    ref, kc, vc, _ = oracle_step(orc, w)
    _tol.check(_f64(out), ref, w.cfg.dtype, "cascade full")
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)


def test_cascade_equals_plain_decode_closely(pa):
    """Same inputs through pa_append_decode and pa_decode_cascade: both are the same
    attention, so they agree to a few output ulps."""
    w = workloads.make("prefix_verify", num_seqs=16)
    plain, _ = gpu_step(pa, w, fused=True)
    casc, _ = gpu_cascade(pa, w)
    diff = (plain.double() - casc.double()).abs().max().item()
    assert diff <= 2e-3, diff


# ------------------------------------------------------------------- more edges
def test_prefill_partial_statistics_match_oracle_partitions(pa, orc):
    """The many-row kernel's partial pass writes each partition's (m, l, acc): the
    normalised partition outputs and log-sum-exps equal the oracle's partitions."""
    lens = [40, 300, 700, 33]
    q_len, S = 33, 3
    q, K, V = _logical_case(24, lens, 8, 2, 128, "bf16", q_len=q_len)
    pc = Paged(orc, K, V, 16, "bf16", perm_seed=16)
    m, l, acc = orc.decode_partitions(q, pc.k, pc.v, pc.tables, pc.lens, 0.0884, "bf16", S,
                                      q_len=q_len)
    qd = _to_dev(q, "bf16")
    nbytes = pa.pa_decode_workspace_size(4, 8, q_len, 128, S)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=DEV)  # garbage-filled
    pa.pa_decode_partial(ws, qd, _to_dev(pc.k, "bf16"), _to_dev(pc.v, "bf16"),
                         torch.from_numpy(pc.tables).to(DEV), torch.from_numpy(pc.lens).to(DEV),
                         0.0884, S, q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    g_acc, g_m, g_l = (t.double().cpu().numpy() for t in pa.workspace_views(ws, 4, 8, q_len, 128, S))
    empty = l == 0
    assert np.array_equal(g_l == 0, empty)
    assert np.all(np.isneginf(g_m[empty])) and np.all(g_acc[empty] == 0)
    ok = ~empty
    _tol.check(g_acc[ok] / g_l[ok][:, None], acc[ok] / l[ok][:, None], "bf16", "partition output")
    lse_g = g_m[ok] * np.log(2.0) + np.log(g_l[ok])
    assert np.abs(lse_g - (m[ok] + np.log(l[ok]))).max() < 1e-4


def test_prefill_longest_chunk_every_element(pa, orc):
    """q_len at the library's limit (4096): one sequence, GQA, every element."""
    w = workloads.make("chunked_prefill", num_seqs=1, q_len=4096, lens=("fixed", (4400,)))
    out, d = gpu_step(pa, w, fused=True)
    ref, kc, vc, _ = oracle_step(orc, w)
    _tol.check(_f64(out), ref, w.cfg.dtype, "q_len 4096")
    assert np.array_equal(_u16(d["k_cache"]), kc)


def test_prefill_bad_block_id_is_reported_not_faulted(pa, orc):
    q, K, V = _logical_case(25, [100, 100], 8, 2, 128, "fp16", q_len=40)
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=17)
    pc.tables[1, 2] = pc.k.shape[0] + 7                  # beyond the pool
    qd = _to_dev(q, "fp16")
    out = torch.empty_like(qd)
    pa.pa_decode(out, qd, _to_dev(pc.k, "fp16"), _to_dev(pc.v, "fp16"),
                 torch.from_numpy(pc.tables).to(DEV), torch.from_numpy(pc.lens).to(DEV), 0.1, 40)
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    assert pa.pa_device_error() == 0                     # cleared
    got = _f64(out)
    assert np.isfinite(got).all()
    ref = pc.decode(orc, q, 0.1, q_len=40)
    _tol.check(got[0], ref[0], "fp16", "unaffected sequence")


def test_prefill_append_reports_positions_beyond_the_table(pa):
    """The table-driven append (q_len > 16) skips and reports new positions past a
    sequence's block table."""
    H, D, q_len = 2, 128, 20
    kc = torch.zeros((8, H, 16, D), dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    q = torch.randn((1, q_len, 2, D), dtype=torch.float16, device=DEV)
    kn = torch.randn((q_len, H, D), dtype=torch.float16, device=DEV)
    vn = torch.randn_like(kn)
    bt = torch.tensor([[3]], dtype=torch.int32, device=DEV)      # one block: 16 positions
    cl = torch.tensor([q_len], dtype=torch.int32, device=DEV)    # needs two
    out = torch.empty_like(q)
    pa.pa_append_decode(out, q, kn, vn, kc, vc, bt, cl, 0.1, q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == pa.PA_ERR_DEVICE_CHECK
    assert torch.equal(kc[3].transpose(0, 1), kn[:16])           # positions 0..15 written
    assert int(kc[torch.arange(8, device=DEV) != 3].abs().sum()) == 0


def test_cascade_without_append_any_lengths(pa, orc):
    """Without an append the cascade is exact for any context lengths, including
    sequences shorter than the shared prefix (each row's causal limit cuts the
    prefix pass)."""
    w = workloads.make("prefix_verify", num_seqs=4, lens=("prefix", 1024, 64, 300))
    d = _dev(w)
    # shorten two sequences into the prefix; their tables keep the prefix blocks
    lens = w.context_lens.clone()
    lens[1] = 500
    lens[3] = 4
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    # the pool as a finished prefill left it (slots before each new position)
    slots = orc.slot_mapping(w.block_tables.numpy(), w.context_lens.numpy(), 16, w.cfg.q_len)
    orc.append_kv(kc, vc, w.bits("k_new"), w.bits("v_new"), slots)
    ref = orc.decode(w.bits("q"), kc, vc, w.block_tables.numpy(), lens.numpy(), w.scale,
                     w.cfg.dtype, q_len=w.cfg.q_len)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.float16).to(DEV)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.float16).to(DEV)
    out = torch.empty_like(d["q"])
    pa.pa_decode_cascade(out, d["q"], kt, vt, d["block_tables"], lens.to(DEV), w.scale,
                         w.cfg.shared_prefix // 16, q_len=w.cfg.q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    _tol.check(_f64(out), ref, w.cfg.dtype, "cascade, short sequences")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("scale", [-0.0884, 0.0], ids=["negative", "zero"])
def test_prefill_nonpositive_scale(pa, orc, dtype, scale):
    """The many-row kernel folds the scale into exp2's argument, which wants a positive
    scale: a negative one negates the score MMA instead, and zero makes every visible
    weight equal (the output is the mean of the visible V rows)."""
    lens = [40, 300, 700]
    q, K, V = _logical_case(24, lens, 8, 2, 128, dtype, q_len=40)
    pc = Paged(orc, K, V, 16, dtype, perm_seed=16)
    ref = pc.decode(orc, q, scale, q_len=40)
    _tol.check(_gpu_decode(pa, pc, q, scale, 40), ref, dtype, f"scale {scale}")
    _tol.check(_gpu_decode(pa, pc, q, scale, 40, num_splits=3), ref, dtype, f"scale {scale}, split 3")


@pytest.mark.parametrize("scale", [-0.0884, 0.0], ids=["negative", "zero"])
def test_cascade_nonpositive_scale(pa, orc, scale):
    """The shared-prefix pass (many-row kernel) and the tail pass (decode kernel) take
    the same non-positive scale."""
    w = workloads.make("prefix_verify", num_seqs=4, q_len=8)
    d = _dev(w)
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    slots = orc.slot_mapping(w.block_tables.numpy(), w.context_lens.numpy(), 16, w.cfg.q_len)
    orc.append_kv(kc, vc, w.bits("k_new"), w.bits("v_new"), slots)
    ref = orc.decode(w.bits("q"), kc, vc, w.block_tables.numpy(), w.context_lens.numpy(), scale,
                     w.cfg.dtype, q_len=w.cfg.q_len)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.float16).to(DEV)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.float16).to(DEV)
    for tail_splits in (1, 2):
        out = torch.empty_like(d["q"])
        pa.pa_decode_cascade(out, d["q"], kt, vt, d["block_tables"], d["context_lens"], scale,
                             w.cfg.shared_prefix // 16, q_len=w.cfg.q_len, tail_splits=tail_splits)
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        _tol.check(_f64(out), ref, w.cfg.dtype, f"cascade scale {scale}, tail splits {tail_splits}")


# ------------------------------------------------- many units per persistent CTA
# units = ceil(q_len * g / 128) * num_kv_heads * num_seqs (* splits), all above the
# 152 SMs, so every persistent CTA walks several units: the rings and barrier
# phases run on across units, the next unit's q replaces the previous one, and
# each epilogue is deferred into the next unit's first chunk.
MANY_UNITS = [
    # dtype, head_dim, h_q, h_kv, q_len, num_seqs
    ("fp16", 128, 12, 4, 200, 10),  # g = 3: q rows written by the softmax threads; 200 units
    ("bf16", 64, 16, 4, 160, 10),   # g = 4: q by TMA; 200 units
    ("bf16", 128, 40, 8, 70, 12),   # g = 5: q by the softmax threads; 288 units
    ("fp16", 64, 32, 8, 48, 14),    # g = 4: q by TMA, 2 row blocks per sequence; 224 units
]


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("case", MANY_UNITS, ids=[f"{c[0]}-d{c[1]}-g{c[2] // c[3]}" for c in MANY_UNITS])
def test_prefill_many_units_per_cta(pa, orc, case, splits):
    dtype, d, h_q, h_kv, q_len, n = case
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(q_len, 1200, size=n)]
    lens[1] = 3       # shorter than the chunk: the first rows see nothing
    lens[2] = q_len   # the chunk is the whole context
    lens[3] = 0       # empty sequence: zeros
    q, K, V = _logical_case(32, lens, h_q, h_kv, d, dtype, q_len=q_len)
    pc = Paged(orc, K, V, 16, dtype, perm_seed=17)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    ref = orc.decode(q, pc.k, pc.v, pc.tables, pc.lens, scale, dtype, q_len=q_len, threads=THREADS)
    _tol.check(_gpu_decode(pa, pc, q, scale, q_len, num_splits=splits), ref, dtype,
               f"{dtype} d{d} g{h_q // h_kv} q_len {q_len} split {splits}")


def test_cascade_prefix_pass_many_units_per_cta(pa, orc):
    """A shared-prefix pass with more units than SMs (128 sequences x 8 query
    positions x 4 heads per KV head = 32 row blocks per KV head, 256 units), then
    the tails: every element against the oracle."""
    w = workloads.make("prefix_verify", q_len=8)
    out, d = gpu_cascade(pa, w, tail_splits=1)
    ref, kc, vc, _ = oracle_step(orc, w)
    _tol.check(_f64(out), ref, w.cfg.dtype, "cascade, many prefix units")
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    # the same through two tail partitions and the combine
    out2, _ = gpu_cascade(pa, workloads.make("prefix_verify", q_len=8), tail_splits=2)
    _tol.check(_f64(out2), ref, w.cfg.dtype, "cascade, tail split 2")


def test_prefill_more_sequences_than_the_ranked_order_holds(pa, orc):
    """Above 256 sequences the kernel takes them in index order and reads the
    context lengths from global memory: 300 short sequences, every element."""
    rng = np.random.default_rng(41)
    lens = [int(x) for x in rng.integers(17, 120, size=300)]
    lens[7] = 0
    lens[8] = 5
    q, K, V = _logical_case(42, lens, 4, 2, 64, "fp16", q_len=17)
    pc = Paged(orc, K, V, 16, "fp16", perm_seed=18)
    ref = orc.decode(q, pc.k, pc.v, pc.tables, pc.lens, 0.125, "fp16", q_len=17, threads=THREADS)
    _tol.check(_gpu_decode(pa, pc, q, 0.125, 17), ref, "fp16", "300 sequences")
    _tol.check(_gpu_decode(pa, pc, q, 0.125, 17, num_splits=3), ref, "fp16", "300 sequences, split 3")


def test_cascade_more_sequences_than_the_ranked_order_holds(pa, orc):
    """The shared-prefix pass over 300 sequences (context lengths from global
    memory), then the tails: every element."""
    w = workloads.make("prefix_verify", num_seqs=300, q_len=2, lens=("prefix", 1024, 16, 80))
    out, d = gpu_cascade(pa, w)
    ref, kc, vc, _ = oracle_step(orc, w)
    _tol.check(_f64(out), ref, w.cfg.dtype, "cascade, 300 sequences")
    assert np.array_equal(_u16(d["k_cache"]), kc)
