"""Seeded random configurations, CUDA path vs the fp64 oracle, every element (needs a
GPU).

Each case draws a dtype, head_dim, block size (8, 16 or 32 tokens), KV head count,
group size, q_len, context
lengths (empty, shorter than q_len and longer), a split count and fused or separate
launches, so that combinations the hand-written cases do not list still meet the
oracle.  The pool is NaN-poisoned outside the written slots.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import _tol
from tests.test_gpu_parity import DEV, _f64, _u16, gpu_step, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    assert pa.pa_device_error() == 0
    return pa


def _case(seed: int, fp8: bool):
    rng = np.random.default_rng(1000 + seed)
    h_kv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8]))
    q_len = int(rng.choice([1, 2, 3, 4, 7, 16, 17, 33, 100, 300]))
    n = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(q_len, 1500, size=n)]
    if n > 1 and rng.random() < 0.5:
        lens[int(rng.integers(n))] = int(rng.integers(0, q_len + 1))  # empty or short
    over = {"num_seqs": n, "num_q_heads": h_kv * g, "num_kv_heads": h_kv, "q_len": q_len,
            "pool_blocks": None,
            "lens": ("fixed", tuple(lens)),
            "dtype": str(rng.choice(["fp16", "bf16"])),
            "head_dim": 128 if fp8 else int(rng.choice([64, 128]))}
    splits = int(rng.choice([1, 2, 5]))
    fused = bool(rng.random() < 0.5)
    over["block_size"] = int(rng.choice([8, 16, 32]))
    return over, splits, fused


@pytest.mark.parametrize("seed", range(24))
def test_random_16bit_cache(pa, orc, seed):
    over, splits, fused = _case(seed, fp8=False)
    w = workloads.make("tiny", seed=seed, **over)
    out, d = gpu_step(pa, w, num_splits=splits, fused=fused)
    ref, kc, vc, _ = oracle_step(orc, w)
    assert np.array_equal(_u16(d["k_cache"]), kc)
    assert np.array_equal(_u16(d["v_cache"]), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{over} splits {splits} fused {fused}")


@pytest.mark.parametrize("seed", range(8))
def test_random_fp8_cache(pa, orc, seed):
    over, splits, fused = _case(seed, fp8=True)
    w = workloads.make("gqa_fp8", seed=seed, **over)
    c = w.cfg
    d = {k: getattr(w, k).to(DEV) for k in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                             "block_tables", "context_lens", "k_scale",
                                             "v_scale")}
    out = torch.empty_like(d["q"])
    if fused:
        pa.pa_decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                         d["block_tables"], d["context_lens"], w.scale, c.q_len, splits,
                         k_new=d["k_new"], v_new=d["v_new"])
    else:
        slots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], c.block_size, c.q_len)
        pa.pa_append_kv_fp8(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], slots,
                            d["k_scale"], d["v_scale"])
        pa.pa_decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                         d["block_tables"], d["context_lens"], w.scale, c.q_len, splits)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    slots = orc.slot_mapping(w.block_tables.numpy(), w.context_lens.numpy(), c.block_size, c.q_len)
    orc.append_kv_fp8(kc, vc, w.bits("k_new"), w.bits("v_new"), slots, c.dtype,
                      w.k_scale.numpy(), w.v_scale.numpy())
    ref = orc.decode_fp8(w.bits("q"), kc, vc, w.k_scale.numpy(), w.v_scale.numpy(),
                         w.block_tables.numpy(), w.context_lens.numpy(), w.scale, c.dtype,
                         q_len=c.q_len)
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(d["v_cache"].cpu().numpy(), vc)
    _tol.check(_f64(out), ref, c.dtype, f"fp8 {over} splits {splits} fused {fused}")
