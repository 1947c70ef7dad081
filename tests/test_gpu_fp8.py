"""FP8 (e4m3) KV cache through the C ABI vs the fp64 oracle (needs a GPU).

The quantising append is compared code for code; attention over the dequantised
cache within the tolerance of tests/_tol.py."""
import os

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
    assert pa.pa_device_error() == 0
    return pa


def _dev(w):
    d = {k: getattr(w, k).to(DEV) for k in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                             "block_tables", "context_lens", "k_scale", "v_scale")}
    return d


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def gpu_step(pa, w, num_splits=1, fused=True):
    d = _dev(w)
    c = w.cfg
    out = torch.empty_like(d["q"])
    if fused:
        pa.pa_decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                         d["block_tables"], d["context_lens"], w.scale, c.q_len, num_splits,
                         k_new=d["k_new"], v_new=d["v_new"])
    else:
        slots = pa.pa_slot_mapping(d["block_tables"], d["context_lens"], c.block_size, c.q_len)
        pa.pa_append_kv_fp8(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], slots,
                            d["k_scale"], d["v_scale"])
        pa.pa_decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                         d["block_tables"], d["context_lens"], w.scale, c.q_len, num_splits)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    return out, d


def oracle_step(orc, w, rows=None, threads=os.cpu_count() or 1):
    c = w.cfg
    kc, vc = w.bits("k_cache").copy(), w.bits("v_cache").copy()
    slots = orc.slot_mapping(w.block_tables.numpy(), w.context_lens.numpy(), c.block_size, c.q_len)
    orc.append_kv_fp8(kc, vc, w.bits("k_new"), w.bits("v_new"), slots, c.dtype,
                      w.k_scale.numpy(), w.v_scale.numpy())
    out = orc.decode_fp8(w.bits("q"), kc, vc, w.k_scale.numpy(), w.v_scale.numpy(),
                         w.block_tables.numpy(), w.context_lens.numpy(), w.scale, c.dtype,
                         q_len=c.q_len, rows=rows, threads=threads)
    return out, kc, vc


def test_quantising_append_matches_oracle_on_every_fp16_value(pa, orc):
    """Every fp16 bit pattern (NaN and infinity included) and a range of scales
    through the hardware e4m3 conversion: codes identical to the oracle's."""
    vals = np.arange(65536, dtype=np.uint16).reshape(512, 1, 128)    # 512 tokens, 1 head
    for scale in (1.0, 0.037, 3.5):
        kc = torch.zeros((32, 1, 16, 128), dtype=torch.uint8, device=DEV)
        vc = torch.zeros_like(kc)
        kn = torch.from_numpy(vals.view(np.int16)).view(torch.float16).to(DEV)
        slots = torch.arange(512, dtype=torch.int64, device=DEV)
        sc = torch.tensor([scale], dtype=torch.float32, device=DEV)
        pa.pa_append_kv_fp8(kc, vc, kn, kn, slots, sc, sc)
        torch.cuda.synchronize()
        ok, ov = np.zeros((32, 1, 16, 128), np.uint8), np.zeros((32, 1, 16, 128), np.uint8)
        orc.append_kv_fp8(ok, ov, vals, vals, np.arange(512), "fp16", [scale], [scale])
        assert np.array_equal(kc.cpu().numpy(), ok), scale
        assert np.array_equal(vc.cpu().numpy(), ov), scale


SMALL = [("llama7b_mha_fp8", {"num_seqs": 3}), ("gqa_fp8", {"num_seqs": 5}),
         ("gqa_fp8", {"num_seqs": 4, "num_q_heads": 8, "num_kv_heads": 4}),      # 2 rows
         ("gqa_fp8", {"num_seqs": 4, "q_len": 4}),                               # 16 rows
         ("llama7b_mha_fp8", {"num_seqs": 2, "num_q_heads": 32, "num_kv_heads": 1,
                              "dtype": "bf16"}),                                 # 32 rows
         ("gqa_fp8", {"num_seqs": 4, "q_len": 2, "dtype": "fp16"}),             # 8 rows, causal
         ("gqa_fp8", {"num_seqs": 5, "num_q_heads": 12, "num_kv_heads": 4}),    # 3 rows
         # more than 16 rows per KV head: the tensor-core many-row kernel, the codes
         # widened to fp16 in shared memory; a bf16 q is converted (row-scaled) by
         # the softmax threads, an fp16 one arrives by TMA when the group divides 128
         ("gqa_fp8", {"num_seqs": 3, "q_len": 40, "lens": ("fixed", (40, 300, 1000))}),
         ("llama7b_mha_fp8", {"num_seqs": 2, "q_len": 24, "num_q_heads": 8,
                              "num_kv_heads": 8, "lens": ("fixed", (30, 700))}),
         ("gqa_fp8", {"num_seqs": 3, "q_len": 100, "dtype": "fp16",
                      "lens": ("fixed", (100, 357, 1500))}),                  # q by TMA
         ("gqa_fp8", {"num_seqs": 2, "q_len": 64, "num_q_heads": 10, "num_kv_heads": 2,
                      "lens": ("fixed", (64, 900))}),                          # g = 5
         ("chunked_prefill_fp8", {"num_seqs": 2, "q_len": 130, "lens": ("fixed", (130, 2000))})]


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("name,over", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_fp8_small_every_element(pa, orc, name, over, splits, fused):
    w = workloads.make(name, **over)
    out, d = gpu_step(pa, w, splits, fused)
    ref, kc, vc = oracle_step(orc, w)
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(d["v_cache"].cpu().numpy(), vc)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{name} {over} splits {splits}")


# The swapped-operand path launches 3-warp CTAs while the units fit in one wave of
# them and 4-warp CTAs above: 7B over FP8 with q_len 4 (1024 units of 4 rows) and
# 96 GQA sequences (768 units) take the 4-warp form.
FULL = [("llama7b_mha_fp8", {}), ("gqa_fp8", {}),
        ("llama7b_mha_fp8", {"q_len": 4, "pool_blocks": None}),
        ("gqa_fp8", {"num_seqs": 96, "pool_blocks": None}),
        ("chunked_prefill_fp8", {})]


@pytest.mark.parametrize("name,over", FULL, ids=["7b", "gqa", "7b-q4", "gqa-96", "chunked"])
def test_fp8_full_size_every_element(pa, orc, name, over):
    w = workloads.make(name, **over)
    out, d = gpu_step(pa, w)
    ref, kc, vc = oracle_step(orc, w)
    _tol.check(_f64(out), ref, w.cfg.dtype, f"{name} {over}")
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(d["v_cache"].cpu().numpy(), vc)


def test_fp8_edge_lengths(pa, orc):
    cfg = workloads.config("gqa_fp8", num_seqs=9, q_len=2,
                           lens=("fixed", (0, 1, 3, 15, 16, 17, 33, 100, 257)), spare_blocks=3)
    w = workloads.make(cfg)
    for splits in (1, 40):
        out, d = gpu_step(pa, w, splits)
        ref, kc, vc = oracle_step(orc, w)
        _tol.check(_f64(out), ref, "bf16", f"edges splits {splits}")


@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_many_rows_edge_lengths(pa, orc, splits):
    """33 query rows per sequence (132 per KV head: the many-row kernel) over contexts
    shorter than, equal to and longer than q_len, empty ones included."""
    cfg = workloads.config("gqa_fp8", num_seqs=9, q_len=33,
                           lens=("fixed", (0, 1, 3, 15, 16, 17, 33, 100, 257)), spare_blocks=3)
    w = workloads.make(cfg)
    out, d = gpu_step(pa, w, splits)
    ref, kc, vc = oracle_step(orc, w)
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    _tol.check(_f64(out), ref, "bf16", f"many-row edges splits {splits}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_many_rows_scales_and_q_magnitudes(pa, orc, dtype):
    """The many-row kernel folds each KV head's K scale into the score scale (a
    negative one negates the scores) and its V scale into the output, and scales
    each q row into fp16 by a power of two: negative, tiny and zero scales, and q
    rows of very different magnitudes."""
    w = workloads.make("gqa_fp8", num_seqs=3, q_len=40, dtype=dtype,
                       lens=("fixed", (40, 333, 1200)))
    ks, vs = w.k_scale.clone(), w.v_scale.clone()
    ks[0], ks[1], ks[2] = -ks[0], 1e-7, 0.0
    vs[3], vs[4] = -vs[3], 0.0
    w.k_scale.copy_(ks)
    w.v_scale.copy_(vs)
    q = w.q.float()
    q[0] *= 300.0 if dtype == "bf16" else 30.0      # large rows (bf16: scaled into fp16)
    q[1, :, :4] *= 1e-3                              # small rows
    w.q.copy_(q.to(w.q.dtype))
    out, d = gpu_step(pa, w)
    ref, kc, vc = oracle_step(orc, w)
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(d["v_cache"].cpu().numpy(), vc)
    _tol.check(_f64(out), ref, dtype, f"scales and magnitudes {dtype}")
