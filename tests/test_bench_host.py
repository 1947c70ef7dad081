"""Host logic of bench.py and the workload recipes, on CPU (no GPU).

The byte and flop counts behind every roofline figure are checked against
independent counts: KV bytes per token from the cache layout, unique tokens from
the distinct slots the block tables reach, causal FLOPs by enumerating visible
(query row, position) pairs.  The clock summary is checked on planted samples and
the traffic record on a copy of the sources that then changes.
"""
import os
import shutil

import numpy as np
import pytest

import bench
import workloads

ELT16 = 2


@pytest.mark.parametrize("name,expect", [("llama7b_mha", 16384), ("gqa", 4096),
                                         ("long_split", 4096), ("prefix_verify", 4096),
                                         ("llama7b_mha_fp8", 8192), ("gqa_fp8", 2048),
                                         ("chunked_prefill", 4096)])
def test_bytes_per_kv_token(name, expect):
    # K and V of one token: 2 * num_kv_heads * head_dim elements of the cache type
    w = workloads.make(name, poison=False)
    c = w.cfg
    elt = 1 if c.kv_fp8 else ELT16
    assert 2 * c.num_kv_heads * c.head_dim * elt == expect
    assert bench.algorithmic_bytes(w)["per_token"] == expect


@pytest.mark.parametrize("name,over", [("tiny", {}), ("prefix_verify", {"num_seqs": 6}),
                                       ("gqa", {"num_seqs": 5})])
def test_unique_tokens_match_distinct_slots(name, over):
    # every (physical block, row) the tables reach for positions < context_len,
    # counted once: a shared prefix's slots are one set for all sequences
    w = workloads.make(name, poison=False, **over)
    c = w.cfg
    tables, lens = w.block_tables.numpy(), w.context_lens.numpy()
    slots = set()
    for i in range(c.num_seqs):
        for pos in range(int(lens[i])):
            slots.add(int(tables[i, pos // c.block_size]) * c.block_size + pos % c.block_size)
    assert w.info["unique_tokens"] == len(slots)
    assert bench.algorithmic_bytes(w)["kv"] == len(slots) * bench.algorithmic_bytes(w)["per_token"]


@pytest.mark.parametrize("q_len,lens", [(1, (5, 0, 17)), (4, (4, 2, 9, 40)), (7, (3, 7, 30))])
def test_attention_flops_enumerate_visible_pairs(q_len, lens):
    # query u of a sequence of length L sees positions t <= L - q_len + u; each visible
    # (row, position) costs 2*D multiply-adds for the score and 2*D for P.V
    w = workloads.make("tiny", poison=False, q_len=q_len, pool_blocks=None,
                       num_seqs=len(lens), lens=("fixed", lens))
    c = w.cfg
    pairs = 0
    for L in w.context_lens.numpy():
        for u in range(q_len):
            pairs += sum(1 for t in range(int(L)) if t <= int(L) - q_len + u)
    assert bench.attention_flops(w) == 4 * c.head_dim * c.num_q_heads * pairs


def test_clock_summary_from_samples(tmp_path, monkeypatch):
    monkeypatch.setenv("PA_BENCH_OUT", str(tmp_path))
    cs = bench.ClockSampler(0)
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line",
            "0, 2055, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    with open(cs.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    cs.proc = object()  # as if nvidia-smi had run
    s = cs.summary()
    assert s["samples"] == 4
    assert s["sm_mhz"] == 2062.5 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    cs.proc = None      # no sampler: no claim
    assert cs.summary() is None


def test_traffic_record_void_once_a_source_changes(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    src = os.path.join(bench.ROOT, "paged_kv_cache_20_gb300", "csrc")
    shutil.copytree(src, root / "paged_kv_cache_20_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.kernel_source_sha("decode")
    (root / "profiles" / "dram_traffic.txt").write_text(
        "# header\n"
        f"kernel=paged_decode_kernel(append+attention) config=gqa src_sha={sha} "
        "dram_bytes_per_launch=123 source=x.md\n")
    assert bench.traffic_record("paged_decode_kernel(append+attention)", "gqa") == 123.0
    assert bench.traffic_record("paged_decode_kernel(append+attention)", "llama7b_mha") is None
    p = root / "paged_kv_cache_20_gb300" / "csrc" / "pa_decode_inst.cuh"
    text = p.read_text()
    # comments and layout do not change what was measured
    p.write_text("/* reworded */\n" + text.replace("\n", "\n  ") + "\n// a note\n")
    assert bench.kernel_source_sha("decode") == sha
    # code does
    p.write_text(text + "\nstatic const int kChanged = 1;\n")
    assert bench.kernel_source_sha("decode") != sha
    assert bench.traffic_record("paged_decode_kernel(append+attention)", "gqa") is None


def test_code_tokens_keep_literals_and_drop_comments():
    src = 'int a = 1; // one\n/* two\nlines */ const char *s = "x // y /* z */"; char c = \'"\';'
    assert bench.code_tokens(src) == 'int a = 1; const char *s = "x // y /* z */"; char c = \'"\';'
    assert bench.code_tokens('s = "q \\" // in"; // out\nt') == 's = "q \\" // in"; t'


def test_workload_recipes_as_documented():
    # GQA: 64 lognormal lengths (median 1500, sigma 0.5, cap 8192), seed 0
    g = workloads.make("gqa", poison=False)
    L = g.context_lens.numpy()
    assert int(L.sum()) == 113339 and L.max() <= 8192 and L.min() >= 1
    assert torch_equal(g, workloads.make("gqa", poison=False))
    assert not torch_equal(g, workloads.make("gqa", poison=False, seed=1))
    # prefix_verify: every sequence repeats the 64 shared blocks of row 0
    p = workloads.make("prefix_verify", poison=False)
    t = p.block_tables.numpy()
    nb = p.cfg.shared_prefix // p.cfg.block_size
    assert nb == 64 and (t[:, :nb] == t[0, :nb]).all()
    private = t[:, nb:][t[:, nb:] >= 0]
    used = set()
    for i, L in enumerate(p.context_lens.numpy()):
        used.update(int(b) for b in t[i, nb:(int(L) + 15) // 16])
    assert not used & set(int(b) for b in t[0, :nb])  # private blocks never shared
    assert len(private) >= len(used)
    # long_split: 4 sequences of 32K tokens, 16 partitions
    s = workloads.make("long_split", poison=False)
    assert (s.context_lens.numpy() == 32768).all() and s.cfg.num_splits == 16


def torch_equal(a, b) -> bool:
    return all(np.array_equal(getattr(a, k).numpy(), getattr(b, k).numpy())
               for k in ("context_lens", "block_tables")) and \
        np.array_equal(a.bits("q"), b.bits("q"))
