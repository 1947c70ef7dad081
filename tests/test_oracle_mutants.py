"""Plausible mistakes planted in copies of the oracle must each fail a pin.

Every mutant is a textual edit of ``oracle/pa_oracle.c`` compiled into a
temporary directory and checked in a child process (a wrong index could read out
of bounds; a crash then fails only that child).  The real oracle is never
modified.  CPU only.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import build as oracle_build  # noqa: E402

MUTANTS = [
    # (name, original text, mistaken text)
    ("gqa_interleaved_heads", "*kvh = *h / group;", "*kvh = *h % c->num_kv_heads;"),
    ("no_tail_mask",
     "*T = (int64_t)c->context_lens[*i] - c->q_len + *u + 1;",
     "*T = ((int64_t)c->context_lens[*i] + c->block_size - 1) / c->block_size * c->block_size - c->q_len + *u + 1;"),
    ("no_causal_offset",
     "*T = (int64_t)c->context_lens[*i] - c->q_len + *u + 1;",
     "*T = (int64_t)c->context_lens[*i];"),
    ("scale_dropped", "return c->scale * dot;", "return dot;"),
    ("max_subtracted_backwards", "s[t] = exp(s[t] - mx);", "s[t] = exp(mx - s[t]);"),
    ("nhd_read_layout",
     "return (size_t)(((physical_block * c->num_kv_heads + h) * c->block_size + block_offset) * c->head_dim);",
     "return (size_t)(((physical_block * c->block_size + block_offset) * c->num_kv_heads + h) * c->head_dim);"),
    ("table_lookup_skipped", "out = physical_block * block_size + block_offset;",
     "out = logical_block * block_size + block_offset;"),
    ("combine_unweighted_denominator", "den += exp(m[w] - M) * l[w];", "den += l[w];"),
    ("partition_off_by_one", "int64_t t1 = t0 + C * block_size;",
     "int64_t t1 = t0 + C * block_size - 1;"),
    ("dot_drops_first_term",
     "    for (int d = 0; d < c->head_dim; d++)\n        dot +=",
     "    for (int d = 1; d < c->head_dim; d++)\n        dot +="),
    ("keys_used_as_values", "o[d] += p * cache_at(c, c->v_cache, c->v_scale, vrow + d, kvh);",
     "o[d] += p * cache_at(c, c->k_cache, c->v_scale, vrow + d, kvh);"),
    ("e4m3_exponent_bias", "v = ldexp((double)(8 + f), e - 10);",
     "v = ldexp((double)(8 + f), e - 9);"),
    ("e4m3_ties_to_odd", "(err == best_err && (c & 1) == 0 && (best & 1) == 1)",
     "(err == best_err && (c & 1) == 1 && (best & 1) == 0)"),
    ("e4m3_no_saturation", "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7E);",
     "if (a >= 480.0)\n        return (uint8_t)(sign | 0x7F);"),
    ("fp8_scales_swapped", "o[d] += p * cache_at(c, c->v_cache, c->v_scale, vrow + d, kvh);",
     "o[d] += p * cache_at(c, c->v_cache, c->k_scale, vrow + d, kvh);"),
    ("fp8_append_multiplies", "k_cache[dst] = orc_e4m3_from_float(kx / k_scale[h]);",
     "k_cache[dst] = orc_e4m3_from_float(kx * k_scale[h]);"),
    ("append_writes_key_into_value", "v_cache[dst] = v_new[src];", "v_cache[dst] = k_new[src];"),
    ("fp16_exponent_bias", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("bf16_subnormal_scale", "v = ldexp((double)f, -133);", "v = ldexp((double)f, -126);"),
    ("softmax_not_normalised", "double p = s[t] / den;", "double p = s[t];"),
    ("slot_position_off_by_one", "int64_t pos = (int64_t)context_lens[i] - q_len + u;",
     "int64_t pos = (int64_t)context_lens[i] - q_len + u + 1;"),
    ("slot_negative_position_not_skipped", "if (pos < 0) {\n                out = -1;",
     "if (pos < -block_size) {\n                out = -1;"),
    ("bf16_table_filled_by_fp16_decoder",
     "bf16_value[b] = orc_bf16_to_double((uint16_t)b);",
     "bf16_value[b] = orc_fp16_to_double((uint16_t)b);"),
    ("e4m3_table_shifted_by_one", "e4m3_value[b] = orc_e4m3_to_double((uint8_t)b);",
     "e4m3_value[b] = orc_e4m3_to_double((uint8_t)(b + 1));"),
    ("copy_blocks_wrong_direction",
     "k_cache[(int64_t)dst[i] * block_elems + e] = k_cache[(int64_t)src[i] * block_elems + e];",
     "k_cache[(int64_t)src[i] * block_elems + e] = k_cache[(int64_t)dst[i] * block_elems + e];"),
]


def _source() -> str:
    with open(oracle_build.SOURCE) as f:
        return f.read()


def _check(lib: str) -> subprocess.CompletedProcess:
    return subprocess.run([sys.executable, "-m", "tests.oracle_pins", lib], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def mutant_results():
    src = _source()
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    jobs = []
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"mutant {name}: pattern not found exactly once"
        path = os.path.join(tmp, f"{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        jobs.append((name, path, os.path.join(tmp, f"lib_{name}.so")))

    def run(job):
        name, path, lib = job
        oracle_build.build(source=path, output=lib, werror=False)
        return name, _check(lib)

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(run, jobs))


def test_real_oracle_passes_every_pin():
    lib = os.path.join(tempfile.mkdtemp(prefix="oracle_real_"), "lib.so")
    oracle_build.build(output=lib)
    res = _check(lib)
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_results, name):
    res = mutant_results[name]
    assert res.returncode != 0, f"mutant {name} passed every pin:\n{res.stdout}{res.stderr}"
