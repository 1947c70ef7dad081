"""Benchmark: paged decode attention (append + attend) on GB300.

One step = one pass of the whole hot path over one batch: slot mapping, append of
the new K/V rows, attention (plus the combine for a split-KV workload), on one
stream, with every input resident in HBM.  The timed step is the fused entry
point pa_append_decode (one launch); the same step as separate launches
(pa_slot_mapping -> pa_append_kv -> pa_decode, or the partial/combine pair) is
timed too and reported as "separate_launches_ms_per_step".

Metric: KV tokens/s = sum of context lengths / step time (a token is counted once
per sequence, whatever the number of heads or query rows), with the achieved HBM
bandwidth of the attention kernel as a fraction of the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Default workload: llama7b_mha (32 seqs, 32/32 heads, head_dim 128, fp16, context
lengths uniform in [512, 4096]).  The other workloads are measured the same way
and reported under "other_configs" (skip with --only).  Under torchrun each rank
runs its own independent batch (different seed) on its own GPU: weak scaling,
no collective on the data path; the barrier and the max-over-ranks reduction are
timing only.

--impl reference times the fp64 CPU oracle (the checker, plain C) on the host
cores on a bounded sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attention: KV tokens/s and achieved HBM GB/s (% of GB300 peak)"
UNIT = "KV tokens/s"
DEFAULT_CONFIG = "llama7b_mha"
# gqa last: the end of the printed line carries it in full even where only the
# line's tail is kept
OTHER_CONFIGS = ["long_split", "prefix_verify", "llama7b_mha_fp8", "gqa_fp8", "chunked_prefill",
                 "chunked_prefill_fp8", "gqa"]
DECODE_MAX_QLEN = 16              # more query rows per sequence go to the prefill kernel
L2_BYTES = 129 << 20             # GB300 L2; every workload's KV cache is several times larger
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
ELT = 2                           # bytes per fp16 / bf16 element


# --------------------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


def algorithmic_bytes(w: workloads.Workload) -> dict:
    """Bytes the step must move at minimum (unique KV once, q, out, tables, lens, append)."""
    c = w.cfg
    kv_elt = 1 if c.kv_fp8 else ELT
    per_token = 2 * c.num_kv_heads * c.head_dim * kv_elt       # K and V of one token, one layer
    lens = w.context_lens.numpy().astype(np.int64)
    nb = (lens + c.block_size - 1) // c.block_size
    kv = w.info["unique_tokens"] * per_token
    q = c.num_seqs * c.q_len * c.num_q_heads * c.head_dim * ELT
    out = q
    tables = int(nb.sum()) * 4 + c.num_seqs * 4
    n_new = c.num_seqs * c.q_len
    append = 2 * n_new * c.num_kv_heads * c.head_dim * (ELT + kv_elt)  # read rows, write slots
    ws = 0
    if c.num_splits > 1:   # partial writes, combine reads, per row: D + 2 floats
        rows = c.num_seqs * c.num_splits * c.q_len * c.num_q_heads
        ws = 2 * rows * (c.head_dim + 2) * 4
    # the attention launch: reads unique KV, q, tables; writes out (or the workspace)
    decode = kv + q + tables + (ws // 2 if c.num_splits > 1 else out)
    # the fused step's attention launch(es): the above, plus the append it performs,
    # plus (split-KV) the combine reading the workspace and writing out
    fused = decode + append + (ws // 2 + out if c.num_splits > 1 else 0)
    return {"per_token": per_token, "kv": kv, "decode_launch": decode, "fused_launch": fused,
            "step": kv + q + out + tables + append + ws + n_new * 8}


def attention_flops(w: workloads.Workload) -> float:
    """Multiply-adds of the attention proper, x2: for every query row, 2*D for its
    scores and 2*D for P.V per visible position (causal window)."""
    c = w.cfg
    lens = w.context_lens.numpy().astype(np.int64)
    u = np.arange(c.q_len, dtype=np.int64)
    visible = np.clip(lens[:, None] - c.q_len + u[None, :] + 1, 0, None)
    return float(4 * c.head_dim * c.num_q_heads * int(visible.sum()))


# the sources each timed kernel is built from (its traffic record is void once any
# of them changes)
_COMMON_SRC = ("pa_device.cuh", "pa_launch.h", "pa_api.cu", "pa_decode.cuh")
KERNEL_SOURCES = {
    "decode": _COMMON_SRC + ("pa_decode_inst.cuh", "pa_decode_fp16.cu", "pa_decode_bf16.cu"),
    "prefill": _COMMON_SRC + ("pa_prefill_tc.cuh", "pa_tc.cuh", "pa_prefill_inst.cuh",
                              "pa_prefill.cu"),
}


def traffic_record(kernel_name: str, config: str):
    """dram bytes per launch from the committed ncu summary, if the kernel source is
    unchanged since the counters were taken (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want_sha = kernel_source_sha("prefill" if "prefill" in kernel_name else "decode")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv = dict(x.split("=", 1) for x in line.split())
        if kv.get("config") == config and kv.get("kernel") == kernel_name and \
                kv.get("src_sha") == want_sha:
            return float(kv["dram_bytes_per_launch"])
    return None


def code_tokens(text: str) -> str:
    """C/C++/CUDA source with its comments removed and whitespace runs collapsed
    (string and character literals kept as written): what the compiler sees, so
    that a change of wording in a comment does not void a measurement."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                                  # literal: copy through its close
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha(kernel: str = "decode") -> str:
    """Hash of the code (comments and layout aside) a timed kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_20_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary); PA_BENCH_OUT overrides
        out_dir = os.environ.get("PA_BENCH_OUT", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"pagedattn_clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- our arm
class Runner:
    """Device buffers and launch sequence for one workload."""

    def __init__(self, pa, w: workloads.Workload, device):
        self.pa, self.w, self.dev = pa, w, device
        c = w.cfg
        names = ["q", "k_new", "v_new", "k_cache", "v_cache", "block_tables", "context_lens"]
        if c.kv_fp8:
            names += ["k_scale", "v_scale"]
        self.d = {k: getattr(w, k).to(device) for k in names}
        self.out = torch.empty_like(self.d["q"])
        self.slots = torch.empty(c.num_seqs * c.q_len, dtype=torch.int64, device=device)
        self.ws = None
        if c.num_splits > 1:
            nbytes = pa.pa_decode_workspace_size(c.num_seqs, c.num_q_heads, c.q_len, c.head_dim,
                                                 c.num_splits)
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        split = 1 if c.num_splits > 1 else 0
        prefill = 1 if c.q_len > DECODE_MAX_QLEN else 0       # separate append launch
        self.mode = "fused"
        self.launches = {"fused": 1 + prefill + split, "separate": 3 + split,
                         "cascade": 3 + prefill}
        if c.shared_prefix:
            self.cascade_ws = torch.empty(
                pa.pa_decode_workspace_size(c.num_seqs, c.num_q_heads, c.q_len, c.head_dim, 2),
                dtype=torch.uint8, device=device)

    @property
    def fused(self) -> bool:
        return self.mode == "fused"

    @fused.setter
    def fused(self, value: bool):
        self.mode = "fused" if value else "separate"

    @property
    def launches_per_step(self) -> int:
        return self.launches[self.mode]

    def step(self, ev_pair=None):
        if self.mode == "fused":
            return self.step_fused(ev_pair)
        if self.mode == "cascade":
            return self.step_cascade(ev_pair)
        return self.step_separate(ev_pair)

    def step_cascade(self, ev_pair=None):
        """pa_decode_cascade with the append: the shared prefix once for all query
        rows, each sequence's own blocks, then the combine."""
        pa, d, c = self.pa, self.d, self.w.cfg
        if ev_pair is not None:
            ev_pair[0].record()
        pa.pa_decode_cascade(self.out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], self.w.scale, c.shared_prefix // c.block_size,
                             q_len=c.q_len, tail_splits=1, k_new=d["k_new"], v_new=d["v_new"],
                             workspace=self.cascade_ws)
        if ev_pair is not None:
            ev_pair[1].record()

    def step_fused(self, ev_pair=None):
        """pa_append_decode: slot mapping, append and attention in one launch (plus the
        combine for a split-KV workload); the events bracket the whole call."""
        pa, d, c = self.pa, self.d, self.w.cfg
        if ev_pair is not None:
            ev_pair[0].record()
        if c.kv_fp8:
            pa.pa_decode_fp8(self.out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"],
                             d["v_scale"], d["block_tables"], d["context_lens"], self.w.scale,
                             c.q_len, c.num_splits, self.ws, k_new=d["k_new"], v_new=d["v_new"])
        else:
            pa.pa_append_decode(self.out, d["q"], d["k_new"], d["v_new"], d["k_cache"],
                                d["v_cache"], d["block_tables"], d["context_lens"], self.w.scale,
                                c.q_len, c.num_splits, self.ws)
        if ev_pair is not None:
            ev_pair[1].record()

    def step_separate(self, ev_pair=None):
        """pa_slot_mapping, pa_append_kv, then the attention launch(es) on their own."""
        pa, d, c = self.pa, self.d, self.w.cfg
        pa.pa_slot_mapping(d["block_tables"], d["context_lens"], c.block_size, c.q_len,
                           out=self.slots)
        if c.kv_fp8:
            pa.pa_append_kv_fp8(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], self.slots,
                                d["k_scale"], d["v_scale"])
            if ev_pair is not None:
                ev_pair[0].record()
            pa.pa_decode_fp8(self.out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"],
                             d["v_scale"], d["block_tables"], d["context_lens"], self.w.scale,
                             c.q_len, c.num_splits, self.ws)
            if ev_pair is not None:
                ev_pair[1].record()
            return
        pa.pa_append_kv(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], self.slots)
        if ev_pair is not None:
            ev_pair[0].record()
        if c.num_splits > 1:
            pa.pa_decode_partial(self.ws, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                 d["context_lens"], self.w.scale, c.num_splits, c.q_len)
            if ev_pair is not None:
                ev_pair[1].record()
            pa.pa_decode_combine(self.out, self.ws, c.num_splits)
        else:
            pa.pa_decode(self.out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                         d["context_lens"], self.w.scale, c.q_len)
            if ev_pair is not None:
                ev_pair[1].record()


def l2_read_through(buf: torch.Tensor) -> None:
    """Read every byte of a buffer of at least twice the L2 (a reduction whose
    result is discarded): the next kernel finds none of the previous step's lines
    in L2, and no dirty lines are left for it to write back."""
    torch.sum(buf)


def time_device(runner: Runner, steps: int, warmup: int, world: int, evict=None):
    """Time exactly `steps` steps twice, after `warmup` untimed ones.
    - Back to back, with one event pair around all of them: the headline.
      Launches follow each other on the stream as in a serving loop.
    - With events around every step and around its attention launch: per-step
      percentiles and per-launch kernel times.  Those events sit between the
      launches, so this pass is slower.
    - With `evict` (a buffer >= 2x L2): a third pass like the second with an
      untimed read-through of that buffer before every step, so no step finds
      the previous one's data in L2; its per-launch kernel times are returned
      as a fifth value.
    Each pass is bracketed by a barrier and a device synchronisation on both
    sides."""
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # back to back
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    a, b = E(), E()
    # Hold the GPU for a moment while the host enqueues every timed step, so the
    # events measure back-to-back device execution, not host launch latency.
    torch.cuda._sleep(int(2e7))
    a.record()
    for _ in range(steps):
        runner.step()
    b.record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    loop_ms = a.elapsed_time(b)
    # instrumented
    evs = [(E(), E(), E(), E()) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e7))
    for s0, s1, k0, k1 in evs:
        s0.record()
        runner.step((k0, k1))
        s1.record()
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [x.elapsed_time(y) for x, y, _, _ in evs]
    kern_ms = [x.elapsed_time(y) for _, _, x, y in evs]
    if evict is None:
        return loop_ms, step_ms, kern_ms, wall
    ev2 = [(E(), E()) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for k0, k1 in ev2:
        l2_read_through(evict)
        runner.step((k0, k1))
    torch.cuda.synchronize()
    barrier(world)
    return loop_ms, step_ms, kern_ms, wall, [x.elapsed_time(y) for x, y in ev2]


def time_graph(runner: Runner, steps: int, warmup: int):
    """The fused step captured once in a CUDA graph, then replayed: the launches'
    host cost leaves the step (each replay is one graph launch)."""
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        runner.step()  # first use of every buffer on the capturing stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        runner.step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [(E(), E()) for _ in range(steps)]
    torch.cuda._sleep(int(2e7))
    for a, b in evs:
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_e2e(runner: Runner, steps: int, warmup: int):
    """Same step through the public API with the inputs in pinned host memory:
    H2D of q, new K/V rows, block tables and context lengths, then the step, then
    D2H of the output, every step inside the timed region.

    The loop is the one a serving engine runs: the step's inputs sit in one pinned
    host buffer and go over in one copy, into one device buffer whose slices are
    the tensors the step reads.  Inputs and outputs are double-buffered, so step
    i+1's H2D copy (one stream) and step i-1's D2H copy (another stream) overlap
    step i's kernels.  Events order each copy after the step that frees its buffer.
    The result is the whole loop's time over the number of steps."""
    w = runner.w
    names = ("q", "k_new", "v_new", "block_tables", "context_lens")
    srcs = {k: getattr(w, k).contiguous() for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (srcs[k].numel() * srcs[k].element_size() + 255) // 256 * 256
    host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in names:
        n = srcs[k].numel() * srcs[k].element_size()
        host_in[offs[k]:offs[k] + n].copy_(srcs[k].view(-1).view(torch.uint8))
    dev_in = [torch.empty(total, dtype=torch.uint8, device=runner.dev) for _ in range(2)]
    views = [{k: dev_in[b][offs[k]:offs[k] + srcs[k].numel() * srcs[k].element_size()]
              .view(srcs[k].dtype).view(srcs[k].shape) for k in names} for b in range(2)]
    outs = [torch.empty_like(runner.out) for _ in range(2)]
    host_out = [torch.empty(runner.out.shape, dtype=runner.out.dtype).pin_memory()
                for _ in range(2)]
    h2d = sum(srcs[k].numel() * srcs[k].element_size() for k in names)
    d2h = host_out[0].numel() * host_out[0].element_size()
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    saved_d = {k: runner.d[k] for k in names}
    saved_out = runner.out

    def loop(n):
        in_ready = [ev(), ev()]    # H2D into buffer b done
        in_free = [ev(), ev()]     # the step reading buffer b done
        out_ready = [ev(), ev()]   # the step writing output b done
        out_free = [ev(), ev()]    # D2H of output b done
        started = [False, False]
        for b in range(min(2, n)):
            with torch.cuda.stream(up):
                dev_in[b].copy_(host_in, non_blocking=True)
                in_ready[b].record(up)
        for i in range(n):
            b = i & 1
            main.wait_event(in_ready[b])
            if started[b]:
                main.wait_event(out_free[b])
            runner.d.update(views[b])
            runner.out = outs[b]
            runner.step()
            in_free[b].record(main)
            out_ready[b].record(main)
            started[b] = True
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                host_out[b].copy_(outs[b], non_blocking=True)
                out_free[b].record(down)
            if i + 2 < n:
                with torch.cuda.stream(up):
                    up.wait_event(in_free[b])
                    dev_in[b].copy_(host_in, non_blocking=True)
                    in_ready[b].record(up)
        main.wait_stream(down)
        main.wait_stream(up)

    try:
        loop(max(2, warmup))
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        up.wait_stream(main)
        down.wait_stream(main)
        loop(steps)
        t1.record(main)
        torch.cuda.synchronize()
        last = outs[(steps - 1) & 1].clone()
    finally:
        runner.d.update(saved_d)
        runner.out = saved_out
    # every D2H copy landed: the last step's output is in its host buffer
    assert torch.equal(host_out[(steps - 1) & 1], last.cpu())
    per = t0.elapsed_time(t1) / steps
    return [per] * steps, h2d, d2h


def cpu_baseline(w: workloads.Workload, budget_s: float = 5.0) -> dict:
    """The oracle as it stands, on the host cores, over the same workload: slot
    mapping, append and attention sequence by sequence, repeated until the time
    budget is spent.  Value in KV tokens/s, with all cores working on each
    sequence's rows; a shorter run on one thread is reported beside it."""
    import oracle
    orc = oracle.get()
    c = w.cfg
    kc, vc = w.bits("k_cache"), w.bits("v_cache")        # append is idempotent: in place
    bt, cl = w.block_tables.numpy(), w.context_lens.numpy()
    slots = orc.slot_mapping(bt, cl, c.block_size, c.q_len)
    qb = w.bits("q")
    rows_per_seq = c.q_len * c.num_q_heads

    def run(threads, budget):
        done_tokens, done_seqs, passes = 0, 0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget and passes < 100:
            for i in range(c.num_seqs):
                sl = slice(i * c.q_len, (i + 1) * c.q_len)
                orc.append_kv(kc, vc, w.bits("k_new")[sl], w.bits("v_new")[sl], slots[sl])
                rows = np.arange(i * rows_per_seq, (i + 1) * rows_per_seq)
                orc.decode(qb, kc, vc, bt, cl, w.scale, c.dtype, q_len=c.q_len, rows=rows,
                           threads=threads)
                done_tokens += int(cl[i])
                done_seqs += 1
                if time.perf_counter() - t0 > budget:
                    break
            passes += 1
        return done_tokens, done_seqs, passes, time.perf_counter() - t0

    threads = os.cpu_count() or 1
    done_tokens, done_seqs, passes, dt = run(threads, budget_s)
    one_tokens, one_seqs, _, one_dt = run(1, budget_s / 2)
    return {"value": done_tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{c.name}: {done_seqs} sequence-steps ({passes} pass(es) over the "
                      f"{c.num_seqs} sequences, {done_tokens} KV tokens), fp64 C oracle, "
                      f"{threads} threads, {dt:.1f} s wall",
            "single_thread": {"value": one_tokens / one_dt, "unit": UNIT, "cores": 1,
                              "sample": f"{one_seqs} sequence-steps ({one_tokens} KV tokens), "
                                        f"{one_dt:.1f} s wall"}}


def measure_config(pa, name, seed, device, steps, warmup, world, peaks, e2e=False,
                   num_seqs=None):
    over = {"num_seqs": num_seqs} if num_seqs else {}
    w = workloads.make(name, seed=seed, poison=False, **over)
    runner = Runner(pa, w, device)
    # the unfused sequence first (reported for comparison), then the fused step
    runner.fused = False
    sep_loop, _, sep_kern_ms, _ = time_device(runner, steps, warmup, world)
    runner.fused = True
    evict = torch.empty(2 * L2_BYTES // 4 + 1024, dtype=torch.float32, device=device).fill_(1.0)
    loop_ms, step_ms, kern_ms, wall, ev_ms = time_device(runner, steps, warmup, world, evict)
    del evict
    assert pa.pa_device_error() == 0, "device error during the timed run"
    ab = algorithmic_bytes(w)
    total_ms = max_over_ranks(loop_ms, world, device)
    tokens = sum_over_ranks(float(w.total_tokens), world, device)
    ms_per_step = total_ms / steps
    kern_avg = statistics.mean(kern_ms)
    split = w.cfg.num_splits > 1
    kern_name = ("paged_decode_kernel(append+partial)+split_combine_kernel" if split
                 else "paged_decode_kernel(append+attention)")
    achieved = ab["fused_launch"] / (kern_avg * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    res = {
        "w": w, "runner": runner, "ms_per_step": ms_per_step, "value": tokens / (ms_per_step * 1e-3),
        "wall_s": wall,
        "step_ms_p10_p50_p90": [float(np.percentile(step_ms, p)) for p in (10, 50, 90)],
        "instrumented_ms_per_step": max_over_ranks(sum(step_ms), world, device) / steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic_record(kern_name, name), "kernel": kern_name,
                     "kernel_us": kern_avg * 1e3,
                     "kernel_us_l2_evicted": statistics.mean(ev_ms) * 1e3,
                     "frac_l2_evicted": ab["fused_launch"] / (statistics.mean(ev_ms) * 1e-3)
                     / 1e9 / peak,
                     "bytes_per_launch": ab["fused_launch"],
                     "bytes_per_kv_token": ab["per_token"],
                     "attention_only_kernel_us": statistics.mean(sep_kern_ms) * 1e3},
        "step_gbs": ab["step"] / (ms_per_step * 1e-3) / 1e9,
        "separate_launches_ms_per_step": max_over_ranks(sep_loop, world, device) / steps,
    }
    if w.cfg.q_len > DECODE_MAX_QLEN:
        # many query rows: the attention is a dense contraction; report it against
        # the tensor-core peak as well
        fl = attention_flops(w)
        tpeak = peaks.get("bf16_tflops")
        res["tensor_roofline"] = {
            "bound": "tensor", "flops_per_step": fl,
            "achieved": fl / (kern_avg * 1e-3) / 1e12,
            "peak": tpeak or 1900.0, "unit": "TFLOP/s",
            "frac": fl / (kern_avg * 1e-3) / 1e12 / (tpeak or 1900.0),
            "peak_source": "measured bf16 dense (burst)" if tpeak else "fallback",
            "kernel": ("append_step_fp8_kernel+paged_prefill_tc_kernel (tcgen05.mma, M = 128, "
                       "e4m3 codes widened to fp16 in shared memory)" if w.cfg.kv_fp8 else
                       "append_step_kernel+paged_prefill_tc_kernel (tcgen05.mma, M = 128)")}
        res["roofline"]["kernel"] = ("append_step_fp8_kernel+paged_prefill_tc_kernel" if w.cfg.kv_fp8
                                     else "append_step_kernel+paged_prefill_kernel")
        res["roofline"]["traffic"] = traffic_record("paged_prefill_tc_kernel", name)
    if w.cfg.shared_prefix:
        runner.mode = "cascade"
        c_loop, _, c_kern, _ = time_device(runner, steps, warmup, world)
        assert pa.pa_device_error() == 0, "device error during the timed cascade run"
        c_step = max_over_ranks(c_loop, world, device) / steps
        res["cascade"] = {"ms_per_step": c_step, "value": tokens / (c_step * 1e-3),
                          "kernel_us": statistics.mean(c_kern) * 1e3,
                          "path": "pa_decode_cascade (shared-prefix pass, tail pass with "
                                  "fused append, combine: 3 launches)"}
        runner.mode = "fused"
    if e2e:
        # the same step as one CUDA graph replay (reported beside the stream timing)
        try:
            g_ms = time_graph(runner, steps, max(3, warmup))
            assert pa.pa_device_error() == 0, "device error during the graph replays"
            g_step = max_over_ranks(sum(g_ms), world, device) / steps
            res["graph"] = {"ms_per_step": g_step, "value": tokens / (g_step * 1e-3),
                            "unit": UNIT,
                            "path": "the fused step captured in a CUDA graph, replayed"}
        except RuntimeError as exc:  # capture refused: report it, keep the bench line
            res["graph"] = {"error": str(exc).splitlines()[0][:200]}
        ms, h2d, d2h = time_e2e(runner, steps, max(3, warmup))
        e_ms = max_over_ranks(sum(ms), world, device) / steps
        res["e2e"] = {"value": tokens / (e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
    return res


def config_obj(w: workloads.Workload, path: str) -> dict:
    c = w.cfg
    return {"workload": c.name, "num_seqs": c.num_seqs, "num_q_heads": c.num_q_heads,
            "num_kv_heads": c.num_kv_heads, "head_dim": c.head_dim, "block_size": c.block_size,
            "kv_dtype": "e4m3 (per-KV-head scales)" if c.kv_fp8 else c.dtype,
            "q_dtype": c.dtype, "q_len": c.q_len, "num_splits": c.num_splits,
            "context_tokens": w.total_tokens, "unique_kv_tokens": w.info["unique_tokens"],
            "pool_blocks": w.num_blocks, "path": path}


def config_l2(w: workloads.Workload) -> str:
    c = w.cfg
    mib = w.info["unique_tokens"] * 2 * c.num_kv_heads * c.head_dim * (1 if c.kv_fp8 else ELT) / 2**20
    return (f"not flushed between the back-to-back steps: the KV cache read each step is "
            f"{mib:.0f} MiB, larger than the {L2_BYTES >> 20} MiB L2; the roofline's "
            f"kernel_us_l2_evicted repeats the kernel timing with a read-through of "
            f"{2 * L2_BYTES >> 20} MiB before every step")


def run_ours(args):
    world, rank, local = dist_env()
    init_dist(world)
    import paged_kv_cache_20_gb300 as pa
    assert torch.cuda.is_available(), "bench needs a GPU"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pa.load()
    peaks = measured_peaks()
    main = args.config
    with ClockSampler(local) as clk:
        r = measure_config(pa, main, rank, device, args.steps, args.warmup, world, peaks,
                           e2e=not args.no_e2e, num_seqs=args.num_seqs)
    clocks = clk.summary()
    others = {}
    if not args.only:
        for name in OTHER_CONFIGS:
            if name == main:
                continue
            o = measure_config(pa, name, rank, device, args.steps, args.warmup, world, peaks)
            others[name] = other_entry(o)
            del o
    copy = None if args.only else measure_copy_blocks(pa, device, peaks)
    cpu = cpu_baseline(r["w"]) if (rank == 0 and not args.no_cpu) else None
    if rank != 0:
        return
    w = r["w"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{w.cfg.dtype} in, fp32 accumulate", "data": "synthetic",
        "config": {**config_obj(w, _path(w)), "l2": config_l2(w)},
        "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r.get("e2e"),
        "gpu_launches": args.steps * r["runner"].launches_per_step,
        "clocks": clocks, "step_p10_p50_p90_ms": r["step_ms_p10_p50_p90"],
        "instrumented_ms_per_step": r["instrumented_ms_per_step"],
        "timing": ("ms_per_step: the timed steps back to back under one event pair; "
                   "step_p10_p50_p90_ms and the roofline's kernel time: a second pass "
                   "with events around every step and launch.  Back to back, each "
                   "launch is a programmatic dependent of the previous one, so its "
                   "start overlaps that launch's tail and ms_per_step can be below "
                   "the per-launch kernel time; the events of the second pass sit "
                   "between launches and remove that overlap"),
        "step_algorithmic_gbs": r["step_gbs"],
        "separate_launches_ms_per_step": r["separate_launches_ms_per_step"],
        "kernel_src_sha": {k: kernel_source_sha(k) for k in KERNEL_SOURCES},
    }
    for extra in ("cascade", "tensor_roofline", "graph"):
        if extra in r:
            line[extra] = r[extra]
    if copy is not None:
        line["copy_blocks"] = copy
    line["other_configs"] = others      # last, gqa last within it
    print(json.dumps(line))


def _sig(x, digits=4):
    """x rounded to `digits` significant digits (keeps the printed line short)."""
    return float(f"{x:.{digits}g}") if isinstance(x, float) else x


def other_entry(o: dict) -> dict:
    """The compact record of one further workload in the JSON line."""
    r, c = o["roofline"], o["w"].cfg
    e = {"value": _sig(o["value"]), "ms_per_step": _sig(o["ms_per_step"]),
         "separate_launches_ms_per_step": _sig(o["separate_launches_ms_per_step"]),
         "kernel_us": _sig(r["kernel_us"]), "kernel_us_l2_evicted": _sig(r["kernel_us_l2_evicted"]),
         "roofline_frac": _sig(r["frac"]), "frac_l2_evicted": _sig(r["frac_l2_evicted"]),
         "frac_of_8tbs": _sig(r["frac_of_8tbs"]), "achieved_gbs": _sig(r["achieved"]),
         "config": {"workload": c.name, "num_seqs": c.num_seqs,
                    "kv_dtype": "e4m3" if c.kv_fp8 else c.dtype}}
    if "cascade" in o:
        e["cascade"] = {"ms_per_step": _sig(o["cascade"]["ms_per_step"]),
                        "kernel_us": _sig(o["cascade"]["kernel_us"])}
    if "tensor_roofline" in o:
        t = o["tensor_roofline"]
        e["tensor_roofline"] = {"achieved_tflops": _sig(t["achieved"]), "frac": _sig(t["frac"]),
                                "peak": t["peak"]}
    return e


def measure_copy_blocks(pa, device, peaks, n_pairs=512, steps=20, warmup=5) -> dict:
    """pa_copy_blocks on a pool of the 7B shape (32 KV heads, 16 x 128 fp16 per
    block and head): n_pairs random source blocks to distinct destinations, K and
    V.  Bytes per launch: each block read once and written once."""
    h_kv, bs, d = 32, 16, 128
    num_blocks = 4 * n_pairs
    k = torch.randn(num_blocks, h_kv, bs, d, device=device, dtype=torch.float16)
    v = torch.randn_like(k)
    perm = torch.randperm(num_blocks, generator=torch.Generator().manual_seed(0))
    src = perm[:n_pairs].to(torch.int32).to(device)
    dst = perm[n_pairs:2 * n_pairs].to(torch.int32).to(device)
    for _ in range(warmup):
        pa.pa_copy_blocks(k, v, src, dst)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        pa.pa_copy_blocks(k, v, src, dst)
    b.record()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0, "device error during the block copies"
    us = a.elapsed_time(b) * 1e3 / steps
    nbytes = 2 * 2 * n_pairs * h_kv * bs * d * ELT
    gbs = nbytes / (us * 1e-6) / 1e9
    peak = peaks.get("hbm_gbs") or FALLBACK_HBM_GBS
    return {"pairs": n_pairs, "bytes_per_launch": nbytes, "us": _sig(us), "gbs": _sig(gbs),
            "frac": _sig(gbs / peak), "pool": "7B shape, fp16, 32 KV heads"}


def _path(w):
    if w.cfg.q_len > DECODE_MAX_QLEN:
        return ("pa_append_decode with q_len > 16: append launch, then the prefill kernel "
                "(persistent CTAs; 128 query rows of a KV head share each K/V chunk)")
    if w.cfg.kv_fp8:
        return "pa_decode_fp8 with k_new/v_new (fused quantising append + attention, one launch)"
    return ("pa_append_decode (fused slot mapping + append + split-KV partial, then combine)"
            if w.cfg.num_splits > 1 else
            "pa_append_decode (fused slot mapping + append + attention, one launch)")


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    orc = oracle.get()
    threads = os.cpu_count() or 1
    name = args.config
    w = workloads.make(name, seed=0, poison=False)
    c = w.cfg
    n_seq = max(1, min(c.num_seqs, args.ref_seqs))       # bounded sample per step
    kc, vc = w.bits("k_cache"), w.bits("v_cache")
    bt, cl = w.block_tables.numpy(), w.context_lens.numpy()
    qb = w.bits("q")
    rows = np.arange(n_seq * c.q_len * c.num_q_heads)
    tokens = int(cl[:n_seq].sum())

    def step():
        slots = orc.slot_mapping(bt[:n_seq], cl[:n_seq], c.block_size, c.q_len)
        orc.append_kv(kc, vc, w.bits("k_new")[:n_seq * c.q_len], w.bits("v_new")[:n_seq * c.q_len],
                      slots)
        orc.decode(qb, kc, vc, bt, cl, w.scale, c.dtype, q_len=c.q_len, rows=rows,
                   threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = tokens / dt
    sample = (f"{name}: first {n_seq} of {c.num_seqs} sequences per step ({tokens} KV tokens), "
              f"fp64 C oracle, {threads} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": config_obj(w, "fp64 CPU oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="scale the main workload down to this many sequences (profiling)")
    ap.add_argument("--ref-seqs", type=int, default=2,
                    help="sequences per step in the reference arm's bounded sample")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
