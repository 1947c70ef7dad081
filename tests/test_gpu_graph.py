"""The fused step captured in a CUDA graph and replayed gives the eager result, bit for
bit (needs a GPU).

Every launch of the library goes to the caller's stream with no host-side
synchronisation and no allocation, so a capture on that stream records the whole
step; the append rewrites the same bits at every replay.
"""
import pytest
import torch

import workloads
from tests.test_gpu_parity import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_20_gb300 as pa
    pa.load()
    assert pa.pa_device_error() == 0
    return pa


CASES = [
    ("gqa", {"num_seqs": 5}),
    ("llama7b_mha", {"num_seqs": 3}),
    ("long_split", {"num_seqs": 1, "lens": ("fixed", (4100,))}),
    ("chunked_prefill", {"num_seqs": 2, "q_len": 100, "lens": ("fixed", (100, 357))}),
    ("gqa_fp8", {"num_seqs": 4}),
]


@pytest.mark.parametrize("name,over", CASES, ids=[c[0] for c in CASES])
def test_fused_step_replays_from_a_cuda_graph(pa, name, over):
    w = workloads.make(name, **over)
    c = w.cfg
    names = ["q", "k_new", "v_new", "k_cache", "v_cache", "block_tables", "context_lens"]
    if c.kv_fp8:
        names += ["k_scale", "v_scale"]
    d = {k: getattr(w, k).to(DEV) for k in names}
    out = torch.empty_like(d["q"])
    ws = None
    if c.num_splits > 1:
        ws = torch.empty(pa.pa_decode_workspace_size(c.num_seqs, c.num_q_heads, c.q_len,
                                                     c.head_dim, c.num_splits),
                         dtype=torch.uint8, device=DEV)

    def step():
        if c.kv_fp8:
            pa.pa_decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                             d["block_tables"], d["context_lens"], w.scale, c.q_len,
                             c.num_splits, ws, k_new=d["k_new"], v_new=d["v_new"])
        else:
            pa.pa_append_decode(out, d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["block_tables"], d["context_lens"], w.scale, c.q_len,
                                c.num_splits, ws)

    step()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(out, eager)
