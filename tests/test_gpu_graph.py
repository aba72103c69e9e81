"""The decode step (kv_append + attention, main kernel and merge) captured in a
CUDA graph and replayed: the same bits as the calls made directly, and the
oracle's result. The library's calls enqueue only kernel launches on the stream
(tensor maps are built on the host and passed by value; the workspace is the
caller's), so the step can be captured once its first direct call has run."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, bf16_host, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_decode", "spec_verify"])
def test_step_replays_from_a_graph(name):
    w = W.make_workload(name)
    eager = DeviceStep(w, torch)
    eager.step()
    torch.cuda.synchronize()

    d = DeviceStep(w, torch)
    ws = pkv.workspace("cuda", pkv.workspace_size(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                                   w.num_kv_heads, w.head_dim))

    def step():
        d.append()
        d.attend(ws=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first call outside the capture (kernel attributes, workspace)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    d.out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(d.out.view(torch.int16), eager.out.view(torch.int16))
    assert torch.equal(d.k_cache.view(torch.int16), eager.k_cache.view(torch.int16))
    if name == "tiny":
        ref, k_ref, _ = oracle.Oracle().step(w)
        assert np.array_equal(bf16_host(d.k_cache), k_ref)
        compare(to_f64(d.out), ref, what="graph replay")
    assert pkv.workspace_error(ws) == 0
