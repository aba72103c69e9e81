"""pkv_decode_step_host: one decode step from a pinned host arena (one copy in,
append, attention, one copy out) gives bit for bit the pool and the output of
the device calls it wraps, and the oracle's result within the tolerance."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def pack(w, d, n_bytes, offs, torch):
    """The step's inputs (device copies in `d`) packed into a pinned host arena."""
    host = torch.zeros(n_bytes, dtype=torch.uint8).pin_memory()
    for name, t in (("q", d.q), ("k_new", d.k_new), ("v_new", d.v_new),
                    ("slot_mapping", d.slots), ("block_tables", d.tables),
                    ("context_lens", d.lens)):
        nb = t.numel() * t.element_size()
        host[offs[name]:offs[name] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    return host


@pytest.mark.parametrize("name,out32", [("tiny", False), ("llama3_8b_decode", False),
                                        ("spec_verify", True)])
def test_host_step_equals_device_calls(name, out32):
    w = W.make_workload(name)
    od = torch.float32 if out32 else torch.bfloat16
    ref_dev = DeviceStep(w, torch, out_dtype=od)
    ref_dev.step()
    torch.cuda.synchronize()

    d = DeviceStep(w, torch, out_dtype=od)
    n, offs = pkv.step_arena_layout(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                    w.num_kv_heads, w.head_dim, w.block_tables.shape[1])
    host = pack(w, d, n, offs, torch)
    dev_arena = torch.empty(n, dtype=torch.uint8, device="cuda")
    out_host = torch.empty(d.out.shape, dtype=od).pin_memory()
    pkv.decode_step_host(host, dev_arena, d.k_cache, d.v_cache, w.num_seqs, w.n_query_per_seq,
                         w.num_q_heads, w.block_tables.shape[1], w.scale, d.out, out_host)
    torch.cuda.synchronize()
    assert torch.equal(d.k_cache.view(torch.int16), ref_dev.k_cache.view(torch.int16))
    assert torch.equal(d.v_cache.view(torch.int16), ref_dev.v_cache.view(torch.int16))
    assert torch.equal(out_host.view(torch.int16 if not out32 else torch.int32),
                       ref_dev.out.cpu().view(torch.int16 if not out32 else torch.int32))
    if name == "tiny":
        ref, _, _ = oracle.Oracle().step(w)
        compare(to_f64(out_host), ref, what="host step")
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0


def test_host_step_rejects_a_short_arena():
    w = W.make_workload("tiny")
    d = DeviceStep(w, torch)
    n, _ = pkv.step_arena_layout(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 w.block_tables.shape[1])
    host = torch.zeros(n - 256, dtype=torch.uint8).pin_memory()
    dev_arena = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    out_host = torch.empty(d.out.shape, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(pkv.PkvError):
        pkv.decode_step_host(host, dev_arena, d.k_cache, d.v_cache, w.num_seqs, 1,
                             w.num_q_heads, w.block_tables.shape[1], w.scale, d.out, out_host)
