"""pkv_decode_step_host: one decode step from a pinned host arena (one copy in,
append, attention, one copy out) gives bit for bit the pool and the output of
the device calls it wraps, and the oracle's result within the tolerance. Its
pipelined form (copies and kernels on three streams, two buffer slots in turn)
gives every step the same bits as the serial one."""
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


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_decode"])
def test_pipelined_steps_equal_serial_steps(name):
    """Six steps through pkv_decode_step_host_pipelined, two buffer slots used in
    turn on three streams, each step with its own queries: every step's host output
    equals, bit for bit, the same step run alone through pkv_decode_step_host, and
    the tiny one matches the oracle. Copies of one step overlap the kernels of the
    next; the slot events keep each arena and output in use until it is free."""
    w = W.make_workload(name)
    n_steps = 6
    rng = np.random.default_rng(31)
    qs = [W.f32_to_bf16_bits(rng.standard_normal(w.q.shape).astype(np.float32))
          for _ in range(n_steps)]
    MB = w.block_tables.shape[1]
    n, offs = pkv.step_arena_layout(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                    w.num_kv_heads, w.head_dim, MB)

    def host_arena(d, q):
        d.q.copy_(torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16))
        return pack(w, d, n, offs, torch)

    # serial reference: each step alone
    ref_dev = DeviceStep(w, torch)
    ref_arena = torch.empty(n, dtype=torch.uint8, device="cuda")
    refs = []
    for q in qs:
        h = host_arena(ref_dev, q)
        oh = torch.empty(ref_dev.out.shape, dtype=torch.bfloat16).pin_memory()
        pkv.decode_step_host(h, ref_arena, ref_dev.k_cache, ref_dev.v_cache, w.num_seqs,
                             w.n_query_per_seq, w.num_q_heads, MB, w.scale, ref_dev.out, oh)
        torch.cuda.synchronize()
        refs.append(oh.clone())

    # pipelined: two slots, three streams
    d = DeviceStep(w, torch)
    hosts = [host_arena(d, q) for q in qs]
    arenas = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [torch.empty(d.out.shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs_h = [torch.full(d.out.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
              for _ in range(n_steps)]
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    events = [tuple(torch.cuda.Event() for _ in range(3)) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(n_steps):
        b = i % 2
        pkv.decode_step_host(hosts[i], arenas[b], d.k_cache, d.v_cache, w.num_seqs,
                             w.n_query_per_seq, w.num_q_heads, MB, w.scale, outs[b], outs_h[i],
                             streams=streams, events=events[b])
    torch.cuda.synchronize()
    for i in range(n_steps):
        assert torch.equal(outs_h[i].view(torch.int16), refs[i].view(torch.int16)), f"step {i}"
    assert torch.equal(d.k_cache.view(torch.int16), ref_dev.k_cache.view(torch.int16))
    if name == "tiny":
        o = oracle.Oracle()
        k, v = o.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
        ref = o.paged_attention(qs[-1], k, v, w.block_tables, w.context_lens, w.n_query_per_seq,
                                w.scale)
        compare(to_f64(outs_h[-1]), ref, what="pipelined host step")
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0


def test_pipelined_steps_e4m3_pools():
    """The pipelined step with per-head scales (E4M3 pools): four steps, two slots,
    every output bit-identical to kv_append_fp8 + paged_decode_attention_fp8 called
    directly on the same inputs, and the codes of the pool the same."""
    w = W.make_workload("llama3_8b_decode")
    k8, v8, ks, vs = W.fp8_pools(w)
    MB = w.block_tables.shape[1]
    n, offs = pkv.step_arena_layout(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads, w.head_dim, MB)
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()

    # direct device calls
    d = DeviceStep(w, torch)
    kc, vc = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pkv.kv_append_fp8(d.k_new, d.v_new, d.slots, kc, vc, ksd, vsd)
    pkv.paged_decode_attention_fp8(d.q, kc, vc, ksd, vsd, d.tables, d.lens, 1, w.scale, d.out)
    torch.cuda.synchronize()
    ref = d.out.cpu()

    host = pack(w, d, n, offs, torch)
    kp, vp = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    arenas = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [torch.empty(d.out.shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs_h = [torch.full(d.out.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
              for _ in range(4)]
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    events = [tuple(torch.cuda.Event() for _ in range(3)) for _ in range(2)]
    for i in range(4):
        pkv.decode_step_host(host, arenas[i % 2], kp, vp, w.num_seqs, 1, w.num_q_heads, MB,
                             w.scale, outs[i % 2], outs_h[i], streams=streams,
                             events=events[i % 2], k_scale=ksd, v_scale=vsd)
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(outs_h[i].view(torch.int16), ref.view(torch.int16)), f"step {i}"
    assert torch.equal(kp, kc) and torch.equal(vp, vc)
    with pytest.raises(ValueError):  # E4M3 pools take the pipelined form
        pkv.decode_step_host(host, arenas[0], kp, vp, w.num_seqs, 1, w.num_q_heads, MB, w.scale,
                             outs[0], outs_h[0], k_scale=ksd, v_scale=vsd)
