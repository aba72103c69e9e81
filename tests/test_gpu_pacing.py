"""Pacing of the attention kernel (PKV_OPT_PACE) changes timing only.

A CTA that runs ahead of the grid's average progress keeps one stage fewer in
flight; the partition of the work into cells, and so the arithmetic, is the
same with pacing on or off. These tests check that the outputs are
bit-identical with pacing off and on (with and without a margin) for a 4-row
bf16 shape, a 32-row shape and an E4M3 pool, and that every call leaves the
workspace's progress counter at zero again.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, bf16_dev, compare, full_reference, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SETTINGS = [(0, 0), (1, 0), (1, 500), (0, 0)]  # (PKV_OPT_PACE, PKV_OPT_PACE_MARGIN)


@pytest.fixture(autouse=True)
def _defaults():
    yield
    pkv.set_option(pkv.PKV_OPT_PACE, 0)
    pkv.set_option(pkv.PKV_OPT_PACE_MARGIN, 0)


def header_words(ws):
    return ws[:32].view(torch.int32).cpu().numpy()


def run_settings(call, out, ws):
    got = []
    for pace, margin in SETTINGS:
        pkv.set_option(pkv.PKV_OPT_PACE, pace)
        pkv.set_option(pkv.PKV_OPT_PACE_MARGIN, margin)
        call()
        torch.cuda.synchronize()
        h = header_words(ws)
        assert h[0] == 0, f"device error word {h[0]} with pacing {pace}"
        assert h[2] == 0 and h[3] == 0 and h[4] == 0, f"counters not reset: {h[:8]}"
        got.append(out.view(torch.int16).clone())
    for g, (pace, margin) in zip(got[1:], SETTINGS[1:]):
        assert torch.equal(g, got[0]), f"pacing {pace}/{margin} changed the output bits"


@pytest.mark.parametrize("name", ["llama3_8b_decode", "spec_verify"])
def test_pacing_is_bit_identical(name):
    w = W.make_workload(name)
    d = DeviceStep(w, torch)
    d.append()
    ws = pkv.workspace("cuda", pkv.workspace_size(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                                   w.num_kv_heads, w.head_dim))
    ws.zero_()
    run_settings(lambda: d.attend(ws=ws), d.out, ws)
    # and the whole output is the oracle's
    compare(to_f64(d.out), full_reference(oracle.Oracle(), w, name), what=name)


def test_pacing_is_bit_identical_fp8():
    w = W.make_workload("llama3_8b_decode")
    k8, v8, ks, vs = W.fp8_pools(w)
    kc = torch.from_numpy(k8).cuda()
    vc = torch.from_numpy(v8).cuda()
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    q = bf16_dev(w.q, torch)
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.context_lens).cuda()
    pkv.kv_append_fp8(bf16_dev(w.k_new, torch), bf16_dev(w.v_new, torch),
                      torch.from_numpy(w.slot_mapping).cuda(), kc, vc, ksd, vsd)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pkv.workspace("cuda", pkv.workspace_size(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads,
                                                   w.head_dim))
    ws.zero_()
    run_settings(lambda: pkv.paged_decode_attention_fp8(q, kc, vc, ksd, vsd, tables, lens, 1,
                                                        w.scale, out, ws=ws), out, ws)
    assert not torch.isnan(out.float()).any()
