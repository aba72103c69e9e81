"""GPU parity of the shared-prefix cascade (pkv_paged_decode_attention_cascade)
against the oracle's plain attention on the same inputs.

The cascade computes the same function as the plain call (each shared prefix
is attended once per group and merged with the members' own blocks by the
online-softmax rule), so the oracle is the unchanged definition:

- one group of consecutive members (8, 4 and 1 query heads per kv head; one
  and two queries per sequence; bf16 and strict fp32 output);
- two groups over one physical prefix, the second using only its first half;
- a member whose queries do not all see the whole prefix (falls back);
- the 70B-mix batch with its 128 sharers moved to the front, on sampled pairs;
- several grid sizes; and a group outside the batch (flagged, others exact).
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, compare, full_reference, report, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _defaults():
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)
    yield
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)


def cascade(d, groups, max_group, out=None, ws=None):
    w = d.w
    out = d.out if out is None else out
    g = torch.from_numpy(np.asarray(groups, dtype=np.int32).reshape(-1, 3)).cuda()
    pkv.paged_decode_attention_cascade(d.q, d.k_cache, d.v_cache, d.tables, d.lens,
                                       w.n_query_per_seq, w.scale, out, g, max_group, ws=ws)
    return out


def cascade_ws(w):
    n = pkv.lib().pkv_workspace_size_cascade(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                             w.num_kv_heads, w.head_dim)
    return pkv.workspace("cuda", int(n))


def check(o, w, groups, max_group, out_dtype=None):
    d = DeviceStep(w, torch, out_dtype=out_dtype)
    d.append()
    ws = cascade_ws(w)
    cascade(d, groups, max_group, ws=ws)
    torch.cuda.synchronize()
    ref, _, _ = o.step(w)
    got = to_f64(d.out)
    compare(got, ref, what=w.name)
    assert pkv.workspace_error(ws) == 0
    return got, ref


@pytest.mark.parametrize("hq,hkv,nq", [(64, 8, 1), (32, 8, 1), (8, 8, 1), (32, 8, 2), (64, 8, 2)])
def test_one_group(o, hq, hkv, nq):
    rng = np.random.default_rng(hq + nq)
    M, S = 37, 45
    lens = np.concatenate([512 + rng.integers(nq, 400, M), rng.integers(nq, 900, S - M)])
    shared = np.arange(S) < M
    w = W.make_custom(S, nq, hq, hkv, 128, lens, seed=90 + hq + nq, shared=shared,
                      prefix_tokens=512)
    check(o, w, [[0, M, 32]], M)


def test_fp32_output_strict(o):
    M, S = 20, 24
    lens = np.concatenate([np.full(M, 600), np.arange(S - M) * 37 + 5])
    w = W.make_custom(S, 1, 32, 8, 128, lens, seed=91, shared=np.arange(S) < M,
                      prefix_tokens=512)
    got, ref = check(o, w, [[0, M, 32]], M, out_dtype=torch.float32)
    assert np.abs(got - ref).max() <= 2e-3


def test_two_groups_one_prefix(o):
    M, S = 30, 34
    rng = np.random.default_rng(3)
    lens = np.concatenate([513 + rng.integers(0, 300, M), [40, 90, 2000, 7]])
    w = W.make_custom(S, 1, 64, 8, 128, lens, seed=92, shared=np.arange(S) < M,
                      prefix_tokens=512)
    # members 0-9 skip all 32 shared blocks, members 10-29 only the first 16
    check(o, w, [[0, 10, 32], [10, 20, 16]], 20)


def test_member_falls_back_when_a_query_misses_part_of_the_prefix(o):
    M, S, nq = 12, 14, 2
    lens = np.concatenate([[513], np.full(M - 1, 700), [30, 60]])   # 513 - 2 < 512
    w = W.make_custom(S, nq, 32, 8, 128, lens, seed=93, shared=np.arange(S) < M,
                      prefix_tokens=512)
    check(o, w, [[0, M, 32]], M)


@pytest.mark.parametrize("ctas", [0, 1, 37])
def test_70b_mix_sharers_first(o, ctas):
    w = W.sharers_first(W.make_workload("llama3_70b_mix"))
    M = int(w.shared.sum())
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, ctas)
    d = DeviceStep(w, torch)
    d.append()
    ws = cascade_ws(w)
    cascade(d, [[0, M, w.meta["prefix_tokens"] // 16]], M, ws=ws)
    torch.cuda.synchronize()
    ref = full_reference(o, w, "llama3_70b_mix/sharers_first")
    got = to_f64(d.out)
    max_abs, max_rel = compare(got, ref, what=f"70b mix cascade, {ctas} CTAs")
    report(f"70b mix cascade, {ctas} CTAs", max_abs, max_rel, got.size)
    assert pkv.workspace_error(ws) == 0


def test_group_outside_the_batch_is_flagged(o):
    M, S = 10, 12
    lens = np.concatenate([np.full(M, 600), [100, 50]])
    w = W.make_custom(S, 1, 32, 8, 128, lens, seed=94, shared=np.arange(S) < M,
                      prefix_tokens=512)
    d = DeviceStep(w, torch)
    d.append()
    ws = cascade_ws(w)
    ws.zero_()
    cascade(d, [[0, M, 32], [S - 1, 5, 4]], M, ws=ws)     # second group runs past the batch
    torch.cuda.synchronize()
    assert pkv.workspace_error(ws) & 32
    ref, _, _ = o.step(w)
    compare(to_f64(d.out), ref, what="valid group")
    ws.zero_()
