"""GPU parity of the fifth-generation tensor-core (tcgen05) kernel against the oracle.

With PKV_OPT_UMMA = 1, kv heads with 17 to 64 query rows (bf16 pools, head_dim
128) run on the tcgen05 kernel: super-stages of up to 8 blocks of one (sequence, kv head), scores with the
tokens on the MMA's M, the softmax one thread per token, P.V into tensor memory.
Every case is compared element by element with the fp64 oracle
(|err| <= 2e-3 + 1e-2 |ref|): row counts across both tile widths (N = 32, 64),
every context length mod 16 and around the 128-token super-stage, grids that cut
segments mid-super-stage, causal draft queries and tree masks, strict fp32 output,
a large running-max jump, and the same calls on the mma.sync kernels (the default,
PKV_OPT_UMMA = 0) for the A/B.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import ATOL, DeviceStep, bf16_dev, compare, full_reference, report, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OPTIONS = (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES, pkv.PKV_OPT_HEADS_PER_CTA,
           pkv.PKV_OPT_TMA_BOX, pkv.PKV_OPT_TAIL, pkv.PKV_OPT_UMMA, pkv.PKV_OPT_PREFETCH)


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _defaults():
    for opt in OPTIONS:
        pkv.set_option(opt, 0)
    pkv.set_option(pkv.PKV_OPT_UMMA, 1)   # the tcgen05 kernel (opt-in)
    yield
    for opt in OPTIONS:
        pkv.set_option(opt, 0)


def run(o, w, out_dtype=None):
    d = DeviceStep(w, torch, out_dtype=out_dtype)
    ref, _, _ = o.step(w)
    ws = torch.zeros(pkv.workspace_size(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                        w.num_kv_heads, w.head_dim), dtype=torch.uint8,
                     device="cuda")
    d.append()
    d.attend(ws=ws)
    torch.cuda.synchronize()
    got = to_f64(d.out)
    stats = compare(got, ref, what=w.name)
    assert pkv.workspace_error(ws) == 0
    return got, ref, stats


# (G, nq): 17..64 score rows per kv head, both tile widths
ROWS = [(8, 4), (16, 2), (32, 1), (6, 3), (9, 2), (16, 4), (64, 1), (12, 4), (20, 3)]


@pytest.mark.parametrize("G,nq", ROWS)
def test_rows_and_lengths(o, G, nq):
    Hkv = 2
    T = [nq, nq + 1, 15, 16, 17, 127, 128, 129, 130, 255, 257, 700]
    w = W.make_custom(len(T), nq, G * Hkv, Hkv, 128, T, seed=500 + 7 * G + nq)
    run(o, w)


def test_every_length_mod_16_around_a_super_stage(o):
    T = list(range(4, 70)) + list(range(120, 140)) + [255, 256, 257, 383, 384, 385]
    w = W.make_custom(len(T), 4, 64, 8, 128, T, seed=510)
    run(o, w)


@pytest.mark.parametrize("ctas", [1, 2, 7, 37, 152, 300, 1000])
def test_grid_sizes(o, ctas):
    """Cells cut segments at any block: partial super-stages at both ends."""
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, ctas)
    T = [3000, 20, 5, 777, 4096, 129, 4, 16, 17, 2500, 130, 1023]
    w = W.make_custom(len(T), 4, 64, 8, 128, T, seed=511)
    run(o, w)


@pytest.mark.parametrize("pf", [1, 2, 9, 100])
def test_prefetch_distances(o, pf):
    """The L2 prefetch cursor (none, 1 block, 8, 99 blocks ahead) changes no result."""
    pkv.set_option(pkv.PKV_OPT_PREFETCH, pf)
    T = [3000, 20, 5, 777, 129, 4, 17, 1023]
    w = W.make_custom(len(T), 4, 64, 8, 128, T, seed=517)
    run(o, w)


def test_fp32_output_strict(o):
    w = W.make_custom(6, 4, 32, 4, 128, [5, 33, 190, 600, 17, 1000], seed=512)
    got, ref, (max_abs, max_rel) = run(o, w, out_dtype=torch.float32)
    assert max_abs <= ATOL
    assert max_rel <= 1e-2


def test_running_max_jumps(o):
    """Queries aligned with late keys: the running max rises by far more than the
    lazy threshold in the middle of a segment, so the accumulator is rescaled."""
    T = [400, 1100, 260]
    w = W.make_custom(len(T), 4, 32, 4, 128, T, seed=513, keep_dense=True)
    q = W.bf16_bits_to_f32(w.q).reshape(len(T), 4, 32, 128)
    rng = np.random.default_rng(3)
    for s, Ts in enumerate(T):
        k = W.bf16_bits_to_f32(w.dense_k[s])              # [Ts, Hkv, D] after the append
        for h in range(4):
            t = int(rng.integers(Ts // 2, Ts - 4))
            q[s, :, 8 * h:8 * h + 8, :] += 6.0 * k[t, h][None, None, :]
    w.q = W.f32_to_bf16_bits(q.reshape(w.q.shape).astype(np.float32))
    run(o, w)


def test_shared_prefix_blocks(o):
    sh = np.array([True, False, True, True, False, True])
    w = W.make_custom(6, 4, 64, 8, 128, [600, 40, 513, 700, 90, 1025], seed=514,
                      shared=sh, prefix_tokens=512)
    run(o, w)


def test_matches_mma_sync_kernel(o):
    """The same call on both kernels: each within tolerance of the oracle."""
    T = [900, 33, 4000, 6, 260, 1300, 77]
    w = W.make_custom(len(T), 4, 64, 8, 128, T, seed=515)
    for umma in (1, 0):
        pkv.set_option(pkv.PKV_OPT_UMMA, umma)
        run(o, w)


def test_spec_verify_full_size(o):
    w = W.make_workload("spec_verify")
    assert pkv.set_option(pkv.PKV_OPT_UMMA, 1) == 1
    d = DeviceStep(w, torch)
    d.step()
    torch.cuda.synchronize()
    got = to_f64(d.out)
    ref = full_reference(o, w, "spec_verify")
    max_abs, max_rel = compare(got, ref, what="spec_verify (tcgen05)")
    report("spec_verify (tcgen05)", max_abs, max_rel, got.size)
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0


def binary_tree_masks(levels):
    masks = []
    for node in range(2 ** levels - 1):
        m, a = 0, node
        while True:
            m |= 1 << a
            if a == 0:
                break
            a = (a - 1) // 2
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


@pytest.mark.parametrize("G,max_q", [(4, 16), (8, 8), (4, 8)])
def test_tree_masks(o, G, max_q):
    """15-node candidate trees scored in runs of up to max_q queries (G * max_q score
    rows per kv head); nodes see the context and their ancestors."""
    masks = binary_tree_masks(4)
    n = masks.size
    ctx = np.array([300, 17, 1000, 129, 64])
    T = (ctx + n).astype(np.int32)
    S = len(T)
    w = W.make_custom(S, n, 8 * G, 8, 128, T, seed=516 + G, keep_full=True)
    qs = (np.arange(S + 1) * n).astype(np.int32)
    tl = np.full(S, n, np.int32)
    split = pkv.split_queries(qs, T, max_q, tree_len=tl)
    tm = np.tile(masks, S)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()

    out = torch.empty((S * n, 8 * G, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(pkv.workspace_size(split["table_row"].size, max_q, 8 * G, 8, 128),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attention_varlen(
        bf16_dev(w.q, torch), bf16_dev(w.k_full, torch), bf16_dev(w.v_full, torch),
        i32(w.block_tables), i32(split["context_lens"]), i32(split["q_start"]), max_q, w.scale,
        out, tree_mask=i32(tm.view(np.int32)), tree_len=i32(split["tree_len"]),
        table_row=i32(split["table_row"]), ws=ws)
    torch.cuda.synchronize()
    ref = o.paged_attention_varlen(w.q, w.k_full, w.v_full, w.block_tables, T, qs, w.scale,
                                   tree_mask=tm, tree_len=tl)
    compare(out.cpu().numpy().astype(np.float64), ref, what=f"tree G={G} runs of {max_q}")
    assert pkv.workspace_error(ws) == 0
