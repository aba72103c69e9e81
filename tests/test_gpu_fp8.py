"""GPU parity of the FP8 (E4M3) KV cache through the C ABI.

- pkv_kv_append_fp8 against the oracle's fp8 append, bit for bit on the whole
  pool: per-head scales, saturating values, padding and out-of-pool slots.
- pkv_paged_decode_attention_fp8 against the oracle's attention over the
  dequantised pool, element by element within 2e-3 + 1e-2*|ref| (bf16 out)
  and max-abs 2e-3 (fp32 out): every length mod 16, 2 to 32 query rows per kv
  head (both consumer orientations), NaN codes in every unused slot, split-K
  at several grid sizes, both TMA box modes, and the full-size 8B-layer and
  speculative-verify workloads on sampled (sequence, kv head) pairs.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import bf16_dev, compare, report, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OPTIONS = (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES, pkv.PKV_OPT_HEADS_PER_CTA,
           pkv.PKV_OPT_TMA_BOX, pkv.PKV_OPT_TAIL)


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _defaults():
    for opt in OPTIONS:
        pkv.set_option(opt, 0)
    yield
    for opt in OPTIONS:
        pkv.set_option(opt, 0)


def u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def f32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


class Fp8Step:
    """A workload's tensors on the GPU with E4M3 pools."""

    def __init__(self, w, seed=5, out_dtype=None):
        self.w = w
        self.k8, self.v8, self.ks, self.vs = W.fp8_pools(w, seed=seed)
        self.q = bf16_dev(w.q, torch)
        self.kc, self.vc = u8_dev(self.k8), u8_dev(self.v8)
        self.kn, self.vn = bf16_dev(w.k_new, torch), bf16_dev(w.v_new, torch)
        self.slots = torch.from_numpy(w.slot_mapping).cuda()
        self.tables = torch.from_numpy(w.block_tables).cuda()
        self.lens = torch.from_numpy(w.context_lens).cuda()
        self.ksd, self.vsd = f32_dev(self.ks), f32_dev(self.vs)
        self.out = torch.empty(self.q.shape, dtype=out_dtype or torch.bfloat16, device="cuda")

    def step(self):
        pkv.kv_append_fp8(self.kn, self.vn, self.slots, self.kc, self.vc, self.ksd, self.vsd)
        pkv.paged_decode_attention_fp8(self.q, self.kc, self.vc, self.ksd, self.vsd, self.tables,
                                       self.lens, self.w.n_query_per_seq, self.w.scale, self.out)
        return self.out

    def reference(self, o, pair_mask=None):
        w = self.w
        k, v = o.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, self.k8, self.v8, self.ks,
                               self.vs)
        out = o.paged_attention_fp8(w.q, k, v, w.block_tables, w.context_lens,
                                    w.n_query_per_seq, w.scale, self.ks, self.vs,
                                    pair_mask=pair_mask)
        return out, k, v


def run(o, w, out_dtype=None, check_pool=True):
    d = Fp8Step(w, out_dtype=out_dtype)
    d.step()
    torch.cuda.synchronize()
    ref, k, v = d.reference(o)
    if check_pool:
        assert np.array_equal(d.kc.cpu().numpy(), k)
        assert np.array_equal(d.vc.cpu().numpy(), v)
    stats = compare(to_f64(d.out), ref, what=w.name)
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0
    return stats


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64), (3, 24)])
def test_append_fp8_bit_exact(o, hkv, d):
    rng = np.random.default_rng(hkv + d)
    NB, n = 40, 300
    k8 = rng.integers(0, 256, size=(NB, 16, hkv, d), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(NB, 16, hkv, d), dtype=np.uint8)
    # values spanning subnormal, normal and saturating quotients
    kn = W.f32_to_bf16_bits((rng.standard_normal((n, hkv, d)) *
                             np.exp(rng.uniform(-8, 6, (n, hkv, 1)))).astype(np.float32))
    vn = W.f32_to_bf16_bits((rng.standard_normal((n, hkv, d)) * 4).astype(np.float32))
    ks = rng.uniform(0.001, 2.0, hkv).astype(np.float32)
    vs = rng.uniform(0.001, 2.0, hkv).astype(np.float32)
    slots = rng.permutation(NB * 16)[:n].astype(np.int64)
    slots[::17] = -1
    slots[5] = NB * 16 + 3                      # outside the pool: skipped
    kd, vd = u8_dev(k8), u8_dev(v8)
    pkv.kv_append_fp8(bf16_dev(kn, torch), bf16_dev(vn, torch), torch.from_numpy(slots).cuda(),
                      kd, vd, f32_dev(ks), f32_dev(vs))
    torch.cuda.synchronize()
    k_ref, v_ref = o.kv_append_fp8(kn, vn, slots, k8, v8, ks, vs)
    assert np.array_equal(kd.cpu().numpy(), k_ref)
    assert np.array_equal(vd.cpu().numpy(), v_ref)


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("hq,hkv,nq", [(8, 2, 1), (32, 8, 1), (64, 8, 1), (16, 8, 1),
                                       (16, 4, 3), (32, 8, 4), (64, 8, 4), (8, 8, 2),
                                       (64, 4, 4), (48, 4, 3)])
def test_attention_fp8_geometries(o, hq, hkv, nq):
    lens = [nq + i for i in range(0, 96, 7)] + [16, 17, 31, 32, 33, 200, 513]
    w = W.make_custom(len(lens), nq, hq, hkv, 128, lens, seed=hq * 10 + nq)
    run(o, w)


def test_attention_fp8_every_length_mod_16(o):
    lens = list(range(1, 49))
    w = W.make_custom(len(lens), 1, 32, 8, 128, lens, seed=3)
    run(o, w)


def test_attention_fp8_fp32_out_strict(o):
    lens = [5, 64, 100, 333, 1000]
    w = W.make_custom(len(lens), 2, 32, 8, 128, lens, seed=4)
    run(o, w, out_dtype=torch.float32)
    d = Fp8Step(w, out_dtype=torch.float32)
    d.step()
    torch.cuda.synchronize()
    ref, _, _ = d.reference(o)
    assert np.abs(to_f64(d.out) - ref).max() <= 2e-3


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_attention_fp8_grid_invariance(o, ctas):
    lens = [3000, 17, 800, 1, 64, 2500]
    w = W.make_custom(len(lens), 1, 32, 8, 128, lens, seed=8)
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, ctas)
    run(o, w)


@pytest.mark.parametrize("box", [1, 2])
def test_attention_fp8_tma_box_modes(o, box):
    lens = [77, 1024, 5, 300]
    w = W.make_custom(len(lens), 4, 64, 8, 128, lens, seed=9)
    pkv.set_option(pkv.PKV_OPT_TMA_BOX, box)
    run(o, w)


def test_attention_fp8_shared_prefix(o):
    lens = [600, 700, 530, 900]
    w = W.make_custom(len(lens), 1, 64, 8, 128, lens, seed=10, shared=[True, True, False, True],
                      prefix_tokens=512)
    run(o, w)


@pytest.mark.parametrize("name", [n for n in W.WORKLOAD_ORDER if W.WORKLOADS[n]["D"] == 128])
def test_attention_fp8_full_size(o, name):
    w = W.make_workload(name)
    d = Fp8Step(w)
    d.step()
    torch.cuda.synchronize()
    ref, k, v = d.reference(o)
    got = to_f64(d.out)
    max_abs, max_rel = compare(got, ref, what=f"{name}, E4M3 pools")
    report(f"{name}, E4M3 pools", max_abs, max_rel, got.size)
    # the append touched only its slots
    kc = d.kc.cpu().numpy().reshape(-1, w.num_kv_heads, w.head_dim)
    assert np.array_equal(kc[w.slot_mapping], k.reshape(-1, w.num_kv_heads, w.head_dim)[w.slot_mapping])
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0
