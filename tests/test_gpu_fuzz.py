"""Seeded random geometries crossed with the tuning options, against the oracle.

Each case draws a geometry and a set of options that no single targeted test
combines:
- head_dim 64 or 128; 1 to 64 query rows per kv head (G x nq); 1 to 12 sequences;
- lengths from nq to 3,000 tokens, sometimes a shared prefix;
- persistent grid size, pipeline depth, heads per CTA, TMA box mode, dynamic
  tail, pacing, CUDA-core consumers; bf16 or fp32 output;
- a second set with the tcgen05 kernel opted in: mostly 17 to 64 rows per kv head
  at head_dim 128 (the rows it takes), with random L2 prefetch distances and grid
  sizes, and some geometries it leaves to the mma.sync kernels.

Then it checks append + attention against the fp64 oracle (the pool bit for bit,
the output within 2e-3 + 1e-2*|ref|), and that the device error word stays 0. Every
option gives the same function up to fp32 rounding order, so the oracle is the
same for all of them.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, bf16_host, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OPTIONS = (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES, pkv.PKV_OPT_HEADS_PER_CTA,
           pkv.PKV_OPT_TMA_BOX, pkv.PKV_OPT_TAIL, pkv.PKV_OPT_PACE, pkv.PKV_OPT_PACE_MARGIN,
           pkv.PKV_OPT_MATH, pkv.PKV_OPT_UMMA, pkv.PKV_OPT_PREFETCH)


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


def draw_case(seed):
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    while True:
        G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        nq = int(rng.integers(1, 5))
        if G * nq <= 64:
            break
    S = int(rng.integers(1, 13))
    T = np.where(rng.random(S) < 0.5, rng.integers(nq, 65, S), rng.integers(nq, 3001, S))
    shared, prefix = None, 0
    if rng.random() < 0.3 and S >= 2:
        prefix = int(rng.choice([16, 32, 64]))
        shared = rng.random(S) < 0.6
        T = np.where(shared, np.maximum(T, prefix + nq), T)
    opts = {
        pkv.PKV_OPT_NUM_CTAS: int(rng.choice([0, 1, 5, 37, 152, 500])),
        pkv.PKV_OPT_STAGES: int(rng.choice([0, 2, 3])),
        pkv.PKV_OPT_HEADS_PER_CTA: int(rng.choice([0, 1, 2])),
        pkv.PKV_OPT_TMA_BOX: int(rng.choice([0, 1])),
        pkv.PKV_OPT_TAIL: int(rng.choice([0, 4])),
        pkv.PKV_OPT_PACE: int(rng.choice([0, 1])),
        pkv.PKV_OPT_MATH: int(rng.choice([0, 1])),
    }
    out32 = bool(rng.random() < 0.3)
    return dict(D=D, Hkv=Hkv, G=G, nq=nq, S=S, T=T.astype(np.int64), shared=shared,
                prefix=prefix, opts=opts, out32=out32)


@pytest.mark.parametrize("seed", range(40))
def test_random_geometry_and_options(o, seed):
    c = draw_case(seed)
    for opt, v in c["opts"].items():
        assert pkv.set_option(opt, v) >= 0
    w = W.make_custom(c["S"], c["nq"], c["G"] * c["Hkv"], c["Hkv"], c["D"], c["T"],
                      seed=6000 + seed, shared=c["shared"], prefix_tokens=c["prefix"])
    d = DeviceStep(w, torch, out_dtype=torch.float32 if c["out32"] else None)
    ref, k_ref, v_ref = o.step(w)
    d.step()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(d.k_cache), k_ref)
    assert np.array_equal(bf16_host(d.v_cache), v_ref)
    compare(to_f64(d.out), ref, what=f"case {seed}: {c['opts']}")
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0


def draw_tcgen05_case(seed):
    rng = np.random.default_rng(7000 + seed)
    D = 128 if rng.random() < 0.85 else 64
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while True:
        G = int(rng.choice([2, 4, 6, 8, 12, 16, 32]))
        nq = int(rng.integers(1, 5))
        if G * nq <= 64 and (G * nq > 16 or rng.random() < 0.15):
            break
    S = int(rng.integers(1, 10))
    T = np.where(rng.random(S) < 0.4, rng.integers(nq, 140, S), rng.integers(nq, 4001, S))
    shared, prefix = None, 0
    if rng.random() < 0.25 and S >= 2:
        prefix = int(rng.choice([16, 128, 256]))
        shared = rng.random(S) < 0.6
        T = np.where(shared, np.maximum(T, prefix + nq), T)
    opts = {
        pkv.PKV_OPT_UMMA: 1,
        pkv.PKV_OPT_NUM_CTAS: int(rng.choice([0, 1, 3, 37, 152, 400])),
        pkv.PKV_OPT_PREFETCH: int(rng.choice([0, 1, 2, 9, 65, 200])),
    }
    out32 = bool(rng.random() < 0.3)
    return dict(D=D, Hkv=Hkv, G=G, nq=nq, S=S, T=T.astype(np.int64), shared=shared,
                prefix=prefix, opts=opts, out32=out32)


@pytest.mark.parametrize("seed", range(24))
def test_random_geometry_tcgen05(o, seed):
    c = draw_tcgen05_case(seed)
    for opt, v in c["opts"].items():
        assert pkv.set_option(opt, v) >= 0
    w = W.make_custom(c["S"], c["nq"], c["G"] * c["Hkv"], c["Hkv"], c["D"], c["T"],
                      seed=8000 + seed, shared=c["shared"], prefix_tokens=c["prefix"])
    d = DeviceStep(w, torch, out_dtype=torch.float32 if c["out32"] else None)
    ref, k_ref, v_ref = o.step(w)
    d.step()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(d.k_cache), k_ref)
    assert np.array_equal(bf16_host(d.v_cache), v_ref)
    compare(to_f64(d.out), ref, what=f"tcgen05 case {seed}: G={c['G']} nq={c['nq']} D={c['D']} "
                                     f"{c['opts']}")
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0
