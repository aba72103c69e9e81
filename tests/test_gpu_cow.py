"""GPU: copy-on-write through the C ABI.

- pkv_copy_blocks against the oracle's block copy, bit for bit on the whole
  pool (random bit patterns, NaNs included), for several head geometries, an
  empty call, skipped pairs and a large batch of pairs.
- A serving loop: the library's block manager forks sampled outputs of one
  prompt and appends for several steps (speculative nq > 1 too); each step
  runs copy -> append -> attention on the GPU and the same copies, appends and
  attention on the oracle's host pools. The pools must agree bit for bit, the
  attention within the parity tolerance, and every live sequence must read
  back its own token rows through its block table.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import bf16_dev, bf16_host, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("hkv,d,npairs", [(2, 64, 1), (8, 128, 257), (1, 8, 33), (3, 24, 100),
                                          (8, 128, 0), (8, 64, 4096)])
def test_copy_blocks_bit_exact(o, hkv, d, npairs):
    rng = np.random.default_rng(hkv * 1000 + d + npairs)
    NB = max(2 * npairs + 8, 16)
    k = rng.integers(0, 1 << 16, size=(NB, 16, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, 16, hkv, d), dtype=np.uint16)
    perm = rng.permutation(NB)
    src = list(perm[:npairs])
    dst = list(perm[npairs:2 * npairs])
    if npairs:
        # skipped pairs: a block past the pool, a negative id, src == dst
        src += [NB + 3, -1, int(perm[-1])]
        dst += [int(perm[-2]), int(perm[-3]), int(perm[-1])]
    kd, vd = bf16_dev(k, torch), bf16_dev(v, torch)
    pkv.copy_blocks(kd, vd, i32_dev(src), i32_dev(dst))
    torch.cuda.synchronize()
    k_ref, v_ref = o.copy_blocks(k, v, src, dst)
    assert np.array_equal(bf16_host(kd), k_ref)
    assert np.array_equal(bf16_host(vd), v_ref)


def normal_rows(rng, n, hkv, d):
    return W.f32_to_bf16_bits(rng.standard_normal((n, hkv, d), dtype=np.float32))


@pytest.mark.parametrize("hq,hkv,d,nq", [(8, 2, 128, 1), (32, 8, 128, 1), (16, 4, 64, 3),
                                         (64, 8, 128, 4)])
def test_serving_loop_with_forks(o, hq, hkv, d, nq):
    rng = np.random.default_rng(hq + 7 * nq + d)
    NB, MB = 640, 96
    scale = float(np.float32(1.0 / np.sqrt(d)))
    bm = pkv.BlockManager(NB)
    k_host = np.full((NB, 16, hkv, d), W.SENTINEL_BF16, dtype=np.uint16)
    v_host = k_host.copy()
    k_dev, v_dev = bf16_dev(k_host, torch), bf16_dev(v_host, torch)
    logical_k, logical_v = {}, {}

    def write(slots, kr, vr):
        nonlocal k_host, v_host
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        pkv.kv_append(bf16_dev(kr, torch), bf16_dev(vr, torch), torch.from_numpy(slots).cuda(),
                      k_dev, v_dev)
        k_host, v_host = o.kv_append(kr, vr, slots, k_host, v_host)

    def add(seq, n):
        assert bm.add_sequence(seq, n)
        t = bm.table(seq)
        slots = [t[i // 16] * 16 + i % 16 for i in range(n)]
        kr, vr = normal_rows(rng, n, hkv, d), normal_rows(rng, n, hkv, d)
        write(slots, kr, vr)
        logical_k[seq], logical_v[seq] = list(kr), list(vr)

    def fork(parent, child):
        bm.fork(parent, child)
        logical_k[child], logical_v[child] = list(logical_k[parent]), list(logical_v[parent])

    add(0, 1000)                      # a prompt whose last block holds 8 tokens
    for c in (1, 2, 3):               # parallel sampling: 63 blocks with count 4
        fork(0, c)
    add(10, 37)
    add(11, 16)                       # a full last block: no copy on its next append
    total_copies = 0
    for step in range(8):
        if step == 3:                 # one output ends; another branches off a sibling
            bm.free(2)
            del logical_k[2], logical_v[2]
            fork(1, 12)
        if step == 5:
            add(13, 0)                # an empty sequence takes its first block now
        seqs = sorted(logical_k)
        res = bm.append_batch(seqs, nq)
        assert res is not None
        slots, copies = res
        total_copies += len(copies)
        if copies:
            src = [a for a, _ in copies]
            dst = [b for _, b in copies]
            pkv.copy_blocks(k_dev, v_dev, i32_dev(src), i32_dev(dst))
            k_host, v_host = o.copy_blocks(k_host, v_host, src, dst)
        kr = normal_rows(rng, len(seqs) * nq, hkv, d)
        vr = normal_rows(rng, len(seqs) * nq, hkv, d)
        write(slots, kr, vr)
        for i, s in enumerate(seqs):
            logical_k[s] += list(kr[i * nq:(i + 1) * nq])
            logical_v[s] += list(vr[i * nq:(i + 1) * nq])

        tables, lens = bm.block_tables(seqs, MB)
        q = W.f32_to_bf16_bits(rng.standard_normal((len(seqs) * nq, hq, d), dtype=np.float32))
        out = torch.empty((len(seqs) * nq, hq, d), dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention(bf16_dev(q, torch), k_dev, v_dev, i32_dev(tables),
                                   i32_dev(lens), nq, scale, out)
        torch.cuda.synchronize()
        ref = o.paged_attention(q, k_host, v_host, tables, lens, nq, scale)
        compare(to_f64(out), ref, what=f"step {step}")
        kd, vd = bf16_host(k_dev), bf16_host(v_dev)
        assert np.array_equal(kd, k_host) and np.array_equal(vd, v_host)
        # every sequence reads back its own rows through its table
        for i, s in enumerate(seqs):
            n = int(lens[i])
            pos = np.arange(n)
            blk = tables[i][pos // 16]
            assert (blk >= 0).all()
            assert np.array_equal(kd[blk, pos % 16], np.stack(logical_k[s])), f"seq {s} K"
            assert np.array_equal(vd[blk, pos % 16], np.stack(logical_v[s])), f"seq {s} V"
        assert bm.check() == 0
    # the first step copies the shared partly filled block for all sharers but the last
    assert total_copies >= 3
