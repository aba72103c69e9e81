"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
rejects invalid arguments on the host before any device work."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_101_gb300 as pkv
from paged_kv_cache_101_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

OK, NULL, SHAPE, DTYPE, ALIGN, RANGE, WORKSPACE, CUDA, UNSUP, NO_BLOCKS, SEQUENCE = range(11)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(pkv_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_workspace_size",
                     "pkv_status_string", "pkv_copy_blocks", "pkv_bm_create", "pkv_bm_append",
                     "pkv_bm_block_tables"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
        assert n in pkv.SIGNATURES, f"{n} has no Python binding"


def test_status_strings_and_version(lib):
    for s in range(11):
        assert pkv.status_string(s) and pkv.status_string(s) != "unknown status"
    assert pkv.status_string(99) == "unknown status"
    assert lib.pkv_version() >= 100


def test_options(lib):
    assert pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 7) == 0
    assert pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0) == 7
    assert pkv.set_option(pkv.PKV_OPT_STAGES, 3) == 0
    assert pkv.set_option(pkv.PKV_OPT_STAGES, 0) == 3
    assert pkv.set_option(42, 1) == -1
    assert pkv.set_option(pkv.PKV_OPT_NUM_CTAS, -5) == -1
    # pacing: 0 = off, 1 = on; margin 0..10000 (1/10000 of the work)
    assert pkv.set_option(pkv.PKV_OPT_PACE, 1) == 0
    assert pkv.set_option(pkv.PKV_OPT_PACE, 2) == -1
    assert pkv.set_option(pkv.PKV_OPT_PACE, 0) == 1
    assert pkv.set_option(pkv.PKV_OPT_PACE_MARGIN, 50) == 0
    assert pkv.set_option(pkv.PKV_OPT_PACE_MARGIN, 10001) == -1
    assert pkv.set_option(pkv.PKV_OPT_PACE_MARGIN, 0) == 50
    # consumers: 0 = tensor cores, 1 = CUDA-core FMA
    assert pkv.set_option(pkv.PKV_OPT_MATH, 1) == 0
    assert pkv.set_option(pkv.PKV_OPT_MATH, 2) == -1
    assert pkv.set_option(pkv.PKV_OPT_MATH, 0) == 1


A = 0x10000  # a 64 KiB-aligned dummy address: never dereferenced on these paths


def append(lib, k=A, v=A, slots=A, n=4, kc=A, vc=A, nb=8, hkv=2, d=64):
    return lib.pkv_kv_append(k, v, slots, n, kc, vc, nb, hkv, d, None)


def test_append_validation(lib):
    assert append(lib, n=0) == OK                      # empty step: no-op
    assert append(lib, k=None) == NULL
    assert append(lib, slots=None) == NULL
    assert append(lib, n=-1) == SHAPE
    assert append(lib, nb=0) == SHAPE
    assert append(lib, hkv=0) == SHAPE
    assert append(lib, d=60) == UNSUP                   # rows move in 16-byte vectors
    assert append(lib, d=2048) == RANGE
    assert append(lib, k=A + 8) == ALIGN
    assert append(lib, vc=A + 2) == ALIGN
    assert append(lib, slots=A + 4) == ALIGN


def copyb(lib, k=A, v=A, nb=8, hkv=2, d=64, src=A, dst=A, n=3):
    return lib.pkv_copy_blocks(k, v, nb, hkv, d, src, dst, n, None)


def test_copy_blocks_validation(lib):
    assert copyb(lib, n=0) == OK                        # nothing to copy: no-op
    assert copyb(lib, k=None) == NULL
    assert copyb(lib, dst=None) == NULL
    assert copyb(lib, n=-1) == SHAPE
    assert copyb(lib, nb=0) == SHAPE
    assert copyb(lib, hkv=0) == SHAPE
    assert copyb(lib, d=12) == UNSUP
    assert copyb(lib, d=2048) == RANGE
    assert copyb(lib, v=A + 8) == ALIGN
    assert copyb(lib, src=A + 2) == ALIGN


def attn(lib, q=A, k=A, v=A, nb=64, bt=A, mb=8, cl=A, S=4, nq=1, hq=8, hkv=2, d=64,
         scale=0.125, out=A, dt=0, ws=A, wsb=1 << 30):
    return lib.pkv_paged_decode_attention(q, k, v, nb, bt, mb, cl, S, nq, hq, hkv, d, scale,
                                          out, dt, ws, wsb, None)


def test_attention_validation(lib):
    assert attn(lib, S=0) == OK                         # empty batch: no-op
    assert attn(lib, q=None) == NULL
    assert attn(lib, bt=None) == NULL
    assert attn(lib, cl=None) == NULL
    assert attn(lib, out=None) == NULL
    assert attn(lib, ws=None) == WORKSPACE
    assert attn(lib, S=-1) == SHAPE
    assert attn(lib, hq=6, hkv=4) == SHAPE              # heads not a multiple of kv heads
    assert attn(lib, nb=0) == SHAPE
    assert attn(lib, mb=0) == SHAPE
    assert attn(lib, nq=0) == SHAPE
    assert attn(lib, nq=5) == UNSUP
    assert attn(lib, d=96) == UNSUP
    assert attn(lib, d=256) == UNSUP
    assert attn(lib, hq=80, hkv=1, nq=1) == UNSUP       # 80 query rows per kv head (max 64)
    assert attn(lib, hq=32, hkv=1, nq=3) == UNSUP       # 96
    assert attn(lib, hq=68, hkv=4, nq=4) == UNSUP       # 17*4 = 68 rows per kv head
    assert attn(lib, dt=2) == DTYPE
    assert attn(lib, q=A + 8) == ALIGN
    assert attn(lib, out=A + 4) == ALIGN
    assert attn(lib, ws=A + 16) == ALIGN
    assert attn(lib, bt=A + 2) == ALIGN
    assert attn(lib, mb=1 << 27) == RANGE


def attn8(lib, q=A, k=A, v=A, nb=64, ks=A, vs=A, bt=A, mb=8, cl=A, S=4, nq=1, hq=8, hkv=2,
          d=128, scale=0.125, out=A, dt=0, ws=A, wsb=1 << 30):
    return lib.pkv_paged_decode_attention_fp8(q, k, v, nb, ks, vs, bt, mb, cl, S, nq, hq, hkv,
                                              d, scale, out, dt, ws, wsb, None)


def test_fp8_validation(lib):
    assert attn8(lib, S=0) == OK
    assert attn8(lib, d=64) == UNSUP                    # E4M3 rows are one 128-byte row
    assert attn8(lib, ks=None) == NULL
    assert attn8(lib, vs=None) == NULL
    assert attn8(lib, vs=A + 2) == ALIGN
    assert attn8(lib, ws=None) == WORKSPACE
    assert attn8(lib, nq=5) == UNSUP
    ap = lib.pkv_kv_append_fp8
    assert ap(A, A, A, 0, A, A, 8, 2, 64, A, A, None) == OK
    assert ap(A, A, A, 4, A, A, 8, 2, 64, None, A, None) == NULL
    assert ap(A, A, A, 4, A, A, 8, 2, 60, A, A, None) == UNSUP
    assert ap(A, A, A, 4, A + 4, A, 8, 2, 64, A, A, None) == ALIGN
    assert ap(A, A, A, -1, A, A, 8, 2, 64, A, A, None) == SHAPE


def test_step_arena_layout(lib):
    n, offs = pkv.step_arena_layout(64, 1, 32, 8, 128, 256)
    sizes = [64 * 32 * 128 * 2, 64 * 8 * 128 * 2, 64 * 8 * 128 * 2, 64 * 8, 64 * 256 * 4, 64 * 4]
    names = ["q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"]
    prev_end = 0
    for name, size in zip(names, sizes):
        o = offs[name]
        assert o % 256 == 0 and o >= prev_end      # aligned, in order, no overlap
        prev_end = o + size
    assert n >= prev_end and n % 256 == 0 and n - prev_end < 256
    assert lib.pkv_step_arena_layout(4, 5, 8, 2, 64, 8, None) == 0     # nq > 4
    assert lib.pkv_step_arena_layout(4, 1, 8, 3, 64, 8, None) == 0     # 8 % 3 != 0
    assert lib.pkv_step_arena_layout(4, 1, 8, 2, 64, 0, None) == 0     # no table columns
    assert lib.pkv_step_arena_layout(0, 1, 8, 2, 64, 8, None) == 0     # empty step: 0 bytes


def step_host(lib, ha=A, da=A, nbytes=1 << 20, k=A, v=A, nb=64, mb=8, S=4, nq=1, hq=8, hkv=2,
              d=64, od=A, oh=A, dt=0, ws=A, wsb=1 << 30):
    return lib.pkv_decode_step_host(ha, da, nbytes, k, v, nb, mb, S, nq, hq, hkv, d, 0.125, od,
                                    oh, dt, ws, wsb, None)


def test_decode_step_host_validation(lib):
    assert step_host(lib, S=0) == OK                    # empty step: nothing enqueued
    assert step_host(lib, S=-1) == SHAPE
    assert step_host(lib, mb=0) == SHAPE
    assert step_host(lib, nq=5) == UNSUP
    assert step_host(lib, d=96) == UNSUP
    assert step_host(lib, ha=None) == NULL
    assert step_host(lib, da=None) == NULL
    assert step_host(lib, oh=None) == NULL
    assert step_host(lib, od=None) == NULL
    assert step_host(lib, k=None) == NULL
    assert step_host(lib, nbytes=1024) == WORKSPACE     # arena smaller than the layout
    assert step_host(lib, da=A + 16) == ALIGN
    assert step_host(lib, dt=2) == DTYPE
    assert step_host(lib, nb=0) == SHAPE
    assert step_host(lib, ws=None) == WORKSPACE


def step_piped(lib, ev=A, S=4, ha=A, nq=1, **kw):
    args = dict(ha=ha, da=A, nbytes=1 << 20, k=A, v=A, nb=64, mb=8, S=S, nq=nq, hq=8, hkv=2, d=64,
                od=A, oh=A, dt=0, ws=A, wsb=1 << 30)
    args.update(kw)
    a = args
    return lib.pkv_decode_step_host_pipelined(
        a["ha"], a["da"], a["nbytes"], a["k"], a["v"], a["nb"], a["mb"], a["S"], a["nq"], a["hq"],
        a["hkv"], a["d"], 0.125, a["od"], a["oh"], a["dt"], a["ws"], a["wsb"], a.get("ks"),
        a.get("vs"), None, None, None, ev, ev, ev)


def test_decode_step_host_pipelined_validation(lib):
    """The pipelined step makes the same checks before anything is enqueued, and
    needs its three events."""
    assert step_piped(lib, S=0) == OK
    assert step_piped(lib, S=-1) == SHAPE
    assert step_piped(lib, nq=5) == UNSUP
    assert step_piped(lib, ha=None) == NULL
    assert step_piped(lib, ev=None) == NULL
    assert step_piped(lib, nbytes=1024) == WORKSPACE
    assert step_piped(lib, da=A + 16) == ALIGN
    assert step_piped(lib, dt=2) == DTYPE
    assert step_piped(lib, ws=None) == WORKSPACE
    assert step_piped(lib, ks=A) == NULL                # one scale without the other
    assert step_piped(lib, ks=A, vs=A) == UNSUP         # E4M3 pools need head_dim 128


def test_workspace_size_rejects_bad_geometry(lib):
    assert lib.pkv_workspace_size(4, 5, 8, 2, 64) == 0
    assert lib.pkv_workspace_size(4, 1, 8, 3, 64) == 0
    assert lib.pkv_workspace_size(4, 1, 8, 2, 80) == 0
    assert lib.pkv_workspace_size(0, 1, 8, 2, 64) == 256


def test_product_path_has_no_cpu_fallback(monkeypatch, tmp_path):
    """With the library missing, the binding raises instead of computing anything."""
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "LIBRARY_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pkv.lib()
