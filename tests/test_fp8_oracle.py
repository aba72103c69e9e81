"""Pins of the oracle's FP8 (E4M3) KV-cache functions against what the format
and the pages fix, and planted mistakes in copies of the oracle, each caught.

- decode of all 256 codes equals the library's float8_e4m3fn conversion, and
  the closed forms of the format (448 the largest, 2^-9 the smallest
  subnormal, 2^-6 the smallest normal, 1.0 = 0x38, NaN = S.1111.111);
- encode: every finite code round-trips; midpoints go to the even code;
  magnitudes beyond 448 saturate; random in-range values agree with the
  library's conversion (which also rounds to nearest even);
- the fp8 append stores encode(x / scale[h]) per kv head: agrees with the
  library on float32 quotients, and every stored value is within half a grid
  step of the quotient;
- fp8 attention equals the pinned bf16 attention when the dequantized values
  are exactly bf16 values (power-of-two scales), bit for bit in fp64.
"""
import os

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


def lib_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).double().numpy()


def lib_encode(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


# ------------------------------------------------------------------ pins
def pin_decode_all_codes(o):
    c = np.arange(256, dtype=np.uint8)
    d, ref = o.e4m3_decode(c), lib_decode(c)
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(d[fin], ref[fin])
    assert np.array_equal(np.signbit(d[fin]), np.signbit(ref[fin]))


def pin_decode_closed_forms(o):
    d = o.e4m3_decode(np.array([0x7E, 0x01, 0x08, 0x38, 0x7F, 0xFF, 0x80, 0xFE, 0x07], np.uint8))
    assert d[0] == 448.0 and d[1] == 2.0 ** -9 and d[2] == 2.0 ** -6 and d[3] == 1.0
    assert np.isnan(d[4]) and np.isnan(d[5])
    assert d[6] == 0.0 and np.signbit(d[6]) and d[7] == -448.0 and d[8] == 7 * 2.0 ** -9


def pin_encode_round_trip_and_ties(o):
    c = np.array([i for i in range(256) if i not in (0x7F, 0xFF)], np.uint8)
    v = o.e4m3_decode(c).astype(np.float32)
    assert np.array_equal(o.e4m3_encode(v), c)
    # midpoints between neighbours go to the even code
    pos = np.arange(0, 0x7E, dtype=np.uint8)               # 0 .. 0x7D and their upper neighbours
    lo, hi = o.e4m3_decode(pos), o.e4m3_decode(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exactly representable
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(o.e4m3_encode(mid), want)
    assert np.array_equal(o.e4m3_encode(-mid), want | 0x80)


def pin_encode_saturates(o):
    x = np.array([449, 464, 470, 479.9, 1e6, np.inf, -500, -np.inf, np.nan], np.float32)
    assert o.e4m3_encode(x).tolist() == [0x7E] * 6 + [0xFE, 0xFE, 0x7F]


def pin_encode_matches_library(o):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200_000) * 40, rng.standard_normal(50_000) * 1e-2,
                        rng.uniform(-2 ** -6, 2 ** -6, 50_000)]).astype(np.float32)
    x = x[np.abs(x) < 448]
    assert np.array_equal(o.e4m3_encode(x), lib_encode(x))


def _append_case(o):
    rng = np.random.default_rng(1)
    NB, Hkv, D, n = 6, 3, 16, 20
    kn = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32) * 3)
    vn = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32) * 3)
    ks = np.array([0.01, 0.5, 3.0], np.float32)
    vs = np.array([0.02, 0.25, 1.5], np.float32)
    slots = rng.permutation(NB * 16)[:n].astype(np.int64)
    slots[3] = -1
    k8 = np.full((NB, 16, Hkv, D), 0x7F, np.uint8)
    v8 = k8.copy()
    k2, v2 = o.kv_append_fp8(kn, vn, slots, k8, v8, ks, vs)
    return kn, vn, ks, vs, slots, k8, k2, v2


def pin_append_matches_library(o):
    kn, vn, ks, vs, slots, k8, k2, v2 = _append_case(o)
    for new, sc, pool in ((kn, ks, k2), (vn, vs, v2)):
        x = W.bf16_bits_to_f32(new) / sc[None, :, None]   # float32 quotient
        ref = k8.copy()
        keep = slots >= 0
        ref.reshape(-1, *ref.shape[2:])[slots[keep]] = lib_encode(np.clip(x, -448, 448))[keep]
        assert np.array_equal(pool, ref)


def pin_append_half_step(o):
    kn, vn, ks, vs, slots, k8, k2, v2 = _append_case(o)
    x = W.bf16_bits_to_f32(kn).astype(np.float64) / ks[None, :, None].astype(np.float64)
    got = o.e4m3_decode(k2.reshape(-1, *k2.shape[2:])[slots[slots >= 0]])
    x = x[slots >= 0]
    a = np.minimum(np.abs(x), 448)
    step = np.where(a < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-30))) - 3))
    assert np.all(np.abs(np.abs(got) - a) <= step / 2 * (1 + 1e-6))
    assert np.all((np.sign(got) == np.sign(x)) | (got == 0))


def pin_attention_equals_bf16_definition(o):
    w = W.make_workload("tiny")
    k8, v8, _, _ = W.fp8_pools(w, seed=3)
    ks = np.array([0.25, 2.0], np.float32)                  # powers of two: exact in bf16
    vs = np.array([0.5, 0.125], np.float32)
    k8[k8 == 0x7F] = 0x38                                   # finite everywhere for the bf16 side
    v8[v8 == 0x7F] = 0x30
    kd = (o.e4m3_decode(k8) * ks[None, None, :, None]).astype(np.float32)
    vd = (o.e4m3_decode(v8) * vs[None, None, :, None]).astype(np.float32)
    kb, vb = W.f32_to_bf16_bits(kd.copy()), W.f32_to_bf16_bits(vd.copy())
    assert np.array_equal(W.bf16_bits_to_f32(kb), kd)       # exact
    for nq in (1, 2):
        lens = np.maximum(w.context_lens, nq)
        q = np.repeat(w.q, nq, axis=0)                      # [S*nq, Hq, D]
        ref = o.paged_attention(q, kb, vb, w.block_tables, lens, nq, w.scale)
        got = o.paged_attention_fp8(q, k8, v8, w.block_tables, lens, nq, w.scale, ks, vs)
        assert np.array_equal(got, ref)


FP8_PINS = [pin_decode_all_codes, pin_decode_closed_forms, pin_encode_round_trip_and_ties,
            pin_encode_saturates, pin_encode_matches_library, pin_append_matches_library,
            pin_append_half_step, pin_attention_equals_bf16_definition]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda f: f.__name__)
def test_fp8_pin(o, pin):
    pin(o)


# ------------------------------------------------------------------ mutants
MUTANTS = {
    "exponent_bias_8": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    "subnormal_step": ("ldexp((double)m, -9)", "ldexp((double)m, -8)"),
    "ties_away": ("double n = nearbyint(ldexp(a, 3 - E));", "double n = round(ldexp(a, 3 - E));"),
    "no_saturation": ("if (field > 15 || (field == 15 && n - 8.0 > 6.0))",
                      "if (field > 15)"),
    "scale_multiplies": ("oracle_e4m3_encode(kx / k_scale[h])", "oracle_e4m3_encode(kx * k_scale[h])"),
    "v_uses_k_scale": ("oracle_e4m3_decode(v_cache[base + d]) * v_scale[h]",
                       "oracle_e4m3_decode(v_cache[base + d]) * k_scale[h]"),
    "mantissa_carry_lost": ("        E += 1;\n        n = 8.0;\n", "        n = 15.0;\n"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fp8_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1, f"mutation site for {name} not found once"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(before, after, 1))
    lib = tmp_path / "mut.so"
    oracle.build(str(path), str(lib), force=True)
    m = oracle.Oracle(oracle.load(str(lib)))
    caught = []
    for pin in FP8_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"


def test_oracle_source_exists():
    assert os.path.exists(oracle.SOURCE)
