"""Pins of the oracle's number codecs against the format definitions,
hand-worked cases and an independent library (torch's float8/bfloat16)."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def test_e2m1_all_codes(golden):
    rows = golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_decode(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e8m0_decode():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert oracle.e8m0_decode(121) == 2.0 ** -6
    assert math.isnan(oracle.e8m0_decode(255))


def _torch_e4m3_table():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_codes_vs_torch():
    ref = _torch_e4m3_table()
    got = oracle.e4m3_decode_array(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_encode_golden(golden):
    for val, byte, *_ in golden("e4m3_cases.txt"):
        assert oracle.e4m3_encode(float(val)) == int(byte, 16), val


def test_e4m3_encode_vs_torch_random_and_midpoints():
    """Values exactly representable in fp32 (so torch's float32 path rounds
    once), |v| < 464 (torch does not saturate beyond that)."""
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.normal(0, 1, 20000) * np.exp2(rng.integers(-12, 9, 20000)),
        rng.uniform(-463.9, 463.9, 5000)]).astype(np.float32)
    v = v[np.abs(v) < 464.0]
    tab = _torch_e4m3_table()
    pos = np.sort(tab[1:127])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)          # every tie point
    v = np.concatenate([v, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(v.astype(np.float64))
    assert np.array_equal(got, ref)


def _bf16_brute(v: float) -> int:
    """Nearest bf16 by exact rational comparison of the two neighbours."""
    x = Fraction(v)
    f32 = np.float32(v)
    cands = set()
    base = int(np.array([f32], dtype=np.float32).view(np.uint32)[0] >> 16)
    for b in (base - 1, base, base + 1, base + 2):
        b &= 0xFFFF
        val = oracle.bf16_to_f64(np.array([b], dtype=np.uint16))[0]
        if np.isfinite(val):
            cands.add((b, Fraction(float(val))))
    best = min(cands, key=lambda c: (abs(c[1] - x), c[0] & 1))
    return best[0]


def test_bf16_encode_vs_exact_rational():
    rng = np.random.default_rng(3)
    v = rng.normal(0, 1, 3000) * np.exp2(rng.integers(-30, 30, 3000))
    # ties: bf16 midpoints, and doubles a hair off a midpoint (catch double rounding)
    b = rng.integers(0x0080, 0x7F00, 500).astype(np.uint16)
    lo = oracle.bf16_to_f64(b)
    hi = oracle.bf16_to_f64(b + 1)
    mid = (lo + hi) / 2
    v = np.concatenate([v, mid, -mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)])
    got = oracle.f64_to_bf16(v)
    for vi, gi in zip(v, got):
        assert gi == _bf16_brute(float(vi)), vi


def test_bf16_encode_vs_torch_on_fp32_values():
    rng = np.random.default_rng(4)
    v = (rng.normal(0, 1, 50000) * np.exp2(rng.integers(-40, 40, 50000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(v.astype(np.float64)), ref)


def test_act_exponent_golden(golden):
    for amax, e, *_ in golden("act_exponent_cases.txt"):
        assert oracle.act_block_exponent(float(amax)) == int(e), amax


def test_act_exponent_is_smallest_by_search():
    """Brute-force definition: the smallest integer e with amax <= 448*2^e."""
    rng = np.random.default_rng(5)
    for amax in np.abs(rng.normal(0, 1, 2000)) * np.exp2(rng.integers(-60, 60, 2000)):
        e = -130
        while not (amax <= 448.0 * 2.0 ** e):
            e += 1
        assert oracle.act_block_exponent(float(amax)) == e


def test_act_quant_rows_vs_torch():
    """Codes are torch's e4m3 rounding of v / 2^e (exact scaling) and the
    scale byte is e + 127; all-zero block -> byte 127."""
    rng = np.random.default_rng(6)
    v = rng.normal(0, 1, (16, 512)).astype(np.float32).astype(np.float64)
    v[3, 128:256] = 0.0
    v[5] *= 1e-20
    q, s = oracle.act_quant(v, 128)
    assert s[3, 1] == 127 and not q[3, 128:256].any()
    for r in range(16):
        for b in range(4):
            blk = v[r, b * 128:(b + 1) * 128]
            e = int(s[r, b]) - 127
            if blk.any():
                e_ref = -130
                while not (np.abs(blk).max() <= 448.0 * 2.0 ** e_ref):
                    e_ref += 1
                assert e == e_ref
            scaled = np.ldexp(blk, -e).astype(np.float32)
            ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[r, b * 128:(b + 1) * 128], ref)


def test_mxfp4_block_golden(golden):
    w = np.zeros((1, 32))
    expect = np.zeros(32, dtype=np.int64)
    for idx, spec, code, *_ in golden("mxfp4_block_cases.txt"):
        kind, _, num = spec.partition("=")
        w[0, int(idx)] = float(num) if kind == "v" else float(num) * 2.0 ** -6
        expect[int(idx)] = int(code)
    packed, scale = oracle.mxfp4_quant(w)
    assert scale[0, 0] == 121
    codes = np.empty(32, dtype=np.int64)
    codes[0::2] = packed[0] & 15
    codes[1::2] = packed[0] >> 4
    assert np.array_equal(codes, expect)
    # and the decode of those bytes gives E2M1 * 2^-6, element 2i in the low nibble
    dec = oracle.mxfp4_decode(packed, scale)[0]
    tab = {int(c): float(v) for c, v in golden("e2m1_values.txt")}
    assert np.array_equal(dec, np.array([tab[c] for c in expect]) * 2.0 ** -6)


def test_mxfp4_quant_error_bound_and_roundtrip():
    """Each decoded value is the nearest E2M1 grid point of v/2^X (checked by
    search over the 8 magnitudes) and exact grid values round-trip."""
    rng = np.random.default_rng(8)
    w = rng.normal(0, 0.02, (64, 256))
    packed, scale = oracle.mxfp4_quant(w)
    dec = oracle.mxfp4_decode(packed, scale)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    X = np.repeat(scale.astype(np.int64) - 127, 32, axis=1)
    u = np.abs(w) / np.exp2(X)
    dist = np.abs(u[..., None] - mags)
    nearest = mags[np.argmin(dist, axis=-1)]
    ok = np.isclose(np.abs(dec) / np.exp2(X), nearest) | (np.min(dist, axis=-1) == np.sort(dist, axis=-1)[..., 1])
    assert ok.all()
    # the block max lands in [4, 8) units before saturation
    amax_u = np.abs(w).reshape(64, 8, 32).max(-1) / np.exp2(scale.astype(np.int64) - 127)
    assert ((amax_u >= 4) & (amax_u < 8)).all()
    p2, s2 = oracle.mxfp4_quant(dec)
    assert np.array_equal(oracle.mxfp4_decode(p2, s2), dec)
