"""Pins of the oracle's fp32-scale activation quantisation (the variant with
s = amax / 448 per 1 x 128 block): hand-worked golden cases, torch's own
float32 division and e4m3 conversion, the exact agreement with the
power-of-two mode when every block's amax is 448 * 2^p, and the e4m3
rounding bound."""
import struct

import numpy as np
import pytest

import oracle


def _bits(f):
    return struct.unpack("<I", struct.pack("<f", float(f)))[0]


def test_golden_cases(golden):
    for amax, sbits, v, code in golden("act_f32s_cases.txt"):
        amax, v = float(amax), float(v)
        blk = np.zeros((1, 128))
        blk[0, 0] = amax            # the block's amax
        blk[0, 1] = v               # the value under test (|v| <= amax)
        q, s = oracle.act_quant(blk, 128, oracle.ACT_SCALE_F32)
        assert s.dtype == np.float32
        assert _bits(s[0, 0]) == int(sbits, 16), (amax, hex(_bits(s[0, 0])))
        assert q[0, 1] == int(code, 16), (amax, v, hex(q[0, 1]))


def test_matches_torch_float32_and_float8_on_bf16_blocks():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    rows, n = 48, 512
    x = rng.standard_normal((rows, n)) * np.exp(rng.uniform(-12, 12, size=(rows, 1)))
    x[3, 128:256] = 0.0                        # an all-zero block
    x[5, :128] = 0.0
    x[5, 7] = 1e-30                            # a block whose only value is tiny
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xf = xb.to(torch.float32)                  # bf16 values are exact in fp32
    q, s = oracle.act_quant(xf.double().numpy(), 128, oracle.ACT_SCALE_F32)
    blocks = xf.view(rows, n // 128, 128)
    amax = blocks.abs().amax(dim=-1)
    s_ref = amax / 448.0
    assert np.array_equal(s.view(np.uint32), s_ref.numpy().view(np.uint32))
    nz = (amax > 0).unsqueeze(-1).expand_as(blocks)
    qt = (blocks / s_ref.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    q_ref = torch.where(nz, qt, torch.zeros_like(qt)).view(rows, n).numpy()
    assert np.array_equal(q, q_ref)


def test_equals_power_of_two_mode_when_amax_is_448_times_a_power_of_two():
    rng = np.random.default_rng(8)
    rows, n = 16, 256
    v = rng.uniform(-1.0, 1.0, size=(rows, n))
    for r in range(rows):
        for b in range(n // 128):
            p = int(rng.integers(-20, 20))
            blk = v[r, b * 128:(b + 1) * 128]
            blk *= 448.0 * 2.0 ** p / np.abs(blk).max()
    # the variant takes the values at fp32 first: compare on fp32-exact values
    vf = v.astype(np.float32).astype(np.float64)
    q0, s0 = oracle.act_quant(vf, 128, oracle.ACT_SCALE_E8M0)
    q1, s1 = oracle.act_quant(vf, 128, oracle.ACT_SCALE_F32)
    assert np.array_equal(q0, q1)
    assert np.array_equal(oracle.act_dequant(q0, s0), oracle.act_dequant(q1, s1))


def test_rounding_bound():
    rng = np.random.default_rng(9)
    v = (rng.standard_normal((32, 384)) * 3.0).astype(np.float32).astype(np.float64)
    q, s = oracle.act_quant(v, 128, oracle.ACT_SCALE_F32)
    d = oracle.act_dequant(q, s)
    sc = np.repeat(s.astype(np.float64), 128, axis=1)
    # e4m3 keeps 3 mantissa bits (relative step 2^-3, half-step 2^-4) down to
    # 2^-6; below it the absolute half-step is 2^-10 (in units of the scale);
    # the fp32 division adds at most one fp32 ulp of v / s
    bound = np.maximum(np.abs(v) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(d - v) <= bound)
    # the block's largest value lands on 448
    amax_pos = np.abs(v).reshape(32, 3, 128).argmax(axis=-1)
    for r in range(32):
        for b in range(3):
            assert oracle.e4m3_decode(int(q[r, b * 128 + amax_pos[r, b]])) in (448.0, -448.0)


def test_forward_variant_stays_close_to_the_power_of_two_mode():
    import synth
    inp = synth.make_inputs("toy")
    f0 = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, 8,
                        act_scale_mode=oracle.ACT_SCALE_E8M0)
    f1 = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, 8,
                        act_scale_mode=oracle.ACT_SCALE_F32)
    assert f1.as_.dtype == np.float32 and f1.hs.dtype == np.float32
    assert np.array_equal(f0.route.ids, f1.route.ids)
    rel = np.linalg.norm(f1.y64 - f0.y64) / np.linalg.norm(f0.y64)
    # both approximate the same product with e4m3 activations (steps of 2^-3
    # relative): their difference is quantisation noise, a few percent at most
    assert 0.0 < rel < 0.08, rel
