"""Pins of the oracle's fp8 expert format (e4m3 weights with one fp32 scale
per 128 x 128 block, the V2.5 experts of "MiMo V2.6 Pro and Flash
architecture teardown", "Why Are the V2.6 Files Half the Size of V2.5?"):
torch's own e4m3 decoding, the block a scale belongs to (element by
element), an FFN whose products are exact integers, and closeness to the
MXFP4 path on the same draws."""
import numpy as np
import pytest

import oracle
import synth


def test_decode_matches_torch_float8():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, size=(256, 384), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C          # no NaN codes in weights
    scales = rng.uniform(0.5, 4.0, size=(2, 3)).astype(np.float32)
    d = oracle.fp8_block_decode(codes, scales)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = ref * np.kron(scales.astype(np.float64), np.ones((128, 128)))
    assert np.array_equal(d, ref)


def test_scale_belongs_to_its_128x128_block():
    R, K = 384, 256
    q = np.full((R, K), 0x38, dtype=np.uint8)      # e4m3 1.0 everywhere
    s = np.array([[2.0 ** (i - 3 * j) for j in range(K // 128)] for i in range(R // 128)], dtype=np.float32)
    d = oracle.fp8_block_decode(q, s)
    for r in range(0, R, 37):
        for c in range(0, K, 29):
            assert d[r, c] == 2.0 ** (r // 128 - 3 * (c // 128)), (r, c)


def _e4m3_int(v):
    # e4m3 codes of the integers -8..8 (exact in e4m3)
    torch = pytest.importorskip("torch")
    return torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_ffn_with_exact_integer_products():
    rng = np.random.default_rng(12)
    n, H, I = 5, 256, 128
    a = rng.integers(-4, 5, size=(n, H)).astype(np.float64)          # exact activations
    w13i = rng.integers(-8, 9, size=(2 * I, H))
    w2i = rng.integers(-8, 9, size=(H, I))
    s13 = np.array([[2.0 ** -(i + j) for j in range(H // 128)] for i in range(2 * I // 128)], dtype=np.float32)
    s2 = np.array([[2.0 ** -(2 * i + j) for j in range(I // 128)] for i in range(H // 128)], dtype=np.float32)
    w13q = _e4m3_int(w13i.astype(np.float32))
    w2q = _e4m3_int(w2i.astype(np.float32))
    h, hq, hs, o = oracle.expert_ffn(a, w13q, s13, w2q, s2, weight_format="fp8")
    W13 = w13i * np.kron(s13.astype(np.float64), np.ones((128, 128)))
    gu = a @ W13.T                                                  # exact (small integers times powers of two)
    g, u = gu[:, :I], gu[:, I:]
    assert np.array_equal(h, g / (1.0 + np.exp(-g)) * u)
    W2 = w2i * np.kron(s2.astype(np.float64), np.ones((128, 128)))
    assert np.allclose(o, oracle.act_dequant(hq, hs) @ W2.T, rtol=0, atol=0)


def test_forward_fp8_close_to_mxfp4_on_the_same_draws():
    x4 = synth.make_inputs("toy")
    x8 = synth.make_inputs("toy", weights="fp8")
    assert x8.w13_q.shape == (16, 512, 512) and x8.w13_s.dtype == np.float32
    f4 = oracle.forward(x4.x, x4.router_w, x4.w13_q, x4.w13_s, x4.w2_q, x4.w2_s, 8)
    f8 = oracle.forward(x8.x, x8.router_w, x8.w13_q, x8.w13_s, x8.w2_q, x8.w2_s, 8, weight_format="fp8")
    assert np.array_equal(f4.route.ids, f8.route.ids)   # same router, same x
    rel = np.linalg.norm(f8.y64 - f4.y64) / np.linalg.norm(f4.y64)
    # MXFP4 keeps 1 mantissa bit (relative steps up to 1/3), e4m3 keeps 3: the two
    # encodings of the same fp32 weights give outputs a few tens of percent apart at most
    assert 0.0 < rel < 0.5, rel
