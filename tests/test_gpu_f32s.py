"""GPU parity of the fp32-scale activation mode (s = amax / 448 per 1 x 128
block, folded into fp32 partial sums per K block in the grouped GEMMs)
against the oracle's same mode, through the C ABI."""
import numpy as np
import pytest

import synth
from parity import full_check, make_layer

pytestmark = pytest.mark.gpu

F32 = 1


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_toy_full_parity_f32_scales():
    inp = synth.make_inputs("toy")
    layer = make_layer(inp, act_scale_mode=F32)
    stats, _, _ = full_check(layer, inp)
    print("toy f32s", stats)


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score
    (1, 512, 16, 256, 8, "none", 0),        # single token
    (300, 512, 16, 256, 8, "none", 0),      # several m-tiles per expert: light and heavy phases
    (200, 384, 8, 256, 2, "normal:1.0", 0), # 128-wide down tiles
    (130, 256, 1, 128, 1, "none", 0),       # one expert, 2 m-tiles
])
def test_shapes_full_parity_f32_scales(shape):
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=300 + T, bias=bias, score_func=score)
    layer = make_layer(inp, act_scale_mode=F32)
    stats, _, _ = full_check(layer, inp)
    print(shape, stats)


def test_flash_decode_sampled_f32_scales():
    inp = synth.make_inputs("flash-decode")
    layer = make_layer(inp, act_scale_mode=F32)
    toks = np.random.default_rng(5).choice(inp.x.shape[0], 16, replace=False)
    stats, _, _ = full_check(layer, inp, tokens=np.sort(toks))
    print("flash-decode f32s", stats)


def test_flash_prefill_sampled_f32_scales():
    """Prefill-sized batch: the fused router's selection, every m-tile in the
    heavy ring (three 128-column half-step partials); routing, dispatch and
    Q1 on every token, the rest on 16 sampled tokens."""
    inp = synth.make_inputs("flash-prefill")
    layer = make_layer(inp, act_scale_mode=F32)
    toks = np.random.default_rng(7).choice(inp.x.shape[0], 16, replace=False)
    stats, _, _ = full_check(layer, inp, tokens=np.sort(toks))
    print("flash-prefill f32s", stats)


def test_scale_getters():
    import fp8_mxfp4_expert_bf16_b300 as moe
    from parity import run_layer
    inp = synth.make_inputs("toy")
    # power-of-two mode: the fp32 getter returns 2^(byte - 127)
    layer = make_layer(inp)
    run_layer(layer, inp)
    _, sb = layer.act_quant()
    sf = layer.block_scales_f32("act")
    assert np.array_equal(sf, np.ldexp(1.0, sb.astype(np.int64) - 127).astype(np.float32))
    _, hb = layer.inter_quant()
    hf = layer.block_scales_f32("inter")
    assert np.array_equal(hf, np.ldexp(1.0, hb.astype(np.int64) - 127).astype(np.float32))
    # fp32 mode: a u8 scale output is refused
    layer2 = make_layer(inp, act_scale_mode=F32)
    run_layer(layer2, inp)
    out = np.empty((inp.x.shape[0], inp.cfg.H // 128), dtype=np.uint8)
    with pytest.raises(moe.MoEError):
        layer2._check(layer2.L.moe_get_act_quant(layer2.h, None, out.ctypes.data))
