"""GPU parity of the fp8 expert format (e4m3 weights with an fp32 scale per
128 x 128 block, folded into fp32 partial sums per K block in the grouped
GEMMs) against the oracle, through the C ABI, with either activation scale
mode."""
import numpy as np
import pytest

import synth
from parity import full_check, make_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("act_scale_mode", [0, 1])
def test_toy_full_parity_fp8_weights(act_scale_mode):
    inp = synth.make_inputs("toy", weights="fp8")
    layer = make_layer(inp, act_scale_mode=act_scale_mode)
    stats, _, _ = full_check(layer, inp)
    print("toy fp8", act_scale_mode, stats)


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score
    (1, 512, 16, 256, 8, "none", 0),        # single token
    (300, 512, 16, 256, 8, "none", 0),      # light and heavy m-tiles
    (200, 384, 8, 256, 2, "normal:1.0", 0), # 128-wide down tiles
    (130, 256, 1, 128, 1, "none", 0),       # one expert, 2 m-tiles
])
def test_shapes_full_parity_fp8_weights(shape):
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=500 + T, bias=bias, score_func=score, weights="fp8")
    layer = make_layer(inp)
    stats, _, _ = full_check(layer, inp)
    print(shape, stats)


def test_flash_decode_sampled_fp8_weights():
    inp = synth.make_inputs("flash-decode", weights="fp8")
    layer = make_layer(inp)
    toks = np.random.default_rng(6).choice(inp.x.shape[0], 16, replace=False)
    stats, _, _ = full_check(layer, inp, tokens=np.sort(toks))
    print("flash-decode fp8", stats)


def test_flash_prefill_sampled_fp8_weights():
    """Prefill-sized batch with fp8 experts: the fused router's selection and
    the heavy promotion ring; routing, dispatch and Q1 on every token, the
    rest on 16 sampled tokens."""
    inp = synth.make_inputs("flash-prefill", weights="fp8")
    layer = make_layer(inp)
    toks = np.random.default_rng(8).choice(inp.x.shape[0], 16, replace=False)
    stats, _, _ = full_check(layer, inp, tokens=np.sort(toks))
    print("flash-prefill fp8", stats)


def test_invalid_fp8_weights_are_rejected():
    import fp8_mxfp4_expert_bf16_b300 as moe
    inp = synth.make_inputs("toy", weights="fp8")
    layer = make_layer(inp)
    bad = inp.w13_q.copy()
    bad[3, 5, 7] = 0x7F                      # e4m3 NaN
    with pytest.raises(moe.MoEError):
        layer.load_weights_fp8(inp.router_w, inp.logit_bias, inp.sel_bias, bad, inp.w13_s, inp.w2_q, inp.w2_s)
    bad_s = inp.w2_s.copy()
    bad_s[1, 0, 0] = -1.0
    with pytest.raises(moe.MoEError):
        layer.load_weights_fp8(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, bad_s)
    # a valid load afterwards works again
    layer.load_weights_fp8(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    y = run_layer(layer, inp)
    assert np.isfinite(y.view(np.uint16).astype(np.float64)).all()
