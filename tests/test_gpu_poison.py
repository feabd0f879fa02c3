"""A forward writes everything it reads.  Every workspace buffer of the
handle (routing and dispatch tables, quantised activation and SwiGLU rows
with their scales, expert outputs) and the output are filled with 0xFF bytes
(NaN as e4m3, E8M0, bf16 and fp32) before the forward; the layer must still
match the oracle on every token, be finite everywhere, and give bit for bit
the output of a freshly initialised handle."""
import numpy as np
import pytest

import synth
from parity import bf16_f64, full_check, make_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("shape,mode,weights", [
    # (T, H, E, I, k, bias), activation scale mode, expert format
    ((64, 512, 16, 256, 8, "none"), 0, "mxfp4"),        # the toy layer
    ((300, 512, 16, 256, 8, "none"), 0, "mxfp4"),       # ragged: light and heavy m-tiles, several per expert
    ((200, 384, 8, 256, 2, "normal:1.0"), 0, "mxfp4"),  # 128-wide down tiles
    ((77, 1024, 40, 384, 6, "zipf:1.1"), 0, "mxfp4"),   # skewed routing, k = 6
    ((300, 512, 16, 256, 8, "none"), 1, "mxfp4"),       # fp32 activation scales (promotion path)
    ((300, 512, 16, 256, 8, "none"), 0, "fp8"),         # fp8 experts (promotion path)
])
def test_poisoned_workspace_does_not_reach_the_output(shape, mode, weights):
    T, H, E, I, k, bias = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=900 + T + 7 * mode, bias=bias, weights=weights)
    clean = make_layer(inp, act_scale_mode=mode)
    y_clean = run_layer(clean, inp)
    clean.close()
    layer = make_layer(inp, act_scale_mode=mode)
    stats, y, _ = full_check(layer, inp, poison=True)
    assert np.isfinite(bf16_f64(y)).all()
    assert np.array_equal(y, y_clean)
    # and again on the same (still poisoned in its padding rows) handle, smaller T
    y_small = run_layer(layer, inp, T=T // 3 + 1, poison=True)
    assert np.isfinite(bf16_f64(y_small)).all()
    print(shape, mode, weights, stats)
