"""Light m-tiles (at most 16 valid rows) put the token rows on the MMA's N
side.  This test builds batches where experts' last m-tiles hold 1..8 and
9..16 rows (both token groups of the epilogue warps, both activation boxes)
beside heavy m-tiles, with 256- and 128-wide down tiles and K-step counts
that do and do not fill the promotion modes' four-step ring units (H = 512:
4 K-steps, I = 256: 2; H = 384 and I = 384: 3), in all four arithmetic
modes, and checks the whole layer against the oracle fed the GPU's ids."""
import numpy as np
import pytest

import synth
from parity import full_check, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("weights,act_scale_mode", [("mxfp4", 0), ("mxfp4", 1), ("fp8", 0), ("fp8", 1)])
@pytest.mark.parametrize("H,I", [(512, 256), (384, 384)])
def test_light_tiles_all_modes(weights, act_scale_mode, H, I):
    T, E, k = 48, 32, 8
    inp = synth.custom_inputs(T, H, E, I, k, seed=2102, bias="normal:0.7", weights=weights)
    layer = make_layer(inp, act_scale_mode=act_scale_mode)
    stats, _, _ = full_check(layer, inp)
    counts, _ = layer.expert_counts()
    last = np.where(counts > 0, counts - 128 * ((counts - 1) // 128), 0)   # rows of each expert's last m-tile
    n_low, n_high, n_heavy = int(((last >= 1) & (last <= 8)).sum()), int(((last >= 9) & (last <= 16)).sum()), \
        int((counts > 16).sum())
    print(weights, act_scale_mode, H, I, stats, "light 1..8:", n_low, "light 9..16:", n_high, "heavy:", n_heavy)
    assert n_low > 0 and n_high > 0 and n_heavy > 0
