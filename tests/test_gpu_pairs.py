"""GPU parity of the SM-pair grouped GEMM (two CTAs of a cluster share one
256-row MMA): batches larger than one dispatch chunk put an expert's heavy
m-tiles in pairs, an odd one left over on the single-SM kernel.  Full
parity against the oracle on shapes that give full pairs, pairs whose
second m-tile is partial, left-over m-tiles and light tails."""
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


def _tile_mix(counts):
    """(pairs, left-over heavy m-tiles, light m-tiles) of the expert counts,
    with 128-row m-tiles, light = at most 16 valid rows."""
    pairs = solo = light = 0
    for c in counts:
        mt = -(-int(c) // 128)
        rem = int(c) - 128 * (mt - 1)
        lt = 1 if mt > 0 and rem <= 16 else 0
        heavy = mt - lt
        pairs += heavy // 2
        solo += heavy % 2
        light += lt
    return pairs, solo, light


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias
    (1024, 512, 8, 256, 2, "normal:0.5"),   # ~256 rows per expert: pairs, left-overs, light tails
    (600, 1024, 4, 384, 2, "none"),         # ~300 rows: a pair + a left-over partial m-tile
    (2048, 256, 4, 128, 3, "zipf:1.1"),     # skewed: one expert with many pairs
    (700, 768, 10, 256, 8, "none"),         # k = 8 of 10, ~560 rows per expert: two pairs + a left-over
])
def test_pair_tiles_full_parity(shape):
    T, H, E, I, k, bias = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=900 + T, bias=bias)
    layer = make_layer(inp)
    stats, _, _ = full_check(layer, inp)
    counts, _ = layer.expert_counts()
    pairs, solo, light = _tile_mix(counts)
    print(shape, stats, "pairs", pairs, "left-over", solo, "light", light)
    assert pairs > 0
    # router, top-k, histogram, scan, row ranks, quantisation, two launches
    # per GEMM (single-SM, then SM-pair), combine
    assert layer.launch_count() == 11

