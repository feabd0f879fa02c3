"""The GPU parity checker's own rules, exercised on the CPU with planted
mistakes: a checker that let a wrong result through would make every GPU
parity claim meaningless.  The oracle's routing of a small seeded batch
stands in for the GPU's answer, and each mistake is made on a copy of it."""
import numpy as np
import pytest

import oracle
import synth
from parity import Y_MAX_ABS_RMS, Y_REL_L2, check_routing, check_y


@pytest.fixture(scope="module")
def routed():
    inp = synth.custom_inputs(64, 256, 16, 128, 4, seed=4242, bias="normal:0.5")
    c = inp.cfg
    r = oracle.route(inp.x, inp.router_w, c.k, c.score_func, inp.logit_bias, inp.sel_bias)
    return r, c.k


def test_routing_identical_passes(routed):
    r, k = routed
    same, order = check_routing(r, r.ids.copy(), r.gates.astype(np.float32), k)
    assert same.all() and order.all()


def test_routing_wrong_expert_with_clear_margin_fails(routed):
    r, k = routed
    t = int(np.argmax(r.margin))                      # the clearest selection
    ids = r.ids.copy()
    unselected = np.setdiff1d(np.arange(r.keys.shape[1]), ids[t])
    ids[t, k - 1] = unselected[np.argmax(r.keys[t, unselected])]   # the best expert left out
    with pytest.raises(AssertionError):
        check_routing(r, ids, r.gates.astype(np.float32), k)


def test_routing_swapped_order_with_clear_gap_fails(routed):
    r, k = routed
    ko = np.take_along_axis(r.keys, r.ids.astype(np.int64), axis=1)
    t = int(np.argmax(ko[:, 0] - ko[:, 1]))           # widest gap between slots 0 and 1
    ids = r.ids.copy()
    ids[t, [0, 1]] = ids[t, [1, 0]]
    with pytest.raises(AssertionError):
        check_routing(r, ids, r.gates.astype(np.float32), k)


def test_routing_near_tie_either_choice_passes(routed):
    """Make slot k-1 and the best unselected expert tie (to within the
    tolerance) in a copy of the keys: either choice is then valid."""
    r, k = routed
    t = 0
    unselected = np.setdiff1d(np.arange(r.keys.shape[1]), r.ids[t])
    e_out = int(unselected[np.argmax(r.keys[t, unselected])])
    keys = r.keys.copy()
    keys[t, e_out] = keys[t, r.ids[t, k - 1]]
    margin = r.margin.copy()
    margin[t] = 0.0
    r2 = oracle.Route(r.ids, r.gates, r.logits, r.scores, keys, margin)
    ids = r.ids.copy()
    ids[t, k - 1] = e_out
    same, _ = check_routing(r2, ids, r.gates.astype(np.float32), k)
    assert not same[t]


def _bf16(v):
    return oracle.f64_to_bf16(np.asarray(v, dtype=np.float64))


def test_y_bars():
    rng = np.random.default_rng(7)
    y = rng.standard_normal((128, 128))
    ref = _bf16(y)
    rms = np.sqrt(np.mean(oracle.bf16_to_f64(ref) ** 2))
    assert check_y(ref, ref) == (0.0, 0.0)
    # one element off by 3x the max-abs bar: fails against the oracle ...
    bad = y.copy()
    bad[3, 5] += 3 * Y_MAX_ABS_RMS * rms
    with pytest.raises(AssertionError):
        check_y(_bf16(bad), ref)
    # ... passes when the oracle fed the GPU's own Q2 codes produces it (a
    # code at a rounding boundary), the relative L2 bar still holding
    check_y(_bf16(bad), ref, _bf16(bad))
    # a small error everywhere breaks the relative L2 bar whatever the Q2 codes
    drift = y * (1 + 3 * Y_REL_L2)
    with pytest.raises(AssertionError):
        check_y(_bf16(drift), ref, _bf16(drift))
    # and the max-abs bar still binds against the Q2-fed reference
    with pytest.raises(AssertionError):
        check_y(_bf16(bad), ref, ref)
    # non-finite output fails
    nan = ref.copy()
    nan[0, 0] = 0x7FC0
    with pytest.raises(AssertionError):
        check_y(nan, ref)
