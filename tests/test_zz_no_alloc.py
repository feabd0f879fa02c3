"""The allocation-free routing entry point, for callers that cannot allocate
device memory on their call path (their device memory belongs to their own
allocator or budget, or a cudaMalloc there could synchronise the device and
stall work in flight).  It is checked through the C ABI against the layer's
own routing (moe_forward) and against the oracle, on two calls in a row.

Its logits are summed over all of H in one pass while moe_forward splits H
for small batches, so the two may select differently where a token's k-th
and (k+1)-th keys are within fp32 rounding; there both must be a valid top-k
of the oracle's keys (the near-tie rule of every parity test), and
everywhere else they must agree exactly, gates within the gate tolerance.

Collected last on purpose: it shares one fixed scratch array inside the
library, and a run that stops at the first failure has run every other test
by then.  It passes on its own in a fresh process too.
"""
import numpy as np
import pytest

import oracle
import synth
from parity import GATE_TOL, TAU_KEY, check_gates, check_routing, make_layer, run_layer

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _tensors(inp):
    import torch
    dev = torch.device("cuda")
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).to(dev)
    wr = torch.from_numpy(inp.router_w.view(np.int16)).view(torch.bfloat16).to(dev)
    lb = torch.from_numpy(inp.logit_bias).to(dev)
    cb = torch.from_numpy(inp.sel_bias).to(dev)
    return x, wr, lb, cb


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score
    (64, 512, 16, 256, 8, "none", 0),          # the toy layer
    (64, 4096, 256, 128, 8, "none", 0),        # Flash router shape (64-expert router tiles)
    (600, 1024, 64, 128, 6, "normal:0.5", 1),  # T > 512: 128-expert router tiles, softmax, logit bias
])
def test_route_noalloc_matches_the_layer_and_the_oracle_twice(shape):
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=7 + T, bias=bias, score_func=score)
    layer = make_layer(inp)
    run_layer(layer, inp)
    ids_ref, gates_ref = layer.routing()
    r = oracle.route(inp.x, inp.router_w, k, score, inp.logit_bias, inp.sel_bias)
    check_routing(r, ids_ref, gates_ref, k)
    clear = r.margin > TAU_KEY * np.abs(r.keys).max(axis=1)

    x, wr, lb, cb = _tensors(inp)
    for call in range(2):
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        gates = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        moe.route_noalloc(x, wr, lb, cb, k, score, ids, gates)
        torch.cuda.synchronize()
        ids_np, gates_np = ids.cpu().numpy(), gates.cpu().numpy()
        # against the oracle: the near-tie rule, gates of the chosen experts
        check_routing(r, ids_np, gates_np, k)
        check_gates(gates_np, oracle.route_with_ids(r, ids_np))
        # against the layer's entry point: the same selection wherever the margin is clear
        same = (ids_np == ids_ref).all(axis=1)
        assert (same | ~clear).all(), f"call {call}: ids differ from moe_forward's on clearly separated tokens"
        np.testing.assert_allclose(gates_np[same], gates_ref[same], atol=GATE_TOL, rtol=0)
    moe.route_noalloc_check_error()
    # NULL biases mean zeros
    if bias == "none":
        ids0, gates0 = moe.route_noalloc(x, wr, None, None, k, score)
        torch.cuda.synchronize()
        assert np.array_equal(ids0.cpu().numpy(), ids_np)
        np.testing.assert_array_equal(gates0.cpu().numpy(), gates_np)


def test_route_noalloc_rejects_sizes_beyond_its_scratch_and_bad_tensors():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    T, H, E = 4097, 128, 256            # T * E = 1,048,832 > 2^20
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.route_noalloc(x, wr, None, None, 8)
    assert ei.value.status == 2 and "scratch" in str(ei.value)
    with pytest.raises(ValueError):
        moe.route_noalloc(x[:8].float(), wr, None, None, 8)            # x not bf16
    with pytest.raises(ValueError):
        moe.route_noalloc(x[:8, ::2], wr[:, ::2], None, None, 8)       # not contiguous


def test_route_noalloc_reports_a_timed_out_wait_once():
    """A kernel wait that gives up is kept in the scratch's error record until
    moe_route_noalloc_check_error reports it (here provoked with the
    library's wait self-test, a 20 ms wait on a barrier nothing completes)."""
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    L = moe.lib()
    inp = synth.custom_inputs(64, 512, 16, 256, 8, seed=71)
    x, wr, lb, cb = _tensors(inp)
    ids1, gates1 = moe.route_noalloc(x, wr, lb, cb, 8)
    assert L.moe_selftest_wait_timeout(None, 20000) == 0
    ids2, gates2 = moe.route_noalloc(x, wr, lb, cb, 8)      # a later call does not clear the record
    with pytest.raises(moe.MoEError) as ei:
        moe.route_noalloc_check_error()
    assert ei.value.status == MOE_ERR_TIMEOUT and "timed out" in str(ei.value)
    moe.route_noalloc_check_error()                          # cleared
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2) and torch.equal(gates1, gates2)
