"""The allocation-free routing entry point (for callers that cannot allocate
device memory on their call path) against the layer's own routing.

Collected last on purpose: it shares one fixed scratch array inside the
library, and a run that stops at the first failure has run every other test
by then.  It passes on its own in a fresh process too.
"""
import numpy as np
import pytest

import synth
from parity import GATE_TOL, make_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score
    (64, 512, 16, 256, 8, "none", 0),          # the toy layer
    (64, 4096, 256, 128, 8, "none", 0),        # Flash router shape (64-expert router tiles)
    (600, 1024, 64, 128, 6, "normal:0.5", 1),  # T > 512: 128-expert router tiles, softmax, logit bias
])
def test_route_noalloc_matches_layer_routing_twice(shape):
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=7 + T, bias=bias, score_func=score)
    layer = make_layer(inp)
    run_layer(layer, inp)
    ids_ref, gates_ref = layer.routing()

    dev = torch.device("cuda")
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).to(dev)
    wr = torch.from_numpy(inp.router_w.view(np.int16)).view(torch.bfloat16).to(dev)
    lb = torch.from_numpy(inp.logit_bias).to(dev)
    cb = torch.from_numpy(inp.sel_bias).to(dev)
    for call in range(2):
        ids = torch.full((T, k), -1, dtype=torch.int32, device=dev)
        gates = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
        moe.route_noalloc(x, wr, lb, cb, k, score, ids, gates)
        torch.cuda.synchronize()
        ids_np, gates_np = ids.cpu().numpy(), gates.cpu().numpy()
        assert np.array_equal(ids_np, ids_ref), f"call {call}: ids differ"
        np.testing.assert_allclose(gates_np, gates_ref, atol=GATE_TOL, rtol=0)
    # NULL biases mean zeros: compare with explicit zero tensors
    if bias == "none":
        ids0, gates0 = moe.route_noalloc(x, wr, None, None, k, score)
        torch.cuda.synchronize()
        assert np.array_equal(ids0.cpu().numpy(), ids_ref)
        np.testing.assert_allclose(gates0.cpu().numpy(), gates_ref, atol=GATE_TOL, rtol=0)


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    T, H, E = 4097, 128, 256            # T * E = 1,048,832 > 2^20
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.route_noalloc(x, wr, None, None, 8)
    assert ei.value.status == 2 and "scratch" in str(ei.value)
