"""GPU parity: the CUDA layer (through the C ABI) against the CPU oracle on
seeded synthetic inputs — small shapes in full, the five workloads at full
size on sampled tokens plus full routing/dispatch."""
import numpy as np
import pytest

import oracle
import synth
from parity import full_check, make_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_toy_full_parity():
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    stats, _, _ = full_check(layer, inp)
    print("toy", stats)


@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score
    (1, 512, 16, 256, 8, "none", 0),        # single token
    (3, 512, 16, 256, 8, "none", 0),        # ragged tiny
    (300, 512, 16, 256, 8, "none", 0),      # several m-tiles per expert, ragged tail
    (200, 384, 8, 256, 2, "normal:1.0", 0), # hidden not a multiple of 256 (128-wide down tiles)
    (130, 256, 1, 128, 1, "none", 0),       # one expert: a dense SwiGLU FFN; 130 rows = 2 m-tiles
    (64, 512, 16, 256, 8, "none", 1),       # softmax scores
    (77, 1024, 40, 384, 6, "zipf:1.1", 0),  # skewed routing, k=6, E not a power of two
    (129, 768, 512, 128, 8, "none", 0),     # E at its maximum
])
def test_shapes_full_parity(shape):
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=100 + T, bias=bias, score_func=score)
    layer = make_layer(inp)
    stats, _, _ = full_check(layer, inp)
    print(shape, stats)


@pytest.mark.parametrize("shape", [(64, 512, 16, 256, 8), (300, 512, 16, 256, 8), (77, 1024, 40, 384, 6)])
def test_structural_invariants(shape):
    T, H, E, I, k = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=700 + T)
    layer = make_layer(inp)
    run_layer(layer, inp)
    ids, gates = layer.routing()
    counts, offsets = layer.expert_counts()
    perm = layer.permutation()
    assert np.allclose(gates.sum(axis=1), 1.0, atol=1e-6)
    assert (gates > 0).all()
    assert all(len(set(r.tolist())) == k for r in ids) and ((0 <= ids) & (ids < E)).all()
    assert counts.sum() == T * k and np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=E))
    assert offsets[0] == 0 and offsets[E] == T * k and (np.diff(offsets) >= 0).all()
    assert np.array_equal(np.sort(perm), np.arange(T * k))


def test_forward_host_matches_device_and_is_deterministic():
    import torch
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    y1 = run_layer(layer, inp)
    y2 = run_layer(layer, inp)
    assert np.array_equal(y1, y2)
    yh = layer.forward_host(np.ascontiguousarray(inp.x))
    assert np.array_equal(yh, y1)
    # a smaller T on the same handle, then back
    y_small = run_layer(layer, inp, T=5)
    assert np.array_equal(y_small, y1[:5])


def test_zero_tokens_is_a_noop():
    import torch
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    x = torch.empty((0, inp.cfg.H), dtype=torch.bfloat16, device="cuda")
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert y.shape == (0, inp.cfg.H)
    layer.check_device_error()


def test_argument_errors():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    inp = synth.make_inputs("toy")
    c = inp.cfg
    layer = moe.MoELayer(c.H, c.I, c.E, c.k, 16)
    x = torch.zeros((4, c.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.forward(x)
    assert ei.value.status == 5                                   # not loaded
    bad = inp.w13_s.copy()
    bad[3, 7, 2] = 0xFF
    with pytest.raises(moe.MoEError) as ei:
        layer.load_weights(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, bad, inp.w2_q, inp.w2_s)
    assert ei.value.status == 1                                   # NaN scale byte
    layer.load_weights(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    with pytest.raises(moe.MoEError) as ei:
        layer.forward(torch.zeros((17, c.H), dtype=torch.bfloat16, device="cuda"))
    assert ei.value.status == 2                                   # T > max_tokens
    xm = torch.zeros((4 * c.H + 8,), dtype=torch.bfloat16, device="cuda")[1:1 + 4 * c.H].view(4, c.H)
    with pytest.raises(moe.MoEError) as ei:
        layer.forward(xm)
    assert ei.value.status == 1                                   # misaligned
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check_device_error()


FULL = ["flash-decode", "pro-decode", "flash-prefill", "pro-prefill-skew"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_sampled(name):
    inp = synth.make_inputs(name)
    T = inp.cfg.T
    rng = np.random.default_rng(1)
    tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 14, replace=False)]))
    layer = make_layer(inp)
    stats, y, _ = full_check(layer, inp, tokens=tokens)
    print(name, stats)
    from parity import bf16_f64
    assert np.isfinite(bf16_f64(y)).all()


def test_forward_captures_in_a_cuda_graph():
    """moe_forward enqueues kernels only (no sync, no readback): it can be
    captured in a CUDA graph, and replays give the eager result."""
    import torch
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    y_eager = run_layer(layer, inp)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, y, s)      # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, y)
    y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    layer.check_device_error()
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), y_eager)


def test_pipelined_host_calls_match_device_forwards():
    """moe_forward_host_async: several batches of different sizes issued
    back to back (copies overlapping the neighbouring forwards through two
    staging slots), each into its own pinned output; after moe_host_sync
    every output equals the device-buffer forward of the same batch."""
    import torch
    inp = synth.custom_inputs(300, 512, 16, 256, 8, seed=1301, bias="normal:0.5")
    layer = make_layer(inp)
    xs = [np.ascontiguousarray(inp.x[a:b]) for a, b in [(0, 300), (0, 1), (17, 117), (0, 300), (5, 264)]]
    pinned_x = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs]
    pinned_y = [torch.full_like(px, -1).pin_memory() for px in pinned_x]
    for px, py in zip(pinned_x, pinned_y):
        layer.forward_host_async(px, py)
    layer.host_sync()
    for x, py in zip(xs, pinned_y):
        ref = layer.forward(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
        torch.cuda.synchronize()
        assert np.array_equal(py.numpy().view(np.uint16), ref.view(torch.int16).cpu().numpy().view(np.uint16))
    layer.check_device_error()

@pytest.mark.parametrize("shape", [
    # T, H, E, I, k, bias, score: batches of at least 4096 tokens select their
    # top-k in the router's epilogue (one CTA per 128 tokens, all experts)
    (4100, 256, 40, 128, 6, "zipf:1.1", 0),       # one expert chunk (N = 48), ragged last token tile
    (4160, 1024, 260, 128, 4, "normal:1.0", 0),   # a 16-wide second chunk, 16 K-steps
    (4096, 256, 384, 128, 8, "normal:0.5", 0),    # chunks of 256 + 128, three ring stages
    (4200, 256, 512, 128, 8, "none", 1),          # E at its maximum, softmax, two stages (the ring wraps)
])
def test_fused_router_shapes(shape):
    T, H, E, I, k, bias, score = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=900 + E, bias=bias, score_func=score)
    layer = make_layer(inp)
    rng = np.random.default_rng(E)
    tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    # routing, gates, dispatch and Q1 on every token; the rest on the sample
    stats, _, _ = full_check(layer, inp, tokens=tokens)
    logits = layer.logits()
    r = oracle.route(inp.x, inp.router_w, k, score, inp.logit_bias, inp.sel_bias)
    err = np.abs(logits.astype(np.float64) - r.logits).max() / np.abs(r.logits).max()
    print(shape, stats, "logit max rel err", err)
    assert err <= 1e-5
