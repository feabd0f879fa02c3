"""Tensor-parallel shards of the expert middle dimension, on one GPU: G shard
handles of the same layer (tp_size = G, tp_rank = 0..G-1, each loaded from
the whole layer's weights) run the same batch.  Routing, dispatch and the
input quantisation must equal the whole layer's bit for bit on every shard;
each shard's SwiGLU codes must be exactly its columns of the whole layer's;
its fp32 partial output must match the oracle's partial for that shard; and
the partials added up and rounded once must match the oracle's layer output
(the parity bars of every test).  Only the all-reduce between GPUs is not
exercised here (one GPU; the orchestration is tested with gloo ranks)."""
import numpy as np
import pytest

import oracle
import synth
from parity import Y_REL_L2, check_y, full_check, make_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _shard(inp, G, r, mode):
    import fp8_mxfp4_expert_bf16_b300 as moe
    c = inp.cfg
    layer = moe.MoELayer(c.H, c.I, c.E, c.k, inp.x.shape[0], c.score_func, act_scale_mode=mode, tp_size=G,
                         tp_rank=r)
    load = layer.load_weights_fp8 if inp.weight_format == "fp8" else layer.load_weights
    load(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    return layer


@pytest.mark.parametrize("G,mode,weights,shape", [
    (2, 0, "mxfp4", (300, 512, 16, 512, 8)),
    (4, 0, "mxfp4", (300, 512, 16, 512, 8)),
    (4, 0, "mxfp4", (64, 1024, 32, 1024, 8)),   # decode-like: light m-tiles only
    (2, 1, "mxfp4", (300, 512, 16, 512, 8)),    # fp32 activation scales
    (2, 0, "fp8", (200, 512, 16, 1024, 8)),     # fp8 experts
])
def test_shards_add_up_to_the_layer(G, mode, weights, shape):
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    T, H, E, I, k = shape
    inp = synth.custom_inputs(T, H, E, I, k, seed=500 + G + 3 * mode, bias="normal:0.5", weights=weights)
    full = make_layer(inp, act_scale_mode=mode)
    _, y_full, f = full_check(full, inp)          # the whole layer against the oracle (fed the GPU's ids)
    ids_f, gates_f = full.routing()
    counts_f, offsets_f = full.expert_counts()
    perm_f = full.permutation()
    aq_f, as_f = full.act_quant()
    hq_f, hs_f = full.inter_quant()
    parts_o = oracle.tp_partials(f, inp.w2_q, inp.w2_s, G, weights)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    Il = I // G
    parts = []
    for r in range(G):
        sh = _shard(inp, G, r, mode)
        y32 = sh.forward_partial(x)
        torch.cuda.synchronize()
        sh.check_device_error()
        ids, gates = sh.routing()
        assert np.array_equal(ids, ids_f) and np.array_equal(gates, gates_f)
        counts, offsets = sh.expert_counts()
        assert np.array_equal(counts, counts_f) and np.array_equal(offsets, offsets_f)
        assert np.array_equal(sh.permutation(), perm_f)
        aq, as_ = sh.act_quant()
        assert np.array_equal(aq, aq_f) and np.array_equal(as_, as_f)
        hq, hs = sh.inter_quant()
        assert np.array_equal(hq, hq_f[:, r * Il:(r + 1) * Il])
        assert np.array_equal(hs, hs_f[:, r * Il // 128:(r + 1) * Il // 128])
        p = y32.cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(p - parts_o[r]) / np.linalg.norm(parts_o[r])
        assert rel <= Y_REL_L2, f"shard {r}: partial output rel L2 {rel:.2e}"
        parts.append(y32)
        sh.close()
    y = moe.sum_partials_bf16(parts)
    torch.cuda.synchronize()
    y_np = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rel, mx = check_y(y_np, f.y)
    a, b = oracle.bf16_to_f64(y_np), oracle.bf16_to_f64(y_full)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 2e-3   # the whole layer on the GPU: bf16 rounding apart
    print(G, mode, weights, shape, "rel L2 vs oracle", rel)


def test_unsharded_partial_rounds_to_the_forward():
    """tp_size 1: the fp32 partial output rounded by moe_sum_partials_bf16 is
    the forward's bf16 output, bit for bit (the same sum, one rounding)."""
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    y = run_layer(layer, inp)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    y32 = layer.forward_partial(x)
    yb = moe.sum_partials_bf16([y32])
    torch.cuda.synchronize()
    assert np.array_equal(yb.view(torch.int16).cpu().numpy().view(np.uint16), y)


def test_shard_config_is_checked():
    import fp8_mxfp4_expert_bf16_b300 as moe
    with pytest.raises(moe.MoEError):
        moe.MoELayer(512, 256, 16, 8, 64, tp_size=4, tp_rank=0)     # 256 / 4 = 64: not a multiple of 128
    with pytest.raises(moe.MoEError):
        moe.MoELayer(512, 256, 16, 8, 64, tp_size=2, tp_rank=2)     # rank outside the group
