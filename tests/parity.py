"""Parity checks of the CUDA layer against the CPU oracle on the same seeded
inputs.  Bars (written here, used by the GPU tests):

  * routing ids, expert counts/offsets, permutation, Q1 codes and scales:
    bit-exact.  Where two keys are closer than TAU_KEY * max|key| their
    order is decided by rounding (the GPU accumulates logits in fp32, the
    oracle in fp64), so two results are both correct: at the selection
    boundary (k-th vs (k+1)-th key) the GPU's set must be a valid top-k of the
    oracle keys within that tolerance; inside the selected set the order must
    be key-descending within the tolerance.  Every other token's set and
    order must match exactly.  Every later step is then compared, on every
    token, with the oracle fed the GPU's selection (``oracle.forward(ids=)``,
    identical to the oracle's own selection wherever the margin is clear):
    dispatch bit-exactly, the rest within the bars below.  Q1 codes and
    scales are compared on every token of the batch.
  * gates: |gpu - oracle| <= 1e-5 (fp32 sigmoid / division vs fp64), every
    token.
  * Q2 (e4m3 SwiGLU codes): equal scale bytes and codes at most one step
    apart; at most 1e-3 of the codes may differ at all (the GPU's fp32
    gate/up sums and the oracle's fp64 sums round differently only near an
    e4m3 rounding boundary).  With fp32 block scales (amax / 448) the scales
    themselves come from those sums: they must agree to Q2_F32_SCALE_REL.
  * y: relative L2 error <= 1e-3 against the oracle's bf16-rounded output,
    and max |error| <= 2e-2 * RMS(y_oracle).  Where a Q2 code sits at an e4m3
    rounding boundary to within the fp32/fp64 difference, both neighbouring
    codes are correct (the reading that decides near-tie routing), and one
    such code moves its token's output by up to a whole e4m3 step of h times
    the down weights.  So, when the intermediates are read back, the max-abs
    bar is measured against the oracle fed the GPU's own Q2 codes and scales
    (identical to the oracle's output wherever the codes agree); the relative
    L2 bar stays against the oracle's own output.
"""
from __future__ import annotations

import numpy as np

import oracle

TAU_KEY = 1e-5
GATE_TOL = 1e-5
Y_REL_L2 = 1e-3
Y_MAX_ABS_RMS = 2e-2
Q2_MISMATCH_FRAC = 1e-3
Q2_F32_SCALE_REL = 1e-4


def bf16_f64(u16):
    return oracle.bf16_to_f64(np.asarray(u16, dtype=np.uint16))


def e4m3_ordinal(codes):
    c = np.asarray(codes, dtype=np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def run_layer(layer, inp, T=None, poison=False):
    """One forward on inp.x (its first T rows).  With ``poison`` every
    workspace buffer and the output are first filled with 0xFF bytes (NaN as
    e4m3, E8M0, bf16 and fp32), so anything the forward reads without having
    written it shows up in the output."""
    import torch
    x_np = inp.x if T is None else inp.x[:T]
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    if poison:
        layer.debug_fill_workspace(0xFF)
        y.view(torch.int16).fill_(-1)
        torch.cuda.synchronize()
    y = layer.forward(x, y)
    torch.cuda.synchronize()
    layer.check_device_error()
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def make_layer(inp, max_tokens=None, score_func=None, act_scale_mode=0):
    import fp8_mxfp4_expert_bf16_b300 as moe
    c = inp.cfg
    layer = moe.MoELayer(c.H, c.I, c.E, c.k, max_tokens or inp.x.shape[0],
                         c.score_func if score_func is None else score_func, act_scale_mode=act_scale_mode)
    load = layer.load_weights_fp8 if getattr(inp, "weight_format", "mxfp4") == "fp8" else layer.load_weights
    load(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    return layer


def check_routing(r, ids_g, gates_g, k):
    """The GPU's selection against the oracle's keys; returns (same_set,
    same_order) boolean masks over tokens (gates are checked by check_gates)."""
    kmax = np.abs(r.keys).max(axis=1)
    tol = TAU_KEY * kmax
    same_set = (np.sort(ids_g, axis=1) == np.sort(r.ids, axis=1)).all(axis=1)
    same_order = (ids_g == r.ids).all(axis=1)
    bad = np.nonzero((r.margin > tol) & ~same_set)[0]
    assert bad.size == 0, f"routing set differs on tokens with a clear margin: {bad[:10]}"
    for t in np.nonzero(~same_set)[0]:
        kth = np.sort(r.keys[t])[::-1][k - 1]
        assert len(set(ids_g[t].tolist())) == k
        assert (r.keys[t, ids_g[t]] >= kth - tol[t]).all(), f"token {t}: invalid near-tie selection"
    # order inside the set: key-descending up to the tolerance; exact where
    # consecutive oracle keys are further apart than that
    kg = np.take_along_axis(r.keys, ids_g.astype(np.int64), axis=1)
    assert (np.diff(kg, axis=1) <= tol[:, None]).all(), "selection order is not key-descending"
    ko = np.take_along_axis(r.keys, r.ids.astype(np.int64), axis=1)
    clear_order = (-np.diff(ko, axis=1) > tol[:, None]).all(axis=1)
    assert (same_order | ~clear_order | ~same_set).all(), "selection order differs where keys are well separated"
    return same_set, same_order


def check_dispatch(layer, f):
    """Counts, offsets and permutation bit-exact against the oracle's dispatch
    of the same selection (f is the oracle fed the GPU's ids)."""
    counts, offsets = layer.expert_counts()
    perm = layer.permutation()
    assert np.array_equal(counts, f.counts)
    assert np.array_equal(offsets, f.offsets)
    assert np.array_equal(perm, f.perm)
    return perm


def check_gates(gates_g, r):
    """GPU gates against the oracle's gates of the same selection, every token."""
    d = np.abs(gates_g.astype(np.float64) - r.gates)
    assert d.max() <= GATE_TOL, f"gate differs by {d.max():.2e} (token {np.unravel_index(d.argmax(), d.shape)})"


def check_act_quant_all(layer, inp):
    """Q1 codes and scales of every token of the batch, bit-exact."""
    aq_g, as_g = layer.act_quant()
    aq_o, as_o = oracle.act_quant(oracle.bf16_to_f64(inp.x), 128, getattr(layer, "act_scale_mode", 0))
    assert as_g.dtype == as_o.dtype
    bad = np.nonzero((aq_g != aq_o).any(axis=1) | (as_g != as_o).any(axis=1))[0]
    assert bad.size == 0, f"Q1 differs on {bad.size} tokens, first {bad[:8]}"


def check_y(y_g, y_o, y_q2=None):
    """y_g against the oracle's output y_o (relative L2) and against y_q2, the
    oracle's output from the GPU's own Q2 codes, when given (max abs)."""
    a = bf16_f64(y_g)
    b = bf16_f64(y_o)
    c = b if y_q2 is None else bf16_f64(y_q2)
    assert np.isfinite(a).all()
    rms = np.sqrt(np.mean(b * b))
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    mx = np.abs(a - c).max() / rms
    assert rel <= Y_REL_L2, f"rel L2 {rel:.3e}"
    assert mx <= Y_MAX_ABS_RMS, f"max abs / rms {mx:.3e}"
    return rel, mx


def slot_map(ids_g, ids_o, t):
    """For token t: oracle slot of each GPU slot (same expert)."""
    pos = {e: j for j, e in enumerate(ids_o[t].tolist())}
    return [pos[e] for e in ids_g[t].tolist()]


def check_q2(layer, f, perm, tokens, ids_g):
    """GPU SwiGLU codes (perm order) vs the oracle's for the listed tokens.
    A block's scale byte may differ by one step only when its amax sits on a
    power-of-two boundary to within the fp32/fp64 difference; such blocks
    (at most Q2_MISMATCH_FRAC of all) are excluded from the code check."""
    hq_g, hs_g = layer.inter_quant()
    k = layer.k
    n_diff = n_tot = n_sdiff = n_blk = 0
    for i, t in enumerate(tokens):
        for j, jo in enumerate(slot_map(ids_g, f.route.ids, t)):
            row = perm[t * k + j]
            if hs_g.dtype == np.float32:
                sg = hs_g[row].astype(np.float64)
                so = f.hs[i, jo].astype(np.float64)
                assert (np.abs(sg - so) <= Q2_F32_SCALE_REL * np.abs(so)).all(), f"Q2 fp32 scale (t={t}, j={j})"
                eq = np.ones(sg.size * 128, dtype=bool)
                n_blk += sg.size
            else:
                sg = hs_g[row].astype(np.int64)
                so = f.hs[i, jo].astype(np.int64)
                assert np.abs(sg - so).max() <= 1, f"Q2 scale differs by more than one step (t={t}, j={j})"
                eq = np.repeat(sg == so, 128)
                n_sdiff += int((sg != so).sum())
                n_blk += sg.size
            d = np.abs(e4m3_ordinal(hq_g[row]) - e4m3_ordinal(f.hq[i, jo]))[eq]
            assert d.size == 0 or d.max() <= 1, f"Q2 code more than one step off (t={t}, j={j})"
            n_diff += int((d > 0).sum())
            n_tot += d.size
    frac = n_diff / max(n_tot, 1)
    assert frac <= Q2_MISMATCH_FRAC, f"Q2 code mismatch fraction {frac:.2e}"
    assert n_sdiff <= Q2_MISMATCH_FRAC * max(n_blk, 1) + 1, f"{n_sdiff} of {n_blk} Q2 scales differ"
    return frac


DOWN_TF_REL = 1e-5


def check_down_teacher_forced(layer, inp, perm, toks, sel, o_g):
    """The down GEMM alone: the oracle recomputes each row's expert output in
    fp64 from the GPU's own Q2 codes and scales (so Q2 rounding differences
    drop out); the GPU's fp32 accumulation must agree to DOWN_TF_REL.
    Returns the relative error and those fp64 outputs, [len(sel), k, H] in
    the GPU's slot order."""
    hq_g, hs_g = layer.inter_quant()
    ids_g, _ = layer.routing()
    c = inp.cfg
    fp8 = getattr(inp, "weight_format", "mxfp4") == "fp8"
    num = den = 0.0
    W2 = {}
    o_tf = np.zeros((len(sel), c.k, c.H))
    for n_i, i in enumerate(sel):
        t = toks[i]
        for j in range(c.k):
            e = int(ids_g[t, j])
            if e not in W2:
                W2[e] = (oracle.fp8_block_decode(inp.w2_q[e], inp.w2_s[e]) if fp8
                         else oracle.mxfp4_decode(inp.w2_q[e], inp.w2_s[e]))
            row = perm[t * c.k + j]
            h = oracle.act_dequant(hq_g[row:row + 1], hs_g[row:row + 1])
            o = (h @ W2[e].T)[0]
            o_tf[n_i, j] = o
            num += float(np.sum((o_g[row].astype(np.float64) - o) ** 2))
            den += float(np.sum(o * o))
    rel = np.sqrt(num / max(den, 1e-300))
    assert rel <= DOWN_TF_REL, f"down GEMM vs fp64 on its own inputs: rel L2 {rel:.3e}"
    return float(rel), o_tf


def full_check(layer, inp, tokens=None, check_intermediates=True, poison=False):
    """Run the GPU layer on all of inp.x; compare routing, dispatch, gates and
    Q1 for all tokens and everything else on ``tokens`` (default all).  The
    later steps are compared with the oracle fed the GPU's selection, so a
    near-tie token that legitimately routed the other way is still checked."""
    c = inp.cfg
    mode = getattr(layer, "act_scale_mode", 0)
    wf = getattr(inp, "weight_format", "mxfp4")
    y_g = run_layer(layer, inp, poison=poison)
    ids_g, gates_g = layer.routing()
    r = oracle.route(inp.x, inp.router_w, c.k, c.score_func, inp.logit_bias, inp.sel_bias)
    same, same_order = check_routing(r, ids_g, gates_g, c.k)
    f = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, c.k, c.score_func,
                       inp.logit_bias, inp.sel_bias, tokens=tokens, act_scale_mode=mode, weight_format=wf,
                       ids=None if same_order.all() else ids_g)
    assert np.array_equal(f.route.ids, ids_g)
    toks = f.tokens
    check_gates(gates_g, f.route)
    perm = check_dispatch(layer, f)
    check_act_quant_all(layer, inp)
    stats = {"near_tie_set_tokens": int((~same).sum()), "near_tie_order_tokens": int((same & ~same_order).sum())}
    y_q2 = None
    if check_intermediates:
        stats["q2_mismatch"] = check_q2(layer, f, perm, toks, ids_g)
        o_g = layer.expert_out()
        rows = np.array([perm[t * c.k + j] for t in toks for j in range(c.k)], dtype=np.int64)
        og = o_g[rows].astype(np.float64)
        oo = f.o.reshape(-1, c.H)
        o_rel = np.linalg.norm(og - oo) / np.linalg.norm(oo)
        assert o_rel <= Y_REL_L2, f"expert output rel L2 {o_rel:.3e}"
        stats["expert_out_rel_l2"] = float(o_rel)
        stats["down_teacher_forced_rel_l2"], o_tf = check_down_teacher_forced(layer, inp, perm, toks,
                                                                               np.arange(toks.size), o_g)
        # the oracle's combine of the outputs from the GPU's own Q2 codes (the
        # oracle's gates; its slots are the GPU's, asserted above)
        y_q2 = oracle.f64_to_bf16(np.einsum("nk,nkh->nh", f.route.gates[toks], o_tf))
    rel, mx = check_y(y_g[toks], f.y, y_q2)
    stats.update(rel_l2=rel, max_abs_over_rms=mx)
    return stats, y_g, f
