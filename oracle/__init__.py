"""CPU oracle for the routed MXFP4/FP8 MoE layer — TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the layer computes.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it; the product path (the CUDA library and its binding) never
does, and the two share no code.  The scalar codecs live in ``codecs.c``
(built with gcc); the dense fp64 contractions are numpy matmuls (a library
primitive used as one step, no blocking or fusion of our own).

Sources (web pages on MiMo-V2.6; each function names the passage it follows):
  [P2] vLLM recipe "XiaomiMiMo/MiMo-V2.6-Pro-RL", section "Overview"
       (384 routed experts top-8; weights stored as mxfp4, computed as
       block-wise FP8 e4m3).
  [P3] devupai "MiMo-V2.6-Flash", sections "No shared expert" and
       "Self-Hosting" (no shared expert; dynamic activation scheme).
  [P5] kgptalkie "MiMo V2.6 Pro and Flash architecture teardown", sections
       "How Is the Backbone Built?" (no shared expert), "How Big Is Each
       Expert?" (sigmoid router plus a per-expert correction bias, 8 experts
       per token, gate/up/down around a 2,048-wide middle) and "Why Are the
       V2.6 Files Half the Size of V2.5?" (MXFP4 layout; router in BF16).

Readings where the pages are silent (each is listed in the design notes):
  * activation function SwiGLU: h = silu(gate) * up, gate rows [0, I) of the
    fused gate/up matrix, up rows [I, 2I);
  * activation blocks are 1 x 128 along K with a power-of-two (E8M0) scale,
    the smallest one that keeps the block's amax within e4m3's 448; the
    variant with an fp32 scale amax / 448 takes the values at fp32 and
    divides in fp32 (an all-zero block: scale 0, zero codes);
  * the correction bias is added to the scores for selection only; the
    router's logit bias is added to the logits;
  * gates are the selected (unbiased) scores renormalised to sum to 1;
  * top-k ties go to the lower expert index;
  * intermediates exact/fp64; the layer output is rounded once to bf16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "codecs.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle_codecs.so")

SCORE_SIGMOID = 0
SCORE_SOFTMAX = 1


def build(force: bool = False) -> str:
    """Compile the oracle's C codecs with gcc (plain -O2, no fast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        d, u32, i32, sz, p = ctypes.c_double, ctypes.c_uint32, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        for name, res, args in [
            ("orc_e2m1_decode", d, [u32]), ("orc_e8m0_decode", d, [u32]),
            ("orc_e4m3_decode", d, [u32]), ("orc_e4m3_encode", u32, [d]),
            ("orc_bf16_encode", u32, [d]), ("orc_bf16_decode", d, [u32]),
            ("orc_e2m1_encode", u32, [d]), ("orc_act_block_exponent", i32, [d]),
            ("orc_e4m3_decode_array", None, [p, sz, p]), ("orc_e4m3_encode_array", None, [p, sz, p]),
            ("orc_bf16_encode_array", None, [p, sz, p]),
            ("orc_act_quant_rows", None, [p, sz, i32, i32, p, p]),
            ("orc_act_quant_rows_f32s", None, [p, sz, i32, i32, p, p]),
            ("orc_mxfp4_quant_rows", None, [p, sz, i32, p, p]),
            ("orc_mxfp4_decode_rows", None, [p, p, sz, i32, p]),
        ]:
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- scalar codecs
def e2m1_decode(code: int) -> float:
    """E2M1 value of a 4-bit code [P5 "Why Are the V2.6 Files Half...", row "Routed experts"]."""
    return _L().orc_e2m1_decode(code)


def e2m1_encode(v: float) -> int:
    return _L().orc_e2m1_encode(v)


def e8m0_decode(b: int) -> float:
    """E8M0 scale byte -> 2^(b-127) [P5 same row: one 8-bit scale per 32 values]."""
    return _L().orc_e8m0_decode(b)


def e4m3_decode(b: int) -> float:
    """e4m3 byte -> value [P2 "Overview": computed as block-wise FP8 e4m3]."""
    return _L().orc_e4m3_decode(b)


def e4m3_encode(v: float) -> int:
    """value -> e4m3 byte, round to nearest even, saturate to +-448."""
    return _L().orc_e4m3_encode(v)


def bf16_encode(v: float) -> int:
    return _L().orc_bf16_encode(v)


def act_block_exponent(amax: float) -> int:
    return _L().orc_act_block_exponent(amax)


# ---------------------------------------------------------------- array codecs
def bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 (bf16 is the top half of an fp32)."""
    u = np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns with a single round-to-nearest-even."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _L().orc_bf16_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode_array(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _L().orc_e4m3_decode_array(_ptr(b), b.size, _ptr(out))
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _L().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


ACT_SCALE_E8M0 = 0
ACT_SCALE_F32 = 1


def act_quant(v: np.ndarray, blk: int = 128, mode: int = ACT_SCALE_E8M0):
    """Per-row 1 x blk e4m3 quantisation.

    [P2 "Overview": block-wise e4m3; P3 "Self-Hosting": dynamic activation
    scheme.]  mode ACT_SCALE_E8M0: a power-of-two scale per block, the
    smallest that keeps the block's amax within 448, returned as E8M0 bytes
    (u8 [rows, n/blk]).  mode ACT_SCALE_F32: s = fp32(amax / 448) per block
    of the values taken at fp32, codes e4m3(fp32(v / s)), returned as
    float32 [rows, n/blk] (0 for an all-zero block).  Codes u8 [rows, n].
    """
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, n = v.shape
    assert n % blk == 0
    q = np.empty((rows, n), dtype=np.uint8)
    if mode == ACT_SCALE_F32:
        s = np.empty((rows, n // blk), dtype=np.float32)
        _L().orc_act_quant_rows_f32s(_ptr(v), rows, n, blk, _ptr(q), _ptr(s))
    else:
        s = np.empty((rows, n // blk), dtype=np.uint8)
        _L().orc_act_quant_rows(_ptr(v), rows, n, blk, _ptr(q), _ptr(s))
    return q, s


def act_dequant(q: np.ndarray, s: np.ndarray, blk: int = 128) -> np.ndarray:
    """Exact value of quantised activations: e4m3(q) * scale, the scale an
    E8M0 byte (2^(s-127)) or an fp32 value, by the dtype of ``s``."""
    vals = e4m3_decode_array(q)
    if s.dtype == np.float32:
        scale = s.astype(np.float64)
    else:
        scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return vals * np.repeat(scale, blk, axis=-1)


def mxfp4_quant(w: np.ndarray):
    """OCP MX v1.0 MXFP4 quantisation of rows [rows, K] -> (packed [rows, K/2], scales [rows, K/32])."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, K = w.shape
    assert K % 32 == 0
    packed = np.empty((rows, K // 2), dtype=np.uint8)
    scale = np.empty((rows, K // 32), dtype=np.uint8)
    _L().orc_mxfp4_quant_rows(_ptr(w), rows, K, _ptr(packed), _ptr(scale))
    return packed, scale


def mxfp4_decode(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Exact values of MXFP4 rows [P5 "Why Are the V2.6 Files Half...", row
    "Routed experts": two 4-bit values per byte, one 8-bit scale per 32]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    K = packed.shape[-1] * 2
    rows = packed.size // (K // 2)
    assert scale.size == rows * (K // 32)
    out = np.empty(packed.shape[:-1] + (K,), dtype=np.float64)
    _L().orc_mxfp4_decode_rows(_ptr(packed), _ptr(scale), rows, K, _ptr(out))
    return out


# ---------------------------------------------------------------- the layer
@dataclass
class Route:
    ids: np.ndarray      # int32 [T, k], selection order (key-descending)
    gates: np.ndarray    # float64 [T, k], renormalised selected scores
    logits: np.ndarray   # float64 [T, E]
    scores: np.ndarray   # float64 [T, E]
    keys: np.ndarray     # float64 [T, E] = scores + correction bias
    margin: np.ndarray   # float64 [T]: k-th selected key minus best unselected key


def route(x_bf16: np.ndarray, router_w_bf16: np.ndarray, k: int, score_func: int = SCORE_SIGMOID,
          logit_bias=None, sel_bias=None) -> Route:
    """Router and top-k gate.

    [P5 "How Big Is Each Expert?": the router scores experts with a sigmoid
    and adds a small correction bias to each score; 8 experts per token.
    P5 "Why Are the V2.6 Files Half...": router weights in BF16.
    P2 "Overview": 384 routed experts, top-8.]
    logits = x . Wr^T (+ logit bias), in fp64 from exact bf16 values;
    scores = sigmoid(logits) (or softmax over experts);
    keys   = scores + correction bias (selection only);
    top-k by key, descending, ties to the lower expert index;
    gates  = selected scores / their sum.
    """
    x = bf16_to_f64(x_bf16)
    w = bf16_to_f64(router_w_bf16)
    T, E = x.shape[0], w.shape[0]
    logits = x @ w.T
    if logit_bias is not None:
        logits = logits + np.asarray(logit_bias, dtype=np.float32).astype(np.float64)[None, :]
    if score_func == SCORE_SIGMOID:
        scores = 1.0 / (1.0 + np.exp(-logits))
    elif score_func == SCORE_SOFTMAX:
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        scores = z / z.sum(axis=1, keepdims=True)
    else:
        raise ValueError("score_func")
    keys = scores.copy()
    if sel_bias is not None:
        keys = keys + np.asarray(sel_bias, dtype=np.float32).astype(np.float64)[None, :]
    # stable sort of -key: descending key, equal keys keep ascending index
    order = np.argsort(-keys, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(scores, ids.astype(np.int64), axis=1)
    gates = sel / sel.sum(axis=1, keepdims=True)
    kth = np.take_along_axis(keys, order[:, k - 1:k], axis=1)[:, 0]
    if k < E:
        nxt = np.take_along_axis(keys, order[:, k:k + 1], axis=1)[:, 0]
        margin = kth - nxt
    else:
        margin = np.full(T, np.inf)
    return Route(ids, gates, logits, scores, keys, margin)


def dispatch(ids: np.ndarray, E: int):
    """Token-to-expert histogram, exclusive scan and stable permutation.

    counts[e] = number of (token, slot) pairs routed to e; offsets = exclusive
    scan (E+1 entries); perm[t*k + j] = offsets[e] + number of tokens t' < t
    that also chose e, i.e. rows are expert-contiguous and token-ascending
    within an expert.  Computed with a stable library sort of the flattened
    (token-major) expert ids.
    """
    flat = ids.reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")
    perm = np.empty(flat.size, dtype=np.int32)
    perm[order] = np.arange(flat.size, dtype=np.int32)
    return counts, offsets, perm


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def fp8_block_decode(q: np.ndarray, s: np.ndarray, blk: int = 128) -> np.ndarray:
    """Exact values of an expert matrix in the fp8 block format: e4m3 codes
    q [R, K] times the fp32 scale of their blk x blk block, s [R/blk, K/blk].

    [P5 "Why Are the V2.6 Files Half the Size of V2.5?", the V2.5 / V2.6
    table, row "Routed experts": V2.5 stores them as FP8 E4M3 with one F32
    scale per 128 x 128 block.]
    """
    vals = e4m3_decode_array(q)
    sc = np.repeat(np.repeat(s.astype(np.float64), blk, axis=-2), blk, axis=-1)
    return vals * sc


def expert_ffn(a: np.ndarray, w13_q, w13_s, w2_q, w2_s, act_scale_mode: int = ACT_SCALE_E8M0,
               weight_format: str = "mxfp4"):
    """One expert's SwiGLU FFN on exact activation values a [n, H].

    [P5 "How Big Is Each Expert?": gate, up and down projections around a
    2,048-wide middle; P5 "Why Are the V2.6 Files Half...": MXFP4 experts.]
    gate/up = a . W13^T with W13 [2I, H] decoded exactly (gate rows first);
    h = silu(gate) * up in fp64; h re-quantised per 1 x 128 block to e4m3
    (scales by ``act_scale_mode``); o = dequant(h) . W2^T with W2 [H, I].
    Returns (h fp64 [n, I], hq u8 [n, I], hs [n, I/128] (E8M0 bytes or fp32),
    o fp64 [n, H]).
    """
    decode = fp8_block_decode if weight_format == "fp8" else mxfp4_decode
    W13 = decode(w13_q, w13_s)
    I2 = W13.shape[0]
    I = I2 // 2
    gu = a @ W13.T
    h = silu(gu[:, :I]) * gu[:, I:]
    hq, hs = act_quant(h, 128, act_scale_mode)
    W2 = decode(w2_q, w2_s)
    o = act_dequant(hq, hs, 128) @ W2.T
    return h, hq, hs, o


@dataclass
class Forward:
    route: Route
    counts: np.ndarray
    offsets: np.ndarray
    perm: np.ndarray
    tokens: np.ndarray      # int64 [n] the tokens whose outputs were computed
    aq: np.ndarray          # u8 [n, H]   Q1 codes of those tokens
    as_: np.ndarray         # [n, H/128] E8M0 bytes (u8) or fp32 scales
    hq: np.ndarray          # u8 [n, k, I] Q2 codes per (token, slot)
    hs: np.ndarray          # [n, k, I/128] E8M0 bytes (u8) or fp32 scales
    h: np.ndarray           # f64 [n, k, I] pre-quantisation SwiGLU output
    o: np.ndarray           # f64 [n, k, H] expert outputs before the gate weighting
    y64: np.ndarray         # f64 [n, H] gate-weighted sum before rounding
    y: np.ndarray           # u16 [n, H] bf16 output


def route_with_ids(r: Route, ids: np.ndarray) -> Route:
    """The same router output with a given selection ``ids`` [T, k] in place
    of the oracle's own top-k: gates = the given experts' scores / their sum.

    Where two keys are closer than the rounding of a device's fp32 logits,
    both selections are correct (the device tests accept either); the layer's
    later steps are then checked against this variant fed the device's
    choice.  The keys and margins stay the oracle's.
    """
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    assert ids.shape == r.ids.shape
    sel = np.take_along_axis(r.scores, ids.astype(np.int64), axis=1)
    gates = sel / sel.sum(axis=1, keepdims=True)
    return Route(ids, gates, r.logits, r.scores, r.keys, r.margin)


def forward(x_bf16, router_w_bf16, w13_q, w13_s, w2_q, w2_s, k: int,
            score_func: int = SCORE_SIGMOID, logit_bias=None, sel_bias=None,
            tokens=None, act_scale_mode: int = ACT_SCALE_E8M0, weight_format: str = "mxfp4",
            ids=None) -> Forward:
    """The whole layer: route, dispatch, quantise, experts, combine.

    Routing, counts, offsets and the permutation cover every token; the
    expert FFNs and the output are computed for ``tokens`` (default: all).
    y[t] = bf16_rne( sum_j gate[t, j] * o[t, j] ), the sum in fp64.
    ``ids`` (optional, int [T, k]) replaces the top-k selection for every
    later step (see ``route_with_ids``).
    """
    T, H = x_bf16.shape
    E = router_w_bf16.shape[0]
    r = route(x_bf16, router_w_bf16, k, score_func, logit_bias, sel_bias)
    if ids is not None:
        r = route_with_ids(r, ids)
    counts, offsets, perm = dispatch(r.ids, E)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    n = toks.size
    aq, as_ = act_quant(bf16_to_f64(x_bf16[toks]), 128, act_scale_mode)
    a = act_dequant(aq, as_, 128)
    I = w2_q.shape[2] * (1 if weight_format == "fp8" else 2)
    hq = np.zeros((n, k, I), dtype=np.uint8)
    hs = np.zeros((n, k, I // 128), dtype=np.float32 if act_scale_mode == ACT_SCALE_F32 else np.uint8)
    h = np.zeros((n, k, I), dtype=np.float64)
    o = np.zeros((n, k, H), dtype=np.float64)
    sel = r.ids[toks]
    for e in np.unique(sel):
        rows, slots = np.nonzero(sel == e)
        h_e, hq_e, hs_e, o_e = expert_ffn(a[rows], w13_q[e], w13_s[e], w2_q[e], w2_s[e], act_scale_mode,
                                          weight_format)
        h[rows, slots] = h_e
        hq[rows, slots] = hq_e
        hs[rows, slots] = hs_e
        o[rows, slots] = o_e
    g = r.gates[toks]
    y64 = np.einsum("nk,nkh->nh", g, o)
    return Forward(r, counts, offsets, perm, toks, aq, as_, hq, hs, h, o, y64, f64_to_bf16(y64))


def tp_partials(f: Forward, w2_q, w2_s, G: int, weight_format: str = "mxfp4"):
    """The layer output split over G tensor-parallel shards of the expert
    middle dimension, as the pages deploy it (vLLM recipe
    "XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview": TP8 on H200, TP4 on MI355X).

    Shard r holds middle columns [r I/G, (r+1) I/G) of every expert: its
    SwiGLU codes are those columns of the layer's Q2 codes (I/G is a multiple
    of 128, so no 1 x 128 block straddles two shards), its down projection
    the same columns of W2, and its partial output
        y_r[t] = sum_j gate[t, j] * dequant(hq[t, j, cols_r]) . W2[e_j][:, cols_r]^T
    in fp64.  The layer output is bf16( sum_r y_r ).  Returns the G partials
    (float64 [n, H] each, for the tokens of ``f``).
    """
    decode = fp8_block_decode if weight_format == "fp8" else mxfp4_decode
    n, k, I = f.hq.shape
    H = f.o.shape[2]
    assert I % (128 * G) == 0
    Il = I // G
    sel = f.route.ids[f.tokens]
    a = act_dequant(f.hq.reshape(n * k, I), f.hs.reshape(n * k, I // 128), 128).reshape(n, k, I)
    parts = []
    for r in range(G):
        cols = slice(r * Il, (r + 1) * Il)
        o = np.zeros((n, k, H), dtype=np.float64)
        for e in np.unique(sel):
            rows, slots = np.nonzero(sel == e)
            W2 = decode(w2_q[e], w2_s[e])
            o[rows, slots] = a[rows, slots][:, cols] @ W2[:, cols].T
        parts.append(np.einsum("nk,nkh->nh", f.route.gates[f.tokens], o))
    return parts
