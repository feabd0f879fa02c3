"""Pins of the oracle's layer steps against definitions computed another way:
brute-force subset search for top-k, a library sort for the permutation,
and small-integer weights whose expert FFN reduces to exact integer matmuls
plus library sigmoid and brute-force rounding."""
import itertools
from collections import Counter

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
import synth


def bf16_bits(v):
    return torch.tensor(np.asarray(v, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(u16):
    return torch.from_numpy(np.asarray(u16, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_helpers_agree_with_torch():
    u = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    a, b = oracle.bf16_to_f64(u), bf16_vals(u)
    fin = np.isfinite(b)
    assert np.array_equal(a[fin], b[fin])


def _keys_independent(x16, w16, lb, cb, score_func):
    logits = bf16_vals(x16) @ bf16_vals(w16).T
    if lb is not None:
        logits = logits + lb.astype(np.float64)
    s = expit(logits) if score_func == 0 else softmax(logits, axis=1)
    return s, s + (0 if cb is None else cb.astype(np.float64))


def _brute_topk(key, k):
    """Smallest sorted index tuple among the k-subsets S with
    min(key[S]) >= max(key[not S]) (the defining property of a top-k set)."""
    E = key.size
    best = None
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if rest and min(key[list(S)]) < max(key[rest]):
            continue
        if best is None or S < best:
            best = S
    return best


@pytest.mark.parametrize("score_func", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_route_matches_brute_force_with_ties(score_func, k):
    rng = np.random.default_rng(10 + k + 7 * score_func)
    T, H, E = 6, 64, 8 if k < 8 else 10
    x = bf16_bits(rng.normal(0, 1, (T, H)))
    w = rng.normal(0, 0.1, (E, H))
    w[3] = w[1]                       # experts 1 and 3 tie on every token
    w[E - 1] = w[0]                   # and 0 with E-1
    w = bf16_bits(w)
    lb = rng.normal(0, 0.3, E).astype(np.float32)
    lb[3], lb[E - 1] = lb[1], lb[0]
    cb = np.zeros(E, dtype=np.float32)
    cb[5] = 0.25                      # a correction bias that changes selection only
    r = oracle.route(x, w, k, score_func, lb, cb)
    s, key = _keys_independent(x, w, lb, cb, score_func)
    for t in range(T):
        expect = _brute_topk(key[t], k)
        assert tuple(sorted(r.ids[t])) == expect
        # selection order: key descending, equal keys by index
        order = sorted(r.ids[t], key=lambda e: (-key[t, e], e))
        assert list(r.ids[t]) == order
        g = s[t, r.ids[t]] / s[t, r.ids[t]].sum()
        np.testing.assert_allclose(r.gates[t], g, rtol=1e-14)
        assert abs(r.gates[t].sum() - 1) < 1e-14
        assert len(set(r.ids[t])) == k


def test_route_all_equal_scores_pick_lowest_indices():
    T, H, E, k = 3, 32, 12, 8
    x = bf16_bits(np.ones((T, H)))
    w = bf16_bits(np.zeros((E, H)))
    r = oracle.route(x, w, k)
    assert (r.ids == np.arange(k)).all()
    np.testing.assert_allclose(r.gates, 1.0 / k)
    assert (r.margin == 0).all()


def test_dispatch_matches_sorted_definition():
    rng = np.random.default_rng(11)
    T, E, k = 50, 12, 4
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.dispatch(ids, E)
    c = Counter(ids.ravel().tolist())
    assert [c.get(e, 0) for e in range(E)] == counts.tolist()
    assert offsets[0] == 0 and offsets[-1] == T * k and (np.diff(offsets) == counts).all()
    triples = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k))
    for row, (e, t, j) in enumerate(triples):
        assert perm[t * k + j] == row
    assert sorted(perm.tolist()) == list(range(T * k))


# ---- expert FFN special case: weights +-m * 2^p, activations small integers
def _pack_codes(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _pm_weight(rng, rows, K, mag_code, scale_byte):
    """Random sign matrix S (+-1) and its MXFP4 encoding with E2M1 magnitude
    code ``mag_code`` and one E8M0 scale byte for every block."""
    S = rng.choice([-1.0, 1.0], (rows, K))
    codes = np.where(S > 0, mag_code, mag_code | 8)
    return S, _pack_codes(codes), np.full((rows, K // 32), scale_byte, dtype=np.uint8)


E2M1 = {2: 1.0, 3: 1.5, 4: 2.0}


def _e4m3_nearest(v):
    """Brute-force nearest e4m3 code (ties to even code) by search over the
    table of all finite values decoded by torch."""
    tab = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = np.array([c for c in range(256) if np.isfinite(tab[c])])
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in np.ndenumerate(v):
        x = min(max(x, -448.0), 448.0)
        d = np.abs(tab[codes] - x)
        m = d.min()
        cand = codes[d == m]
        if len(cand) > 1:
            even = cand[(cand & 1) == 0]
            cand = even if len(even) else cand
            # equal distance to +0/-0 only at x == 0: keep the sign of x
            if len(cand) > 1:
                cand = cand[[(c >> 7) == int(np.signbit(x)) for c in cand]]
        out[i] = cand[0]
    return out, tab


def _q2_brute(h):
    """1 x 128 requantisation by search: smallest e with amax <= 448 * 2^e."""
    n, I = h.shape
    q = np.empty((n, I), dtype=np.uint8)
    s = np.empty((n, I // 128), dtype=np.uint8)
    deq = np.empty_like(h)
    for r in range(n):
        for b in range(I // 128):
            blk = h[r, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            e = 0
            if amax > 0:
                e = -140
                while not (amax <= 448.0 * 2.0 ** e):
                    e += 1
            codes, tab = _e4m3_nearest(blk / 2.0 ** e)
            q[r, b * 128:(b + 1) * 128] = codes
            s[r, b] = e + 127
            deq[r, b * 128:(b + 1) * 128] = tab[codes] * 2.0 ** e
    return q, s, deq


@pytest.mark.parametrize("E,k", [(1, 1), (2, 2), (3, 2)])
def test_expert_ffn_small_integer_case(E, k):
    """x in {-3..3}: Q1 is exact.  W13/W2 are +-m*2^p: gate/up are exact
    integer matmuls.  SwiGLU by scipy's expit, Q2 by brute force, down-proj and
    combine in fp64.  Different gate and up sign matrices pin the row order;
    non-square matrices pin the orientation of every operand."""
    rng = np.random.default_rng(20 + E)
    T, H, I = 5, 256, 256
    x = rng.integers(-3, 4, (T, H)).astype(np.float64)
    x[:, 0] = 3
    x16 = bf16_bits(x)
    wr = bf16_bits(rng.normal(0, 0.05, (E, H)))
    W13_list, W2_list = [], []
    w13_q = np.empty((E, 2 * I, H // 2), np.uint8)
    w13_s = np.empty((E, 2 * I, H // 32), np.uint8)
    w2_q = np.empty((E, H, I // 2), np.uint8)
    w2_s = np.empty((E, H, I // 32), np.uint8)
    for e in range(E):
        mc, sb = [(2, 127), (3, 125), (4, 126)][e]
        S13, w13_q[e], w13_s[e] = _pm_weight(rng, 2 * I, H, mc, sb)
        S2, w2_q[e], w2_s[e] = _pm_weight(rng, H, I, [3, 2, 4][e], [129, 127, 124][e])
        W13_list.append(S13 * E2M1[mc] * 2.0 ** (sb - 127))
        W2_list.append(S2 * E2M1[[3, 2, 4][e]] * 2.0 ** ([129, 127, 124][e] - 127))
    f = oracle.forward(x16, wr, w13_q, w13_s, w2_q, w2_s, k)
    # independent routing
    s = expit(bf16_vals(x16) @ bf16_vals(wr).T)
    ids = np.argsort(-s, axis=1, kind="stable")[:, :k]
    assert np.array_equal(f.route.ids, ids)
    # Q1 exact: the decoded activations equal x
    assert np.array_equal(oracle.act_dequant(f.aq, f.as_), x)
    y = np.zeros((T, H))
    for t in range(T):
        sel = s[t, ids[t]]
        for j, e in enumerate(ids[t]):
            gu = x[t:t + 1] @ W13_list[e].T
            g, u = gu[:, :I], gu[:, I:]
            hval = g * expit(g) * u
            q, sc, deq = _q2_brute(hval)
            np.testing.assert_allclose(f.h[t, j], hval[0], rtol=1e-13, atol=1e-300)
            assert np.array_equal(f.hq[t, j], q[0]) and np.array_equal(f.hs[t, j], sc[0])
            y[t] += sel[j] / sel.sum() * (deq @ W2_list[e].T)[0]
    np.testing.assert_allclose(f.y64, y, rtol=1e-12, atol=1e-9 * np.abs(y).max())
    assert np.array_equal(f.y, oracle.f64_to_bf16(f.y64))


def test_forward_token_subset_matches_full():
    inp = synth.make_inputs("toy")
    full = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, 8,
                          logit_bias=inp.logit_bias, sel_bias=inp.sel_bias)
    sub = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, 8,
                         logit_bias=inp.logit_bias, sel_bias=inp.sel_bias, tokens=[5, 17, 63])
    assert np.array_equal(sub.y, full.y[[5, 17, 63]])
    assert np.array_equal(sub.perm, full.perm)


def test_page_byte_accounting(golden):
    """Expert sizes printed on the teardown page pin 3*H*I parameters per
    expert and 4.25 bits per MXFP4 weight."""
    g = {r[0]: float(r[1]) for r in golden("page_accounting.txt")}
    I = int(g["intermediate"])
    for hid, key in [("flash_hidden", "flash_expert_params_millions"), ("pro_hidden", "pro_expert_params_millions")]:
        params = 3 * int(g[hid]) * I
        assert round(params / 1e6, 1) == g[key]
        assert synth.expert_weight_bytes(int(g[hid]), I) * 8 == params * g["bits_per_weight"]
    assert round(g["flash_expert_weights_billions"] * 1e9 * g["bits_per_weight"] / 8 / 1e9, 1) == g["flash_expert_gb"]


def test_generator_mxfp4_matches_oracle_quantiser():
    w = synth.expert_f32(3, 7, 2, 32, 512, 0.02)
    p, s = synth.mxfp4_experts(3, 7, 2, 32, 512, 0.02)
    po, so = oracle.mxfp4_quant(w.reshape(-1, 512).astype(np.float64))
    assert np.array_equal(po.reshape(p.shape), p) and np.array_equal(so.reshape(s.shape), s)


def test_generator_is_deterministic_and_seeded():
    a = synth.make_inputs("toy")
    b = synth.make_inputs("toy")
    assert np.array_equal(a.x, b.x) and np.array_equal(a.w13_q, b.w13_q) and np.array_equal(a.w2_s, b.w2_s)
    x = bf16_vals(a.x)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    c = synth.make_inputs(synth.Config("s1", 64, 512, 16, 256, 8, 1, "none"))
    assert not np.array_equal(a.x, c.x)


def test_forward_structural_invariants():
    """Gates sum to 1, k distinct experts per token, counts sum to T*k,
    offsets are the exclusive scan ending at T*k, the permutation is a
    bijection that lists each expert's (token, slot) pairs contiguously."""
    inp = synth.custom_inputs(37, 256, 12, 128, 5, seed=41, bias="normal:1.0")
    T, k, E = 37, 5, 12
    f = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, k,
                       logit_bias=inp.logit_bias)
    r = f.route
    assert np.allclose(r.gates.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert all(len(set(row.tolist())) == k for row in r.ids)
    assert f.counts.sum() == T * k
    assert f.offsets[0] == 0 and f.offsets[E] == T * k and (np.diff(f.offsets) >= 0).all()
    assert np.array_equal(np.sort(f.perm), np.arange(T * k))
    flat = r.ids.reshape(-1)
    for e in range(E):
        rows = f.perm[flat == e]
        assert np.array_equal(np.sort(rows), np.arange(f.offsets[e], f.offsets[e + 1]))


# ----------------------------------------------------------- routing override
def _small_layer(seed, T=6, H=128, E=8, I=128, k=2):
    inp = synth.custom_inputs(T, H, E, I, k, seed=seed, bias="normal:0.3")
    c = inp.cfg
    args = (inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    kw = dict(score_func=c.score_func, logit_bias=inp.logit_bias, sel_bias=inp.sel_bias)
    return inp, args, kw


def test_forward_with_its_own_ids_is_the_plain_forward():
    inp, args, kw = _small_layer(41)
    f0 = oracle.forward(*args, 2, **kw)
    f1 = oracle.forward(*args, 2, **kw, ids=f0.route.ids.copy())
    for name in ["counts", "offsets", "perm", "aq", "as_", "hq", "hs", "h", "o", "y64", "y"]:
        assert np.array_equal(getattr(f0, name), getattr(f1, name)), name
    assert np.array_equal(f0.route.gates, f1.route.gates)


def test_forward_with_other_ids_reuses_each_token_expert_output():
    """An expert's output for a token depends only on that (token, expert)
    pair: with the override (1st, 3rd choice) the 1st slot equals the plain
    top-2 forward's slot 0 and the 2nd slot equals the plain top-3 forward's
    slot 2; gates renormalise the chosen scores; dispatch follows the ids."""
    inp, args, kw = _small_layer(42)
    f2 = oracle.forward(*args, 2, **kw)
    f3 = oracle.forward(*args, 3, **kw)
    ids = np.stack([f3.route.ids[:, 0], f3.route.ids[:, 2]], axis=1).astype(np.int32)
    fo = oracle.forward(*args, 2, **kw, ids=ids)
    assert np.array_equal(fo.route.ids, ids)
    assert np.array_equal(fo.o[:, 0], f2.o[:, 0]) and np.array_equal(fo.hq[:, 0], f2.hq[:, 0])
    assert np.array_equal(fo.o[:, 1], f3.o[:, 2]) and np.array_equal(fo.hq[:, 1], f3.hq[:, 2])
    s = np.take_along_axis(f3.route.scores, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(fo.route.gates, s / s.sum(axis=1, keepdims=True), rtol=1e-15)
    assert np.array_equal(fo.counts, np.bincount(ids.reshape(-1), minlength=inp.cfg.E))
    flat = ids.reshape(-1)
    for e in range(inp.cfg.E):   # rows of expert e: contiguous, token-ascending
        rows = fo.perm[flat == e]
        assert np.array_equal(rows, np.arange(fo.offsets[e], fo.offsets[e + 1]))
    np.testing.assert_allclose(fo.y64, np.einsum("nk,nkh->nh", fo.route.gates, fo.o), rtol=1e-14)


def test_forward_with_permuted_slots_keeps_the_output_when_all_experts_are_chosen():
    """k = E: every selection order is the same set, so y cannot change
    (fp64 sums in another order: equal to 1e-12) while gates and expert
    outputs move with their slots."""
    inp, args, kw = _small_layer(43, E=4, k=4)
    f0 = oracle.forward(*args, 4, **kw)
    ids = f0.route.ids[:, ::-1].copy()
    f1 = oracle.forward(*args, 4, **kw, ids=ids)
    np.testing.assert_allclose(f1.y64, f0.y64, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(f1.route.gates, f0.route.gates[:, ::-1], rtol=1e-15)
    assert np.array_equal(f1.o, f0.o[:, ::-1])


# ----------------------------------------------------------- tensor-parallel split
@pytest.mark.parametrize("weights", ["mxfp4", "fp8"])
def test_tp_partials_add_up_to_the_layer(weights):
    """Splitting the expert middle dimension over G shards and adding the
    partial outputs gives the whole layer's fp64 output (G = 1: the same
    operations, so bit for bit)."""
    inp = synth.custom_inputs(5, 256, 4, 512, 2, seed=44, weights=weights)
    c = inp.cfg
    f = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, c.k, c.score_func,
                       inp.logit_bias, inp.sel_bias, weight_format=weights)
    (p1,) = oracle.tp_partials(f, inp.w2_q, inp.w2_s, 1, weights)
    assert np.array_equal(p1, f.y64)
    for G in (2, 4):
        parts = oracle.tp_partials(f, inp.w2_q, inp.w2_s, G, weights)
        assert len(parts) == G
        np.testing.assert_allclose(sum(parts), f.y64, rtol=1e-12, atol=1e-14)
        assert not np.allclose(parts[0], f.y64)          # each shard holds only part of the sum
    with pytest.raises(AssertionError):
        oracle.tp_partials(f, inp.w2_q, inp.w2_s, 3, weights)   # 512 / 3 is not a multiple of 128
