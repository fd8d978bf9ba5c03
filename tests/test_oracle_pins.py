"""Pins for the CPU oracle: each oracle function against something other than itself.

Closed forms, printed values, special cases that reduce to a dense SwiGLU FFN or a full
softmax, brute force over all k-subsets, and an independent per-token evaluation.  Each
check is a plain function so that `test_planted_mistakes_are_caught` can re-run it against
an oracle with a plausible mistake planted in it (on the CPU) and see it fail.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "printed_values.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _arrays_fn(W):
    return lambda name, e: W[name][e]


def _rand_layer(seed, T, d, d_ff, E, n_shared=0, d_ffs=0):
    r = _rng(seed)
    W = {"W1": r.normal(0, d ** -0.5, (E, d, d_ff)), "W2": r.normal(0, d ** -0.5, (E, d, d_ff)),
         "W3": r.normal(0, d_ff ** -0.5, (E, d_ff, d))}
    if n_shared:
        W.update({"Ws1": r.normal(0, d ** -0.5, (n_shared, d, d_ffs)),
                  "Ws2": r.normal(0, d ** -0.5, (n_shared, d, d_ffs)),
                  "Ws3": r.normal(0, d_ffs ** -0.5, (n_shared, d_ffs, d))})
    x = r.normal(0, 1, (T, d))
    Wg = r.normal(0, d ** -0.5, (d, E))
    return x, Wg, W


def dense_swiglu_loops(x, W1, W2, W3):
    """A dense SwiGLU FFN written out as scalar loops, independent of the oracle's code:
    y = ((x W1) * silu(x W2)) W3, silu(v) = v / (1 + e^-v)."""
    T, d = len(x), len(x[0])
    dff, dout = len(W1[0]), len(W3[0])
    out = []
    for t in range(T):
        h = []
        for n in range(dff):
            u = sum(float(x[t][i]) * float(W1[i][n]) for i in range(d))
            v = sum(float(x[t][i]) * float(W2[i][n]) for i in range(d))
            h.append(u * v / (1.0 + math.exp(-v)))
        out.append([sum(h[n] * float(W3[n][c]) for n in range(dff)) for c in range(dout)])
    return np.array(out)


# ---------------------------------------------------------------------------- checks


def check_router_logits_closed_form():
    # W_g with a single non-zero entry w at (i, e): logit[:, e] = w x[:, i], zero elsewhere.
    # A transposed operand or a wrong reduction axis fails this.
    x = _rng(1).normal(size=(5, 6))
    Wg = np.zeros((6, 4))
    Wg[2, 3] = 0.5
    l = orc.router_logits(x, Wg)
    assert l.shape == (5, 4) and l.dtype == np.float32
    expect = np.zeros((5, 4), np.float32)
    expect[:, 3] = (0.5 * x[:, 2]).astype(np.float32)
    assert np.array_equal(l, expect)
    # bias is added per expert (column)
    lb = np.array([1.0, -2.0, 0.25, 3.0], np.float32)
    l2 = orc.router_logits(x, Wg, lb)
    assert np.array_equal(l2, (expect + lb).astype(np.float32))


def check_scores_closed_forms():
    s = orc.scores(np.array([[0.0, math.log(3.0)]], np.float32), "softmax")
    assert np.allclose(s, [[0.25, 0.75]], rtol=1e-7)
    s = orc.scores(np.zeros((2, 7), np.float32), "softmax")
    assert np.allclose(s, 1.0 / 7)
    l = _rng(2).normal(size=(3, 9)).astype(np.float32)
    assert np.allclose(orc.scores(l, "softmax"), orc.scores((l + np.float32(5)).astype(np.float32), "softmax"), atol=1e-6)
    s = orc.scores(np.array([[0.0, math.log(3.0), -math.log(3.0)]], np.float32), "sigmoid")
    assert np.allclose(s, [[0.5, 0.75, 0.25]], rtol=1e-7)


def check_topk_bruteforce():
    r = _rng(3)
    for trial in range(40):
        E = int(r.integers(1, 8))
        k = int(r.integers(1, E + 1))
        key = r.permutation(E).astype(np.float32)[None, :] * np.float32(0.37) - np.float32(1)
        idx = orc.select_topk(key, k)[0]
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(key[0, list(c)]))
        assert set(idx.tolist()) == set(best)
        assert all(key[0, idx[j]] > key[0, idx[j + 1]] for j in range(k - 1))
    # equal keys: the lower expert id wins
    idx = orc.select_topk(np.array([[1.0, 2.0, 2.0, 0.0, 2.0]], np.float32), 3)
    assert idx.tolist() == [[1, 2, 4]]


def check_gate_invariants():
    r = _rng(4)
    for scoring in ("softmax", "sigmoid"):
        l = r.normal(0, 2, (50, 16)).astype(np.float32)
        out = orc.route(l.astype(np.float64), np.eye(16), 4, scoring)   # W_g = I: logits = x
        g = out["gate"]
        assert np.all(g >= 0)
        assert np.allclose(g.sum(axis=1), 1.0, atol=1e-14)


def check_gates_two_formulations():
    # softmax over all E, then renormalise over the chosen k ("Field Manual" 2.1) equals
    # exp(l_e) / sum over the chosen k of exp(l_e') ("8.6" section 2).
    r = _rng(5)
    l = r.normal(0, 3, (64, 12)).astype(np.float32)
    out = orc.route(l.astype(np.float64), np.eye(12), 3, "softmax")
    lf = l.astype(np.float64)
    sel = np.take_along_axis(lf, out["idx"].astype(np.int64), axis=1)
    direct = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    assert np.allclose(out["gate"], direct, rtol=1e-12, atol=0)


def check_k_equals_E_is_dense_softmax():
    # k = E: the gates are the full softmax, the layer a dense softmax-weighted ensemble.
    r = _rng(6)
    l = r.normal(0, 1, (20, 6)).astype(np.float32)
    out = orc.route(l.astype(np.float64), np.eye(6), 6, "softmax")
    full = np.exp(l.astype(np.float64))
    full /= full.sum(axis=1, keepdims=True)
    g_by_expert = np.zeros_like(full)
    np.put_along_axis(g_by_expert, out["idx"].astype(np.int64), out["gate"], axis=1)
    assert np.allclose(g_by_expert, full, rtol=1e-12)


def check_dispatch():
    r = _rng(7)
    T, k, E = 37, 3, 5
    idx = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    d = orc.dispatch(idx, E)
    # brute force: walk the flattened pairs expert by expert, in pair order
    perm = [t for e in range(E) for t in range(T) for j in range(k) if idx[t, j] == e]
    counts = [sum(1 for t in range(T) for j in range(k) if idx[t, j] == e) for e in range(E)]
    assert d["perm_tok"].tolist() == perm
    assert d["counts"].tolist() == counts
    assert int(d["counts"].sum()) == T * k
    assert d["offsets"].tolist() == [sum(counts[:e]) for e in range(E + 1)]
    pos = d["inv_pos"]
    assert sorted(pos.reshape(-1).tolist()) == list(range(T * k))   # a bijection
    for t in range(T):
        for j in range(k):
            p = int(pos[t, j])
            assert perm[p] == t and d["offsets"][idx[t, j]] <= p < d["offsets"][idx[t, j] + 1]


def check_swiglu_scalar_closed_form():
    # x = 1, W1 = 2, W2 = 3, W3 = 5: y = 5 * 2 * silu(3) = 10 * 3 / (1 + e^-3).
    # Swapping W1 and W2 gives 5 * 3 * silu(2), which differs.
    y = orc.swiglu_expert(np.array([[1.0]]), np.array([[2.0]]), np.array([[3.0]]), np.array([[5.0]]))
    assert abs(y[0, 0] - 10.0 * 3.0 / (1.0 + math.exp(-3.0))) < 1e-12


def check_swiglu_vs_loops():
    r = _rng(8)
    x = r.normal(size=(3, 5))
    W1, W2, W3 = r.normal(size=(5, 4)), r.normal(size=(5, 4)), r.normal(size=(4, 5))
    assert np.allclose(orc.swiglu_expert(x, W1, W2, W3), dense_swiglu_loops(x, W1, W2, W3), rtol=1e-12, atol=1e-12)


def check_E1_k1_is_dense_swiglu():
    # One expert, top-1: the gate is exactly 1 and the layer is a dense SwiGLU FFN.
    x, Wg, W = _rand_layer(9, T=6, d=5, d_ff=7, E=1)
    out = orc.forward(x, Wg, _arrays_fn(W), 1, 1, "softmax")
    assert np.array_equal(out["gate"], np.ones((6, 1)))
    ref = dense_swiglu_loops(x, W["W1"][0], W["W2"][0], W["W3"][0])
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def check_grouped_equals_bruteforce():
    cases = [dict(T=9, d=6, d_ff=5, E=4, k=2, scoring="softmax"),
             dict(T=7, d=4, d_ff=3, E=6, k=3, scoring="sigmoid"),
             dict(T=11, d=5, d_ff=4, E=5, k=1, scoring="softmax", n_shared=1, d_ffs=3),
             dict(T=4, d=3, d_ff=2, E=8, k=2, scoring="softmax"),           # some experts empty
             dict(T=5, d=4, d_ff=3, E=3, k=3, scoring="sigmoid", n_shared=2, d_ffs=2)]
    for i, c in enumerate(cases):
        x, Wg, W = _rand_layer(10 + i, c["T"], c["d"], c["d_ff"], c["E"], c.get("n_shared", 0), c.get("d_ffs", 0))
        lb = _rng(30 + i).normal(0, 1, c["E"]).astype(np.float32) if i % 2 else None
        sb = _rng(40 + i).normal(0, 1, c["E"]).astype(np.float32) if i == 3 else None
        g = orc.forward(x, Wg, _arrays_fn(W), c["E"], c["k"], c["scoring"], lb, sb, c.get("n_shared", 0))
        b = orc.forward_bruteforce(x, Wg, _arrays_fn(W), c["E"], c["k"], c["scoring"], lb, sb, c.get("n_shared", 0))
        assert np.allclose(g["y"], b, rtol=1e-12, atol=1e-12)
        # per-token evaluation from the routing
        ft = orc.forward_tokens(x, g["idx"], g["gate"], _arrays_fn(W), c.get("n_shared", 0))
        assert np.allclose(g["y"], ft, rtol=1e-12, atol=1e-12)


def check_shared_only():
    # Routed W3 = 0: every routed expert outputs 0 and the layer is the shared expert alone.
    x, Wg, W = _rand_layer(20, T=6, d=4, d_ff=3, E=3, n_shared=1, d_ffs=5)
    W["W3"] = np.zeros_like(W["W3"])
    out = orc.forward(x, Wg, _arrays_fn(W), 3, 2, "sigmoid", n_shared=1)
    ref = dense_swiglu_loops(x, W["Ws1"][0], W["Ws2"][0], W["Ws3"][0])
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def check_selection_bias():
    # A bias used only for choosing ("Field Manual" 3.3): a huge bias forces expert 2 into
    # every token's set, but the gates are the unbiased scores renormalised.
    r = _rng(21)
    l = r.normal(0, 1, (30, 6)).astype(np.float32)
    sb = np.array([0, 0, 100, 0, 0, 0], np.float32)
    out = orc.route(l.astype(np.float64), np.eye(6), 2, "softmax", sel_bias=sb)
    assert np.all(out["idx"][:, 0] == 2)
    s = np.exp(l.astype(np.float64))
    sel = np.take_along_axis(s, out["idx"].astype(np.int64), axis=1)
    assert np.allclose(out["gate"], sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


def check_selection_bias_sigmoid_uses_scores():
    # Sigmoid routing adds the bias to the score ([RA] "Load balancing"): logits (3, 0, -1),
    # bias (0, 0.6, 0.3) -> keys sigmoid(l) + b = (0.9526, 1.1, 0.5689): top-2 = experts 1, 0.
    # On logits + bias (3, 0.6, -0.7) the order would be 0, 1 instead.
    l = np.array([[3.0, 0.0, -1.0]])
    sb = np.array([0.0, 0.6, 0.3], np.float32)
    out = orc.route(l, np.eye(3), 2, "sigmoid", sel_bias=sb)
    assert out["idx"].tolist() == [[1, 0]]
    s1, s0 = 0.5, 1.0 / (1.0 + math.exp(-3.0))
    assert np.allclose(out["gate"], [[s1 / (s0 + s1), s0 / (s0 + s1)]], rtol=1e-12)
    # softmax routing adds it to the logit: keys (3, 0.6, -0.7) -> experts 0, 1
    out = orc.route(l, np.eye(3), 2, "softmax", sel_bias=sb)
    assert out["idx"].tolist() == [[0, 1]]
    # a zero bias changes nothing
    r = _rng(22)
    x = r.normal(size=(40, 5))
    Wg = r.normal(size=(5, 7))
    for sc in ("softmax", "sigmoid"):
        a = orc.route(x, Wg, 3, sc)
        b = orc.route(x, Wg, 3, sc, sel_bias=np.zeros(7, np.float32))
        assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["gate"], b["gate"])


def check_sel_bias_update_closed_form():
    # T = 10 tokens, k = 2, E = 4: share T k / E = 5 per expert.  Overloaded -> - gamma,
    # underloaded -> + gamma, exactly at the share -> unchanged ([FM] 3.3).
    b = np.array([0.5, -0.25, 0.0, 1.0], np.float32)
    out = orc.update_sel_bias(b, np.array([9, 5, 4, 2]), 10, 2, 0.125)
    assert out.dtype == np.float32
    assert out.tolist() == [0.375, -0.25, 0.125, 1.125]
    # shares that are not integers: T k / E = 7 / 3
    out = orc.update_sel_bias(np.zeros(3, np.float32), np.array([3, 2, 2]), 7, 1, 1.0)
    assert out.tolist() == [-1.0, 1.0, 1.0]


def check_bias_controller_balances():
    # Loads skewed by a fixed per-expert logit offset; repeated route -> count -> update
    # steps drive the most-loaded expert towards its share (the controller's purpose).
    r = _rng(23)
    T, E, k = 512, 8, 2
    l = (r.normal(0, 1, (T, E)) + np.linspace(-2, 2, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    def max_over_mean(bias):
        idx = orc.route(l.astype(np.float64), np.eye(E), k, "softmax", sel_bias=bias)["idx"]
        c = np.bincount(idx.ravel(), minlength=E)
        return c, c.max() / (T * k / E)
    c, start = max_over_mean(b)
    for _ in range(300):
        b = orc.update_sel_bias(b, c, T, k, 0.02)
        c, m = max_over_mean(b)
    assert start > 2.0 and m < 1.2, (start, m)


def check_switch_top1_no_renorm():
    # Switch: top-1, y = p_i(x) E_i(x) with p the softmax probability itself ([RA] "The router").
    x, Wg, W = _rand_layer(24, T=5, d=4, d_ff=3, E=4)
    out = orc.forward(x, Wg, _arrays_fn(W), 4, 1, "softmax_norenorm")
    l = orc.router_logits(x, Wg).astype(np.float64)
    for t in range(5):
        ex = [math.exp(v) for v in l[t]]
        e = int(np.argmax(l[t]))
        p = ex[e] / sum(ex)
        assert out["idx"][t, 0] == e and abs(out["gate"][t, 0] - p) < 1e-12 and p < 1.0
        ref = p * dense_swiglu_loops(x[t:t + 1], W["W1"][e], W["W2"][e], W["W3"][e])[0]
        assert np.allclose(out["y"][t], ref, rtol=1e-12, atol=1e-12)
    # with k = E nothing is left out: the plain and renormalised gates coincide
    a = orc.route(x, Wg, 4, "softmax_norenorm")
    b = orc.route(x, Wg, 4, "softmax")
    assert np.array_equal(a["idx"], b["idx"]) and np.allclose(a["gate"], b["gate"], rtol=1e-12)


def check_load_stats():
    # hand example: E = 4, k = 2, three tokens choosing (0,1), (0,2), (0,3): counts 3,1,1,1,
    # mean load 6/4 -> max/mean 2; f = counts / T; every token's logits (ln 3, 0, 0, 0) give the
    # softmax (1/2, 1/6, 1/6, 1/6) = P; L_aux = alpha E sum f P.
    idx = np.array([[0, 1], [0, 2], [0, 3]], np.int32)
    l = np.tile(np.array([math.log(3.0), 0, 0, 0], np.float32), (3, 1))
    st = orc.load_stats(idx, l, 4, "softmax", 0.01)
    assert st["counts"].tolist() == [3, 1, 1, 1] and st["max_over_mean"] == 2.0
    assert np.allclose(st["f"], [1.0, 1 / 3, 1 / 3, 1 / 3], rtol=1e-15)
    assert np.allclose(st["P"], [0.5, 1 / 6, 1 / 6, 1 / 6], rtol=1e-6)
    assert abs(st["aux_loss"] - 0.01 * 4 * (0.5 + 3 * (1 / 3) * (1 / 6))) < 1e-9
    # uniform scores with top-1 routing: L_aux = alpha whatever the assignment ([MM] 3.1, E = 64)
    E, T = 64, 256
    idx = (np.arange(T) % E).reshape(T, 1).astype(np.int32)
    st = orc.load_stats(idx, np.zeros((T, E), np.float32), E, "softmax", 0.01)
    assert abs(st["aux_loss"] - 0.01) < 1e-15 and st["max_over_mean"] == 1.0
    # sigmoid scores: P is the mean sigmoid score
    st = orc.load_stats(idx[:2], np.zeros((2, E), np.float32), E, "sigmoid", 1.0)
    assert np.allclose(st["P"], 0.5, rtol=1e-15)


def check_capacity_dropping():
    # The printed example ([RA] "Capacity and token dropping"): 4,096 tokens, 64 experts,
    # top-8, capacity factor 1.0 -> 512 slots; an expert picked 600 times drops 88, and the
    # 88 dropped are its last 88 tokens in token order.
    T, E, k = 4096, 64, 8
    assert orc.capacity_slots(T, k, E, 1.0) == 512
    r = _rng(25)
    idx = np.empty((T, k), np.int32)
    hot = set(r.choice(T, 600, replace=False).tolist())
    others = np.array([e for e in range(E) if e != 7])
    for t in range(T):
        pick = r.choice(others, k - 1 if t in hot else k, replace=False).tolist()
        idx[t] = ([7] + pick) if t in hot else pick
    d = orc.dispatch(idx, E, 512)
    assert d["counts"][7] == 600
    kept7 = d["offsets"][8] - d["offsets"][7]
    assert kept7 == 512 and d["counts"][7] - kept7 == 88
    hot_sorted = sorted(hot)
    assert all(d["inv_pos"][t, 0] >= 0 for t in hot_sorted[:512])
    assert all(d["inv_pos"][t, 0] == -1 for t in hot_sorted[512:])
    kept = np.minimum(d["counts"], 512)
    assert int((d["inv_pos"] == -1).sum()) == int((d["counts"] - kept).sum())
    assert d["offsets"][-1] == kept.sum() == len(d["perm_tok"])
    # positions of kept pairs are a bijection onto 0 .. kept - 1, and point back to their token
    flat = d["inv_pos"].reshape(-1)
    live = flat[flat >= 0]
    assert sorted(live.tolist()) == list(range(int(kept.sum())))
    tok = np.repeat(np.arange(T), k)[flat >= 0]
    assert np.array_equal(d["perm_tok"][live], tok)
    # slots in whole numbers: ceil(T k c / E)
    assert orc.capacity_slots(10, 2, 3, 1.0) == 7 and orc.capacity_slots(8, 1, 4, 1.25) == 3


def check_capacity_grouped_equals_bruteforce():
    # Dropped pairs contribute nothing: the grouped evaluation with a capacity equals the
    # naive per-expert loop that skips a token once its expert is full.
    x, Wg, W = _rand_layer(26, T=24, d=6, d_ff=5, E=4)
    Wg[:, 1] += 0.8                     # skew towards expert 1 so that it overflows
    for c in (0.5, 1.0, 1.25):
        g = orc.forward(x, Wg, _arrays_fn(W), 4, 2, "softmax", capacity_factor=c)
        b = orc.forward_bruteforce(x, Wg, _arrays_fn(W), 4, 2, "softmax", capacity_factor=c)
        assert np.allclose(g["y"], b, rtol=1e-12, atol=1e-12)
        assert (g["inv_pos"] == -1).any()
    # a capacity no expert reaches changes nothing
    g = orc.forward(x, Wg, _arrays_fn(W), 4, 2, "softmax", capacity_factor=100.0)
    n = orc.forward(x, Wg, _arrays_fn(W), 4, 2, "softmax")
    assert np.array_equal(g["y"], n["y"]) and np.array_equal(g["inv_pos"], n["inv_pos"])


def check_expert_choice():
    # Balanced by construction ([FM] 5.1): every expert takes exactly m tokens; the grouped
    # evaluation equals the naive per-expert full sort; gates are the token's softmax score.
    x, Wg, W = _rand_layer(27, T=20, d=6, d_ff=5, E=4)
    m = orc.expert_choice_slots(20, 2, 4, 0.0)
    assert m == 10
    g = orc.expert_choice_forward(x, Wg, _arrays_fn(W), 4, m)
    assert np.array_equal(np.diff(g["offsets"]), [m] * 4)
    assert ((g["pos_of"] >= 0).sum(axis=0) == m).all()
    b = orc.expert_choice_bruteforce(x, Wg, _arrays_fn(W), 4, m)
    assert np.allclose(g["y"], b, rtol=1e-12, atol=1e-12)
    s = orc.scores(orc.router_logits(x, Wg), "softmax")
    for e in range(4):
        toks = g["perm_tok"][e * m:(e + 1) * m]
        assert list(toks) == sorted(toks)
        assert np.allclose(g["gate"][e * m:(e + 1) * m], s[toks, e], rtol=1e-15)
        # the chosen tokens are the m largest of the column
        assert s[toks, e].min() >= np.sort(s[:, e])[-m]
    # every expert takes every token (m = T): the softmax-weighted dense ensemble, which is
    # token choice with k = E
    full = orc.expert_choice_forward(x, Wg, _arrays_fn(W), 4, 20)
    dense = orc.forward(x, Wg, _arrays_fn(W), 4, 4, "softmax")
    assert np.allclose(full["y"], dense["y"], rtol=1e-12, atol=1e-12)
    # one expert that takes every token: gate 1, a dense SwiGLU FFN
    x1, Wg1, W1 = _rand_layer(28, T=5, d=4, d_ff=3, E=1)
    one = orc.expert_choice_forward(x1, Wg1, _arrays_fn(W1), 1, 5)
    assert np.allclose(one["y"], dense_swiglu_loops(x1, W1["W1"][0], W1["W2"][0], W1["W3"][0]), rtol=1e-12)
    # slots: ceil(T k c / E), at most T
    assert orc.expert_choice_slots(100, 2, 8, 1.25) == 32 and orc.expert_choice_slots(10, 4, 2, 2.0) == 10


def check_printed_values():
    G = json.load(open(GOLDEN))
    for c in G["combinations"]:
        assert orc.n_combinations(c["E"], c["k"]) == c["value"] == math.comb(c["E"], c["k"])
    for c in G["expert_params"]:
        assert orc.expert_params(c["d"], c["d_ff"]) == c["value"]
    for c in G["router_params"]:
        assert orc.moe_ffn_params(c["E"], c["d"], 0) == c["value"]
    h = G["total_active"][0]
    P_e = orc.expert_params(h["d"], h["d_ff"])
    assert h["L"] * h["E"] * P_e == h["routed"]
    tot, act = orc.total_active_params(h["N0"], h["L"], h["E"], h["k"], P_e)
    assert (tot, act) == (h["total"], h["active"])
    assert tot - h["L"] * h["gap_experts"] * P_e == act
    v3 = G["total_active"][1]
    assert v3["L"] * v3["E"] * orc.expert_params(v3["d"], v3["d_ff"]) == v3["routed"]
    f = G["flops"][0]
    assert abs(2 * f["active"] / 1e9 - f["gflops_per_token_printed"]) / f["gflops_per_token_printed"] < f["rel_tol"]
    f = G["flops"][1]
    d = f["d"]
    assert orc.flops_per_token(d, 8 * d // 3, f["E"], f["k"]) == 16 * d * d * f["k"] + 2 * d * f["E"]
    m = G["moe_ffn_params"][0]
    d, E = m["d"], m["E"]
    experts = orc.moe_ffn_params(E, d, 8 * d // 3) - d * E
    assert abs(experts - m["experts_printed"]) / m["experts_printed"] < m["rel_tol"]
    assert abs(orc.expert_params(d, 8 * d // 3) - m["dense_printed"]) / m["dense_printed"] < m["rel_tol"]
    p = G["p_unused"][0]
    assert abs(100 * orc.p_expert_unused(p["E"], p["k"], p["batch"]) - p["printed_percent"]) < p["abs_tol_percent"]
    c = G["capacity"][0]
    cap = orc.capacity(c["tokens"], c["E"], c["k"], c["factor"])
    assert cap == c["slots"] and orc.dropped(c["picks"], int(cap)) == c["dropped"]
    a = G["aux_loss"][0]
    u = np.full(a["E"], 1.0 / a["E"])
    assert abs(orc.aux_loss(u, u, a["alpha"]) - a["uniform_value"]) < 1e-15
    b = G["dispatch_bytes"][0]
    assert orc.dispatch_bytes(b["T"], b["k"], b["d"], b["elem_bytes"]) == b["value"]


CHECKS = [check_router_logits_closed_form, check_scores_closed_forms, check_topk_bruteforce,
          check_gate_invariants, check_gates_two_formulations, check_k_equals_E_is_dense_softmax,
          check_dispatch, check_swiglu_scalar_closed_form, check_swiglu_vs_loops,
          check_E1_k1_is_dense_swiglu, check_grouped_equals_bruteforce, check_shared_only,
          check_selection_bias, check_selection_bias_sigmoid_uses_scores, check_sel_bias_update_closed_form,
          check_bias_controller_balances, check_switch_top1_no_renorm, check_load_stats,
          check_capacity_dropping, check_capacity_grouped_equals_bruteforce, check_expert_choice,
          check_printed_values]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


# ---------------------------------------------------------------- planted mistakes

def _swapped_swiglu(X, W1, W2, W3):             # W1 and W2 exchanged
    u, v = X @ W2, X @ W1
    return (u * orc.silu(v)) @ W3


def _no_renorm(s, idx):                        # gates not renormalised over the chosen k
    return np.take_along_axis(np.asarray(s, np.float64), idx.astype(np.int64), axis=-1)


def _mirrored_experts(x, Wg, logit_bias=None):   # logits written to the wrong expert columns
    l = (np.asarray(x, np.float64) @ np.asarray(Wg, np.float64)[:, ::-1]).astype(np.float32)
    return l if logit_bias is None else (l + np.asarray(logit_bias, np.float32)).astype(np.float32)


def _unstable_dispatch(idx, E):                # pairs of one expert in reverse order
    out = orc.__dict__["_orig_dispatch"](idx, E)
    T, k = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat[::-1], kind="stable")
    order = (T * k - 1 - order)
    perm = order // k
    inv = np.empty(T * k, np.int32)
    inv[order] = np.arange(T * k)
    out["perm_tok"], out["inv_pos"] = perm.astype(np.int32), inv.reshape(T, k)
    return out


def _no_shared(x64, get_w, n_shared):          # shared expert dropped
    return None


def _silu_sign(v):                             # Swish with the wrong sign in the exponent
    return v / (1.0 + np.exp(v))


def _topk_ascending(key32, k):                 # smallest instead of largest
    return np.argsort(np.asarray(key32, np.float32), axis=-1, kind="stable")[:, :k].astype(np.int32)


def _bias_update_wrong_sign(sel_bias, counts, T, k, gamma):   # overloaded experts pushed up
    return orc.__dict__["_orig_update_sel_bias"](sel_bias, counts, T, k, -gamma)


def _bias_on_logits(l32, scoring, sel_bias=None):             # sigmoid bias added to logits
    return orc.__dict__["_orig_selection_keys"](l32, "softmax", sel_bias)


def _aux_without_E(f, P, alpha):                               # the factor E left out
    return float(alpha * np.sum(np.asarray(f) * np.asarray(P)))


def _drop_earliest(idx, E, slots=None):                       # an expert keeps its LAST pairs
    if slots is None:
        return orc.__dict__["_orig_dispatch"](idx, E)
    rev = orc.__dict__["_orig_dispatch"](idx[::-1].copy(), E, slots)
    T, k = idx.shape
    inv = rev["inv_pos"][::-1].copy()
    return {"counts": rev["counts"], "offsets": rev["offsets"], "perm_tok": rev["perm_tok"], "inv_pos": inv}


def _ec_lowest(x64, Wg64, E, m, logit_bias=None):               # experts take their m LOWEST scores
    r = orc.__dict__["_orig_expert_choice_route"](-np.asarray(x64), Wg64, E, m, logit_bias)
    return r


PLANTS = [
    ("swiglu_expert", _swapped_swiglu, [check_swiglu_scalar_closed_form, check_swiglu_vs_loops]),
    ("gates_from_scores", _no_renorm, [check_gate_invariants, check_gates_two_formulations]),
    ("router_logits", _mirrored_experts, [check_router_logits_closed_form]),
    ("dispatch", _unstable_dispatch, [check_dispatch]),
    ("shared_experts", _no_shared, [check_shared_only]),
    ("silu", _silu_sign, [check_swiglu_scalar_closed_form, check_E1_k1_is_dense_swiglu]),
    ("select_topk", _topk_ascending, [check_topk_bruteforce]),
    ("update_sel_bias", _bias_update_wrong_sign, [check_sel_bias_update_closed_form, check_bias_controller_balances]),
    ("selection_keys", _bias_on_logits, [check_selection_bias_sigmoid_uses_scores]),
    ("aux_loss", _aux_without_E, [check_load_stats]),
    ("dispatch", _drop_earliest, [check_capacity_dropping, check_capacity_grouped_equals_bruteforce]),
    ("expert_choice_route", _ec_lowest, [check_expert_choice]),
]


@pytest.mark.parametrize("name,bad,checks", PLANTS, ids=[p[0] for p in PLANTS])
def test_planted_mistakes_are_caught(monkeypatch, name, bad, checks):
    monkeypatch.setitem(orc.__dict__, "_orig_" + name, getattr(orc, name))
    monkeypatch.setattr(orc, name, bad)
    for check in checks:
        with pytest.raises(AssertionError):
            check()
