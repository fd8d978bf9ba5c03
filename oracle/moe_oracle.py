"""CPU oracle for the forward pass of a top-k Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE.  Only the tests, `__graft_entry__.smoke()` and the CPU-baseline /
reference legs of `bench.py` may import or run this module.  It shares no code with the
CUDA library (it imports nothing from the product package), and the library never imports
it.  Inputs come from the seeded generator in `workloads/`, which both sides use.

It is a plain, slow, obviously-correct restatement of the layer as the pages define it:

    MoE(x) = f_shared(x) + sum_{e in TopK(x)} g_e(x) f_e(x)
    f_e(x) = ((x W1_e) * Swish(x W2_e)) W3_e,   Swish = SiLU (beta = 1)

Sources (page title, section):
  [MM]  "8.6 - Mixture of Experts (MoE)": section 2 (SwiGLU expert, router x W_g, top-k by
        largest logit, gates exp(l_e) / sum over the chosen k, layer output), section 2.1
        (FLOP and parameter counts), section 3.1 (auxiliary loss), section 3.2 (capacity),
        section 4 (combinations), section 4.1 (shared expert).
  [FM]  "Mixture-of-Experts Internals: A Systems Engineer's Field Manual": section 2.1
        (softmax over all E, top-k, renormalise over the chosen k), section 3.2 (Switch
        auxiliary loss), section 3.3 (bias used only for selection), section 4.2 (dispatch
        volume), section 5.1 (expert choice: each expert takes its top-m tokens).
  [RA]  "Mixture-of-Experts, from the router to the all-to-all": "The router" (sigmoid
        scores normalised over the chosen k; Switch's top-1 y = p_i(x) E_i(x) without
        renormalisation), "Experts, fine-grained and shared" (P_e =
        3 d d_ff, combination counts), "Why total and active parameters come apart",
        "Capacity and token dropping", "Load balancing" (auxiliary loss, a bias used only
        for choosing and its update).
  [T26] "T2.6 What MoE changes": "Routing creates an assignment problem" (per-expert counts,
        maximum load over mean load), "In practice" (what to monitor).
  [TR]  "Mixture of Experts: What Actually Happens When a Token Hits the Router": Step 3
        (the masked per-expert loop; sort by expert, one matmul per expert, scatter back),
        Step 4 (down(silu(gate(x)) * up(x)), weighted sum).

Precision.  The router logits are formed in float64 from the stored (float32 or bfloat16)
values and rounded once to float32: the top-k decision is taken on float32 values on both
sides, as the pages keep the router in float32.  Biases are added in float32.  Scores,
gates, the experts and the combine are float64.

Pins (tests/test_oracle_pins.py): every function here is checked against something other
than itself: closed forms, printed values, special cases that reduce to a dense SwiGLU FFN
or a full softmax, brute force over all k-subsets, and an independent per-token evaluation.
The numeric values of y for the five synthetic workloads are not printed by the pages; they
are trusted through those pins.
"""
from __future__ import annotations

import math
from typing import Callable, Dict, Optional, Sequence

import numpy as np

from workloads import to_f64

# --------------------------------------------------------------------------------------
# Router: logits, scores, top-k, gates
# --------------------------------------------------------------------------------------


def router_logits(x64: np.ndarray, Wg64: np.ndarray,
                  logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Router logits l = x W_g (+ bias), as float32 [T, E].

    [MM] section 2: router(x) = x W_g with W_g of shape d x E.  [FM] section 2.1 writes the
    same map as W_r x with W_r = W_g^T.  The per-expert bias of the skewed workload is added
    to the logits, so it shifts both the scores and the selection."""
    l = (np.asarray(x64, np.float64) @ np.asarray(Wg64, np.float64)).astype(np.float32)
    if logit_bias is not None:
        l = (l + np.asarray(logit_bias, np.float32)).astype(np.float32)
    return l


def scores(l32: np.ndarray, scoring: str) -> np.ndarray:
    """Per-expert scores in float64.

    softmax (and softmax_norenorm): s = softmax(l) over all E experts ([FM] section 2.1;
    [RA] "The router").  sigmoid: s_e = 1 / (1 + exp(-l_e)), DeepSeek-V3's scoring ([RA]
    "The router")."""
    l = np.asarray(l32, np.float64)
    if scoring in ("softmax", "softmax_norenorm"):
        m = l.max(axis=-1, keepdims=True)
        e = np.exp(l - m)
        return e / e.sum(axis=-1, keepdims=True)
    if scoring == "sigmoid":
        return 1.0 / (1.0 + np.exp(-l))
    raise ValueError(scoring)


def select_topk(key32: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys per row, in descending key order; equal keys go to the
    lower expert id.  [MM] section 2: the k experts with the largest gate logits."""
    key = np.asarray(key32, np.float32)
    order = np.argsort(-key, axis=-1, kind="stable")
    return order[:, :k].astype(np.int32)


def gates_from_scores(s64: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g_j = s_{I_j} / sum_{j'} s_{I_j'}: the chosen scores renormalised to sum to 1.

    [FM] section 2.1 (renormalised gates; zero outside the chosen set) and [RA] "The router"
    (sigmoid scores normalised among the selected)."""
    sel = np.take_along_axis(np.asarray(s64, np.float64), idx.astype(np.int64), axis=-1)
    return sel / sel.sum(axis=-1, keepdims=True)


def selection_keys(l32: np.ndarray, scoring: str, sel_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """The float32 values the top-k is taken over.

    Without a selection bias: the logits l (softmax and sigmoid are monotone, so the chosen
    set and its order are those of the scores).  With a per-expert bias b used for choosing
    only: [FM] section 3.3 adds b to the routing logit (softmax routing); [RA] "Load
    balancing" (a bias instead of a loss) adds b to the score s (DeepSeek-V3's sigmoid routing).  So the key is
    l + b for softmax scoring and sigmoid(l) + b for sigmoid scoring, each sum rounded to
    float32 (the sigmoid itself is rounded to float32 first)."""
    l = np.asarray(l32, np.float32)
    if sel_bias is None:
        return l
    b = np.asarray(sel_bias, np.float32)
    if scoring == "sigmoid":
        s32 = scores(l, "sigmoid").astype(np.float32)
        return (s32 + b).astype(np.float32)
    return (l + b).astype(np.float32)


def route(x64: np.ndarray, Wg64: np.ndarray, k: int, scoring: str,
          logit_bias: Optional[np.ndarray] = None,
          sel_bias: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Router logits -> scores -> top-k -> gates for every token.

    Selection runs on selection_keys (a bias used for choosing only, [FM] section 3.3, [RA]
    "Load balancing"; the gates come from the unbiased scores).  Returns idx [T, k]
    int32, gate [T, k] float64, logits [T, E] float32."""
    l = router_logits(x64, Wg64, logit_bias)
    idx = select_topk(selection_keys(l, scoring, sel_bias), k)
    s = scores(l, scoring)
    if scoring == "softmax_norenorm":
        # Switch: y = p_i(x) E_i(x), the softmax probability itself ([RA] "The router")
        g = np.take_along_axis(s, idx.astype(np.int64), axis=-1)
    else:
        g = gates_from_scores(s, idx)
    return {"idx": idx, "gate": g, "logits": l}


def update_sel_bias(sel_bias: np.ndarray, counts: np.ndarray, T: int, k: int, gamma: float) -> np.ndarray:
    """One step of the bias controller ([FM] section 3.3; [RA] "Load balancing"):
    an expert that received more than its share T k / E of the last batch's assignments
    (overloaded) has its bias lowered by gamma, one that received less (underloaded) has it
    raised by gamma; an expert at exactly its share keeps its bias.  The comparison is done
    in integers (counts[e] E against T k); the update in float32."""
    b = np.asarray(sel_bias, np.float32).copy()
    c = np.asarray(counts, np.int64)
    E = len(b)
    share = np.int64(T) * np.int64(k)
    g = np.float32(gamma)
    over = c * E > share
    under = c * E < share
    b[over] = (b[over] - g).astype(np.float32)
    b[under] = (b[under] + g).astype(np.float32)
    return b


# --------------------------------------------------------------------------------------
# Dispatch: histogram, offsets, permutation
# --------------------------------------------------------------------------------------


def capacity_slots(T: int, k: int, E: int, factor: float) -> int:
    """Slots per expert when a capacity factor c is set: ceil(T k c / E) ([MM] section 3.2:
    capacity = T k / E * c; [RA] "Capacity and token dropping").  Computed in double as
    (T k) * c / E with c the float32 value the library is given, then rounded up to whole
    slots."""
    return int(math.ceil(float(T * k) * float(np.float32(factor)) / float(E)))


def dispatch(idx: np.ndarray, E: int, slots: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Group the (token, slot) pairs by expert ([TR] Step 3: sort tokens by assigned expert
    into contiguous blocks).

    counts[e]   = number of pairs routed to expert e (its load, before any dropping)
    offsets[e]  = sum of the kept pairs of the experts before e; offsets[E] = pairs kept
    perm_tok[p] = token of the p-th kept pair in expert order (pairs of one expert keep the
                  order of their flattened index t k + j)
    inv_pos[t, j] = position p of pair (t, j), or -1 if the pair was dropped.

    With `slots` (a capacity), an expert keeps its first `slots` pairs in token order and
    drops the rest ([RA] "Capacity and token dropping": a token that finds its expert full
    is dropped from it)."""
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    kept = counts if slots is None else np.minimum(counts, slots).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(kept)]).astype(np.int32)
    full_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    e_of = flat[order]
    rank = np.arange(T * k, dtype=np.int64) - full_offsets[e_of]
    keep = rank < kept[e_of]
    inv = np.full(T * k, -1, dtype=np.int32)
    inv[order[keep]] = (offsets[e_of[keep]] + rank[keep]).astype(np.int32)
    perm_tok = (order[keep] // k).astype(np.int32)
    return {"counts": counts, "offsets": offsets, "perm_tok": perm_tok,
            "inv_pos": inv.reshape(T, k)}


# --------------------------------------------------------------------------------------
# Experts
# --------------------------------------------------------------------------------------


def silu(v: np.ndarray) -> np.ndarray:
    """Swish with beta = 1 (SiLU): v * sigmoid(v)."""
    return v / (1.0 + np.exp(-v))


def swiglu_expert(X64: np.ndarray, W1: np.ndarray, W2: np.ndarray, W3: np.ndarray) -> np.ndarray:
    """f(x) = ((x W1) * Swish(x W2)) W3 for every row of X, in float64 ([MM] section 2).
    W2 is the gated projection ([TR] Step 4 writes down(silu(gate(x)) * up(x)))."""
    u = X64 @ W1
    v = X64 @ W2
    return (u * silu(v)) @ W3


WeightFn = Callable[[str, int], np.ndarray]   # (name, expert) -> float64 matrix


def weights_from_arrays(arrays: Dict[str, np.ndarray], dtype: str) -> WeightFn:
    """Adapter: stacked stored arrays {"W1": [E, d, d_ff], ...} -> float64 per expert."""
    def get(name: str, e: int) -> np.ndarray:
        return to_f64(arrays[name][e], dtype)
    return get


def experts_grouped(x_perm64: np.ndarray, offsets: np.ndarray, get_w: WeightFn) -> np.ndarray:
    """Each expert e runs once on its contiguous block rows offsets[e]:offsets[e+1] of the
    permuted activations ([TR] Step 3, one dense matmul per expert).  Empty experts are
    skipped.  Returns y_perm [T k, d] float64."""
    E = len(offsets) - 1
    y = np.zeros((x_perm64.shape[0], get_w("W3", 0).shape[1] if E else 0), np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_expert(x_perm64[a:b], get_w("W1", e), get_w("W2", e), get_w("W3", e))
    return y


def shared_experts(x64: np.ndarray, get_w: WeightFn, n_shared: int) -> Optional[np.ndarray]:
    """Sum of the always-on shared experts, gate 1 ([MM] section 4.1; [FM] section 6.2)."""
    if n_shared <= 0:
        return None
    ys = np.zeros((x64.shape[0], x64.shape[1]), np.float64)
    for s in range(n_shared):
        ys += swiglu_expert(x64, get_w("Ws1", s), get_w("Ws2", s), get_w("Ws3", s))
    return ys


def combine(y_perm64: np.ndarray, inv_pos: np.ndarray, gate64: np.ndarray,
            shared64: Optional[np.ndarray] = None) -> np.ndarray:
    """y[t] = sum_j g[t, j] y_perm[inv_pos[t, j]] (+ shared[t]): scatter the expert outputs
    back to token order and weight them by the gates ([MM] section 2; [TR] Step 3/4).  Pairs
    dropped at dispatch (inv_pos = -1) contribute zero ([MM] section 3.2)."""
    T, k = inv_pos.shape
    y = np.zeros((T, y_perm64.shape[1]), np.float64)
    for j in range(k):
        kept = inv_pos[:, j] >= 0                 # a dropped pair contributes nothing
        y[kept] += gate64[kept, j:j + 1] * y_perm64[inv_pos[kept, j]]
    if shared64 is not None:
        y += shared64
    return y


def forward(x64: np.ndarray, Wg64: np.ndarray, get_w: WeightFn, E: int, k: int,
            scoring: str, logit_bias=None, sel_bias=None, n_shared: int = 0,
            capacity_factor: float = 0.0) -> Dict[str, np.ndarray]:
    """The whole layer, evaluated the grouped way: route, dispatch (with capacity_slots per
    expert when capacity_factor > 0), one SwiGLU per expert over its block, combine (+ shared
    experts).  All results are returned for comparison."""
    r = route(x64, Wg64, k, scoring, logit_bias, sel_bias)
    T = x64.shape[0]
    slots = capacity_slots(T, k, E, capacity_factor) if capacity_factor > 0 else None
    dsp = dispatch(r["idx"], E, slots)
    x_perm = x64[dsp["perm_tok"]]
    y_perm = experts_grouped(x_perm, dsp["offsets"], get_w)
    ys = shared_experts(x64, get_w, n_shared)
    y = combine(y_perm, dsp["inv_pos"], r["gate"], ys)
    out = dict(r)
    out.update(dsp)
    out.update({"y_perm": y_perm, "y": y, "y_shared": ys})
    return out


def forward_tokens(x_rows64: np.ndarray, idx_rows: np.ndarray, gate_rows: np.ndarray,
                   get_w: WeightFn, n_shared: int = 0, kept_rows: Optional[np.ndarray] = None) -> np.ndarray:
    """The layer output for a few tokens, given their routing, by the definition
    MoE(x) = sum_j g_j f_{I_j}(x) (+ shared): each chosen expert evaluated on the token
    itself ([MM] section 2).  Tokens that share an expert are evaluated together.  kept_rows
    [n, k] bool, if given, leaves out the pairs dropped at dispatch."""
    n, k = idx_rows.shape
    y = np.zeros((n, x_rows64.shape[1]), np.float64)
    for e in np.unique(idx_rows):
        sel = idx_rows == e
        if kept_rows is not None:
            sel = sel & kept_rows
        rows, slots = np.nonzero(sel)
        if rows.size == 0:
            continue
        fe = swiglu_expert(x_rows64[rows], get_w("W1", int(e)), get_w("W2", int(e)), get_w("W3", int(e)))
        y[rows] += gate_rows[rows, slots][:, None] * fe
    ys = shared_experts(x_rows64, get_w, n_shared)
    return y if ys is None else y + ys


def forward_bruteforce(x64: np.ndarray, Wg64: np.ndarray, get_w: WeightFn, E: int, k: int,
                       scoring: str, logit_bias=None, sel_bias=None, n_shared: int = 0,
                       capacity_factor: float = 0.0) -> np.ndarray:
    """The naive evaluation ([TR] Step 3): loop over experts, mask the tokens that chose
    each, run the expert on them, weight by the gate and accumulate.  No sort, no offsets,
    no permutation: an independent evaluation of the same sum, for tiny inputs.  With a
    capacity, an expert takes the tokens that chose it in token order and skips the rest
    once it is full ([RA] "Capacity and token dropping")."""
    r = route(x64, Wg64, k, scoring, logit_bias, sel_bias)
    T = x64.shape[0]
    slots = capacity_slots(T, k, E, capacity_factor) if capacity_factor > 0 else None
    y = np.zeros_like(x64, dtype=np.float64)
    for e in range(E):
        taken = 0
        for t in range(T):
            for j in range(k):
                if r["idx"][t, j] == e:
                    if slots is not None and taken >= slots:
                        continue
                    taken += 1
                    f = swiglu_expert(x64[t:t + 1], get_w("W1", e), get_w("W2", e), get_w("W3", e))[0]
                    y[t] += r["gate"][t, j] * f
    ys = shared_experts(x64, get_w, n_shared)
    return y if ys is None else y + ys


# --------------------------------------------------------------------------------------
# Expert-choice routing
# --------------------------------------------------------------------------------------


def expert_choice_slots(T: int, k: int, E: int, factor: float) -> int:
    """Tokens each expert takes under expert choice: m = ceil(T k c / E) with c the capacity
    factor (1 when none is given), at most T.  [FM] section 5.1: each expert chooses its
    top-m tokens, exactly m per expert; the capacity formula is that of [MM] section 3.2."""
    c = factor if factor > 0 else 1.0
    return min(T, capacity_slots(T, k, E, c))


def expert_choice_route(x64: np.ndarray, Wg64: np.ndarray, E: int, m: int,
                        logit_bias: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Expert choice ([FM] section 5.1; [RA] "Load balancing": each expert takes its top
    tokens, so load is balanced by construction).  The token-to-expert scores are the softmax
    over the experts of each token's router logits; expert e takes the m tokens with the
    largest s[t, e] (decided on float32 values; equal values go to the lower token id) and
    weights its output for token t by s[t, e].  A token may be taken by any number of
    experts, including none.

    Returns offsets [E+1] (= e m), perm_tok [E m] (each expert's tokens in ascending token
    order), gate [E m] float64, pos_of [T, E] int32 (the position of (t, e), or -1),
    logits, scores."""
    l = router_logits(x64, Wg64, logit_bias)
    s = scores(l, "softmax")
    key = s.astype(np.float32)
    T = l.shape[0]
    perm, gate = [], []
    pos_of = np.full((T, E), -1, dtype=np.int32)
    for e in range(E):
        order = np.argsort(-key[:, e], kind="stable")
        toks = np.sort(order[:m])
        for r, t in enumerate(toks):
            pos_of[t, e] = e * m + r
        perm.append(toks)
        gate.append(s[toks, e])
    return {"offsets": (np.arange(E + 1) * m).astype(np.int32),
            "perm_tok": np.concatenate(perm).astype(np.int32) if E else np.zeros(0, np.int32),
            "gate": np.concatenate(gate) if E else np.zeros(0), "pos_of": pos_of, "logits": l, "scores": s}


def expert_choice_forward(x64: np.ndarray, Wg64: np.ndarray, get_w: WeightFn, E: int, m: int,
                          logit_bias=None, n_shared: int = 0) -> Dict[str, np.ndarray]:
    """The layer under expert choice, grouped: each expert runs once on its m tokens, and
    y[t] = sum over the experts that took t of s[t, e] f_e(x_t) (+ shared experts), summed in
    expert order."""
    r = expert_choice_route(x64, Wg64, E, m, logit_bias)
    y_perm = experts_grouped(x64[r["perm_tok"]], r["offsets"], get_w)
    T = x64.shape[0]
    y = np.zeros((T, x64.shape[1]), np.float64)
    for e in range(E):
        p = r["pos_of"][:, e]
        took = p >= 0
        y[took] += r["gate"][p[took]][:, None] * y_perm[p[took]]
    ys = shared_experts(x64, get_w, n_shared)
    if ys is not None:
        y = y + ys
    out = dict(r)
    out.update({"y_perm": y_perm, "y": y})
    return out


def expert_choice_bruteforce(x64: np.ndarray, Wg64: np.ndarray, get_w: WeightFn, E: int, m: int,
                             logit_bias=None, n_shared: int = 0) -> np.ndarray:
    """Expert choice evaluated naively: for every expert, rank all tokens by their score for
    it with a full sort, keep the first m, run the expert on each kept token alone and add
    s[t, e] times its output to that token."""
    l = router_logits(x64, Wg64, logit_bias)
    s = scores(l, "softmax")
    T = x64.shape[0]
    y = np.zeros((T, x64.shape[1]), np.float64)
    for e in range(E):
        ranked = sorted(range(T), key=lambda t: (-float(np.float32(s[t, e])), t))
        for t in ranked[:m]:
            f = swiglu_expert(x64[t:t + 1], get_w("W1", e), get_w("W2", e), get_w("W3", e))[0]
            y[t] += s[t, e] * f
    ys = shared_experts(x64, get_w, n_shared)
    return y if ys is None else y + ys


# --------------------------------------------------------------------------------------
# Counting helpers (printed quantities on the pages)
# --------------------------------------------------------------------------------------


def n_combinations(E: int, k: int) -> int:
    """Number of distinct k-expert sets out of E: E! / (k! (E-k)!), in exact integers
    ([MM] section 4; [RA] "Experts, fine-grained and shared")."""
    if k < 0 or k > E:
        return 0
    num, den = 1, 1
    for i in range(k):
        num *= E - i
        den *= i + 1
    return num // den


def expert_params(d: int, d_ff: int) -> int:
    """Weights of one SwiGLU expert: P_e = 3 d d_ff ([RA] "Experts, fine-grained and shared")."""
    return 3 * d * d_ff


def moe_ffn_params(E: int, d: int, d_ff: int) -> int:
    """Weights of one MoE FFN sub-layer: E (3 d d_ff) + d E ([MM] section 2.1)."""
    return E * expert_params(d, d_ff) + d * E


def total_active_params(N0: int, L: int, E: int, k: int, P_e: int):
    """(N_total, N_active) = (N0 + L E P_e, N0 + L k P_e)
    ([RA] "Why total and active parameters come apart")."""
    return N0 + L * E * P_e, N0 + L * k * P_e


def flops_per_token(d: int, d_ff: int, E: int, k: int, n_shared: int = 0, d_ff_shared: int = 0) -> int:
    """Forward FLOPs per token: router 2 d E plus 6 d d_ff per evaluated SwiGLU expert
    (two d x d_ff and one d_ff x d matrix-vector product; [MM] section 2.1 gives 16 d^2 k
    when d_ff = 8d/3)."""
    return 2 * d * E + 6 * d * d_ff * k + 6 * d * d_ff_shared * n_shared


def p_expert_unused(E: int, k: int, batch: int) -> float:
    """Chance that one expert is chosen by none of `batch` tokens that each pick k of E
    uniformly: ((E - k) / E)^batch ([RA] "Why total and active parameters come apart")."""
    return ((E - k) / E) ** batch


def capacity(tokens: int, E: int, k: int, factor: float) -> float:
    """Expert capacity tokens k / E * factor ([MM] section 3.2; [RA] "Capacity and token
    dropping")."""
    return tokens * k / E * factor


def dropped(picks: int, cap: int) -> int:
    """Assignments an expert drops when picked more often than its capacity allows."""
    return max(0, picks - cap)


def aux_loss(f: np.ndarray, P: np.ndarray, alpha: float) -> float:
    """Switch load-balancing loss alpha E sum_i f_i P_i ([MM] section 3.1; [FM] section 3.2)."""
    f = np.asarray(f, np.float64)
    P = np.asarray(P, np.float64)
    return float(alpha * len(f) * np.sum(f * P))


def load_stats(idx: np.ndarray, l32: np.ndarray, E: int, scoring: str, alpha: float) -> Dict[str, np.ndarray]:
    """Forward load statistics of one batch, by their definitions:
      f_e = (1/T) #{tokens that chose e}                 ([MM] section 3.1; [FM] section 3.2)
      P_e = (1/T) sum_t s_e(x_t), s the layer's scores (softmax over all E, or sigmoid)
      L_aux = alpha E sum_e f_e P_e
      max/mean load = max_e c_e / (T k / E), c_e the assignments of expert e ([T26] "Routing
                     creates an assignment problem": maximum load divided by mean load)."""
    T, k = idx.shape
    c = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            c[idx[t, j]] += 1
    f = c / T
    P = scores(l32, scoring).mean(axis=0)
    return {"f": f, "P": P, "aux_loss": aux_loss(f, P, alpha), "max_over_mean": float(c.max() / (T * k / E)),
            "counts": c}


def dispatch_bytes(T: int, k: int, d: int, elem_bytes: int) -> int:
    """Bytes of one dispatch exchange: T k d elements ([FM] section 4.2)."""
    return T * k * d * elem_bytes


def min_adjacent_gap(key32: np.ndarray, m: int) -> np.ndarray:
    """Per row, the smallest difference between consecutive keys among the m largest (ranks
    1..m in descending order).  Used to redraw tokens whose top-k could flip on rounding."""
    key = np.asarray(key32, np.float32).astype(np.float64)
    srt = -np.sort(-key, axis=-1)[:, :m]
    if m < 2:
        return np.full(key.shape[0], np.inf)
    return np.min(srt[:, :-1] - srt[:, 1:], axis=-1)
