"""Seeded oracle cases: workload inputs whose routing is unambiguous in float32.

TEST INFRASTRUCTURE (see moe_oracle.py): used by the tests, smoke() and bench.py's CPU legs.

The top-k decision is an integer result decided by float32 logits.  The GPU sums the d
products in another order than the oracle, so two logits closer than the rounding noise
could swap.  A token row is therefore redrawn (attempt + 1 in the generator key) until
all adjacent gaps among its m = min(k+1, E) largest selection keys are at least `min_gap`
in the oracle's float32 logits.  Then the chosen set and its order are unique and must match
bit for bit.
"""
from __future__ import annotations

import functools
from typing import Optional

import numpy as np

import workloads as wl
from . import moe_oracle as orc


def gapped_attempts(shape: wl.MoEShape, seed: int = 0, min_gap: float = 1e-3,
                    sel_bias: Optional[np.ndarray] = None, max_rounds: int = 200) -> np.ndarray:
    """Per-token attempt counters for which every token's top-(k+1) keys are >= min_gap apart."""
    T, k, E = shape.T, shape.k, shape.E
    m = min(k + 1, E)
    Wg = wl.to_f64(wl.gen_router(shape, seed), shape.dtype)
    lb = wl.gen_logit_bias(shape, seed)
    attempts = np.zeros(T, dtype=np.int64)
    rows = np.arange(T)
    x = wl.gen_x(shape, seed, attempts)
    for _ in range(max_rounds):
        xr = wl.to_f64(x[rows], shape.dtype)
        l = orc.router_logits(xr, Wg, lb)
        key = orc.selection_keys(l, shape.scoring, sel_bias)
        bad = rows[orc.min_adjacent_gap(key, m) < min_gap]
        if bad.size == 0:
            return attempts
        attempts[bad] += 1
        x[bad] = wl.gen_x(shape, seed, attempts, rows=bad)
        rows = bad
    raise RuntimeError("could not separate the router logits of %d tokens" % rows.size)


def expert_choice_gapped_attempts(shape: wl.MoEShape, m: int, seed: int = 0, min_rel_gap: float = 1e-4,
                                  max_rounds: int = 200) -> np.ndarray:
    """Per-token attempt counters for expert choice: for every expert, the m-th and (m+1)-th
    largest float32 scores s[:, e] differ by at least min_rel_gap of the m-th, so every
    expert's set of m tokens is unique (the GPU's scores differ from the oracle's by a few
    ulps).  The two tokens at an expert's boundary are redrawn until that holds."""
    T, E = shape.T, shape.E
    Wg = wl.to_f64(wl.gen_router(shape, seed), shape.dtype)
    lb = wl.gen_logit_bias(shape, seed)
    attempts = np.zeros(T, dtype=np.int64)
    x = wl.gen_x(shape, seed, attempts)
    if m >= T:
        return attempts
    for _ in range(max_rounds):
        l = orc.router_logits(wl.to_f64(x, shape.dtype), Wg, lb)
        key = orc.scores(l, "softmax").astype(np.float32).astype(np.float64)
        bad = set()
        for e in range(E):
            order = np.argsort(-key[:, e], kind="stable")
            a, b = key[order[m - 1], e], key[order[m], e]
            if a - b < min_rel_gap * a:
                bad.update((int(order[m - 1]), int(order[m])))
        if not bad:
            return attempts
        rows = np.array(sorted(bad))
        attempts[rows] += 1
        x[rows] = wl.gen_x(shape, seed, attempts, rows=rows)
    raise RuntimeError("could not separate the expert-choice boundaries")


class Case:
    """Host inputs of one workload plus float64 views for the oracle.

    Expert matrices are drawn lazily per expert (and cached), so sampled checks on the
    largest workloads only materialise the experts they touch."""

    def __init__(self, shape: wl.MoEShape, seed: int = 0, gap: bool = True,
                 sel_bias: Optional[np.ndarray] = None):
        self.shape = shape
        self.seed = seed
        self.sel_bias = sel_bias
        self.ec_m = (orc.expert_choice_slots(shape.T, shape.k, shape.E, shape.capacity_factor)
                     if shape.scoring == "expert_choice" else None)
        if not gap:
            self.attempts = np.zeros(shape.T, np.int64)
        elif self.ec_m is not None:
            self.attempts = expert_choice_gapped_attempts(shape, self.ec_m, seed)
        else:
            self.attempts = gapped_attempts(shape, seed, sel_bias=sel_bias)
        self.x = wl.gen_x(shape, seed, self.attempts)
        self.W_g = wl.gen_router(shape, seed)
        self.logit_bias = wl.gen_logit_bias(shape, seed)
        self._cache = {}

    def f64(self, a: np.ndarray) -> np.ndarray:
        return wl.to_f64(a, self.shape.dtype)

    def stored_expert(self, name: str, e: int) -> np.ndarray:
        key = (name, e)
        if key not in self._cache:
            self._cache[key] = wl.gen_expert(self.shape, name, e, self.seed)
        return self._cache[key]

    @functools.lru_cache(maxsize=64)
    def _w64(self, name: str, e: int) -> np.ndarray:
        return self.f64(self.stored_expert(name, e))

    def get_w(self, name: str, e: int) -> np.ndarray:
        return self._w64(name, e)

    def route(self):
        s = self.shape
        return orc.route(self.f64(self.x), self.f64(self.W_g), s.k, s.scoring,
                         self.logit_bias, self.sel_bias)

    def forward(self):
        s = self.shape
        if self.ec_m is not None:
            return orc.expert_choice_forward(self.f64(self.x), self.f64(self.W_g), self.get_w, s.E, self.ec_m,
                                             self.logit_bias, s.n_shared)
        return orc.forward(self.f64(self.x), self.f64(self.W_g), self.get_w, s.E, s.k, s.scoring,
                           self.logit_bias, self.sel_bias, s.n_shared, s.capacity_factor)
