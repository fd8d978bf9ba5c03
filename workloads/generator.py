"""Seeded synthetic inputs for the top-k MoE FFN forward pass.

This module is shared by the tests, the benchmark and the CPU oracle's callers.  It only
draws random numbers and rounds them to the storage dtype; it holds none of the MoE
arithmetic (no logits, no scores, no selection, no expert evaluation).

Every tensor is drawn from a counter-based generator: numpy's Philox4x32-10 keyed by
(seed, tensor id, attempt, index), so any slice (one token row, one expert's matrix) can be
regenerated on its own, in any order, on any thread, and always comes out the same.

Distributions follow the workload descriptions: token activations x ~ N(0, 1); every weight
matrix ~ N(0, 1/fan_in) (variance 1/fan_in, i.e. standard deviation 1/sqrt(fan_in)); the
per-expert logit bias of the skewed workload ~ N(0, 1.5) read as standard deviation 1.5.
Values are drawn as float32 standard normals, scaled in float32, and stored either as
float32 or rounded to bfloat16 with round-to-nearest-even (kept as uint16 bit patterns,
since numpy has no bfloat16 type).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterable, Optional

import numpy as np

# Tensor ids: part of the generator key, so each tensor has its own stream.
TENSOR_IDS = {
    "x": 1, "W_g": 2, "logit_bias": 3, "W1": 4, "W2": 5, "W3": 6,
    "Ws1": 7, "Ws2": 8, "Ws3": 9, "sel_bias": 10,
}


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Sizes and options of one MoE FFN layer workload."""
    name: str
    T: int            # tokens
    d: int            # model width
    d_ff: int         # routed expert width
    E: int            # routed experts
    k: int            # experts chosen per token
    dtype: str        # "f32" or "bf16" (x, W_g, expert weights and y)
    scoring: str      # "softmax" (softmax over E, top-k, renormalise) or "sigmoid"
    n_shared: int = 0
    d_ff_shared: int = 0
    logit_bias_std: float = 0.0   # > 0: a per-expert bias added to the logits
    capacity_factor: float = 0.0  # > 0: each expert keeps at most ceil(T k c / E) assignments

    def replace(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)


# The five workloads the library is measured and checked on.
WORKLOADS: Dict[str, MoEShape] = {
    # Tiny fp32 layer that the oracle runs in well under a second.
    "tiny_f32": MoEShape("tiny_f32", T=64, d=128, d_ff=256, E=8, k=2, dtype="f32",
                         scoring="softmax"),
    # Mixtral-8x7B-shaped prefill layer (d=4096, 8 experts, top-2).
    "mixtral_prefill": MoEShape("mixtral_prefill", T=4096, d=4096, d_ff=14336, E=8, k=2,
                                dtype="bf16", scoring="softmax"),
    # Same layer at decode batch size: weight-bandwidth bound.
    "mixtral_decode": MoEShape("mixtral_decode", T=16, d=4096, d_ff=14336, E=8, k=2,
                               dtype="bf16", scoring="softmax"),
    # Hunyuan-A13B-shaped fine-grained layer, load skewed by a per-expert logit bias.
    "hunyuan_a13b": MoEShape("hunyuan_a13b", T=8192, d=4096, d_ff=3072, E=64, k=8,
                             dtype="bf16", scoring="softmax", logit_bias_std=1.5),
    # DeepSeek-V3-shaped layer: 256 routed experts with sigmoid scores, top-8, one shared.
    "deepseek_v3": MoEShape("deepseek_v3", T=8192, d=7168, d_ff=2048, E=256, k=8,
                            dtype="bf16", scoring="sigmoid", n_shared=1, d_ff_shared=2048),
}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _key(seed: int, tensor: str, index: int, attempt: int = 0) -> np.ndarray:
    tid = TENSOR_IDS[tensor]
    assert 0 <= index < (1 << 32) and 0 <= attempt < (1 << 16)
    hi = (tid << 48) | (attempt << 32) | index
    return np.array([seed & ((1 << 64) - 1), hi], dtype=np.uint64)


def standard_normal(seed: int, tensor: str, index: int, n: int, attempt: int = 0) -> np.ndarray:
    """n float32 draws of N(0, 1) from the stream keyed by (seed, tensor, attempt, index)."""
    g = np.random.Generator(np.random.Philox(key=_key(seed, tensor, index, attempt)))
    return g.standard_normal(n, dtype=np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values (float32 array, or uint16 bfloat16 bits) as float64."""
    if dtype == "bf16":
        return bf16_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _store(z: np.ndarray, std: float, dtype: str) -> np.ndarray:
    v = z * np.float32(std)
    return bf16_round(v) if dtype == "bf16" else v.astype(np.float32)


def gen_matrix(seed: int, tensor: str, index: int, rows: int, cols: int, std: float,
               dtype: str, attempt: int = 0) -> np.ndarray:
    """One [rows, cols] matrix drawn from its own stream, stored in `dtype`."""
    z = standard_normal(seed, tensor, index, rows * cols, attempt)
    return _store(z, std, dtype).reshape(rows, cols)


def gen_x(shape: MoEShape, seed: int = 0, attempts: Optional[np.ndarray] = None,
          rows: Optional[Iterable[int]] = None) -> np.ndarray:
    """Token activations x [T, d] ~ N(0, 1); row t is keyed by (t, attempts[t]).

    `attempts` lets a caller redraw individual token rows (a redrawn row uses attempt+1).
    `rows` restricts the output to those token rows (in the given order)."""
    T, d = shape.T, shape.d
    idx = list(range(T)) if rows is None else list(rows)
    att = np.zeros(T, dtype=np.int64) if attempts is None else np.asarray(attempts)
    out = np.empty((len(idx), d), dtype=np.uint16 if shape.dtype == "bf16" else np.float32)

    def one(i):
        t = idx[i]
        out[i] = gen_matrix(seed, "x", t, 1, d, 1.0, shape.dtype, int(att[t]))[0]

    if len(idx) > 256:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(len(idx))))
    else:
        for i in range(len(idx)):
            one(i)
    return out


def gen_router(shape: MoEShape, seed: int = 0) -> np.ndarray:
    """Router matrix W_g [d, E] ~ N(0, 1/d)."""
    return gen_matrix(seed, "W_g", 0, shape.d, shape.E, 1.0 / np.sqrt(shape.d), shape.dtype)


def gen_logit_bias(shape: MoEShape, seed: int = 0) -> Optional[np.ndarray]:
    """Per-expert logit bias [E] float32 ~ N(0, std^2), or None when the workload has none."""
    if shape.logit_bias_std <= 0:
        return None
    return standard_normal(seed, "logit_bias", 0, shape.E) * np.float32(shape.logit_bias_std)


def gen_sel_bias(shape: MoEShape, std: float, seed: int = 0) -> np.ndarray:
    """A per-expert selection bias [E] float32 ~ N(0, std^2) (a state of the balancing
    controller, for tests that route with such a bias)."""
    return standard_normal(seed, "sel_bias", 0, shape.E) * np.float32(std)


def expert_dims(shape: MoEShape, which: str):
    """(rows, cols, std) of one expert matrix: W1/W2 are [d, d_ff], W3 is [d_ff, d]."""
    if which in ("W1", "W2"):
        return shape.d, shape.d_ff, 1.0 / np.sqrt(shape.d)
    if which == "W3":
        return shape.d_ff, shape.d, 1.0 / np.sqrt(shape.d_ff)
    if which in ("Ws1", "Ws2"):
        return shape.d, shape.d_ff_shared, 1.0 / np.sqrt(shape.d)
    if which == "Ws3":
        return shape.d_ff_shared, shape.d, 1.0 / np.sqrt(shape.d_ff_shared)
    raise KeyError(which)


def gen_expert(shape: MoEShape, which: str, e: int, seed: int = 0) -> np.ndarray:
    """Expert e's matrix `which` (W1, W2, W3 for routed experts; Ws1, Ws2, Ws3 for shared)."""
    rows, cols, std = expert_dims(shape, which)
    return gen_matrix(seed, which, e, rows, cols, std, shape.dtype)


def gen_experts(shape: MoEShape, which: str, seed: int = 0,
                experts: Optional[Iterable[int]] = None) -> np.ndarray:
    """Stacked matrices [n, rows, cols] for the given experts (all of them by default)."""
    n_all = shape.n_shared if which.startswith("Ws") else shape.E
    ids = list(range(n_all)) if experts is None else list(experts)
    rows, cols, _ = expert_dims(shape, which)
    out = np.empty((len(ids), rows, cols), dtype=np.uint16 if shape.dtype == "bf16" else np.float32)

    def one(i):
        out[i] = gen_expert(shape, which, ids[i], seed)

    if len(ids) > 1 and rows * cols * len(ids) > (1 << 22):
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(len(ids))))
    else:
        for i in range(len(ids)):
            one(i)
    return out


def workload_arrays(shape: MoEShape, seed: int = 0, attempts: Optional[np.ndarray] = None,
                    with_experts: bool = True) -> Dict[str, np.ndarray]:
    """All host inputs of one workload (experts optional, they dominate the size)."""
    out = {"x": gen_x(shape, seed, attempts), "W_g": gen_router(shape, seed)}
    lb = gen_logit_bias(shape, seed)
    if lb is not None:
        out["logit_bias"] = lb
    if with_experts:
        for w in ("W1", "W2", "W3"):
            out[w] = gen_experts(shape, w, seed)
        if shape.n_shared > 0:
            for w in ("Ws1", "Ws2", "Ws3"):
                out[w] = gen_experts(shape, w, seed)
    return out
