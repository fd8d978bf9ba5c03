"""Helpers shared by the GPU tests: upload seeded inputs, run the library, compare to the oracle."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np
import pytest
import torch

import workloads as wl

BF16_TOL = 2e-2    # max|err| <= 2e-2 * rms(ref) for bfloat16 weights and activations
F32_TOL = 1e-4     # max|err| <= 1e-4 * rms(ref) for the float32 layer
GATE_ATOL = 1e-5   # gates: computed in float32 on the GPU from the same float32 logits as the oracle


def require_cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for a gpu-marked test")
    from mixture_experts_sparse_02_b300 import moe   # fails loudly if libmoe.so is missing
    return moe


def tdtype(shape) -> torch.dtype:
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def to_dev(a: np.ndarray, shape) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if shape.dtype == "bf16" and a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to("cuda")


def from_dev_stored(t: torch.Tensor, shape) -> np.ndarray:
    """Device tensor (bf16 or f32) back to the stored host form (uint16 bits or float32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.uint16).numpy() if hasattr(torch, "uint16") else t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def upload_experts(shape, seed: int = 0, keep: Iterable[int] = (), keep_shared: bool = True) -> Dict:
    """Draw every expert matrix, copy it to the device, and keep host copies of the experts in
    `keep` (the ones the oracle needs).  Returns {"W1": tensor [E, d, d_ff], ..., "host": {...}}."""
    dt = tdtype(shape)
    out = {}
    keep = set(int(e) for e in keep)
    host = {}
    jobs = [(w, e) for w in ("W1", "W2", "W3") for e in range(shape.E)]
    if shape.n_shared > 0:
        jobs += [(w, s) for w in ("Ws1", "Ws2", "Ws3") for s in range(shape.n_shared)]
    for w in ("W1", "W2", "W3", "Ws1", "Ws2", "Ws3"):
        n = shape.n_shared if w.startswith("Ws") else shape.E
        if n == 0:
            continue
        rows, cols, _ = wl.expert_dims(shape, w)
        out[w] = torch.empty((n, rows, cols), dtype=dt, device="cuda")

    def one(job):
        w, e = job
        a = wl.gen_expert(shape, w, e, 0 if seed is None else seed)
        out[w][e].copy_(torch.from_numpy(a).view(dt) if shape.dtype == "bf16" else torch.from_numpy(a))
        if (w.startswith("Ws") and keep_shared) or (not w.startswith("Ws") and e in keep):
            host[(w, e)] = a

    with ThreadPoolExecutor(16) as ex:
        list(ex.map(one, jobs))
    torch.cuda.synchronize()
    out["host"] = host
    return out


def host_weight_fn(host: Dict, shape):
    def get(name, e):
        return wl.to_f64(host[(name, e)], shape.dtype)
    return get


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return float(np.max(np.abs(got.astype(np.float64) - ref))) / max(rms, 1e-300)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bfloat16 values (8 significant bits): the largest
    distance between a real number and its round-to-nearest bfloat16 value v."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, np.finfo(np.float64).tiny)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def layer_out_err(got: np.ndarray, ref: np.ndarray, shape) -> float:
    """Error of a stored output (the layer output y, or the expert outputs y_perm) against the
    oracle, in units of rms(ref).

    float32 layers: max|y - ref| / rms(ref).  bfloat16 layers: the value is stored in
    bfloat16, so it carries up to half a bfloat16 ulp of its own value beyond any arithmetic
    error; that rounding alone reaches ~2.4% of rms(ref) at the largest outputs of these
    shapes.  The rule is therefore applied to the value before that final rounding, through
    the lower bound max(|y - ref| - ulp(y)/2) / rms(ref): it can only fail if the unrounded
    value misses the rule."""
    got = np.asarray(got, np.float64)
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    d = np.abs(got - ref)
    if shape.dtype == "bf16":
        d = d - bf16_half_ulp(got)
    return float(np.max(d)) / max(rms, 1e-300)


def y_tol(shape) -> float:
    return BF16_TOL if shape.dtype == "bf16" else F32_TOL


# (test, what, raw max|err|/rms, figure the rule is applied to, tolerance) of every check_close
# call in this session; tests/conftest.py prints a summary at the end of the run.
RECORDS: List[Tuple[str, str, float, float, float]] = []


def check_close(got, ref: np.ndarray, shape, what: str = "y") -> Tuple[float, float]:
    """Assert the output rule of the layer's dtype on a result (device tensor or array) against
    the oracle and record both figures: the raw max|err|/rms(ref), and the figure the rule is
    applied to (a bfloat16 tensor: after half a bfloat16 ulp of the stored value, see
    layer_out_err; a float32 tensor, such as y_perm: the raw figure)."""
    stored_bf16 = isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16
    if isinstance(got, torch.Tensor):
        got = dev_to_f64(got)
    got = np.asarray(got, np.float64)
    raw = max_rel_err(got, ref)
    err = layer_out_err(got, ref, shape) if stored_bf16 else raw
    tol = y_tol(shape)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORDS.append((test, what, raw, err, tol))
    assert err <= tol, ("%s: max|err| = %.3g rms(ref) raw, %.3g rms(ref) after half a bf16 ulp of the stored "
                        "value; tolerance %g" % (what, raw, err, tol))
    return raw, err
