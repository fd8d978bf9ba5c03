"""GPU parity where the 2e-2 rms rule cannot hold for any bfloat16 evaluation.

The bf16 layer stores the SwiGLU output h in bfloat16 between its two GEMMs (as the x_perm
rows and y are stored).  With a short W3 contraction (small d_ff) and outputs far above their
rms, that one rounding of h alone moves y by more than 2e-2 rms(ref) against the float64
oracle.  The other parity suites therefore avoid such shapes.  Here they are run on purpose,
and two things are checked:
  - the layer against the oracle's arithmetic with h rounded once to bfloat16 (through float32,
    as the kernels round their float32 accumulators), under the usual output rule;
  - that the layer's error against the plain float64 oracle is the one that rounding explains:
    at most the model's own error plus a quarter of the rule.
"""
import os

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import Case
from oracle import moe_oracle as orc

from gpu_util import RECORDS, check_close, layer_out_err, max_rel_err, require_cuda, tdtype, to_dev, upload_experts

pytestmark = pytest.mark.gpu

S = wl.MoEShape
SHAPES = [
    # heavy dropping with a strong bias: outputs up to ~12 x rms, W3 contraction of 128
    S("cap_skewed_e64_dff128", T=512, d=256, d_ff=128, E=64, k=8, dtype="bf16", scoring="softmax",
      logit_bias_std=1.5, capacity_factor=1.25),
    # expert choice over 256 experts with a W3 contraction of 64: outputs up to ~17 x rms
    S("ec_e256_dff64", T=1024, d=256, d_ff=64, E=256, k=8, dtype="bf16", scoring="expert_choice"),
]


def _bf16(a64):
    """float64 values rounded to float32, then to bfloat16 (round to nearest even), as float64."""
    return wl.to_f64(wl.bf16_round(np.asarray(a64, np.float32)), "bf16")


def _expert_bf16_h(X64, W1, W2, W3):
    """One SwiGLU expert with its hidden activation h stored in bfloat16."""
    return _bf16((X64 @ W1) * orc.silu(X64 @ W2)) @ W3


def _model(case, ref):
    """The oracle's layer on its own routing, with every h (routed and shared) rounded once."""
    s, get_w = case.shape, case.get_w
    x64 = case.f64(case.x)
    off = ref["offsets"]
    y_perm = np.zeros((ref["perm_tok"].shape[0], s.d), np.float64)
    for e in range(s.E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            y_perm[a:b] = _expert_bf16_h(x64[ref["perm_tok"][a:b]], get_w("W1", e), get_w("W2", e), get_w("W3", e))
    ys = None
    if s.n_shared:
        ys = sum(_expert_bf16_h(x64, get_w("Ws1", i), get_w("Ws2", i), get_w("Ws3", i)) for i in range(s.n_shared))
    if case.ec_m is None:
        return orc.combine(y_perm, ref["inv_pos"], ref["gate"], ys)
    y = np.zeros((s.T, s.d), np.float64)
    for e in range(s.E):
        p = ref["pos_of"][:, e]
        took = p >= 0
        y[took] += ref["gate"][p[took]][:, None] * y_perm[p[took]]
    return y if ys is None else y + ys


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_layer_matches_bf16_h_model(shape):
    moe = require_cuda()
    s = shape
    case = Case(s, 0)
    ref = case.forward()
    W = upload_experts(s, 0, keep=range(s.E))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    moe.forward(cfg, to_dev(case.x, s), to_dev(case.W_g, s), W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb,
                Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"))
    assert moe.get_device_error() == 0
    y_model = _model(case, ref)
    check_close(y, y_model, s, "y vs the bf16-h model")
    got = y.float().cpu().numpy().astype(np.float64)
    err_gpu = layer_out_err(got, ref["y"], s)
    err_model = layer_out_err(_bf16(y_model), ref["y"], s)
    RECORDS.append((os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                    "y vs the float64 oracle (the bf16-h model's own error %.3g)" % err_model,
                    max_rel_err(got, ref["y"]), err_gpu, err_model + 0.25 * 2e-2))
    assert err_gpu <= err_model + 0.25 * 2e-2, (err_gpu, err_model)
