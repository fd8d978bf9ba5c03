"""The bounds-checking build (libmoe_debug.so, compiled with MOE_DEBUG_BOUNDS).

Its kernels also report, in bit ERR_BOUNDS of the device error word, any index they read from
offsets, perm_tok, inv_pos or pos_of that is out of range (and skip that access, as the normal
build does silently).  A correct run must leave the word at 0: the debug build runs the whole
layer on small cases through the C ABI, in a child process that loads it (MOE_LIBRARY=debug),
against the oracle.  A combine call given one out-of-range position shows the report: the
debug build sets the bit, the normal build skips the position without a word.  Nothing is
ever read or written out of bounds: the checked index is skipped before it is used.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_util import require_cuda

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ERR_BOUNDS = 1 << 6

CHILD = r'''
import os, sys
sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import workloads as wl
from oracle import Case
from mixture_experts_sparse_02_b300 import moe
from gpu_util import check_close, tdtype, to_dev, upload_experts
assert moe.LIB_PATH.endswith("libmoe_debug.so"), moe.LIB_PATH
S = wl.MoEShape
shapes = [
    S("dbg_ragged", T=300, d=256, d_ff=200, E=8, k=2, dtype="bf16", scoring="softmax", logit_bias_std=1.0),
    S("dbg_shared_e64", T=200, d=192, d_ff=128, E=64, k=6, dtype="bf16", scoring="sigmoid", n_shared=1, d_ff_shared=64),
    S("dbg_capacity", T=1000, d=256, d_ff=192, E=8, k=2, dtype="bf16", scoring="softmax", logit_bias_std=0.7,
      capacity_factor=1.25),
    S("dbg_chunked", T=4500, d=64, d_ff=64, E=8, k=4, dtype="bf16", scoring="softmax"),
    S("dbg_f32", T=70, d=40, d_ff=24, E=48, k=5, dtype="f32", scoring="softmax", logit_bias_std=1.0),
    S("dbg_expert_choice", T=128, d=128, d_ff=64, E=8, k=2, dtype="bf16", scoring="expert_choice"),
]
for s in shapes:
    case = Case(s, 0)
    ref = case.forward()
    W = upload_experts(s, 0)
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    moe.forward(cfg, to_dev(case.x, s), to_dev(case.W_g, s), W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb,
                Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"))
    word = moe.get_device_error()
    assert word == 0, (s.name, hex(word))
    check_close(y, ref["y"], s)
    print("%s: word 0, %d kernels" % (s.name, moe.last_launch_count()))
# one out-of-range position handed to moe_combine: reported, and skipped
s = shapes[0]
T, k, d = s.T, s.k, s.d
cfg = moe.config_from_shape(s)
y_perm = torch.ones((T * k, d), dtype=torch.float32, device="cuda")
inv = torch.arange(T * k, dtype=torch.int32, device="cuda").reshape(T, k)
inv[7, 1] = T * k + 5
gate = torch.full((T, k), 0.5, dtype=torch.float32, device="cuda")
y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
moe.combine(cfg, y_perm, inv, gate, y)
word = moe.get_device_error()
assert word & ERR_BOUNDS_BIT, hex(word)
assert float(y[7, 0]) == 0.5 and float(y[8, 0]) == 1.0
print("bad position: word %s" % hex(word))
'''.replace("ERR_BOUNDS_BIT", str(ERR_BOUNDS))


def test_debug_build_runs_clean_and_reports_bad_indices():
    require_cuda()
    lib = os.path.join(ROOT, "mixture_experts_sparse_02_b300", "libmoe_debug.so")
    assert os.path.exists(lib), "libmoe_debug.so is not built (python -m mixture_experts_sparse_02_b300.build --debug-bounds)"
    env = dict(os.environ, MOE_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "bad position" in r.stdout


def test_normal_build_skips_a_bad_position_silently():
    moe = require_cuda()
    T, k, d = 64, 2, 128
    cfg = moe.config(T, d, 64, 8, k)
    y_perm = torch.ones((T * k, d), dtype=torch.float32, device="cuda")
    inv = torch.arange(T * k, dtype=torch.int32, device="cuda").reshape(T, k)
    inv[7, 1] = T * k + 5
    gate = torch.full((T, k), 0.5, dtype=torch.float32, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.combine(cfg, y_perm, inv, gate, y)
    assert moe.get_device_error() == 0
    assert float(y[7, 0]) == 0.5 and float(y[8, 0]) == 1.0
