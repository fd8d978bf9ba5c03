"""The dynamic tile schedule of the CTA-pair GEMMs under concurrency and reuse.

Each launch of a CTA-pair GEMM takes its tiles from a counter pair of its own (a slot of a
256-slot array in the library's device image) and resets it before it completes.  These tests
check that two layers in flight on two streams at once (each with its own workspace) give
exactly the results they give alone, and that more launches than there are slots (the slots
wrap around) keep giving the same results.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import require_cuda, tdtype, to_dev, upload_experts

pytestmark = pytest.mark.gpu

S = wl.MoEShape
# ~1024 rows per expert: the token-wide kernel (both GEMMs); ~256 rows: the same with wide
# tiles; a shared expert: the 256-row pair kernel on its dense block.
SHAPES = [
    S("sched_big", T=2048, d=256, d_ff=384, E=4, k=2, dtype="bf16", scoring="softmax"),
    S("sched_wide_shared", T=512, d=256, d_ff=256, E=16, k=8, dtype="bf16", scoring="sigmoid",
      n_shared=1, d_ff_shared=128),
]


def _setup(moe, s, seed):
    W = upload_experts(s, 0)
    x = to_dev(wl.gen_x(s, seed), s)
    Wg = to_dev(wl.gen_router(s, 0), s)
    cfg = moe.config_from_shape(s)
    return W, x, Wg, cfg


def _forward(moe, s, W, x, Wg, cfg, stream=None, ws=None, y=None):
    ws = ws if ws is not None else torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    y = y if y is not None else torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    moe.forward(cfg, x, Wg, W["W1"], W["W2"], W["W3"], y, ws, Ws1=W.get("Ws1"), Ws2=W.get("Ws2"),
                Ws3=W.get("Ws3"), stream=stream)
    return y, ws


@pytest.mark.parametrize("s", SHAPES, ids=[s.name for s in SHAPES])
def test_two_streams_in_flight_match_one_stream(s):
    moe = require_cuda()
    W, xa, Wg, cfg = _setup(moe, s, 0)
    xb = to_dev(wl.gen_x(s, 7), s)
    ref_a, _ = _forward(moe, s, W, xa, Wg, cfg)
    ref_b, _ = _forward(moe, s, W, xb, Wg, cfg)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = [_forward(moe, s, W, xa, Wg, cfg, stream=streams[0]), _forward(moe, s, W, xb, Wg, cfg, stream=streams[1])]
    for _ in range(3):
        for i, (x, st) in enumerate(((xa, streams[0]), (xb, streams[1]))):
            y, ws = bufs[i]
            _forward(moe, s, W, x, Wg, cfg, stream=st, ws=ws, y=y)
    for st in streams:
        st.synchronize()
    assert moe.get_device_error() == 0
    assert torch.equal(bufs[0][0], ref_a)
    assert torch.equal(bufs[1][0], ref_b)


def test_more_launches_than_counter_slots():
    moe = require_cuda()
    s = SHAPES[0]
    W, x, Wg, cfg = _setup(moe, s, 0)
    first, ws = _forward(moe, s, W, x, Wg, cfg)
    y = torch.empty_like(first)
    for _ in range(150):   # two CTA-pair launches per layer: 300 launches > 256 slots
        _forward(moe, s, W, x, Wg, cfg, ws=ws, y=y)
    torch.cuda.synchronize()
    assert moe.get_device_error() == 0
    assert torch.equal(y, first)
    assert np.isfinite(y.float().cpu().numpy()).all()
