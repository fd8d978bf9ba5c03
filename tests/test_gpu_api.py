"""The measurement entry points behave like moe_forward: moe_forward_host (x and y in host
memory, copies inside the call), moe_forward_host_async (the same without the wait, on two
streams) and moe_forward_profiled (events at the stage boundaries)."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import Case

from gpu_util import check_close, require_cuda, tdtype, to_dev, upload_experts

pytestmark = pytest.mark.gpu

S = wl.MoEShape
SHAPES = [
    S("api_bf16_shared", T=300, d=256, d_ff=192, E=16, k=2, dtype="bf16", scoring="sigmoid", n_shared=1,
      d_ff_shared=128, logit_bias_std=1.0),
    S("api_f32", T=64, d=64, d_ff=96, E=8, k=2, dtype="f32", scoring="softmax"),
    S("api_expert_choice", T=256, d=128, d_ff=128, E=8, k=2, dtype="bf16", scoring="expert_choice"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_host_and_profiled_match_forward(shape):
    moe = require_cuda()
    s = shape
    case = Case(s, 0)
    ref = case.forward()
    W = upload_experts(s, 0, keep=range(s.E))
    x, Wg = to_dev(case.x, s), to_dev(case.W_g, s)
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    Ws = dict(Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    moe.forward(cfg, x, Wg, W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb, **Ws)
    assert moe.get_device_error() == 0
    check_close(y, ref["y"], s)
    # host buffers: pinned x in, pinned y out; the call waits for its stream
    xh = x.cpu().pin_memory()
    yh = torch.zeros((s.T, s.d), dtype=tdtype(s)).pin_memory()
    moe.forward_host(cfg, xh, Wg, W["W1"], W["W2"], W["W3"], yh, ws, logit_bias=lb, **Ws)
    assert torch.equal(yh, y.cpu())
    # the asynchronous call on two streams with two workspaces, as a serving loop would
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [ws, torch.empty_like(ws)]
    ys = [torch.zeros((s.T, s.d), dtype=tdtype(s)).pin_memory() for _ in range(2)]
    for i in range(4):
        moe.forward_host_async(cfg, xh, Wg, W["W1"], W["W2"], W["W3"], ys[i % 2], wss[i % 2], logit_bias=lb,
                               stream=streams[i % 2], **Ws)
    for st in streams:
        st.synchronize()
    assert torch.equal(ys[0], y.cpu()) and torch.equal(ys[1], y.cpu())
    # events at the stage boundaries: same output, the 7 events recorded in order
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_NUM_STAGES + 1)]
    y2 = torch.empty_like(y)
    moe.forward(cfg, x, Wg, W["W1"], W["W2"], W["W3"], y2, ws, logit_bias=lb, events=evs, **Ws)
    torch.cuda.synchronize()
    assert torch.equal(y2, y)
    spans = [evs[i].elapsed_time(evs[i + 1]) for i in range(moe.MOE_NUM_STAGES)]
    assert all(t >= 0 for t in spans)
    assert abs(sum(spans) - evs[0].elapsed_time(evs[-1])) < 1e-3 + 1e-3 * sum(spans)
