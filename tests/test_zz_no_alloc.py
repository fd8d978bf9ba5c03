"""moe_dispatch_static, the dispatch call that allocates nothing.

Some callers cannot allocate device memory: a plug-in whose host framework owns all device
memory and hands it no scratch, or a latency-critical path that must not call cudaMalloc
(which may synchronise the device).  For them the library keeps dispatch's scratch, the
per-chunk count and position tables, in a fixed 1 MiB device array of its own.  This checks,
through the C ABI, that two calls in a row give exactly what the workspace-based moe_dispatch
gives (dispatch is integer work, so the tolerance is zero).  Every case here takes the chunked
dispatch path (more than 16384 pairs, or more than 256 experts), the one that uses the array;
one case fills the array exactly.  The refusal of larger sizes needs no GPU and is checked in
test_abi_host.py.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import require_cuda

pytestmark = pytest.mark.gpu

CASES = [  # (T, d, E, k, capacity factor)
    (8192, 128, 256, 8, 0.0),      # DeepSeek-V3-shaped routing: 65536 pairs over 256 experts
    (16384, 64, 256, 8, 0.0),      # ceil(T k / 256) * E = 131072: both tables fill the 1 MiB array
    (40000, 64, 8, 2, 0.0),        # Mixtral-shaped routing, 80000 pairs
    (8192, 64, 64, 8, 1.25),       # capacity: pairs beyond ceil(T k c / E) per expert are dropped
    (333, 64, 300, 6, 0.0),        # few pairs, but more than 256 experts
]


def _outputs(T, d, E, k):
    def z(*shape):
        return torch.full(shape, -7, dtype=torch.int32, device="cuda")
    return dict(counts=z(E), offsets=z(E + 1), perm=z(T * k), inv=z(T, k),
                x_perm=torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("T,d,E,k,cf", CASES)
def test_static_dispatch_matches_workspace_dispatch(T, d, E, k, cf):
    moe = require_cuda()
    rng = np.random.default_rng(T + E)
    # k distinct experts per token, skewed so that some experts overflow a capacity
    w = rng.random((T, E)) * np.linspace(1.0, 3.0, E)[None, :]
    idx_np = np.argsort(-w, axis=1)[:, :k].astype(np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    x = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    cfg = moe.config(T, d, 64, E, k, capacity_factor=cf)
    ref = _outputs(T, d, E, k)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    moe.dispatch(cfg, idx, x, ref["counts"], ref["offsets"], ref["perm"], ref["inv"], ref["x_perm"], ws)
    assert moe.last_launch_count() == 4          # histogram, scan, permute, gather: the chunked path
    if cf > 0:
        assert int((ref["inv"] < 0).sum()) > 0   # the capacity did drop pairs
    for _ in range(2):
        got = _outputs(T, d, E, k)
        moe.dispatch_static(cfg, idx, x, got["counts"], got["offsets"], got["perm"], got["inv"], got["x_perm"])
        assert moe.last_launch_count() == 4
        torch.cuda.synchronize()
        for name in ref:
            assert torch.equal(got[name], ref[name]), name
    assert moe.get_device_error() == 0
