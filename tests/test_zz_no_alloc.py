"""moe_dispatch_static, the dispatch call that allocates nothing.

Some callers cannot allocate device memory (a plug-in whose host framework owns all device
memory, a latency-critical path that must not call cudaMalloc).  For them the library keeps
dispatch's scratch in a fixed device array of its own.  This checks, through the C ABI, that
two calls in a row give exactly what the workspace-based moe_dispatch gives (dispatch is
integer work, so the tolerance is zero), and that sizes beyond the array are refused.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import require_cuda

pytestmark = pytest.mark.gpu

CASES = [  # (T, d, E, k): the Mixtral-shaped and DeepSeek-V3-shaped routing sizes, small d
    (4096, 256, 8, 2),
    (8192, 128, 256, 8),
    (333, 64, 64, 6),
]


def _outputs(T, d, E, k):
    def z(*shape):
        return torch.full(shape, -7, dtype=torch.int32, device="cuda")
    return dict(counts=z(E), offsets=z(E + 1), perm=z(T * k), inv=z(T, k),
                x_perm=torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("T,d,E,k", CASES)
def test_static_dispatch_matches_workspace_dispatch(T, d, E, k):
    moe = require_cuda()
    rng = np.random.default_rng(T + E)
    idx_np = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)   # k distinct experts per token
    idx = torch.from_numpy(idx_np).cuda()
    x = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    cfg = moe.config(T, d, 64, E, k)
    ref = _outputs(T, d, E, k)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    moe.dispatch(cfg, idx, x, ref["counts"], ref["offsets"], ref["perm"], ref["inv"], ref["x_perm"], ws)
    for _ in range(2):
        got = _outputs(T, d, E, k)
        moe.dispatch_static(cfg, idx, x, got["counts"], got["offsets"], got["perm"], got["inv"], got["x_perm"])
        torch.cuda.synchronize()
        for name in ref:
            assert torch.equal(got[name], ref[name]), name
    assert moe.get_device_error() == 0


def test_static_dispatch_rejects_sizes_beyond_its_array():
    moe = require_cuda()
    # ceil(T*k / 256) * E = 1025 * 256 > 131072
    cfg = moe.config(1025 * 32, 64, 64, 256, 8)
    with pytest.raises(moe.MoEError) as e:
        moe.dispatch_static(cfg, 0x100000, 0x100000, 0x100000, 0x100000, 0x100000, 0x100000, 0x100000, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
