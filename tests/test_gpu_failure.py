"""Failure detection on the GPU without a fault: a grouped tensor-core GEMM whose TMA producer
issues nothing (moe_test_pipeline_fault) must give up on its bounded waits, report through
the device error word, free its tensor memory and return, leaving the context usable."""
import time

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import Case

from gpu_util import check_close, require_cuda, to_dev, upload_experts

pytestmark = pytest.mark.gpu

ERR_WAIT_MMA = 1 << 3
ERR_WAIT_EPILOGUE = 1 << 4


@pytest.mark.parametrize("variant", ["single", "pair", "tpair", "tpairw"])
def test_starved_pipeline_times_out_and_reports(variant, monkeypatch):
    moe = require_cuda()
    monkeypatch.setenv("MOE_GEMM_KERNEL", variant)
    s = wl.MoEShape("starve", T=300, d=256, d_ff=256, E=4, k=2, dtype="bf16", scoring="softmax")
    case = Case(s, 0)
    ref = case.forward()
    W = upload_experts(s, 0, keep=range(s.E))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    xp = to_dev(case.x[ref["perm_tok"]], s)
    off = torch.from_numpy(ref["offsets"]).cuda()
    y_perm = torch.empty((s.T * s.k, s.d), dtype=torch.float32, device="cuda")
    assert moe.get_device_error() == 0
    moe.test_pipeline_fault(20_000_000)          # 20 ms per wait
    t0 = time.time()
    moe.experts(cfg, xp, off, W["W1"], W["W2"], W["W3"], y_perm, ws)
    word = moe.get_device_error()                # waits for the stream: the kernel came back
    elapsed = time.time() - t0
    assert word & ERR_WAIT_MMA and word & ERR_WAIT_EPILOGUE, hex(word)
    assert elapsed < 5.0
    assert moe.get_device_error() == 0           # read and cleared
    # the context is fine and the next launch is unaffected
    moe.experts(cfg, xp, off, W["W1"], W["W2"], W["W3"], y_perm, ws)
    assert moe.get_device_error() == 0
    check_close(y_perm, ref["y_perm"], s, "y_perm")


def test_fault_hook_rejects_bad_limits():
    moe = require_cuda()
    for bad in (0, 3_000_000_000):
        with pytest.raises(moe.MoEError) as e:
            moe.test_pipeline_fault(bad)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG
