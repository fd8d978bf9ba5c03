"""GPU parity for auxiliary-loss-free balancing: routing with a selection-only bias, and the
bias controller's update, through the C ABI against the CPU oracle.

Pages: "Mixture-of-Experts Internals: A Systems Engineer's Field Manual", section 3.3; "Mixture-
of-Experts, from the router to the all-to-all", "Load balancing".
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import Case
from oracle import moe_oracle as orc

from gpu_util import GATE_ATOL, check_close, require_cuda, tdtype, to_dev, upload_experts

pytestmark = pytest.mark.gpu

S = wl.MoEShape
# (shape, standard deviation of the selection bias): softmax biases act on logits (~N(0,1)),
# sigmoid biases on scores in (0, 1).
SEL_CASES = [
    (S("sel_softmax_e16", T=200, d=256, d_ff=136, E=16, k=2, dtype="bf16", scoring="softmax"), 0.5),
    (S("sel_sigmoid_e64_shared", T=150, d=192, d_ff=128, E=64, k=6, dtype="bf16", scoring="sigmoid",
       n_shared=1, d_ff_shared=64), 0.05),
    (S("sel_sigmoid_e8", T=120, d=128, d_ff=128, E=8, k=2, dtype="bf16", scoring="sigmoid",
       logit_bias_std=1.0), 0.1),
    (S("sel_softmax_e40_f32", T=70, d=48, d_ff=32, E=40, k=4, dtype="f32", scoring="softmax"), 0.5),
]


@pytest.fixture(scope="module")
def moe():
    return require_cuda()


@pytest.mark.parametrize("shape,std", SEL_CASES, ids=[c[0].name for c in SEL_CASES])
def test_route_and_forward_with_selection_bias(moe, shape, std):
    s = shape
    sb_np = wl.gen_sel_bias(s, std, 0)
    case = Case(s, 0, sel_bias=sb_np)
    ref = case.forward()
    plain = orc.route(case.f64(case.x), case.f64(case.W_g), s.k, s.scoring, case.logit_bias)
    assert not np.array_equal(plain["idx"], ref["idx"])          # the bias does move traffic
    sb = torch.from_numpy(sb_np).cuda()
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    x, Wg = to_dev(case.x, s), to_dev(case.W_g, s)
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    moe.route(cfg, x, Wg, idx, gate, logit_bias=lb, sel_bias=sb, ws=ws)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.max(np.abs(gate.cpu().numpy() - ref["gate"])) <= GATE_ATOL
    W = upload_experts(s, 0, keep=range(s.E))
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    moe.forward(cfg, x, Wg, W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb, sel_bias=sb, Ws1=W.get("Ws1"),
                Ws2=W.get("Ws2"), Ws3=W.get("Ws3"), topk_idx_out=idx, counts_out=counts)
    assert moe.get_device_error() == 0
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    check_close(y, ref["y"], s)


@pytest.mark.parametrize("T,k,E", [(10, 2, 4), (4096, 2, 8), (8192, 8, 256), (333, 6, 64), (7, 1, 3)])
def test_update_sel_bias_matches_oracle(moe, T, k, E):
    r = np.random.default_rng(T + E)
    counts_np = r.multinomial(T * k, np.ones(E) / E).astype(np.int32)
    if (T * k) % E == 0:
        counts_np[0] = T * k // E             # one expert exactly at its share keeps its bias
    sb_np = (r.standard_normal(E) * 0.3).astype(np.float32)
    cfg = moe.config(T, 64, 64, E, k)
    counts = torch.from_numpy(counts_np).cuda()
    sb = torch.from_numpy(sb_np).cuda()
    for gamma in (1e-3, 0.25):
        moe.update_sel_bias(cfg, counts, gamma, sb)
        sb_np = orc.update_sel_bias(sb_np, counts_np, T, k, gamma)
        assert np.array_equal(sb.cpu().numpy(), sb_np)
    assert moe.last_launch_count() == 1


def test_bias_controller_balances_skewed_layer(moe):
    """Route -> counts -> update on the GPU, step after step, on a layer whose loads a
    per-expert logit bias skews: the most loaded expert comes down towards its share."""
    s = S("skewed", T=2048, d=256, d_ff=64, E=64, k=8, dtype="bf16", scoring="softmax", logit_bias_std=1.5)
    case = Case(s, 0, gap=False)
    x, Wg = to_dev(case.x, s), to_dev(case.W_g, s)
    lb = torch.from_numpy(case.logit_bias).cuda()
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=torch.bfloat16, device="cuda")
    sb = torch.zeros((s.E,), dtype=torch.float32, device="cuda")
    share = s.T * s.k / s.E
    history = []
    for _ in range(300):
        moe.route(cfg, x, Wg, idx, gate, logit_bias=lb, sel_bias=sb, ws=ws)
        moe.dispatch(cfg, idx, x, counts, offsets, perm, inv, x_perm, ws)
        history.append(int(counts.max()) / share)
        moe.update_sel_bias(cfg, counts, 0.02, sb)
    assert moe.get_device_error() == 0
    assert history[0] > 3.0 and np.median(history[-50:]) < 1.2, (history[0], history[-50:])


# Switch-style gating: softmax over all E, top-k, gates = the probabilities themselves.
PLAIN_SHAPES = [
    S("switch_top1_e16", T=300, d=256, d_ff=192, E=16, k=1, dtype="bf16", scoring="softmax_norenorm"),
    S("plain_top2_e64", T=200, d=192, d_ff=128, E=64, k=2, dtype="bf16", scoring="softmax_norenorm",
      logit_bias_std=1.0),
    S("plain_top2_f32", T=64, d=64, d_ff=96, E=8, k=2, dtype="f32", scoring="softmax_norenorm"),
]


@pytest.mark.parametrize("shape", PLAIN_SHAPES, ids=[s.name for s in PLAIN_SHAPES])
def test_switch_style_gates(moe, shape):
    s = shape
    case = Case(s, 0)
    ref = case.forward()
    assert np.all(ref["gate"].sum(axis=1) < 1.0)
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    x, Wg = to_dev(case.x, s), to_dev(case.W_g, s)
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    moe.route(cfg, x, Wg, idx, gate, logit_bias=lb, ws=ws)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.max(np.abs(gate.cpu().numpy() - ref["gate"])) <= GATE_ATOL
    W = upload_experts(s, 0, keep=range(s.E))
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    moe.forward(cfg, x, Wg, W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb, topk_idx_out=idx)
    assert moe.get_device_error() == 0
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    check_close(y, ref["y"], s)


STATS_SHAPES = [
    S("stats_softmax_e8", T=4096, d=512, d_ff=64, E=8, k=2, dtype="bf16", scoring="softmax"),
    S("stats_sigmoid_e256", T=1000, d=256, d_ff=64, E=256, k=8, dtype="bf16", scoring="sigmoid",
      logit_bias_std=1.0),
    S("stats_skewed_e64", T=777, d=128, d_ff=64, E=64, k=8, dtype="bf16", scoring="softmax", logit_bias_std=1.5),
    S("stats_plain_e12_f32", T=50, d=40, d_ff=16, E=12, k=1, dtype="f32", scoring="softmax_norenorm"),
]


@pytest.mark.parametrize("shape", STATS_SHAPES, ids=[s.name for s in STATS_SHAPES])
def test_load_stats(moe, shape):
    s = shape
    case = Case(s, 0)
    r = case.route()
    ref = orc.load_stats(r["idx"], r["logits"], s.E, s.scoring, 0.01)
    lb = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    x, Wg = to_dev(case.x, s), to_dev(case.W_g, s)
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=tdtype(s), device="cuda")
    moe.route(cfg, x, Wg, idx, gate, logit_bias=lb, ws=ws)
    moe.dispatch(cfg, idx, x, counts, offsets, perm, inv, x_perm, ws)
    f = torch.empty((s.E,), dtype=torch.float32, device="cuda")
    P = torch.empty_like(f)
    summary = torch.empty((2,), dtype=torch.float32, device="cuda")
    moe.load_stats(cfg, x, Wg, counts, 0.01, f, P, summary, logit_bias=lb, ws=ws)
    assert moe.last_launch_count() == 3
    assert moe.get_device_error() == 0
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(f.cpu().numpy(), (ref["counts"].astype(np.float32) / np.float32(s.T)))
    assert np.allclose(P.cpu().numpy(), ref["P"], rtol=2e-4, atol=1e-7)
    got = summary.cpu().numpy()
    assert abs(got[0] - ref["aux_loss"]) <= 2e-4 * ref["aux_loss"]
    assert abs(got[1] - ref["max_over_mean"]) <= 1e-6 * ref["max_over_mean"]
    # identical on a second call
    P2 = torch.empty_like(P)
    moe.load_stats(cfg, x, Wg, counts, 0.01, f, P2, summary, logit_bias=lb, ws=ws)
    assert torch.equal(P, P2)
