"""GPU parity: the CUDA library through its C ABI against the CPU oracle, on seeded inputs.

Routing indices, per-expert counts, offsets and the permutation must match bit for bit; the
layer output within max|err| <= 2e-2 rms(ref) (bfloat16) or 1e-4 rms(ref) (float32).
Small cases run the whole oracle; the five full-size workloads are checked on every
routing decision and on sampled tokens' outputs, through the same moe_forward call that
bench.py times.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import Case
from oracle import moe_oracle as orc

from gpu_util import (GATE_ATOL, check_close, dev_to_f64, from_dev_stored, host_weight_fn, require_cuda, tdtype,
                      to_dev, upload_experts)

pytestmark = pytest.mark.gpu

S = wl.MoEShape
SMALL = [
    wl.WORKLOADS["tiny_f32"],
    S("bf16_softmax_ragged", T=300, d=512, d_ff=384, E=8, k=2, dtype="bf16", scoring="softmax"),
    S("bf16_skewed_e64", T=257, d=256, d_ff=320, E=64, k=8, dtype="bf16", scoring="softmax", logit_bias_std=1.5),
    S("bf16_sigmoid_shared_e256", T=200, d=384, d_ff=256, E=256, k=8, dtype="bf16", scoring="sigmoid",
      n_shared=1, d_ff_shared=192),
    S("bf16_k_equals_E", T=65, d=128, d_ff=136, E=4, k=4, dtype="bf16", scoring="softmax"),
    S("bf16_E1_k1", T=130, d=64, d_ff=64, E=1, k=1, dtype="bf16", scoring="softmax"),
    S("bf16_single_token", T=1, d=256, d_ff=256, E=16, k=4, dtype="bf16", scoring="softmax"),
    S("bf16_two_shared_k1", T=96, d=192, d_ff=200, E=40, k=1, dtype="bf16", scoring="sigmoid",
      n_shared=2, d_ff_shared=72),
    S("f32_sigmoid_shared", T=50, d=96, d_ff=80, E=12, k=3, dtype="f32", scoring="sigmoid",
      n_shared=2, d_ff_shared=48),
    S("f32_e48", T=70, d=40, d_ff=24, E=48, k=5, dtype="f32", scoring="softmax", logit_bias_std=1.0),
    S("bf16_e32_router", T=150, d=320, d_ff=96, E=32, k=4, dtype="bf16", scoring="softmax", logit_bias_std=0.5),
    S("f32_e2", T=90, d=64, d_ff=32, E=2, k=1, dtype="f32", scoring="sigmoid"),
    # the limits the ABI accepts: E = 1024 experts (the GEMMs' group tables hold exactly that
    # many) and k = 32 experts per token
    S("bf16_e1024_limit", T=512, d=128, d_ff=256, E=1024, k=8, dtype="bf16", scoring="softmax"),
    S("bf16_k32_limit", T=96, d=128, d_ff=128, E=64, k=32, dtype="bf16", scoring="sigmoid"),
]

# Shapes for running every grouped-GEMM kernel on the same inputs: 128-row single-CTA tiles,
# 256-row CTA-pair tiles, and token-wide CTA-pair tiles of 16..256 tokens, with and without
# wide last tiles of up to 288 tokens.  They cover ragged groups that end inside a tile, empty
# experts, a group larger than one pair tile, N not a multiple of the tile width, and shared
# experts accumulating.
GEMM_SHAPES = [
    S("gemm_ragged_e6", T=1000, d=512, d_ff=776, E=6, k=2, dtype="bf16", scoring="softmax", logit_bias_std=1.0),
    S("gemm_skewed_e64", T=257, d=256, d_ff=320, E=64, k=8, dtype="bf16", scoring="softmax", logit_bias_std=1.5),
    S("gemm_two_shared", T=300, d=384, d_ff=200, E=40, k=1, dtype="bf16", scoring="sigmoid",
      n_shared=2, d_ff_shared=72),
    # 280 rows per shared expert: one wide token tile, accumulated by the second shared expert
    S("gemm_wide_shared", T=280, d=256, d_ff=200, E=8, k=2, dtype="bf16", scoring="softmax",
      n_shared=2, d_ff_shared=72),
    # 1024 expert groups, most of them a few rows: the largest group table of every kernel
    S("gemm_e1024", T=512, d=128, d_ff=256, E=1024, k=8, dtype="bf16", scoring="softmax"),
    # d = 200: the W1/W2 contraction ends in a partial k-block (8 of 64 columns, the rest
    # zero-filled by TMA); d_ff = 136: a partial second column tile; blocks of 287..323 rows
    # (one wide token tile, and full tiles with 33..67-row tails)
    S("gemm_d200_ktail", T=600, d=200, d_ff=136, E=4, k=2, dtype="bf16", scoring="softmax"),
]

# Expert block sizes on every boundary of the kernels' row tiles: empty; around the 16-row
# steps of the token-wide tiles; 128 and 256 +- 1; one wide token tile (257..288: a full tile
# plus up to 32 rows); a full tile and a short one (289, 300); a full and a wide tile (544);
# three tiles (545).
TILE_BOUNDARY_COUNTS = [0, 1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 272, 273, 288, 289, 300, 544, 545, 31]


@pytest.fixture(scope="module")
def moe():
    return require_cuda()


def _device_inputs(case):
    s = case.shape
    d = {"x": to_dev(case.x, s), "W_g": to_dev(case.W_g, s)}
    d["logit_bias"] = None if case.logit_bias is None else torch.from_numpy(case.logit_bias).cuda()
    return d


def _forward(moe, case, W, din):
    s = case.shape
    cfg = moe.config_from_shape(s)
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    moe.forward(cfg, din["x"], din["W_g"], W["W1"], W["W2"], W["W3"], y, ws, logit_bias=din["logit_bias"],
                Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"), topk_idx_out=idx, counts_out=counts)
    assert moe.last_launch_count() == _expected_launches(s)
    assert moe.get_device_error() == 0
    return y, idx, counts


def _expected_launches(s):
    """Kernels one moe_forward launches: router (logits + top-k when E > 32), dispatch (histogram,
    scan, permute, gather; one kernel for the first three up to 16384 pairs over <= 256 experts),
    W1/W2, W3, two per shared expert, combine."""
    small = s.T * s.k <= 16384 and s.E <= 256
    return (1 if s.E <= 32 else 2) + (2 if small else 4) + 2 + 2 * s.n_shared + 1


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_forward_small(moe, shape):
    case = Case(shape, 0)
    ref = case.forward()
    W = upload_experts(shape, 0, keep=range(shape.E))
    y, idx, counts = _forward(moe, case, W, _device_inputs(case))
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    check_close(y, ref["y"], shape)
    # run-to-run identical
    y2, _, _ = _forward(moe, case, W, _device_inputs(case))
    assert torch.equal(y, y2)


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_stages_small(moe, shape):
    """Each ABI call alone, fed the oracle's own intermediate results."""
    s = shape
    case = Case(s, 0)
    ref = case.forward()
    din = _device_inputs(case)
    W = upload_experts(s, 0, keep=range(s.E))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    # route
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    moe.route(cfg, din["x"], din["W_g"], idx, gate, logit_bias=din["logit_bias"], ws=ws)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.max(np.abs(gate.cpu().numpy() - ref["gate"])) <= GATE_ATOL
    # dispatch (oracle indices in)
    idx_ref = torch.from_numpy(ref["idx"]).cuda()
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=tdtype(s), device="cuda")
    moe.dispatch(cfg, idx_ref, din["x"], counts, offsets, perm, inv, x_perm, ws)
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(perm.cpu().numpy(), ref["perm_tok"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv_pos"])
    assert np.array_equal(from_dev_stored(x_perm, s), case.x[ref["perm_tok"]])
    # experts (oracle x_perm and offsets in)
    xp_ref = to_dev(case.x[ref["perm_tok"]], s)
    off_ref = torch.from_numpy(ref["offsets"]).cuda()
    y_perm = torch.empty((s.T * s.k, s.d), dtype=torch.float32, device="cuda")
    moe.experts(cfg, xp_ref, off_ref, W["W1"], W["W2"], W["W3"], y_perm, ws)
    check_close(y_perm, ref["y_perm"], s, "y_perm")
    # combine (oracle y_perm, inv_pos, gates in)
    yp_ref = torch.from_numpy(ref["y_perm"].astype(np.float32)).cuda()
    inv_ref = torch.from_numpy(ref["inv_pos"]).cuda()
    g_ref = torch.from_numpy(ref["gate"].astype(np.float32)).cuda()
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    moe.combine(cfg, yp_ref, inv_ref, g_ref, y, x=din["x"], Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"),
                ws=ws)
    check_close(y, ref["y"], s)
    assert moe.get_device_error() == 0


@pytest.mark.parametrize("variant", ["single", "pair", "tpair", "tpairw"])
@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=[s.name for s in GEMM_SHAPES])
def test_gemm_kernels(moe, shape, variant, monkeypatch):
    """Each grouped-GEMM kernel, forced, against the oracle: the experts call alone (oracle
    x_perm and offsets in) and the whole layer; results are run-to-run identical."""
    monkeypatch.setenv("MOE_GEMM_KERNEL", variant)
    s = shape
    case = Case(s, 0)
    ref = case.forward()
    W = upload_experts(s, 0, keep=range(s.E))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    xp_ref = to_dev(case.x[ref["perm_tok"]], s)
    off_ref = torch.from_numpy(ref["offsets"]).cuda()
    y_perm = torch.empty((s.T * s.k, s.d), dtype=torch.float32, device="cuda")
    moe.experts(cfg, xp_ref, off_ref, W["W1"], W["W2"], W["W3"], y_perm, ws)
    assert moe.get_device_error() == 0
    check_close(y_perm, ref["y_perm"], s, "y_perm")
    y_perm2 = torch.empty_like(y_perm)
    moe.experts(cfg, xp_ref, off_ref, W["W1"], W["W2"], W["W3"], y_perm2, ws)
    assert torch.equal(y_perm, y_perm2)
    y, idx, _ = _forward(moe, case, W, _device_inputs(case))
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    check_close(y, ref["y"], s)


@pytest.mark.parametrize("variant", ["single", "pair", "tpair", "tpairw"])
def test_gemm_tile_boundaries(moe, variant, monkeypatch):
    """The experts call on rows already grouped by expert, with block sizes on every tile
    boundary, against the oracle's grouped evaluation (every output row compared)."""
    monkeypatch.setenv("MOE_GEMM_KERNEL", variant)
    counts = np.array(TILE_BOUNDARY_COUNTS, dtype=np.int64)
    s = S("gemm_tile_boundaries", T=int(counts.sum()), d=384, d_ff=320, E=len(counts), k=1, dtype="bf16",
          scoring="softmax")
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = wl.gen_x(s, 0)                      # the rows of x_perm, in expert order
    W = upload_experts(s, 0, keep=range(s.E))
    ref = orc.experts_grouped(wl.to_f64(x, s.dtype), offsets, host_weight_fn(W["host"], s))
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    y_perm = torch.full((s.T, s.d), float("nan"), dtype=torch.float32, device="cuda")
    moe.experts(cfg, to_dev(x, s), torch.from_numpy(offsets).cuda(), W["W1"], W["W2"], W["W3"], y_perm, ws)
    assert moe.get_device_error() == 0
    got = dev_to_f64(y_perm)
    assert np.isfinite(got).all()           # every row written
    check_close(got, ref, s, "y_perm")


def _routed_to(counts, d, seed):
    """A layer input whose top-1 routing gives expert e exactly counts[e] tokens, in a shuffled
    token order (so every expert's rows are scattered over x): x is a seeded draw whose first E
    features are replaced by 4 at the token's expert and 0 elsewhere, and W_g is the identity on
    those features, so the logits are that one-hot row (a gap of 4 between the first and the
    second score)."""
    E = len(counts)
    owner = np.repeat(np.arange(E), counts)
    np.random.default_rng(seed).shuffle(owner)
    T = len(owner)
    s = S("fwd_tile_boundaries", T=T, d=d, d_ff=320, E=E, k=1, dtype="bf16", scoring="softmax")
    x = wl.gen_x(s, seed).copy()
    x[:, :E] = 0
    x[np.arange(T), owner] = wl.bf16_round(np.float32(4.0))
    W_g = np.zeros((d, E), dtype=x.dtype)
    W_g[np.arange(E), np.arange(E)] = wl.bf16_round(np.float32(1.0))
    return s, x, W_g, owner


@pytest.mark.parametrize("variant", ["tpair", "tpairw", "pair", "single"])
def test_forward_tile_boundaries(moe, variant, monkeypatch):
    """The whole layer through moe_forward with expert blocks on every tile boundary (the block
    sizes of test_gemm_tile_boundaries) and each expert's tokens scattered over x: the routing
    exact, the output against the oracle's layer, and equal bit for bit to the separate route,
    dispatch, experts and combine calls."""
    monkeypatch.setenv("MOE_GEMM_KERNEL", variant)
    s, x, W_g, owner = _routed_to(np.array(TILE_BOUNDARY_COUNTS, dtype=np.int64), 384, 0)
    assert s.dtype == "bf16" and x.dtype == np.uint16
    W = upload_experts(s, 0, keep=range(s.E))
    get_w = host_weight_fn(W["host"], s)
    ref = orc.forward(wl.to_f64(x, s.dtype), wl.to_f64(W_g, s.dtype), get_w, s.E, s.k, s.scoring)
    assert np.array_equal(ref["idx"][:, 0], owner)
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    xd, Wgd = to_dev(x, s), to_dev(W_g, s)
    y = torch.empty((s.T, s.d), dtype=tdtype(s), device="cuda")
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    moe.forward(cfg, xd, Wgd, W["W1"], W["W2"], W["W3"], y, ws, topk_idx_out=idx)
    assert moe.get_device_error() == 0
    assert moe.last_launch_count() == _expected_launches(s)
    assert np.array_equal(idx.cpu().numpy()[:, 0], owner)
    check_close(y, ref["y"], s)
    # the same layer through the separate calls (x_perm written by the dispatch)
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=tdtype(s), device="cuda")
    y_perm = torch.empty((s.T * s.k, s.d), dtype=torch.float32, device="cuda")
    y_sep = torch.empty_like(y)
    moe.route(cfg, xd, Wgd, idx, gate, ws=ws)
    moe.dispatch(cfg, idx, xd, counts, offsets, perm, inv, x_perm, ws)
    moe.experts(cfg, x_perm, offsets, W["W1"], W["W2"], W["W3"], y_perm, ws)
    moe.combine(cfg, y_perm, inv, gate, y_sep, ws=ws)
    assert moe.get_device_error() == 0
    assert np.array_equal(counts.cpu().numpy(), np.array(TILE_BOUNDARY_COUNTS))
    assert torch.equal(y, y_sep)


FULL = ["mixtral_prefill", "mixtral_decode", "hunyuan_a13b", "deepseek_v3"]


def _sample_tokens(idx, counts, T, n_random, seed=1):
    r = np.random.default_rng(seed)
    hot = int(np.argmax(counts))
    nz = np.nonzero(counts)[0]
    cold = int(nz[np.argmin(counts[nz])])
    pick = [0, T - 1]
    for e in (hot, cold):
        pick += list(np.nonzero((idx == e).any(axis=1))[0][:2])
    pick += list(r.choice(T, size=min(n_random, T), replace=False))
    return np.unique(np.array(pick, dtype=np.int64))


def _check_blocks(counts, T):
    """Expert blocks whose every row is compared at full size: the hottest and the coldest
    non-empty expert, and, where the layer has them, one block of 257..288 rows (one wide
    token tile) and one of at most 256 rows (one token tile).  Decode-sized layers: all."""
    nz = np.nonzero(counts)[0]
    if T <= 64:
        return [int(e) for e in nz]
    pick = [int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])]
    for lo, hi in ((257, 288), (1, 256)):
        cand = [int(e) for e in nz if lo <= counts[e] <= hi and int(e) not in pick]
        if cand:
            pick.append(cand[len(cand) // 2])
    return pick


@pytest.mark.parametrize("name", FULL)
def test_full_size(moe, name):
    """The five workloads at full size through the same moe_forward call that bench.py times:
    routing, counts, offsets and the permutation bit-exact; the layer output on sampled tokens;
    and every row of whole expert blocks of the experts call (the hottest, the coldest, a
    wide-tile block, a one-tile block) against float64 evaluations of those blocks."""
    s = wl.WORKLOADS[name]
    case = Case(s, 0)
    r = case.route()
    dsp = orc.dispatch(r["idx"], s.E)
    sample = _sample_tokens(r["idx"], dsp["counts"], s.T, 12 if s.E >= 256 else 24)
    blocks = _check_blocks(dsp["counts"], s.T)
    W = upload_experts(s, 0, keep=set(np.unique(r["idx"][sample]).tolist()) | set(blocks))
    din = _device_inputs(case)
    y, idx, counts = _forward(moe, case, W, din)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert np.array_equal(counts.cpu().numpy(), dsp["counts"])
    get_w = host_weight_fn(W["host"], s)
    x64 = case.f64(case.x[sample])
    y_ref = orc.forward_tokens(x64, r["idx"][sample], r["gate"][sample], get_w, s.n_shared)
    check_close(y[torch.from_numpy(sample).cuda()], y_ref, s, "y (%d sampled tokens)" % len(sample))
    # routing and dispatch outputs of the separate calls, at full size
    cfg = moe.config_from_shape(s)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    gate = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    moe.route(cfg, din["x"], din["W_g"], idx, gate, logit_bias=din["logit_bias"], ws=ws)
    assert np.max(np.abs(gate.cpu().numpy() - r["gate"])) <= GATE_ATOL
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=tdtype(s), device="cuda")
    moe.dispatch(cfg, idx, din["x"], counts, offsets, perm, inv, x_perm, ws)
    assert np.array_equal(offsets.cpu().numpy(), dsp["offsets"])
    assert np.array_equal(perm.cpu().numpy(), dsp["perm_tok"])
    assert np.array_equal(inv.cpu().numpy(), dsp["inv_pos"])
    rows = np.random.default_rng(2).choice(s.T * s.k, size=min(64, s.T * s.k), replace=False)
    assert np.array_equal(from_dev_stored(x_perm[torch.from_numpy(rows).cuda()], s), case.x[dsp["perm_tok"][rows]])
    # the experts call at full size (every expert block, the kernels bench.py runs); every row of
    # the chosen blocks against the oracle's float64 evaluation of the block
    y_perm = torch.full((s.T * s.k, s.d), float("nan"), dtype=torch.float32, device="cuda")
    moe.experts(cfg, x_perm, offsets, W["W1"], W["W2"], W["W3"], y_perm, ws)
    assert moe.get_device_error() == 0
    for e in blocks:
        a, b = int(dsp["offsets"][e]), int(dsp["offsets"][e + 1])
        ref_rows = orc.swiglu_expert(case.f64(case.x[dsp["perm_tok"][a:b]]), get_w("W1", e), get_w("W2", e),
                                     get_w("W3", e))
        check_close(y_perm[a:b], ref_rows, s, "y_perm of expert %d (%d rows)" % (e, b - a))
    assert moe.get_device_error() == 0
    # every element of the forward's output equals that of the separate calls, whose expert
    # blocks were checked above
    y_sep = torch.empty_like(y)
    moe.combine(cfg, y_perm, inv, gate, y_sep, x=din["x"], Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"),
                ws=ws)
    assert moe.get_device_error() == 0
    assert torch.equal(y, y_sep), "moe_forward differs from route/dispatch/experts/combine"


def test_empty_batch(moe):
    s = S("empty", T=0, d=128, d_ff=128, E=8, k=2, dtype="bf16", scoring="softmax")
    cfg = moe.config_from_shape(s)
    dummy = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    moe.forward(cfg, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert moe.last_launch_count() == 0


@pytest.mark.parametrize("T,k,E", [(64, 2, 8), (3000, 8, 64)], ids=["single_block", "chunked"])
def test_bad_expert_id_sets_device_error(moe, T, k, E):
    s = S("bad_ids", T=T, d=64, d_ff=64, E=E, k=k, dtype="bf16", scoring="softmax")
    cfg = moe.config_from_shape(s)
    x = torch.randn((s.T, s.d), device="cuda").to(torch.bfloat16)
    idx = torch.arange(s.T * s.k, device="cuda", dtype=torch.int32).reshape(s.T, s.k) % s.E
    idx[5, 1] = s.E + 3          # out of range: flagged by the kernel, the pair is skipped
    counts = torch.empty((s.E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((s.E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.zeros((s.T * s.k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((s.T * s.k, s.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    moe.get_device_error()
    moe.dispatch(cfg, idx, x, counts, offsets, perm, inv, x_perm, ws)
    w = moe.get_device_error()
    assert w & 1
    assert int(counts.sum()) == s.T * s.k - 1
    assert int(inv[5, 1]) == -1
    assert moe.get_device_error() == 0   # cleared by the previous read
