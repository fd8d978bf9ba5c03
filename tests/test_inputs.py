"""The seeded input generator and the gap rule (CPU only)."""
import numpy as np

import workloads as wl
from oracle import Case, gapped_attempts
from oracle import moe_oracle as orc


def test_bf16_round_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, 1.0 + 2 ** -7], np.float32)
    bits = wl.bf16_round(vals)
    # 1 + 2^-8 is half-way between 1 and 1 + 2^-7: ties to the even mantissa (1.0);
    # 1 + 3 * 2^-8 is half-way between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6.
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x3F81]
    assert np.array_equal(wl.bf16_to_f32(bits), np.array([1, 1, 1 + 2 ** -6, -2.5, 0, 1 + 2 ** -7], np.float32))


def test_counter_based_and_reproducible():
    a = wl.standard_normal(0, "W1", 3, 1000)
    b = wl.standard_normal(0, "W1", 3, 1000)
    c = wl.standard_normal(0, "W2", 3, 1000)
    d = wl.standard_normal(0, "W1", 4, 1000)
    e = wl.standard_normal(1, "W1", 3, 1000)
    assert np.array_equal(a, b)
    for other in (c, d, e):
        assert not np.array_equal(a, other)
    # rows drawn alone equal rows drawn with the rest
    s = wl.WORKLOADS["tiny_f32"]
    x = wl.gen_x(s, 0)
    assert np.array_equal(wl.gen_x(s, 0, rows=[5, 2]), x[[5, 2]])
    W = wl.gen_experts(s, "W3", 0)
    assert np.array_equal(wl.gen_experts(s, "W3", 0, experts=[6]), W[[6]])


def test_distributions():
    s = wl.WORKLOADS["tiny_f32"].replace(T=512, d=256, d_ff=512, dtype="bf16")
    x = wl.to_f64(wl.gen_x(s, 0), "bf16")
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    W1 = wl.to_f64(wl.gen_expert(s, "W1", 0), "bf16")
    assert abs(W1.std() * np.sqrt(s.d) - 1.0) < 0.01
    W3 = wl.to_f64(wl.gen_expert(s, "W3", 0), "bf16")
    assert abs(W3.std() * np.sqrt(s.d_ff) - 1.0) < 0.01
    sk = wl.WORKLOADS["hunyuan_a13b"]
    lb = wl.gen_logit_bias(sk, 0)
    assert lb.dtype == np.float32 and lb.shape == (64,)
    assert 1.0 < lb.std() < 2.0


def test_gap_rule_holds_after_redraw():
    s = wl.WORKLOADS["hunyuan_a13b"].replace(T=2048, d=512)
    att = gapped_attempts(s, 0)
    assert att.sum() > 0          # some tokens needed a redraw at this size
    c = Case(s, 0)
    l = orc.router_logits(c.f64(c.x), c.f64(c.W_g), c.logit_bias)
    assert orc.min_adjacent_gap(l, s.k + 1).min() >= 1e-3
