"""The output-rounding allowance used by the bfloat16 parity checks (host only)."""
import numpy as np

import workloads as wl
from gpu_util import bf16_half_ulp, layer_out_err


def test_half_ulp_bounds_round_to_nearest():
    r = np.random.default_rng(0)
    v = (r.standard_normal(200000) * np.exp(r.uniform(-20, 20, 200000))).astype(np.float32)
    rounded = wl.bf16_to_f32(wl.bf16_round(v)).astype(np.float64)
    gap = np.abs(rounded - v.astype(np.float64))
    assert np.all(gap <= bf16_half_ulp(rounded))
    # tight: some values sit almost exactly half an ulp away
    assert np.max(gap / bf16_half_ulp(rounded)) > 0.99


def test_half_ulp_values():
    assert bf16_half_ulp(np.array([1.0]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([1.5]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([-3.0]))[0] == 2.0 ** -7
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0


class _S:
    def __init__(self, dtype):
        self.dtype = dtype


def test_layer_out_err_allows_only_the_final_rounding():
    r = np.random.default_rng(1)
    ref = r.standard_normal(4096) * 3
    rms = np.sqrt(np.mean(ref ** 2))
    exact = wl.bf16_to_f32(wl.bf16_round(ref.astype(np.float32))).astype(np.float64)
    assert layer_out_err(exact, ref, _S("bf16")) <= 1e-12     # correctly rounded: no error left
    off = ref.copy()
    off[17] += 0.05 * rms                                      # a 5%-of-rms arithmetic error
    got = wl.bf16_to_f32(wl.bf16_round(off.astype(np.float32))).astype(np.float64)
    assert layer_out_err(got, ref, _S("bf16")) > 2e-2
    assert layer_out_err(got.astype(np.float32), ref, _S("f32")) > 2e-2
