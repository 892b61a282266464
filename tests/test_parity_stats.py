"""The parity report's own arithmetic (CPU): the bf16 ulp used to count elements that
differ from the oracle by more than one unit, and the fields of a comparison."""

import numpy as np
import torch

from gpu_util import bf16_ulp, stats


def test_bf16_ulp_is_the_gap_to_the_next_bf16_value():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        [1.0, -1.0, 2.0, 0.5, 3.0, 65504.0, 2.0 ** -126]])
    a = torch.from_numpy(v.astype(np.float32)).bfloat16()
    nxt = (a.view(torch.int16) + 1).view(torch.bfloat16)        # next value away from zero
    gap = (nxt.double() - a.double()).abs().numpy()
    np.testing.assert_array_equal(bf16_ulp(a.double().numpy()), gap)
    # the subnormal range and zero: the smallest subnormal step
    assert bf16_ulp(0.0) == 2.0 ** -133 and bf16_ulp(2.0 ** -130) == 2.0 ** -133


def test_stats_fields():
    o = np.array([1.0, 2.0, -4.0, 0.0])
    g = o + np.array([2.0 ** -7, 2.0 ** -5, 0.0, 0.0])   # one ulp, two ulps, exact, exact
    s = stats(g, o)
    rms = np.sqrt(np.mean(o * o))
    assert s["n_gt_1ulp"] == 1 and s["n"] == 4
    assert s["max_abs"] == 2.0 ** -5
    assert np.isclose(s["max_over_rms"], 2.0 ** -5 / rms)
    assert np.isclose(s["max_scaled"], max(2.0 ** -7 / (rms + 1), 2.0 ** -5 / (rms + 2)))
    assert np.isclose(s["rel_l2"], np.hypot(2.0 ** -7, 2.0 ** -5) / np.linalg.norm(o))
