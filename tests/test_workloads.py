"""The seeded input generators: the bf16 rounding of the drawn values matches torch's
fp32 -> bf16 conversion (round to nearest, ties to even), and the draws are reproducible."""

import numpy as np
import torch

from workloads import CONFIGS, bf16_bits_to_f64, f32_to_bf16_bits, gen_bf16, gen_logits


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    a = (rng.standard_normal(200000) * 10.0 ** rng.integers(-40, 38, 200000)).astype(np.float32)
    # exact ties (the 16 dropped bits are 0x8000) with even and odd kept parts
    ties = (np.arange(1000, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    a = np.concatenate([a, ties.view(np.float32), np.float32([0.0, -0.0, 3.3895e38, 1e-45])])
    ours = f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).bfloat16().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_draws_are_reproducible_and_distinct():
    c = CONFIGS["tiny"]
    a, b = gen_bf16(c, "x", (c.T, c.d)), gen_bf16(c, "x", (c.T, c.d))
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, gen_bf16(c, "dy", (c.T, c.d)))
    v = bf16_bits_to_f64(a)
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1.0) < 0.02
    np.testing.assert_array_equal(gen_logits(c), gen_logits(c))
