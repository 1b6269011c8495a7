"""CPU pins of the secondary cosine metric used by the GPU parity tests."""
import numpy as np
import torch

from tests._metrics import COSINE_MIN, cosine_to_rounded


def test_output_rounding_alone_scores_one():
    ref = np.random.default_rng(3).standard_normal(4096) * 7.0
    got = torch.from_numpy(ref).to(torch.bfloat16)
    assert cosine_to_rounded(got, ref) == 1.0
    assert cosine_to_rounded(np.zeros(8), np.zeros(8)) == 1.0


def test_a_one_ulp_error_everywhere_fails_and_a_sign_error_fails():
    ref = np.random.default_rng(4).standard_normal(4096)
    r16 = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64)
    assert cosine_to_rounded(r16 * (1 + 2.0 ** -7), ref) >= COSINE_MIN     # a common scale keeps the angle
    noisy = r16 * (1 + 2.0 ** -7 * torch.from_numpy(np.random.default_rng(5).choice([-1.0, 1.0], 4096)))
    assert cosine_to_rounded(noisy, ref) < COSINE_MIN
    flipped = r16.clone()
    flipped[0] = -flipped[0] * 50
    assert cosine_to_rounded(flipped, ref) < COSINE_MIN
