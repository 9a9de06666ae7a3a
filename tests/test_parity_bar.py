"""The parity bar itself (tests/helpers.compare), on the CPU: it accepts a
correctly rounded bf16 output at any magnitude and rejects errors a wrong
kernel would make (an element off by one bf16 step above 4, a near-zero
element off by 3e-4, a dropped term in a row)."""
import numpy as np
import pytest
import torch

from tests.helpers import compare


def bf16(x):
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)


def test_correctly_rounded_outputs_pass_at_every_magnitude():
    rng = np.random.default_rng(0)
    ref = rng.normal(size=(64, 8, 128)) * np.array([0.01, 0.1, 1, 3, 5, 9, 20, 0.001])[None, :,
                                                                                      None]
    compare(bf16(ref), ref, "rounded")


def test_one_step_off_above_four_fails():
    ref = np.full((1, 1, 4), 5.3)
    g = bf16(ref).float()
    g[0, 0, 2] += 2.0 ** -5  # one bf16 step at [4, 8)
    with pytest.raises(AssertionError):
        compare(g.to(torch.bfloat16), ref, "expected-fail: step")


def test_near_zero_element_fails_the_relative_floor():
    ref = np.array([[[1e-3, 0.5, -0.25, 0.75]]])
    g = bf16(ref).float()
    g[0, 0, 0] += 3e-4  # 3e-4 / max(1e-3, 1e-2) = 3e-2 > 2e-2
    with pytest.raises(AssertionError):
        compare(g.to(torch.bfloat16), ref, "expected-fail: floor")


def test_dropped_term_fails():
    rng = np.random.default_rng(1)
    w = rng.random(8)
    w /= w.sum()
    v = rng.normal(size=(8, 64))
    ref = (w[:, None] * v).sum(0)[None, None, :]
    wrong = ((w[:-1, None] * v[:-1]).sum(0) / w[:-1].sum())[None, None, :]
    with pytest.raises(AssertionError):
        compare(bf16(wrong), ref, "expected-fail: dropped")
