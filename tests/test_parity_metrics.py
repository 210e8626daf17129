"""The GPU parity metrics catch one wrong output row (CPU only).

At the 8 192-row headline shape a single row that is entirely wrong (its
values swapped for another row's, as a wrong value slice or a mis-merged
split would leave it) stays inside the whole-tensor rel-L2 bound of FP8 dots
but fails the per-row bound.  The "GPU output" here is a perturbed copy of
a reference array; no oracle is involved.
"""

import numpy as np
import torch

from tests.parity import TOL, assert_close, compare


def _fake_outputs(seed, noise):
    rng = np.random.default_rng(seed)
    ref = rng.standard_normal((64, 2, 64, 512))
    lse = rng.standard_normal((64, 2, 64))
    got = ref * (1 + noise * rng.standard_normal(ref.shape))
    return ref, lse, got


def test_single_wrong_row_fails_the_row_bound_only():
    ref, lse, got = _fake_outputs(0, 0.03)
    m = compare(torch.from_numpy(got), torch.from_numpy(lse), ref, lse, "fp8")
    assert_close(m, "fp8")  # a uniformly noisy output passes
    got[17, 1, 33] = ref[3, 0, 5]  # one row replaced by another row's values
    m = compare(torch.from_numpy(got), torch.from_numpy(lse), ref, lse, "fp8")
    assert m["rel_l2"] <= TOL["fp8"]["rel_l2"]
    assert m["row_rel_l2_max"] > 1.0 > TOL["fp8"]["row_rel_l2"]


def test_zero_reference_row_is_held_to_an_absolute_bound():
    ref, lse, got = _fake_outputs(1, 0.0)
    ref[2, 0, 1] = 0.0
    got[2, 0, 1] = 0.5
    m = compare(torch.from_numpy(got), torch.from_numpy(lse), ref, lse, "bf16")
    assert m["row_rel_l2_max"] > TOL["bf16"]["row_rel_l2"]
