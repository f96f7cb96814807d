"""The bf16 validity check of the step-by-step chain comparison (tests/parity.py) on the
CPU: the oracle's own roundings pass, roundings of float32-perturbed inputs pass, and a
value moved by one bf16 ulp away from a rounding boundary fails."""
import numpy as np
import pytest

from oracle import eagle3_oracle as O
from parity import assert_bf16_valid


def _bits(x):
    return (O.round_bf16(x).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("seed", range(4))
def test_bf16_validity_check(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((4, 256)) * 3
    assert_bf16_valid(_bits(x), x, "oracle's own rounding")
    xp = (x * (1 + 1e-6 * rng.standard_normal(x.shape))).astype(np.float32).astype(np.float64)
    assert_bf16_valid(_bits(xp), x, "float32-perturbed input")
    # one ulp up on the largest value of a row, which is far from any boundary
    bad = _bits(x)
    r = 2
    i = int(np.argmax(np.abs(x[r]) * (np.abs(x[r] / O.round_bf16(x[r]) - 1) < 1e-3)))
    bad[r, i] += 1
    with pytest.raises(AssertionError):
        assert_bf16_valid(bad, x, "planted")
