"""The per-element bound the bf16 forward is held to where 1e-2 cannot hold (helpers.
bf16_forward_allowed), checked against a direct simulation of the arithmetic the method
prescribes, independent of the kernels: weights p = exp(s - m) in fp64, each rounded to bf16
before the weighted sum of V, the normaliser summing the unrounded weights, and the result rounded
to bf16.  Rows with a few dominant keys (scores scaled up, as the N = 32768 workload's queries
are) are where the bound exceeds 1e-2."""
import numpy as np
import pytest
import torch

from helpers import BF16_O_MAX_ABS, bf16_forward_allowed


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def simulate(s, v):
    """Exact and simulated O for score rows s [R, n] and values v [n, d] (fp64 in, fp64 out)."""
    p = np.exp(s - s.max(1, keepdims=True))
    l = p.sum(1, keepdims=True)
    exact = (p / l) @ v
    oabs = (p / l) @ np.abs(v)
    simulated = bf16((bf16(p) @ v) / l)
    return exact, oabs, simulated


@pytest.mark.parametrize("score_scale", [1.0, 4.0, 8.0])
def test_bound_covers_the_prescribed_arithmetic(score_scale):
    rng = np.random.default_rng(int(score_scale * 10))
    n, d = 512, 64
    worst, over = 0.0, 0
    for _ in range(40):
        s = score_scale * rng.standard_normal((64, n)) * 1.5
        v = bf16(rng.standard_normal((n, d)) * 1.5)
        exact, oabs, sim = simulate(s, v)
        err = np.abs(sim - exact)
        allowed = bf16_forward_allowed(exact, oabs)
        worst = max(worst, float((err / allowed).max()))
        over += int((err > BF16_O_MAX_ABS).sum())
    assert worst <= 1.0, worst
    if score_scale >= 4.0:
        # peaky rows: the stated 1e-2 is exceeded by the arithmetic itself, the bound is not
        assert over > 0


def test_half_ulp_above_four_exceeds_the_stated_bound():
    # bf16 values in [4, 8) are 2^-5 apart: a value midway between two of them is 2^-6 from both
    x = 4.0 + 2.0 ** -6
    assert abs(float(bf16(np.array([x]))[0]) - x) == pytest.approx(2.0 ** -6)
    assert 2.0 ** -6 > BF16_O_MAX_ABS
    # and the bound admits it
    assert bf16_forward_allowed(np.array([x]), np.array([x]))[0] >= 2.0 ** -6


def test_bound_is_the_stated_one_where_that_is_larger():
    # small outputs of non-peaky rows: the worst case of the arithmetic is below 1e-2
    o, oabs = np.array([0.0, 0.1, 0.3]), np.array([0.0, 0.1, 0.5])
    assert np.all(bf16_forward_allowed(o, oabs) == BF16_O_MAX_ABS)
    # from |O| ~ 1 on, with all the weight on keys of that size, the worst case exceeds it
    assert bf16_forward_allowed(np.array([1.0]), np.array([1.0]))[0] > BF16_O_MAX_ABS
