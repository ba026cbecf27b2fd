"""Pins of the oracle's numeric building blocks (CPU only).

Each check compares the oracle with something other than itself: exact
rational arithmetic, a library routine in higher precision, a textbook special
case or a limit of the formula.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O

sympy = pytest.importorskip("sympy")


def _rn32(fr: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (ties to even)."""
    x = np.float32(float(fr))
    cands = [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.array(c).view(np.uint32)) & 1))


def test_sigmoid_constants_are_the_exact_roundings():
    l2e = Fraction(str(sympy.N(1 / sympy.log(2), 50)))
    ln2 = Fraction(str(sympy.N(sympy.log(2), 50)))
    assert O.LOG2E == _rn32(l2e)
    assert Fraction(float(O.LN2_HI)) == Fraction(355, 512)
    assert O.LN2_LO == _rn32(ln2 - Fraction(355, 512))
    for k, c in enumerate(O.INV_FACT, start=1):
        assert c == _rn32(Fraction(1, math.factorial(k))), k


def _ulp_err(got32, ref64):
    ref32 = ref64.astype(np.float32)
    ulp = np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(got32.astype(np.float64) - ref64) / ulp


def test_exp_f32_within_two_ulp_of_float64_exp():
    y = np.concatenate([np.linspace(-87, 88, 400001, dtype=np.float32),
                        np.random.default_rng(1).uniform(-87, 88, 200000).astype(np.float32)])
    err = _ulp_err(O.exp_f32(y), np.exp(y.astype(np.float64)))
    assert err.max() <= 2.0, err.max()


def test_sigmoid_f32_accuracy_and_special_values():
    x = np.linspace(-16, 16, 300001, dtype=np.float32)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    assert _ulp_err(O.sigmoid_f32(x), ref).max() <= 3.0
    assert O.sigmoid_f32(np.float32(0.0)) == np.float32(0.5)
    assert O.sigmoid_f32(np.float32(100.0)) == np.float32(1.0)
    big_neg = O.sigmoid_f32(np.array([-50.0, -87.0, -200.0], np.float32))
    assert np.all(big_neg > 0) and np.all(big_neg < 1e-20)
    # monotone non-decreasing on a fine grid
    s = O.sigmoid_f32(x)
    assert np.all(np.diff(s.astype(np.float64)) >= 0)


def test_round_bf16_matches_torch_on_float32_inputs():
    g = np.random.default_rng(2)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * np.float32(3),
        (g.standard_normal(1000) * 1e30).astype(np.float32),
        (g.standard_normal(1000) * 1e-30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, -3.0e38], np.float32),
    ])
    # exact ties of the bf16 grid (low 16 bits = 0x8000) exercise ties-to-even
    ties = ((g.integers(0x3F00, 0x4100, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even_by_hand():
    one = 1.0
    assert O.round_bf16(np.array([one + 2.0 ** -8]))[0] == 1.0            # tie -> even (1.0)
    assert O.round_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6
    assert O.round_bf16(np.array([one + 2.0 ** -8 + 2.0 ** -30]))[0] == one + 2.0 ** -7
    assert O.round_bf16(np.array([2.0 ** -133]))[0] == 2.0 ** -133        # bf16 subnormal
    assert np.isinf(O.round_bf16(np.array([3.4e38]))[0])


# --- SituGLU -----------------------------------------------------------------

def test_situ_zero_gate_or_up_gives_zero():
    g = np.linspace(-50, 50, 1001)
    assert np.all(O.situ(np.zeros_like(g), g, 4.0, 8.0) == 0.0)
    assert np.all(O.situ(g, np.zeros_like(g), 4.0, 8.0) == 0.0)
    assert np.all(O.situ(g, np.zeros_like(g), 4.0, 0.0) == 0.0)


def test_situ_large_beta_is_silu_gated_and_up_passes_through():
    g = np.linspace(-20, 20, 4001)
    u = np.linspace(3, -5, 4001)
    silu = torch.nn.functional.silu(torch.from_numpy(g)).numpy()      # g * sigmoid(g)
    got = O.situ(g, u, 1e7, 0.0)          # beta -> inf, linear_beta unset
    assert np.allclose(got, silu * u, rtol=1e-9, atol=1e-12)
    got_neg = O.situ(g, u, 1e7, -3.0)     # any linear_beta <= 0 means unset
    assert np.array_equal(got, got_neg)


def test_situ_saturation_limits():
    beta, lb = 4.0, 8.0
    assert O.situ(np.array([1e4]), np.array([1e4]), beta, lb)[0] == pytest.approx(beta * lb, rel=1e-12)
    assert O.situ(np.array([1e4]), np.array([-1e4]), beta, lb)[0] == pytest.approx(-beta * lb, rel=1e-12)
    assert abs(O.situ(np.array([-1e4]), np.array([5.0]), beta, lb)[0]) < 1e-300
    # bounded by beta * linear_beta everywhere
    g = np.random.default_rng(3).normal(0, 30, 100000)
    u = np.random.default_rng(4).normal(0, 30, 100000)
    assert np.all(np.abs(O.situ(g, u, beta, lb)) < beta * lb)


def test_situ_small_argument_expansion():
    # beta*tanh(g/beta) = g - g^3/(3 beta^2) + O(g^5): relative deviation from
    # silu(g)*up -> 0 like (g^2 + u^2)/(3 beta^2) for small g, u.
    beta, lb = 4.0, 8.0
    g = np.array([1e-3, -2e-3, 5e-4])
    u = np.array([3e-3, 1e-3, -4e-3])
    silu = g / (1 + np.exp(-g))
    rel = O.situ(g, u, beta, lb) / (silu * u) - 1
    bound = (g ** 2) / (3 * beta ** 2) + (u ** 2) / (3 * lb ** 2)
    assert np.all(np.abs(rel) <= 1.01 * bound + 1e-15)


def test_situ_up_factor_is_odd():
    g = np.random.default_rng(5).normal(0, 5, 1000)
    u = np.random.default_rng(6).normal(0, 20, 1000)
    for lb in (8.0, 0.0):
        assert np.array_equal(O.situ(g, -u, 4.0, lb), -O.situ(g, u, 4.0, lb))


def test_situ_requires_beta():
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(ValueError):
            O.situ(np.ones(2), np.ones(2), bad, 8.0)


def test_situ_and_mul_gate_is_first_half():
    # with beta -> inf and linear_beta unset the result is bf16(silu(gate) * up);
    # up = 1 makes it bf16(silu(gate)), which a swapped layout would not give.
    g = np.random.default_rng(7).normal(0, 3, (16, 64)).astype(np.float32)
    x = np.concatenate([g, np.ones_like(g)], axis=1)
    xb = O.f64_to_bf16_bits(x.astype(np.float64))
    got = O.bf16_to_f64(O.situ_and_mul(xb, 1e7, 0.0))
    gb = torch.from_numpy(O.bf16_to_f64(xb[:, :64]))
    ref = torch.nn.functional.silu(gb).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, ref)


def test_masked_situ_leaves_padded_rows_untouched():
    import workloads as W
    x, counts = W.masked_situ_input(6, 10, 32, seed=3)
    counts = counts.copy()
    counts[0], counts[1] = -5, 99            # clamped to 0 and T_max (R-11)
    init = W.sentinel_like((6, 10, 16))
    out = O.masked_situ_and_mul(x, counts, init, 4.0, 8.0)
    for e in range(6):
        n = min(max(int(counts[e]), 0), 10)
        assert np.all(out[e, n:] == W.SENTINEL)
        if n:
            assert np.array_equal(out[e, :n], O.situ_and_mul(x[e, :n], 4.0, 8.0))
