"""Pins of the two error measures every parity verdict goes through, to values fixed by
arithmetic alone:

- oracle.rel_rms, the relative RMS error ||x - ref||_2 / ||ref||_2 of the [FLA] issue's
  accuracy budget (comment of Oct 3: "relative RMS" of each gradient against an fp32
  reference), and
- tests/helpers.bias, the relative signed projection sum((got - ref) ref) / sum(ref^2) that
  reads the [AIT] PR's truncation effect (about -0.3 % of the output, Technical details) as
  -3e-3.

Each case is chosen so that a plausible slip fails it: a missing square root, a mean taken
in one term but a sum in the other, a max-norm instead of the 2-norm, a flipped sign, or a
NaN that compares as a pass."""
import math

import numpy as np

import oracle
from helpers import bias


def test_rel_rms_of_a_power_of_two_relative_error_is_exact():
    # ref * (1 + 2^-10) - ref == ref * 2^-10 exactly for small-integer ref, and the squared
    # norms scale by an exact power of 4, so the ratio is exactly 2^-10 (a missing sqrt
    # gives 2^-20).
    ref = np.arange(1, 65, dtype=np.float64).reshape(4, 16)
    eps = 2.0**-10
    assert oracle.rel_rms(ref * (1 + eps), ref) == eps
    assert oracle.rel_rms(ref * (1 - eps), ref) == eps


def test_rel_rms_one_element_error_hand_value():
    # ||(0, 1)|| / ||(3, 4)|| = 1/5.  A mean in the numerator only gives sqrt(1/2)/5; a mean in
    # the denominator only gives sqrt(2)/5; a max-norm denominator gives 1/4.
    assert oracle.rel_rms(np.array([3.0, 5.0]), np.array([3.0, 4.0])) == 0.2


def test_rel_rms_error_orthogonal_to_the_reference():
    # error (0, 1, 1, 1) against ref (1, 0, 0, 0): sqrt(3) / 1
    got = oracle.rel_rms(np.array([1.0, 1.0, 1.0, 1.0]), np.array([1.0, 0.0, 0.0, 0.0]))
    assert abs(got - math.sqrt(3.0)) <= 1e-15


def test_rel_rms_is_symmetric_in_the_error_sign_and_scale_free():
    rng = np.random.default_rng(5)
    ref = rng.standard_normal((8, 33))
    d = 1e-3 * rng.standard_normal((8, 33))
    a = oracle.rel_rms(ref + d, ref)
    assert abs(a - oracle.rel_rms(ref - d, ref)) <= 1e-15
    assert abs(a - oracle.rel_rms(4.0 * (ref + d), 4.0 * ref)) <= 1e-15
    # and it is the 2-norm ratio over the whole tensor, not an average of per-row ratios
    rows = np.mean([np.linalg.norm(d[i]) / np.linalg.norm(ref[i]) for i in range(8)])
    assert abs(a - np.linalg.norm(d) / np.linalg.norm(ref)) <= 1e-15
    assert abs(a - rows) > 1e-6


def test_rel_rms_zero_reference_and_nan():
    # a zero reference gives the absolute error norm (documented behaviour)
    assert oracle.rel_rms(np.array([3.0, 4.0]), np.zeros(2)) == 5.0
    assert oracle.rel_rms(np.zeros(3), np.zeros(3)) == 0.0
    # a NaN anywhere in x makes the measure NaN, which no tolerance check passes
    e = oracle.rel_rms(np.array([1.0, np.nan]), np.array([1.0, 2.0]))
    assert math.isnan(e) and not (e <= 1.0)


def test_bias_reads_a_multiplicative_shrink_with_its_sign():
    rng = np.random.default_rng(6)
    ref = rng.standard_normal((16, 128))
    assert abs(bias(ref * (1 - 0.003), ref) - (-0.003)) <= 1e-15
    assert abs(bias(ref * (1 + 0.003), ref) - 0.003) <= 1e-15
    assert bias(ref, ref) == 0.0


def test_bias_ignores_error_orthogonal_to_the_reference():
    # the error (0, 1) is orthogonal to ref (1, 0): no signed bias, although rel_rms is 1
    ref = np.array([1.0, 0.0])
    got = np.array([1.0, 1.0])
    assert bias(got, ref) == 0.0
    assert oracle.rel_rms(got, ref) == 1.0
    # hand value: ref (1, 2), got (1.5, 2) -> (0.5 * 1) / (1 + 4) = 0.1
    assert abs(bias(np.array([1.5, 2.0]), np.array([1.0, 2.0])) - 0.1) <= 1e-15
