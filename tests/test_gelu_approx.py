"""The erf approximation the bf16 kernels use for GELU and its derivative,
against the exact functions (CPU, fp64).

"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer": the expert activation is the GELU u * Phi(u), Phi the
standard normal CDF (exact erf).  The bf16 first-GEMM epilogue and the
backward pass evaluate erf with the rational approximation of Abramowitz &
Stegun, Handbook of Mathematical Functions, formula 7.1.26:
    erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),
    t = 1 / (1 + p z), z >= 0,
    p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
    -1.453152027, 1.061405429,
with |error| <= 1.5e-7 as the handbook states.  These tests evaluate that
published formula in fp64 (not the kernels' fp32 arrangement of it, which the
GPU test of the first GEMM's output covers) and pin the error figures the
kernels' documentation quotes:
  * |erf error| <= 1.5e-7 on z in [0, 12];
  * GELU:  |error| <= 7e-8 * |u| (so <= 5.6e-7 on [-8, 8]);
  * GELU' = Phi(u) + u phi(u): |error| <= 7e-8 (half the erf error; the
    u phi(u) term is exact).
"""
import numpy as np
from scipy.special import erf

P = 0.3275911
A = (0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429)


def erfc_as7126(z):
    """q(t) exp(-z^2) ~ 1 - erf(z) for z >= 0."""
    t = 1.0 / (1.0 + P * z)
    q = 0.0
    for a in reversed(A):
        q = (q + a) * t
    return q * np.exp(-z * z)


def phi_as7126(u):
    """Normal CDF from the approximation: 1 - h for u >= 0, h for u < 0."""
    h = 0.5 * erfc_as7126(np.abs(u) / np.sqrt(2.0))
    return np.where(u >= 0, 1.0 - h, h)


def test_erf_error_bound():
    z = np.linspace(0.0, 12.0, 1_200_001)
    err = np.abs((1.0 - erfc_as7126(z)) - erf(z))
    assert err.max() <= 1.5e-7
    assert err.max() >= 1.0e-7  # the bound is close to tight: the coefficients are the handbook's


def test_gelu_error_bound():
    u = np.linspace(-8.0, 8.0, 1_600_001)
    exact = 0.5 * u * (1.0 + erf(u / np.sqrt(2.0)))
    approx = u * phi_as7126(u)
    err = np.abs(approx - exact)
    assert np.all(err <= 7e-8 * np.abs(u) + 1e-300)
    assert err.max() <= 5.6e-7
    # a planted mistake (one coefficient's sign flipped) breaks the bound
    global A
    saved = A
    try:
        A = (saved[0], saved[1], saved[2], -saved[3], saved[4])
        assert np.max(np.abs(u * phi_as7126(u) - exact)) > 1e-3
    finally:
        A = saved


def test_gelu_derivative_error_bound():
    u = np.linspace(-10.0, 10.0, 2_000_001)
    dens = np.exp(-0.5 * u * u) / np.sqrt(2.0 * np.pi)
    exact = 0.5 * (1.0 + erf(u / np.sqrt(2.0))) + u * dens
    approx = phi_as7126(u) + u * dens
    err = np.abs(approx - exact)
    assert err.max() <= 7e-8
    # and the derivative is the slope of the GELU: central differences agree
    g = lambda v: 0.5 * v * (1.0 + erf(v / np.sqrt(2.0)))  # noqa: E731
    v = np.linspace(-6.0, 6.0, 1201)
    fd = (g(v + 1e-5) - g(v - 1e-5)) / 2e-5
    ex = 0.5 * (1.0 + erf(v / np.sqrt(2.0))) + v * np.exp(-0.5 * v * v) / np.sqrt(2.0 * np.pi)
    assert np.max(np.abs(fd - ex)) <= 1e-8
