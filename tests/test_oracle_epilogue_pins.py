"""Pins of the oracle's fused epilogue (CPU only).

The epilogue is D = act(alpha * rs[i] * cs[j] * (A.B)[i][j] + beta * C_prev[i][j]
+ bias[j]), act in {none, ReLU, GELU}: the bias / ReLU / GELU epilogues that
"tensor-cores-cutlass-and-cute" lists among cuBLASLt's features (its
comparison with cuBLAS), with the order of the terms read as scale, add,
activate.  The pins below fix it against things other than its own formula:
tabulated values of the normal CDF, PyTorch's own tanh-form GELU (a library
routine, for the tanh form's constants), identities of GELU and ReLU, the
page-1 worked example (D = 16 i j), and planted mistakes that must fail a pin.
"""
import math

import numpy as np
import pytest

from test_oracle_pins import load_worked_example, worked_example_operands

# Standard normal CDF at 1, 2, 3 as printed in statistical tables.
PHI_TABLE = {1.0: 0.8413447461, 2.0: 0.9772498681, 3.0: 0.9986501020}


def test_gelu_table_values(oracle_mod):
    x = np.array(sorted(PHI_TABLE))
    g = oracle_mod.activation(x, oracle_mod.ACT_GELU)
    for xi, gi in zip(x, g):
        assert abs(gi - xi * PHI_TABLE[xi]) < 1e-9
    # Phi(-x) = 1 - Phi(x): GELU(-x) = -x (1 - Phi(x))
    gn = oracle_mod.activation(-x, oracle_mod.ACT_GELU)
    for xi, gi in zip(x, gn):
        assert abs(gi + xi * (1.0 - PHI_TABLE[xi])) < 1e-9


def test_gelu_identities(oracle_mod):
    x = np.linspace(-8.0, 8.0, 1601)
    g = oracle_mod.activation(x, oracle_mod.ACT_GELU)
    assert oracle_mod.activation(np.array([0.0]), oracle_mod.ACT_GELU)[0] == 0.0
    # x Phi(x) - (-x) Phi(-x) = x (Phi(x) + Phi(-x)) = x
    assert np.max(np.abs(g - g[::-1] - x)) < 1e-12
    # GELU lies between min(x, 0) and max(x, 0) and tends to ReLU
    assert np.all(g <= np.maximum(x, 0) + 1e-15) and np.all(g >= np.minimum(x, 0) - 1e-15)
    assert abs(oracle_mod.activation(np.array([20.0]), 2)[0] - 20.0) < 1e-12
    assert abs(oracle_mod.activation(np.array([-20.0]), 2)[0]) < 1e-12
    # the slope bound used by the acceptance measure is the true maximum
    d = np.diff(g) / np.diff(x)
    assert d.max() <= oracle_mod.GELU_MAX_SLOPE + 1e-6
    assert d.max() >= oracle_mod.GELU_MAX_SLOPE - 1e-3


def test_gelu_tanh_form(oracle_mod):
    """The tanh form is odd-symmetric like the erf form (g(x) - g(-x) = x),
    zero at zero, tends to ReLU, stays within 1e-3 of the erf form, and its
    slope stays under the bound the acceptance measure uses."""
    x = np.linspace(-8.0, 8.0, 3201)
    g = oracle_mod.activation(x, oracle_mod.ACT_GELU_TANH)
    ge = oracle_mod.activation(x, oracle_mod.ACT_GELU)
    assert oracle_mod.activation(np.array([0.0]), oracle_mod.ACT_GELU_TANH)[0] == 0.0
    assert np.max(np.abs(g - g[::-1] - x)) < 1e-12
    assert np.max(np.abs(g - ge)) < 1e-3
    assert np.max(np.abs(g - ge)) > 1e-5  # a different function, not the erf form again
    assert abs(oracle_mod.activation(np.array([20.0]), 3)[0] - 20.0) < 1e-12
    d = np.diff(g) / np.diff(x)
    assert d.max() <= oracle_mod.GELU_MAX_SLOPE + 2e-3


def _torch_gelu_tanh(x):
    """PyTorch's own tanh-form GELU (``approximate="tanh"``) in fp64: a
    library routine written independently of the oracle, used here as the
    fixed point the oracle's constants (sqrt(2/pi) and 0.044715) must meet."""
    torch = pytest.importorskip("torch")
    return torch.nn.functional.gelu(torch.from_numpy(np.asarray(x, dtype=np.float64)),
                                    approximate="tanh").numpy()


def test_gelu_tanh_matches_library(oracle_mod):
    """Over [-10, 10] the oracle's tanh form agrees with PyTorch's to rounding
    (both in fp64).  A wrong constant does not: 0.0447 for 0.044715 moves the
    value by up to 8.7e-6, sqrt(2/pi) cut to 4 digits by more, seven orders of
    magnitude above this pin's tolerance."""
    x = np.linspace(-10.0, 10.0, 20001)
    g = oracle_mod.activation(x, oracle_mod.ACT_GELU_TANH)
    ref = _torch_gelu_tanh(x)
    assert np.max(np.abs(g - ref)) <= 1e-13 * np.maximum(1.0, np.abs(x)).max()


@pytest.mark.parametrize("mistake", ["cubic_constant_truncated", "sqrt_2_over_pi_truncated",
                                     "cubic_term_squared", "half_dropped"])
def test_planted_gelu_tanh_mistakes_are_caught(oracle_mod, mistake):
    """Each slip in the tanh form fails the library pin above by orders of
    magnitude more than its tolerance (the planted versions are computed here,
    on the CPU, from the same formula with the slip in it)."""
    x = np.linspace(-10.0, 10.0, 20001)
    c, a, h = math.sqrt(2.0 / math.pi), 0.044715, 0.5
    p = 3
    if mistake == "cubic_constant_truncated":
        a = 0.0447
    elif mistake == "sqrt_2_over_pi_truncated":
        c = 0.7979
    elif mistake == "cubic_term_squared":
        p = 2
    else:
        h = 1.0
    bad = h * x * (1.0 + np.tanh(c * (x + a * x ** p)))
    ref = _torch_gelu_tanh(x)
    assert np.max(np.abs(bad - ref)) > 1e-6
    # the oracle is not the planted version
    g = oracle_mod.activation(x, oracle_mod.ACT_GELU_TANH)
    assert np.max(np.abs(g - bad)) > 1e-6


def test_relu(oracle_mod):
    x = np.array([-3.0, -0.0, 0.0, 1e-30, 2.5])
    assert list(oracle_mod.activation(x, oracle_mod.ACT_RELU)) == [0.0, 0.0, 0.0, 1e-30, 2.5]


def _worked(oracle_mod, dtype=0):
    A, B = worked_example_operands(dtype)
    Cref, Den = oracle_mod.gemm(A, B, dtype, 16, 8, 16, 16, 8)
    _, table = load_worked_example()
    return Cref[0], Den[0], table


def test_scaled_worked_example(oracle_mod):
    Cref, Den, table = _worked(oracle_mod)
    rs = np.arange(1, 17, dtype=np.float64)        # row i scaled by i + 1
    cs = np.array([2.0 ** -j for j in range(8)])   # column j by 2^-j
    D, DenD = oracle_mod.epilogue(Cref, Den, alpha=3.0, row_scale=rs, col_scale=cs)
    i = np.arange(16)[:, None]
    j = np.arange(8)[None, :]
    assert np.array_equal(D, 3.0 * (i + 1) * 2.0 ** -j * 16 * i * j)
    assert np.array_equal(D, 3.0 * rs[:, None] * cs[None, :] * table)
    assert np.array_equal(DenD, np.abs(D))


def test_bias_is_added_after_scaling(oracle_mod):
    """alpha = 2, bias = 1: 2 * 16 i j + 1, not 2 * (16 i j + 1)."""
    Cref, Den, table = _worked(oracle_mod)
    D, _ = oracle_mod.epilogue(Cref, Den, alpha=2.0, bias=np.ones(8))
    assert np.array_equal(D, 2.0 * table + 1.0)
    assert D[3, 5] == 481.0 and D[15, 7] == 3361.0


def test_beta_and_previous_c(oracle_mod):
    """A = 0 (every product zero): D = beta * C_prev + bias exactly, and with
    alpha = 0 the product does not enter at all."""
    Cref, Den, table = _worked(oracle_mod)
    Cp = np.arange(128, dtype=np.float64).reshape(16, 8) - 64.0
    D, DenD = oracle_mod.epilogue(np.zeros_like(Cref), np.zeros_like(Den), beta=-0.5, C_prev=Cp,
                                  bias=np.full(8, 0.25))
    assert np.array_equal(D, -0.5 * Cp + 0.25)
    assert np.array_equal(DenD, np.abs(-0.5 * Cp) + 0.25)
    D0, _ = oracle_mod.epilogue(Cref, Den, alpha=0.0, beta=1.0, C_prev=Cp)
    assert np.array_equal(D0, Cp)


def test_activation_applies_last(oracle_mod):
    """ReLU of (16 i j - 100): zero exactly where 16 i j < 100."""
    Cref, Den, table = _worked(oracle_mod)
    D, _ = oracle_mod.epilogue(Cref, Den, bias=np.full(8, -100.0), act=oracle_mod.ACT_RELU)
    assert np.array_equal(D, np.maximum(table - 100.0, 0.0))
    assert D[1, 1] == 0.0 and D[3, 5] == 140.0
    G, DenG = oracle_mod.epilogue(Cref, Den, alpha=1 / 64, bias=np.full(8, -1.0),
                                  act=oracle_mod.ACT_GELU)
    # 16 * 4 * 1 / 64 - 1 = 0 -> GELU(0) = 0; 16 * 8 * 1 / 64 - 1 = 1 -> Phi(1)
    assert G[4, 1] == 0.0 and abs(G[8, 1] - PHI_TABLE[1.0]) < 1e-9
    assert np.all(DenG >= 1.128 * (np.abs(table / 64) + 1.0))


@pytest.mark.parametrize("mistake", ["scales_swapped", "bias_before_scale", "act_before_bias",
                                     "beta_sign"])
def test_planted_epilogue_mistakes_are_caught(oracle_mod, mistake):
    """Each plausible slip in the epilogue changes at least one pinned value."""
    Cref, Den, table = _worked(oracle_mod)
    rs = np.arange(1, 17, dtype=np.float64)
    cs = np.array([2.0 ** -j for j in range(8)])
    Cp = np.full((16, 8), 3.0)
    bias = np.linspace(-50, 50, 8)
    good, _ = oracle_mod.epilogue(Cref, Den, alpha=0.5, beta=0.25, C_prev=Cp, bias=bias,
                                  row_scale=rs, col_scale=cs, act=oracle_mod.ACT_RELU)
    scale = 0.5 * rs[:, None] * cs[None, :]
    if mistake == "scales_swapped":
        # row scale applied per column and column scale per row (square corner)
        t8, rs8, cs8 = table[:8, :8], rs[:8], cs[:8]
        right, _ = oracle_mod.epilogue(Cref[:8, :8], Den[:8, :8], row_scale=rs8, col_scale=cs8)
        wrong = cs8[:, None] * rs8[None, :] * t8
        assert not np.allclose(wrong, right)
        assert np.array_equal(right, rs8[:, None] * cs8[None, :] * t8)
        return
    elif mistake == "bias_before_scale":
        bad = np.maximum(scale * (table + bias) + 0.25 * Cp, 0)
    elif mistake == "act_before_bias":
        bad = np.maximum(scale * table + 0.25 * Cp, 0) + bias
    else:
        bad = np.maximum(scale * table - 0.25 * Cp + bias, 0)
    assert not np.allclose(bad, good)
    # and the right composition is the one the oracle computes
    assert np.array_equal(good, np.maximum(scale * table + 0.25 * Cp + bias, 0))
