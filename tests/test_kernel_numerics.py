"""Host-side checks of the numerical claims the tensor-core kernels rest on
(no GPU): the softcap series used by the softmax's second pass. The GPU
parity tests check the kernels' outputs against the oracle; these check
the mathematics the kernel comments state, from first principles."""
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_latent_attention_cache_gb300", "csrc")


def _tanh_maclaurin(n_terms):
    """Odd Maclaurin coefficients of tanh, from the Bernoulli numbers:
    tanh x = sum_{n>=1} 2^(2n) (2^(2n) - 1) B_(2n) x^(2n-1) / (2n)!."""
    sympy = pytest.importorskip("sympy")
    out = []
    for n in range(1, n_terms + 1):
        b = sympy.bernoulli(2 * n)
        c = sympy.Rational(2) ** (2 * n) * (sympy.Rational(2) ** (2 * n) - 1) * b / sympy.factorial(2 * n)
        out.append(Fraction(int(c.p), int(c.q)))
    return out


def _kernel_series_coefficients():
    """The coefficients the read-phase host code scales by softcap and
    scale (the `t[5]` table in pa_tc.cu)."""
    src = open(os.path.join(CSRC, "pa_tc.cu")).read()
    m = re.search(r"const double t\[5\] = \{([^}]*)\}", src)
    assert m, "series table not found"
    vals = []
    for item in m.group(1).split(","):
        item = item.strip()
        num, _, den = item.partition("/")
        f = Fraction(num.strip())
        if den:
            f /= Fraction(den.strip())
        vals.append(f)
    return vals


def test_softcap_series_coefficients_are_tanhs():
    assert _kernel_series_coefficients() == _tanh_maclaurin(5)


def test_softcap_series_truncation_bound():
    """Through y^9 the series is within 3e-9 of tanh on |y| <= 1/4 (the
    kernel's switch point), and the first omitted term bounds the error."""
    c = [float(x) for x in _tanh_maclaurin(6)]
    y = np.linspace(-0.25, 0.25, 200001)
    y2 = y * y
    series = y * (c[0] + y2 * (c[1] + y2 * (c[2] + y2 * (c[3] + y2 * c[4]))))
    err = np.abs(series - np.tanh(y))
    assert err.max() < 3e-9
    next_term = abs(c[5]) * 0.25 ** 11
    assert err.max() <= next_term * (1 + 1e-6)
    # increasing on the interval, as the max-of-raw-scores shortcut needs
    d = c[0] + y2 * (3 * c[1] + y2 * (5 * c[2] + y2 * (7 * c[3] + y2 * 9 * c[4])))
    assert d.min() > 0.9


def test_softcap_series_in_scaled_units():
    """The kernel evaluates s = v * (a1 + v^2 (a3 + ...)) with
    a_(2i+1) = softcap * log2(e) * t_(2i+1) * (scale / softcap)^(2i+1); in
    float32 that stays within a few ulp of softcap*log2(e)*tanh(v*scale/softcap)
    on the raw scores v where |v * scale / softcap| <= 1/4."""
    t = [float(x) for x in _tanh_maclaurin(5)]
    for softcap, scale in [(50.0, 1 / math.sqrt(192)), (3.0, 1 / math.sqrt(192)), (0.5, 0.3)]:
        ci, co = scale / softcap, softcap * math.log2(math.e)
        a = np.array([co * t[i] * ci ** (2 * i + 1) for i in range(5)], dtype=np.float32)
        vlim = 0.25 / ci
        v = np.linspace(-vlim, vlim, 20001).astype(np.float32)
        v2 = v * v
        q = np.float32(a[4])
        for ai in (a[3], a[2], a[1], a[0]):
            q = (q * v2 + ai).astype(np.float32)
        s = (v * q).astype(np.float32)
        exact = co * np.tanh(v.astype(np.float64) * ci)
        ulp = np.spacing(np.float32(co * math.tanh(0.25)))
        assert np.abs(s - exact).max() <= 4 * ulp
