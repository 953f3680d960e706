"""Randomised properties of the CPU oracle over small shapes and the whole
double range (hypothesis; a bounded number of examples so the CPU suite
stays quick).  Each property is checked against something other than the
oracle: exact rationals, numpy, or the other packed format."""
import math
from fractions import Fraction

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

FAST = settings(max_examples=40, deadline=None)


def _ternary(draw, N, K):
    return np.array(draw(st.lists(st.integers(-1, 1), min_size=N * K, max_size=N * K)),
                    dtype=np.int8).reshape(N, K)


@FAST
@given(st.data(), st.integers(1, 5), st.integers(1, 3))
def test_both_formats_round_trip_and_agree(data, N, G):
    K = 128 * G
    W = _ternary(data.draw, N, K)
    wp, bad = oracle.pack(W)
    p5, bad5 = oracle.pack_t5(W)
    assert bad == 0 and bad5 == 0
    back, _ = oracle.unpack(wp, K)
    back5, _ = oracle.unpack_t5(p5, K)
    assert np.array_equal(back, W) and np.array_equal(back5, W)


@FAST
@given(st.data(), st.integers(1, 3), st.integers(1, 4), st.integers(1, 2))
def test_linear_f64_matches_exact_rationals(data, T, N, G):
    K = 128 * G
    W = _ternary(data.draw, N, K)
    seed = data.draw(st.integers(0, 2 ** 16))
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=seed)
    x = synth.activations(T, K, seed=seed + 1, outlier_frac=0.02)
    xf = synth.bf16_bits_to_f32(x)
    fmt = data.draw(st.sampled_from(["2bit", "t5"]))
    wp = oracle.pack(W)[0] if fmt == "2bit" else oracle.pack_t5(W)[0]
    y, m = oracle.linear_f64(wp, s, x, T, K, N)
    for t in range(T):
        for n in range(N):
            tot, mag = Fraction(0), Fraction(0)
            for g in range(G):
                sg = Fraction(float(s[n, g]))
                part = sum((int(W[n, k]) * Fraction(float(xf[t, k]))
                            for k in range(128 * g, 128 * g + 128)), Fraction(0))
                parta = sum((abs(int(W[n, k]) * Fraction(float(xf[t, k])))
                             for k in range(128 * g, 128 * g + 128)), Fraction(0))
                tot += sg * part
                mag += abs(sg) * parta
            assert y[t, n] == pytest.approx(float(tot), rel=1e-12, abs=1e-12)
            assert m[t, n] == pytest.approx(float(mag), rel=1e-12, abs=1e-12)


@settings(max_examples=300, deadline=None)
@given(st.floats(allow_nan=False, allow_infinity=True, width=64))
def test_f64_to_bf16_is_nearest_even_everywhere(d):
    bits = int(oracle.f64_to_bf16(np.array([d]))[0])
    g = float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])
    if d == 0.0:
        assert g == 0.0 and math.copysign(1.0, g) == math.copysign(1.0, d)
        return
    a = abs(d)
    top = Fraction(2) ** 128 - Fraction(2) ** 119  # halfway between the largest finite and 2^128
    if math.isinf(a) or Fraction(a) >= top:
        assert math.isinf(g) and math.copysign(1.0, g) == math.copysign(1.0, d)
        return
    # neighbours on the bf16 grid: step 2^(e-8) in [2^(e-1), 2^e), 2^-133 below 2^-126
    _, e = math.frexp(a)
    step = Fraction(2) ** max(e - 8, -133)
    lo = (Fraction(a) // step) * step
    hi = lo + step
    dl, dh = Fraction(a) - lo, hi - Fraction(a)
    want = lo if dl < dh else hi if dh < dl else (lo if (lo / step) % 2 == 0 else hi)
    assert Fraction(abs(g)) == want
    assert math.copysign(1.0, g) == math.copysign(1.0, d)  # sign kept, also on a zero result
