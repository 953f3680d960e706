"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a hand-derived fixture, a brute-force
loop written independently here (Python integers / fractions, numpy's own
float16 and bfloat16 widening), a closed form, or an invariant.  A dropped
term, a wrong sign or group index, a transposed operand or a wrong bit order
in the oracle fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


def _bf16_value(bits):
    """bf16 bits -> exact Python float, independently of the oracle."""
    return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])


def _bf16_bits_exact(values):
    """Python floats that are exactly representable in bf16 -> bf16 bits."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def _brute_linear(W, s, xb):
    """y[t][n] = sum_g s[n,g] * sum_{k in g} w[n,k] x[t,k], with exact rationals."""
    N, K = W.shape
    T = xb.shape[0]
    G = K // 128
    y = np.zeros((T, N))
    for t in range(T):
        xs = [Fraction(_bf16_value(b)) for b in xb[t]]
        for n in range(N):
            tot = Fraction(0)
            for g in range(G):
                part = Fraction(0)
                for k in range(g * 128, (g + 1) * 128):
                    w = int(W[n, k])
                    if w:
                        part += w * xs[k]
                tot += Fraction(float(s[n, g])) * part
            y[t, n] = float(tot)
    return y


# ---------------------------------------------------------------- packing

def test_pack_layout_golden_words():
    for name, ws, word in _read_fixture("pack_layout.txt"):
        w = np.array([int(v) for v in ws.split(",")], dtype=np.int8).reshape(1, 16)
        wp, bad = oracle.pack(w)
        assert bad == 0
        assert int(wp[0, 0]) == int(word, 16), name
        back, bad2 = oracle.unpack(wp, 16)
        assert bad2 == 0 and np.array_equal(back, w), name


def test_pack_word_and_row_order():
    # Two rows, K = 48: word index n*(K/16) + k/16.  One nonzero weight per row
    # at a hand-chosen position; every other weight is 0 (no bits set).
    W = np.zeros((2, 48), dtype=np.int8)
    W[0, 17] = -1   # word 1 of row 0, byte 0, i = 1 -> 0x0000000A
    W[1, 40] = 1    # word 2 of row 1, byte 2, i = 0 -> 0x00010000
    wp, _ = oracle.pack(W)
    expect = np.zeros((2, 3), dtype=np.uint32)
    expect[0, 1] = 0x0000000A
    expect[1, 2] = 0x00010000
    assert np.array_equal(wp, expect)


def test_pack_unpack_round_trip_random():
    W = synth.ternary_weights(7, 256, 0.4, seed=11)
    wp, bad = oracle.pack(W)
    assert bad == 0
    back, bad2 = oracle.unpack(wp, 256)
    assert bad2 == 0 and np.array_equal(back, W)


def test_pack_counts_invalid_values():
    W = np.zeros((1, 16), dtype=np.int8)
    W[0, 3] = 2
    W[0, 9] = -5
    wp, bad = oracle.pack(W)
    assert bad == 2
    assert int(wp[0, 0]) == 0  # invalid values stored as 0


def test_unpack_counts_invalid_pair():
    # weight 3 of byte 0: negative bit (bit 7) set without its nonzero bit (bit 5)
    wp = np.array([[0x00000080]], dtype=np.uint32)
    W, bad = oracle.unpack(wp, 16)
    assert bad == 1 and W[0, 3] == 0 and not W.any()


# ---------------------------------------------------------------- bf16 rungs

@pytest.mark.parametrize("T,K,N", [(1, 128, 3), (3, 256, 5), (2, 384, 4)])
def test_linear_f64_brute_force(T, K, N):
    W = synth.ternary_weights(N, K, 0.4, seed=T * 100 + N)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=T + N)
    x = synth.activations(T, K, seed=N, outlier_frac=0.02)
    wp, _ = oracle.pack(W)
    y, m = oracle.linear_f64(wp, s, x, T, K, N)
    yb = _brute_linear(W, s, x)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-15)
    # m = sum |s w x|, brute-forced with numpy's own widenings
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    sf = np.repeat(s.astype(np.float64), 128, axis=1)
    mb = np.abs(xf[:, None, :] * (W[None, :, :] * sf[None, :, :])).sum(-1)
    np.testing.assert_allclose(m, mb, rtol=1e-12)


def test_linear_f64_zero_weights_give_zero():
    T, K, N = 2, 256, 6
    W = np.zeros((N, K), dtype=np.int8)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=1)
    x = synth.activations(T, K, seed=2)
    wp, _ = oracle.pack(W)
    y, m = oracle.linear_f64(wp, s, x, T, K, N)
    assert np.all(y == 0.0) and np.all(m == 0.0)


def test_linear_f64_all_plus_one_is_scaled_group_sums():
    T, K, N = 2, 384, 3
    W = np.ones((N, K), dtype=np.int8)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=3)
    x = synth.activations(T, K, seed=4)
    wp, _ = oracle.pack(W)
    y, _ = oracle.linear_f64(wp, s, x, T, K, N)
    xf = [[_bf16_value(b) for b in row] for row in x]
    for t in range(T):
        for n in range(N):
            expect = math.fsum(float(s[n, g]) * math.fsum(xf[t][g * 128:(g + 1) * 128])
                               for g in range(K // 128))
            assert y[t, n] == pytest.approx(expect, rel=1e-13, abs=1e-15)


def test_linear_f64_one_hot_selects_one_weight():
    T, K, N = 1, 512, 8
    W = synth.ternary_weights(N, K, 1.0 / 3.0, seed=5)
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=6)
    wp, _ = oracle.pack(W)
    for k0 in (0, 127, 128, 300, 511):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k0] = _bf16_bits_exact([1.0])[0]
        y, _ = oracle.linear_f64(wp, s, x, T, K, N)
        expect = s[:, k0 // 128].astype(np.float64) * W[:, k0]
        assert np.array_equal(y[0], expect), k0


def test_linear_f64_negation_and_additivity():
    T, K, N = 2, 256, 5
    W = synth.ternary_weights(N, K, 0.4, seed=7)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=8)
    wp, _ = oracle.pack(W)
    rng = np.random.default_rng(9)
    a = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    b = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    ya, _ = oracle.linear_f64(wp, s, _bf16_bits_exact(a), T, K, N)
    yb, _ = oracle.linear_f64(wp, s, _bf16_bits_exact(b), T, K, N)
    yab, _ = oracle.linear_f64(wp, s, _bf16_bits_exact(a + b), T, K, N)
    yneg, _ = oracle.linear_f64(wp, s, _bf16_bits_exact(-a), T, K, N)
    np.testing.assert_allclose(yab, ya + yb, rtol=1e-12, atol=1e-12)
    assert np.array_equal(yneg, -ya)


def test_linear_f64_sampled_matches_full():
    T, K, N = 3, 256, 9
    c = synth.case("x", T, K=K, N=N, seed=12)
    wp, _ = oracle.pack(c.W)
    y, m = oracle.linear_f64(wp, c.scales, c.x, T, K, N)
    ti = np.array([0, 2, 1, 2], dtype=np.int32)
    ni = np.array([8, 0, 4, 8], dtype=np.int32)
    ys, ms = oracle.linear_f64_sampled(wp, c.scales, c.x, K, N, ti, ni)
    assert np.array_equal(ys, y[ti, ni]) and np.array_equal(ms, m[ti, ni])


# ---------------------------------------------------------------- s8 quantiser

def test_quant_s8_golden_ties():
    for name, xs_txt, q_txt, scale_txt in _read_fixture("quant_ties.txt"):
        xv = [float(v) for v in xs_txt.split(",")]
        qv = np.array([int(v) for v in q_txt.split(",")], dtype=np.int8)
        q, xs = oracle.quant_s8(_bf16_bits_exact(xv).reshape(1, -1), 1, len(xv))
        assert np.array_equal(q[0], qv), name
        assert float(xs[0]) == float(scale_txt), name


def test_quant_s8_properties_random():
    T, K = 5, 1024
    x = synth.activations(T, K, seed=21, outlier_frac=0.01)
    q, xs = oracle.quant_s8(x, T, K)
    xf = synth.bf16_bits_to_f32(x)
    for t in range(T):
        a = float(np.max(np.abs(xf[t])))
        # x_scale is the fp32 quotient a/127 (numpy's IEEE float32 division)
        assert xs[t] == np.float32(a) / np.float32(127.0)
        # the absmax channel maps to +-127
        k = int(np.argmax(np.abs(xf[t])))
        assert abs(int(q[t, k])) == 127 and np.sign(q[t, k]) == np.sign(xf[t, k])
        # every code is within half a step of x / x_scale
        err = np.abs(q[t].astype(np.float64) - xf[t].astype(np.float64) / float(xs[t]))
        assert np.all(err <= 0.5 + 1e-6)
        assert np.all(np.abs(q[t]) <= 127)


def test_quant_s8_integer_rows_are_identity():
    # Integer rows holding +-127 quantise to themselves (x_scale = 1).
    rng = np.random.default_rng(22)
    x = rng.integers(-127, 128, size=(3, 256)).astype(np.float32)
    x[:, 7] = 127.0
    x[1, 7] = -127.0
    q, xs = oracle.quant_s8(_bf16_bits_exact(x), 3, 256)
    assert np.all(xs == 1.0)
    assert np.array_equal(q.astype(np.float32), x)


# ---------------------------------------------------------------- s8 linear

@pytest.mark.parametrize("T,K,N", [(1, 128, 4), (3, 256, 5)])
def test_linear_s8_brute_force(T, K, N):
    W = synth.ternary_weights(N, K, 0.4, seed=31 + T)
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=32)
    x = synth.activations(T, K, seed=33, outlier_frac=0.01)
    wp, _ = oracle.pack(W)
    q, xs = oracle.quant_s8(x, T, K)
    y, m, acc = oracle.linear_s8(wp, s, q, xs, T, K, N, want_acc=True)
    G = K // 128
    for t in range(T):
        for n in range(N):
            tot = Fraction(0)
            for g in range(G):
                a = sum(int(q[t, k]) * int(W[n, k]) for k in range(g * 128, (g + 1) * 128))
                assert acc[t, n, g] == a
                tot += Fraction(float(s[n, g])) * a
            expect = float(Fraction(float(xs[t])) * tot)
            assert y[t, n] == pytest.approx(expect, rel=1e-12, abs=1e-300)


def test_linear_s8_unit_scale_integer_trick():
    # scales = 1 and integer activations containing +-127: q = x, x_scale = 1,
    # so y must equal the exact integer dot product.
    T, K, N = 2, 384, 6
    W = synth.ternary_weights(N, K, 0.4, seed=41)
    s = np.ones((N, K // 128), dtype=np.float16)
    rng = np.random.default_rng(42)
    x = rng.integers(-127, 128, size=(T, K)).astype(np.float32)
    x[:, 0] = 127.0
    wp, _ = oracle.pack(W)
    q, xs = oracle.quant_s8(_bf16_bits_exact(x), T, K)
    y, _, _ = oracle.linear_s8(wp, s, q, xs, T, K, N)
    exact = x.astype(np.int64) @ W.astype(np.int64).T
    assert np.array_equal(y, exact.astype(np.float64))


def test_linear_s8_sampled_matches_full():
    T, K, N = 2, 256, 7
    c = synth.case("x", T, K=K, N=N, seed=43)
    wp, _ = oracle.pack(c.W)
    q, xs = oracle.quant_s8(c.x, T, K)
    y, m, acc = oracle.linear_s8(wp, c.scales, q, xs, T, K, N, want_acc=True)
    ti = np.array([1, 0, 1], dtype=np.int32)
    ni = np.array([6, 3, 0], dtype=np.int32)
    ys, ms, accs = oracle.linear_s8_sampled(wp, c.scales, q, xs, K, N, ti, ni, want_acc=True)
    assert np.array_equal(ys, y[ti, ni]) and np.array_equal(ms, m[ti, ni])
    assert np.array_equal(accs, acc[ti, ni])


# ---------------------------------------------------------------- invalid codes

def _brute_s8(W, s, q, xs):
    """y = xs * sum_g s * sum_{k in g} q w with exact rationals; the integer
    accumulators acc[t, n, g] beside it."""
    N, K = W.shape
    T, G = q.shape[0], K // 128
    y = np.zeros((T, N))
    acc = np.zeros((T, N, G), dtype=np.int64)
    for t in range(T):
        for n in range(N):
            tot = Fraction(0)
            for g in range(G):
                a = sum(int(q[t, k]) * int(W[n, k]) for k in range(g * 128, (g + 1) * 128))
                acc[t, n, g] = a
                tot += Fraction(float(s[n, g])) * a
            y[t, n] = float(Fraction(float(xs[t])) * tot)
    return y, acc


def test_invalid_2bit_pairs_read_as_zero_in_both_rungs():
    # The library documents that its kernels read the invalid pair
    # (nz = 0, neg = 1) as weight 0; the oracle's definitions must too.
    T, K, N = 2, 256, 3
    W = synth.ternary_weights(N, K, 0.2, seed=61)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=62)
    x = synth.activations(T, K, seed=63)
    wp, _ = oracle.pack(W)
    # turn three nonzero weights into the invalid pair: keep only the
    # negative bit (nonzero bit at P[i] = {0,1,4,5}[k%4], negative bit 2 above)
    Wz = W.copy()
    for n, start in [(0, 5), (1, 130), (2, 200)]:
        k = start + int(np.flatnonzero(W[n, start:])[0])  # first nonzero weight from start
        p = 8 * ((k % 16) // 4) + [0, 1, 4, 5][k % 4]
        wp[n, k // 16] = (int(wp[n, k // 16]) & ~(1 << p)) | (1 << (p + 2))
        Wz[n, k] = 0
    back, bad = oracle.unpack(wp, K)
    assert bad == 3 and np.array_equal(back, Wz)
    y, _ = oracle.linear_f64(wp, s, x, T, K, N)
    np.testing.assert_allclose(y, _brute_linear(Wz, s, x), rtol=1e-12, atol=1e-15)
    q, xs = oracle.quant_s8(x, T, K)
    y8, _, acc = oracle.linear_s8(wp, s, q, xs, T, K, N, want_acc=True)
    yb, accb = _brute_s8(Wz, s, q, xs)
    assert np.array_equal(acc, accb)
    np.testing.assert_allclose(y8, yb, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- base-3 packing

def _t5_digits(v):
    """The five base-3 digits of v, least significant first, from numpy's
    own base conversion."""
    return [int(d) for d in reversed(np.base_repr(v, 3).zfill(5))]


def test_t5_golden_bytes():
    for name, ws, byte in _read_fixture("t5_bytes.txt"):
        w5 = [int(v) for v in ws.split(",")]
        W = np.zeros((1, 128), dtype=np.int8)
        W[0, 10:15] = w5  # byte 2 of the group holds weights 10..14
        p, bad = oracle.pack_t5(W)
        assert bad == 0 and p.shape == (1, 26)
        assert int(p[0, 2]) == int(byte), name
        assert all(int(b) == 121 for j, b in enumerate(p[0]) if j != 2), name
        back, bad2 = oracle.unpack_t5(p, 128)
        assert bad2 == 0 and np.array_equal(back, W), name


def test_t5_closed_form_groups_and_padding():
    # A group of 128 equal weights: 25 full bytes and a last byte holding
    # three weights plus two padding digits written as weight 0 (digit 1).
    for w, full, last in [(0, 121, 1 + 3 + 9 + 27 + 81),
                          (-1, 0, 27 + 81),
                          (1, 242, 2 + 6 + 18 + 27 + 81)]:
        W = np.full((2, 256), w, dtype=np.int8)
        p, _ = oracle.pack_t5(W)
        rows = p.reshape(2, 2, 26)
        assert np.all(rows[:, :, :25] == full), w
        assert np.all(rows[:, :, 25] == last), w
    # storage: 26 bytes and one fp16 scale per 128 weights = 1.75 bits per
    # weight, the average the page gives for this format
    assert (26 + 2) * 8 / 128 == 1.75


def test_t5_unpack_every_byte_value_against_base_repr():
    K = 256
    for v in range(256):
        p = np.full((1, 2 * 26), 121, dtype=np.uint8)  # all weights 0
        p[0, 26 + 7] = v                               # group 1, byte 7: k = 163..167
        W, bad = oracle.unpack_t5(p, K)
        expect = np.zeros((1, K), dtype=np.int8)
        if v <= 242:
            expect[0, 163:168] = [d - 1 for d in _t5_digits(v)]
            assert bad == 0, v
        else:
            assert bad == 1, v                         # invalid byte: weights read 0
        assert np.array_equal(W, expect), v


def test_t5_last_byte_ignores_padding_digits():
    # digits 3 and 4 of byte 25 lie past the group: any value there leaves
    # the group's weights unchanged
    W = synth.ternary_weights(1, 128, 0.4, seed=64)
    p, _ = oracle.pack_t5(W)
    low = int(p[0, 25]) % 27
    for pad in range(9):
        q = p.copy()
        q[0, 25] = low + 27 * pad
        back, bad = oracle.unpack_t5(q, 128)
        assert bad == 0 and np.array_equal(back, W), pad


def test_t5_pack_counts_invalid_values():
    W = np.zeros((1, 128), dtype=np.int8)
    W[0, 0] = 3
    W[0, 127] = -2
    p, bad = oracle.pack_t5(W)
    assert bad == 2 and np.all(p == 121)  # stored as weight 0


def test_t5_round_trip_and_agreement_with_2bit_code():
    N, K = 9, 640
    W = synth.ternary_weights(N, K, 0.4, seed=65)
    p, bad = oracle.pack_t5(W)
    assert bad == 0 and p.shape == (N, 5 * 26)
    back, bad2 = oracle.unpack_t5(p, K)
    assert bad2 == 0 and np.array_equal(back, W)
    wp, _ = oracle.pack(W)
    back2, _ = oracle.unpack(wp, K)
    assert np.array_equal(back, back2)


@pytest.mark.parametrize("T,K,N", [(1, 128, 3), (3, 384, 4)])
def test_t5_linear_f64_brute_force_and_equal_to_2bit(T, K, N):
    W = synth.ternary_weights(N, K, 0.4, seed=66 + T)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=67)
    x = synth.activations(T, K, seed=68, outlier_frac=0.02)
    p, _ = oracle.pack_t5(W)
    y, m = oracle.linear_f64(p, s, x, T, K, N)
    np.testing.assert_allclose(y, _brute_linear(W, s, x), rtol=1e-12, atol=1e-15)
    # the same weights in the 2-bit code give the same sums in the same order
    wp, _ = oracle.pack(W)
    y2, m2 = oracle.linear_f64(wp, s, x, T, K, N)
    assert np.array_equal(y, y2) and np.array_equal(m, m2)
    ti = np.array([T - 1, 0], dtype=np.int32)
    ni = np.array([0, N - 1], dtype=np.int32)
    ys, ms = oracle.linear_f64_sampled(p, s, x, K, N, ti, ni)
    assert np.array_equal(ys, y[ti, ni]) and np.array_equal(ms, m[ti, ni])


def test_t5_linear_s8_brute_force_and_equal_to_2bit():
    T, K, N = 3, 256, 5
    W = synth.ternary_weights(N, K, 0.4, seed=69)
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=70)
    x = synth.activations(T, K, seed=71, outlier_frac=0.01)
    p, _ = oracle.pack_t5(W)
    q, xs = oracle.quant_s8(x, T, K)
    y, m, acc = oracle.linear_s8(p, s, q, xs, T, K, N, want_acc=True)
    yb, accb = _brute_s8(W, s, q, xs)
    assert np.array_equal(acc, accb)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-300)
    wp, _ = oracle.pack(W)
    y2, m2, acc2 = oracle.linear_s8(wp, s, q, xs, T, K, N, want_acc=True)
    assert np.array_equal(y, y2) and np.array_equal(m, m2) and np.array_equal(acc, acc2)
    ti = np.array([2, 0], dtype=np.int32)
    ni = np.array([4, 1], dtype=np.int32)
    ys, ms, accs = oracle.linear_s8_sampled(p, s, q, xs, K, N, ti, ni, want_acc=True)
    assert np.array_equal(ys, y[ti, ni]) and np.array_equal(accs, acc[ti, ni])


def test_t5_invalid_bytes_read_as_zero_in_both_rungs():
    T, K, N = 2, 256, 2
    W = synth.ternary_weights(N, K, 0.2, seed=72)
    s = synth.scales_uniform(N, K, 0.01, 0.05, seed=73)
    x = synth.activations(T, K, seed=74)
    p, _ = oracle.pack_t5(W)
    Wz = W.copy()
    p[0, 3] = 243          # group 0, byte 3: k = 15..19
    p[1, 26 + 25] = 255    # group 1, last byte: k = 253..255
    Wz[0, 15:20] = 0
    Wz[1, 253:256] = 0
    back, bad = oracle.unpack_t5(p, K)
    assert bad == 2 and np.array_equal(back, Wz)
    y, _ = oracle.linear_f64(p, s, x, T, K, N)
    np.testing.assert_allclose(y, _brute_linear(Wz, s, x), rtol=1e-12, atol=1e-15)
    q, xs = oracle.quant_s8(x, T, K)
    y8, _, acc = oracle.linear_s8(p, s, q, xs, T, K, N, want_acc=True)
    yb, accb = _brute_s8(Wz, s, q, xs)
    assert np.array_equal(acc, accb)
    np.testing.assert_allclose(y8, yb, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- rotation

def test_f64_to_bf16_golden():
    for name, val, bits in _read_fixture("bf16_round.txt"):
        got = oracle.f64_to_bf16(np.array([float.fromhex(val)]))
        assert int(got[0]) == int(bits, 16), name


def _bf16_neighbours(d):
    """The two bf16 values around a positive normal double d, by exact
    rational arithmetic: the grid step is 2^(e-8) for d in [2^(e-1), 2^e)."""
    m, e = math.frexp(d)
    step = Fraction(2) ** (e - 8)
    lo = (Fraction(d) // step) * step
    return lo, lo + step, step


def test_f64_to_bf16_random_against_exact_rationals():
    rng = np.random.default_rng(91)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-60, 60, size=4000))
    got = synth.bf16_bits_to_f32(oracle.f64_to_bf16(v)).astype(np.float64)
    for d, g in zip(v, got):
        a = abs(float(d))
        lo, hi, step = _bf16_neighbours(a)
        dl, dh = Fraction(a) - lo, hi - Fraction(a)
        if dl < dh:
            want = lo
        elif dh < dl:
            want = hi
        else:  # tie: the neighbour whose last fraction bit is 0
            want = lo if (lo / step) % 2 == 0 else hi
        assert Fraction(abs(float(g))) == want and np.sign(g) == np.sign(d), (d, g)


@pytest.mark.parametrize("B", [2, 16, 64, 1024])
def test_rotate_matches_scipy_hadamard(B):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    T, K = 3, 2048
    x = synth.activations(T, K, seed=92, outlier_frac=0.01)
    exact, xr = oracle.rotate(x, T, K, block=B)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    H = scipy_linalg.hadamard(B).astype(np.float64) / math.sqrt(B)
    ref = (xf.reshape(T, K // B, B) @ H.T).reshape(T, K)
    np.testing.assert_allclose(exact, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(xr, oracle.f64_to_bf16(exact))


def test_rotate_closed_forms():
    B, K = 1024, 2048
    # one-hot input e_j in block 1: the output is column j of H / 32, exactly
    for j in (0, 1, 5, 513, 1023):
        xb = np.zeros((1, K), dtype=np.float32)
        xb[0, B + j] = 1.0
        exact, _ = oracle.rotate(_bf16_bits_exact(xb), 1, K)
        signs = np.array([(-1) ** bin(i & j).count("1") for i in range(B)], dtype=np.float64)
        assert not exact[0, :B].any()
        assert np.array_equal(exact[0, B:], signs / 32.0), j
    # a constant block of ones sums to 1024/32 = 32 in output 0 and cancels elsewhere
    xb = np.zeros((1, K), dtype=np.float32)
    xb[0, :B] = 1.0
    exact, xr = oracle.rotate(_bf16_bits_exact(xb), 1, K)
    assert exact[0, 0] == 32.0 and not exact[0, 1:].any()
    assert int(xr[0, 0]) == 0x4200  # 32.0 in bf16


def test_rotate_is_orthonormal_and_blockwise():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    T, K, B = 2, 3072, 1024
    x = synth.activations(T, K, seed=93, outlier_frac=0.02)
    exact, _ = oracle.rotate(x, T, K)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    # Parseval: the norm of each block is kept
    np.testing.assert_allclose((exact.reshape(T, 3, B) ** 2).sum(-1),
                               (xf.reshape(T, 3, B) ** 2).sum(-1), rtol=1e-12)
    # rotating back with H / 32 returns the input
    H = scipy_linalg.hadamard(B).astype(np.float64) / 32.0
    back = (exact.reshape(T, 3, B) @ H.T).reshape(T, K)
    np.testing.assert_allclose(back, xf, rtol=0, atol=1e-12)
    # a change inside block 1 leaves blocks 0 and 2 bit-identical
    x2 = x.copy()
    x2[:, B + 7] ^= 0x0040
    exact2, _ = oracle.rotate(x2, T, K)
    assert np.array_equal(exact2[:, :B], exact[:, :B])
    assert np.array_equal(exact2[:, 2 * B:], exact[:, 2 * B:])
    assert not np.array_equal(exact2[:, B:2 * B], exact[:, B:2 * B])


# ---------------------------------------------------------------- generators

def test_synth_distributions():
    W = synth.ternary_weights(64, 4096, 0.4, seed=0)
    frac0 = float(np.mean(W == 0))
    assert abs(frac0 - 0.4) < 0.01
    assert abs(float(np.mean(W == 1)) - 0.3) < 0.01
    s = synth.scales_lognormal(64, 4096, -3.5, 0.3, seed=0).astype(np.float64)
    assert abs(np.mean(np.log(s)) + 3.5) < 0.05
    x = synth.bf16_bits_to_f32(synth.activations(4, 5120, seed=0, outlier_frac=0.01))
    big = np.abs(x).max(axis=0) > 10
    assert 30 <= int(big.sum()) <= 51  # 51 outlier channels; a few may draw small values
