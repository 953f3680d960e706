"""The number facts the kernels' exactness rests on, checked exhaustively on
the CPU.  fp8 roundings are written out here from their definition (round to
nearest, ties to even, on the format's grid) and cross-checked against
torch's own float8 conversions.

- The 2-bit code turns into the e4m3 encoding of w / 8 with one mask.
- s8 rung: every int8 code q in [-127, 127] is the exact sum of two e4m3
  values 16 * floor((q + 8) / 16) and the remainder in [-8, 7] (the int8
  decode variant's split), and of 16 * rint(q / 16) and the remainder in
  [-8, 8] (the s8 quantiser's split, through its fp32 magic-number steps).
- s8 quantiser: the code rint(x * (1/scale)) equals rint(x / scale) (the
  quotient rounded once) wherever the product lies at least 2^-15 from a
  half-integer, for every finite bf16 x up to the row's absmax, and the
  product is never farther than 1.91e-5 from the rounded quotient.
- bf16 rungs: a bf16 value scaled into (-2^15, 2^15) splits as h1 = e5m2(v),
  h2 = e5m2(v - h1), h3 = e5m2(v - h1 - h2) with h1 + h2 + h3 == v whenever
  |v| >= 2^-7, every nonzero piece a normal e5m2 value and every fp32
  difference exact.  With the group absmax scaled into [2^14, 2^15) that
  covers every element within 21 binades of the absmax's binade; the rest
  are the "leftovers" the kernels add exactly on the CUDA cores.
- The old two-piece e4m3 split fails the bf16 bar on an input with the
  group's absmax on a zero weight; the three-piece split with leftovers
  meets it on the same input, in an emulation of the kernels' arithmetic.
- The per-group sums the tensor core accumulates on the s8 rung stay within
  11 significant bits, so their fp32 accumulation is exact.
"""
from fractions import Fraction

import numpy as np
import torch

import synth

E4M3 = torch.float8_e4m3fn
E5M2 = torch.float8_e5m2


def _e4m3(values):
    """float values -> their e4m3 roundings as float64 (round to nearest even)."""
    return torch.tensor(np.asarray(values, dtype=np.float32)).to(E4M3).to(torch.float64).numpy()


def rne_e5m2(v):
    """Round float64 values to e5m2 (1 sign, 5 exponent bits with bias 15, 2
    mantissa bits; subnormal step 2^-16), nearest with ties to even.  Values
    here stay below the largest finite e5m2 (57344)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14.0)                 # subnormals share the 2^-14 binade's step
    q = np.exp2(e - 2.0)                     # step of the binade: 3 significant bits
    r = a / q                                # exact: q is a power of two
    n = np.floor(r)
    frac = r - n
    n = n + ((frac > 0.5) | ((frac == 0.5) & (np.fmod(n, 2.0) == 1.0)))
    out = np.sign(v) * n * q
    assert np.all(np.abs(out) <= 57344.0)
    return out


def _all_bf16_between(lo, hi):
    """Every finite bf16 value with lo <= |v| < hi, both signs."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    v = (bits << 16).view(np.float32).astype(np.float64)
    v = v[(v >= lo) & (v < hi)]
    return np.concatenate([v, -v])


def test_weight_code_bytes_are_e4m3_of_w_over_8():
    # byte after the mask: 0x00 -> 0, 0x20 -> +1/8, 0xA0 -> -1/8, and the
    # invalid pair's 0x80 -> -0 (contributes nothing)
    b = torch.tensor([0x00, 0x20, 0xA0, 0x80], dtype=torch.uint8).view(E4M3).to(torch.float64)
    assert b.tolist() == [0.0, 0.125, -0.125, 0.0]
    assert np.signbit(b.numpy()[3])


def test_int8_codes_split_into_two_exact_e4m3_pieces():
    q = np.arange(-127, 128)
    h = np.floor((q + 8) / 16).astype(np.int64)
    assert h.min() == -8 and h.max() == 8
    p1, p2 = 16 * h, q - 16 * h
    assert p2.min() == -8 and p2.max() == 7
    assert np.array_equal(_e4m3(p1), p1.astype(np.float64))
    assert np.array_equal(_e4m3(p2), p2.astype(np.float64))
    assert np.array_equal(p1 + p2, q)


def test_int8_codes_split_by_rint_in_fp32():
    # the s8 quantiser's steps on fp32 values: t = q / 16 + 1.5 * 2^23 (one
    # rounding: q / 16 is exact), p1 = 16 t - 16 * 1.5 * 2^23 (exact), p2 = q - p1
    q = np.arange(-127, 128).astype(np.float32)
    t = q * np.float32(0.0625) + np.float32(12582912.0)
    p1 = t * np.float32(16.0) - np.float32(201326592.0)
    p2 = q - p1
    qi = np.arange(-127, 128)
    h = np.rint(qi / 16.0)                      # ties to even
    assert np.array_equal(p1.astype(np.int64), 16 * h.astype(np.int64))
    assert p1.min() == -128 and p1.max() == 128 and np.all(p1 % 16 == 0)
    assert p2.min() == -8 and p2.max() == 8
    assert np.array_equal(_e4m3(p1), p1.astype(np.float64))
    assert np.array_equal(_e4m3(p2), p2.astype(np.float64))
    assert np.array_equal((p1 + p2).astype(np.int64), qi)


def _bf16_magnitudes_up_to(a):
    codes = np.arange(0, 0x7F80, dtype=np.uint32)
    mags = (codes << 16).view(np.float32)
    return mags[mags <= a]


def test_quant_product_and_check_matches_the_division():
    # scales on the product path (scale = absmax / 127 normal), absmax values
    # in bf16 from 2^-118 up to the largest finite bf16
    rng = np.random.default_rng(8)
    codes = np.unique(np.concatenate([rng.integers(0x0480, 0x7F80, size=40),
                                      [0x3F80, 0x42FE, 0x7F7F, 0x0480]])).astype(np.uint32)
    margin = np.float32(2.0 ** -15)
    for c in codes:
        a = (np.uint32(c) << 16).view(np.float32)
        scale = np.float32(a) / np.float32(127.0)
        assert scale >= np.float32(2.0 ** -126)           # the kernel's fast-path test
        inv = np.float32(1.0) / scale
        v = _bf16_magnitudes_up_to(a)
        v = np.concatenate([v, -v])
        quot = v / scale                                  # rounded once (IEEE)
        q0 = v * inv                                      # rounded product
        prod = v.astype(np.float64) * np.float64(inv)     # exact product (FMA-contracted form)
        assert np.abs(q0.astype(np.float64) - quot).max() < 1.91e-5
        assert np.abs(prod - quot).max() < 1.91e-5
        for qq in (q0.astype(np.float64), prod):
            r = np.rint(q0)
            safe = np.abs(qq - r) < 0.5 - margin
            assert np.array_equal(r[safe], np.rint(quot)[safe])
            # and the product path never leaves [-127, 127]
            assert np.abs(r).max() <= 127


def test_rne_e5m2_agrees_with_torch():
    # every bf16 value below the e5m2 range's top, including subnormals and ties
    v = _all_bf16_between(0.0, 49152.0)
    mine = rne_e5m2(v)
    ref = torch.tensor(v.astype(np.float32)).to(E5M2).to(torch.float64).numpy()
    assert np.array_equal(mine, ref)
    # hand-picked ties: 1.125 lies between 1.0 and 1.25 (even: 1.0); 1.375 -> 1.5
    assert rne_e5m2([1.125, 1.375, 2.0 ** -17, 3 * 2.0 ** -17]).tolist() == \
        [1.0, 1.5, 0.0, 2.0 ** -15]


def _round3_fp32(x):
    """The kernels' round3 in fp32: (x + c) - c with c = 1.5 * 2^(exp(x) + 21)."""
    x = np.asarray(x, dtype=np.float32)
    e = x.view(np.uint32) & np.uint32(0x7F800000)
    c = ((e + np.uint32(21 << 23)) | np.uint32(0x00400000)).view(np.float32)
    return ((x + c) - c).astype(np.float64)


def test_round3_is_rne_to_e5m2_on_the_pieces_range():
    # every fp32 value with at most 12 significant bits in [2^-14, 2^15), both
    # signs: round3 equals e5m2 round to nearest even (and 0 stays 0)
    mant = np.arange(0, 1 << 11, dtype=np.uint32) << np.uint32(12)
    exps = np.arange(127 - 14, 127 + 15, dtype=np.uint32) << np.uint32(23)
    bits = (exps[:, None] | mant[None, :]).ravel()
    v = bits.view(np.float32)
    v = np.concatenate([v, -v, np.zeros(1, np.float32)])
    assert np.array_equal(_round3_fp32(v), rne_e5m2(v.astype(np.float64)))


def _three_pieces_round3(v):
    v32 = v.astype(np.float32)
    h1 = _round3_fp32(v32)
    r1 = v32 - h1.astype(np.float32)
    h2 = _round3_fp32(r1)
    r2 = r1 - h2.astype(np.float32)
    return h1, h2, r2.astype(np.float64)


def test_kernel_split_formula_matches_the_definition():
    v = _all_bf16_between(2.0 ** -7, 2.0 ** 15)
    h1, h2, h3, _, _ = _three_pieces(v)
    g1, g2, g3 = _three_pieces_round3(v)
    assert np.array_equal(g1, h1) and np.array_equal(g2, h2) and np.array_equal(g3, h3)
    assert np.array_equal(rne_e5m2(g3), g3)  # the last piece is an e5m2 value


def _three_pieces(v):
    """The kernels' split in fp32: pieces and the two fp32 remainders."""
    v32 = v.astype(np.float32)
    h1 = rne_e5m2(v32.astype(np.float64))
    r1 = (v32 - h1.astype(np.float32)).astype(np.float64)
    h2 = rne_e5m2(r1)
    r2 = (r1.astype(np.float32) - h2.astype(np.float32)).astype(np.float64)
    h3 = rne_e5m2(r2)
    return h1, h2, h3, r1, r2


def test_bf16_three_piece_e5m2_split_exact_in_window():
    v = _all_bf16_between(2.0 ** -7, 2.0 ** 15)
    h1, h2, h3, r1, r2 = _three_pieces(v)
    assert np.array_equal(r1, v - h1)             # fp32 differences are exact
    assert np.array_equal(r2, v - h1 - h2)
    assert np.array_equal(h1 + h2 + h3, v)        # the pieces sum to v exactly
    for h in (h1, h2, h3):                         # every nonzero piece is normal
        nz = h != 0
        assert np.all(np.abs(h[nz]) >= 2.0 ** -14)
    # the window is needed: below 2^-7 some values lose bits
    lo = _all_bf16_between(2.0 ** -12, 2.0 ** -7)
    g1, g2, g3, _, _ = _three_pieces(lo)
    assert not np.array_equal(g1 + g2 + g3, lo)


def test_group_scale_puts_the_absmax_in_range_and_sets_the_leftover_limit():
    # m 2^p in [2^14, 2^15) with p = 14 - floor(log2 m); leftover limit
    # tau = f 2^-10 with f = 2^(floor(log2 m) - 11): |x| >= tau <=> |x 2^p| >= 2^-7
    for m in (1.0, 3.0, 80.0, 2.0 ** 100, 1.5 * 2 ** -120, 2.0 ** -133):
        el = int(np.floor(np.log2(m)))
        p = 14 - el
        assert 2.0 ** 14 <= Fraction(m) * Fraction(2) ** p < 2.0 ** 15
        f = Fraction(2) ** (el - 11)
        assert f == Fraction(2) ** (3 - p)
        tau = f * Fraction(1, 1024)
        assert tau * Fraction(2) ** p == Fraction(1, 128)


def _bf16(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32)))


def _emulate_group_three_piece(x, w, s):
    """The kernels' arithmetic for one group and one output: pieces of the
    in-window elements (exact products, accumulated in fp64 here: the fp32
    accumulation error is bounded separately), leftovers added exactly."""
    x = x.astype(np.float64)
    m = np.abs(x).max()
    el = int(np.floor(np.log2(m)))
    p = 14 - el
    tau = 2.0 ** (el - 21)
    left = (x != 0) & (np.abs(x) < tau)
    v = np.where(left, 0.0, x * 2.0 ** p)
    h1, h2, h3, _, _ = _three_pieces(v)
    f = 2.0 ** (3 - p)
    d = np.sum((w / 8.0) * h1) + np.sum((w / 8.0) * h2) + np.sum((w / 8.0) * h3)
    return s * (f * d + np.sum(w[left] * x[left]))


def _emulate_group_two_piece_e4m3(x, w, s):
    """The earlier split: absmax into [128, 256), two e4m3 pieces."""
    x = x.astype(np.float64)
    el = int(np.floor(np.log2(np.abs(x).max())))
    p = 7 - el
    v = x * 2.0 ** p
    h1 = _e4m3(v)
    h2 = _e4m3((v.astype(np.float32) - h1.astype(np.float32)))
    return s * 2.0 ** (3 - p) * np.sum((w / 8.0) * (h1 + h2))


def test_absmax_on_a_zero_weight_two_piece_fails_three_piece_meets_the_bar():
    # one group: x = 80 on a zero weight, 0.01 on 127 weights of +1, s = 0.03
    x = _bf16(np.array([80.0] + [0.01] * 127))
    w = np.array([0] + [1] * 127, dtype=np.float64)
    s = 0.03
    exact = s * np.sum(w * x.astype(np.float64))
    bar = 1e-3 * np.sum(np.abs(s * w * x)) + 1e-6
    assert abs(_emulate_group_two_piece_e4m3(x, w, s) - exact) > 10 * bar
    assert _emulate_group_three_piece(x, w, s) == exact


def test_dynamic_range_and_leftovers_emulated_exactly():
    rng = np.random.default_rng(5)
    for span in (20, 40, 120):
        x = _bf16(np.exp2(-rng.uniform(0, span, 128)) * rng.choice([-1, 1], 128))
        x[rng.integers(0, 128)] = _bf16(np.array([2.0 ** 30]))[0]
        w = rng.choice([-1, 0, 1], 128).astype(np.float64)
        exact = 0.02 * np.sum(w * x.astype(np.float64))
        bar = 1e-3 * np.sum(np.abs(0.02 * w * x)) + 1e-6
        assert abs(_emulate_group_three_piece(x, w, 0.02) - exact) <= 1e-12 * bar


def test_s8_group_sums_fit_the_accumulator():
    # One 128-wide group of MMA products per accumulator before the fp32 fold:
    # p1 * w/8 are multiples of 2 with |p1| <= 128, so |sum| <= 2048;
    # p2 * w/8 are multiples of 1/8 with |p2| <= 8, so |sum| <= 128.
    # Either sum takes at most 2^11 steps of its quantum: exact in fp32 (and
    # in any accumulator that keeps 12 or more significant bits).
    for quantum, bound in ((2.0, 128 * 128 / 8), (1 / 8, 128 * 8 / 8)):
        assert bound / quantum <= 2 ** 11
