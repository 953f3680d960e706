"""The number facts the kernels' exactness rests on, checked exhaustively on
the CPU with torch's own float8_e4m3fn conversion (round to nearest even, as
the device conversion with saturation does for values in range).

- The 2-bit code turns into the e4m3 encoding of w / 8 with one mask.
- s8 rung: every int8 code q in [-127, 127] is the exact sum of two e4m3
  values 16 * floor((q + 8) / 16) and the remainder in [-8, 7].
- bf16 rungs: a bf16 value scaled into (-256, 256) splits as h1 = e4m3(y),
  h2 = e4m3(y - h1) with h1 + h2 == y whenever |y| >= 2^-2, and within
  2^-10 of y below that.
- The per-group sums the tensor core accumulates stay within 11 significant
  bits, so their fp32 accumulation is exact.
"""
import numpy as np
import torch

E4M3 = torch.float8_e4m3fn


def _e4m3(values):
    """float values -> their e4m3 roundings as float64 (round to nearest even)."""
    return torch.tensor(np.asarray(values, dtype=np.float32)).to(E4M3).to(torch.float64).numpy()


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


def _all_bf16_below(limit):
    """Every finite bf16 value with |v| < limit (both signs, zero once)."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # positive finite patterns
    v = (bits << 16).view(np.float32)
    v = v[v < limit]
    return np.concatenate([v, -v[1:]])


def test_bf16_two_piece_split_exact_above_a_quarter():
    y = _all_bf16_below(256.0)
    h1 = _e4m3(y)
    r = (y.astype(np.float32) - h1.astype(np.float32)).astype(np.float64)  # fp32, as on the device
    assert np.array_equal(r, y.astype(np.float64) - h1)                     # that difference is exact
    h2 = _e4m3(r)
    err = np.abs(h1 + h2 - y.astype(np.float64))
    big = np.abs(y) >= 0.25
    assert not err[big].any()
    assert err[~big].max() <= 2.0 ** -10


def test_s8_group_sums_fit_the_accumulator():
    # One 128-wide group of MMA products per accumulator before the fp32 fold:
    # p1 * w/8 are multiples of 2 with |p1| <= 128, so |sum| <= 2048;
    # p2 * w/8 are multiples of 1/8 with |p2| <= 8, so |sum| <= 128.
    # Either sum takes at most 2^11 steps of its quantum: exact in fp32 (and
    # in any accumulator that keeps 12 or more significant bits).
    for quantum, bound in ((2.0, 128 * 128 / 8), (1 / 8, 128 * 8 / 8)):
        assert bound / quantum <= 2 ** 11
