"""GPU parity of the fused Hadamard rotation (TERN_ROTATE=1) against the
oracle: every rung runs the layer on the blockwise-rotated activations,
rotated inside its own activation staging.

The oracle's reference is linear(rotate(x)) with rotate's exact value rounded
once to bf16.  The kernels rotate in fp32 butterflies, which may round an
element whose exact value lies within the fp32 sum bound of a bf16 rounding
boundary the other way (one bf16 step).  So:
- integer-valued x in [-8, 8]: every butterfly sum is an exact fp32 integer,
  both sides round the same exact value, and the usual bars hold (the s8 rung
  bit-exact in its integers);
- general x: the bf16 bar widened by sum_k |s w| * 2 * bound_k, bound_k the
  rotation's own error bound for element k (half a bf16 step plus the fp32 sum
  bound of ten butterfly stages).
"""
import os

import numpy as np
import pytest

import oracle
import synth
from helpers import (BF16_ABS, BF16_REL, assert_bf16_parity, assert_s8_parity, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tl():
    import torch
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    torch.cuda.init()
    return tl


class rotated:
    """TERN_ROTATE=1 and a forced rung for the duration of a block."""

    def __init__(self, tl, rung):
        self.tl, self.rung = tl, rung

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in ("TERN_ROTATE", "TERN_RUNG")}
        os.environ["TERN_ROTATE"] = "1"
        os.environ["TERN_RUNG"] = self.rung
        self.tl.tern_reload_env()

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        self.tl.tern_reload_env()


def _run_rotated(tl, case, rung):
    import torch
    W, s, x = to_device(case)
    Wp = tl.tern_pack(W)
    with rotated(tl, rung):
        y = tl.tern_linear(Wp, s, x)
        assert tl.tern_last_rung() == rung
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    return y.cpu().numpy().astype(np.float64)


def _rotation_bound(xb, exact):
    T, K = exact.shape
    absx = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)).reshape(T, K // 1024, 1024)
    acc = np.repeat(10 * 2.0 ** -24 * absx.sum(-1) / 32, 1024, axis=1).reshape(T, K)
    _, e = np.frexp(np.abs(exact) + acc)
    return np.exp2(np.maximum(e - 9, -134).astype(np.float64)) + acc


def _integer_case(T, K, N, seed):
    c = synth.case("rot-int", T, seed=seed, K=K, N=N)
    rng = np.random.default_rng(seed + 17)
    xi = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    c.x = synth.f32_to_bf16_bits(xi)
    return c


CASES = [("gemv", 1, 2048, 1000), ("gemv", 1, 5120, 4200), ("small_t", 5, 3072, 777),
         ("small_t_tiled", 13, 2048, 1300), ("s8", 37, 5120, 640), ("s8", 20, 2048, 300),
         ("bf16", 37, 5120, 640)]


@pytest.mark.parametrize("rung,T,K,N", CASES)
def test_rotated_integer_activations_match_exactly(tl, rung, T, K, N):
    c = _integer_case(T, K, N, seed=T * 31 + K)
    y = _run_rotated(tl, c, rung)
    exact, xr = oracle.rotate(c.x, T, K)
    # integer inputs: every fp32 butterfly sum is exact, so the kernels round
    # the same exact value as the oracle and must reproduce its bf16 bits
    wp, bad = oracle.pack(c.W)
    assert bad == 0
    if rung == "s8":
        q, xs = oracle.quant_s8(xr, T, K)
        y_ref, m, _ = oracle.linear_s8(wp, c.scales, q, xs, T, K, N)
        assert_s8_parity(y, y_ref, m, f"rotated {rung} T={T} K={K} N={N}")
    else:
        y_ref, m = oracle.linear_f64(wp, c.scales, xr, T, K, N)
        assert_bf16_parity(y, y_ref, m, f"rotated {rung} T={T} K={K} N={N}")


@pytest.mark.parametrize("rung,T,K,N", [c for c in CASES if c[0] != "s8"])
def test_rotated_general_activations_within_derived_bar(tl, rung, T, K, N):
    c = synth.case("rot", T, seed=T * 13 + N, K=K, N=N)
    y = _run_rotated(tl, c, rung)
    exact, xr = oracle.rotate(c.x, T, K)
    wp, _ = oracle.pack(c.W)
    y_ref, m = oracle.linear_f64(wp, c.scales, xr, T, K, N)
    sw = np.abs(c.W.astype(np.float64)) * np.repeat(
        c.scales.astype(np.float64), 128, axis=1)        # |s w| [N, K]
    widen = (2.0 * _rotation_bound(c.x, exact)) @ sw.T   # [T, N]
    err = np.abs(y - y_ref)
    bar = BF16_REL * m + BF16_ABS + widen
    assert (err <= bar).all(), f"rotated {rung}: worst excess {float((err - bar).max())!r}"
    # the widening is slack, not the rule: nearly every output is also inside
    # the plain bf16 bar
    assert np.mean(err <= BF16_REL * m + BF16_ABS) > 0.99


def test_rotation_changes_the_result(tl):
    # the switch is live: the rotated call differs from the plain one and
    # matches the oracle on rotated activations (integer inputs: exact)
    import torch
    c = _integer_case(3, 2048, 512, seed=5)
    W, s, x = to_device(c)
    Wp = tl.tern_pack(W)
    plain = tl.tern_linear(Wp, s, x).cpu().numpy()
    with rotated(tl, "small_t"):
        rot = tl.tern_linear(Wp, s, x).cpu().numpy()
    torch.cuda.synchronize()
    assert not np.allclose(plain, rot)
    _, xr = oracle.rotate(c.x, 3, 2048)
    wp, _ = oracle.pack(c.W)
    y_ref, m = oracle.linear_f64(wp, c.scales, xr, 3, 2048, 512)
    assert_bf16_parity(rot, y_ref, m, "rotated small_t")
