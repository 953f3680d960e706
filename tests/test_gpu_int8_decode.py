"""GPU parity of the int8-activation decode variant (TERN_DECODE_ACT=int8):
the T <= 16 rungs run the s8 definition (per-token int8 codes of
tern_quant_act_s8, exact integer group sums, y = xs * sum_g s * acc) and are
held to the s8 rung's bars against the oracle."""
import os

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_s8_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tl():
    import torch
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    torch.cuda.init()
    return tl


class int8_decode:
    def __init__(self, tl, rung):
        self.tl, self.rung = tl, rung

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in ("TERN_DECODE_ACT", "TERN_RUNG")}
        os.environ["TERN_DECODE_ACT"] = "int8"
        os.environ["TERN_RUNG"] = self.rung
        self.tl.tern_reload_env()

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        self.tl.tern_reload_env()


def _run(tl, case, rung):
    import torch
    W, s, x = to_device(case)
    Wp = tl.tern_pack(W)
    with int8_decode(tl, rung):
        y = tl.tern_linear(Wp, s, x)
        assert tl.tern_last_rung() == rung
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("rung,T", [("gemv", 1), ("small_t", 3), ("small_t", 8),
                                    ("small_t_tiled", 13), ("small_t_tiled", 16)])
@pytest.mark.parametrize("K,N", [(640, 300), (5120, 4200)])
def test_int8_decode_matches_the_s8_definition(tl, rung, T, K, N):
    c = synth.case("i8", T, K=K, N=N, seed=T * 7 + K, outliers=True)
    y = _run(tl, c, rung)
    wp, _ = oracle.pack(c.W)
    q, xs = oracle.quant_s8(c.x, T, K)
    y_ref, m, _ = oracle.linear_s8(wp, c.scales, q, xs, T, K, N)
    assert_s8_parity(y, y_ref, m, f"int8 decode {rung} T={T} K={K} N={N}")


@pytest.mark.parametrize("rung,T", [("gemv", 1), ("small_t", 5), ("small_t_tiled", 12)])
def test_int8_decode_integer_sums_exact(tl, rung, T):
    # unit scales and integer rows that each contain +-127: xs = 1 and q = x,
    # so y must be sum_k q w exactly (below 2^24, exact in fp32)
    K, N = 17408, 640
    c = synth.case("i8int", T, K=K, N=N, seed=T + 1)
    rng = np.random.default_rng(T)
    xi = rng.integers(-127, 128, size=(T, K)).astype(np.float32)
    xi[:, 7] = 127.0
    c.x = synth.f32_to_bf16_bits(xi)
    c.scales = np.ones_like(c.scales)
    y = _run(tl, c, rung)
    exact = xi.astype(np.float64) @ c.W.astype(np.float64).T
    assert np.array_equal(y, exact)


def test_int8_decode_zero_token_and_full_size_sampled(tl):
    # a zero token gives y = 0; the rest of a full gate+up call on samples
    from helpers import sample_indices
    c = synth.config_verify("gu", 4)
    c.x[2, :] = 0
    y = _run(tl, c, "small_t")
    assert not y[2].any()
    wp, _ = oracle.pack(c.W)
    q, xs = oracle.quant_s8(c.x, c.T, c.K)
    ti, ni = sample_indices(c.T, c.N, 4096, seed=11)
    y_ref, m, _ = oracle.linear_s8_sampled(wp, c.scales, q, xs, c.K, c.N, ti, ni)
    assert_s8_parity(y[ti, ni], y_ref, m, "int8 decode gate+up T=4 sampled")
