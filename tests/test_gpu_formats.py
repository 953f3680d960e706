"""GPU parity of the base-3 weight conversion and the activation rotation,
through the C ABI, against the CPU oracle.

- tern_repack_t5: base-3 bytes (five weights per byte) -> the 2-bit layout,
  bit-exact against the oracle's unpack_t5 followed by its pack; invalid
  bytes counted exactly.
- tern_rotate_bf16: against the oracle's exact fp64 rotation, within half a
  bf16 step plus the fp32 sum bound of ten butterfly stages
  (10 * 2^-24 * sum |x| over the block / 32).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_bf16_parity, packed_to_numpy, sample_indices, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tl():
    import torch
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    torch.cuda.init()
    return tl


# ---------------------------------------------------------------- base-3 repack

def _t5_bytes(N, K, seed, invalid):
    W = synth.ternary_weights(N, K, 0.4, seed=seed)
    P, _ = oracle.pack_t5(W)
    if invalid:
        rng = np.random.default_rng(seed + 1)
        flat = P.reshape(-1)
        idx = rng.choice(flat.size, size=invalid, replace=False)
        flat[idx] = rng.integers(243, 256, size=invalid)
    return P


# (7, 128): one CTA, 182 bytes, a tail that is not a whole 16-byte chunk;
# (300, 1280): 3000 groups, a partial last CTA; (129, 2048): 2064 groups.
@pytest.mark.parametrize("N,K,invalid", [(7, 128, 3), (300, 1280, 50), (129, 2048, 0)])
def test_repack_t5_bit_exact(tl, N, K, invalid):
    import torch
    P = _t5_bytes(N, K, seed=N + K, invalid=invalid)
    W_ref, nbad = oracle.unpack_t5(P, K)
    assert nbad == invalid
    wp_ref, _ = oracle.pack(W_ref)
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wp = tl.tern_repack_t5(torch.from_numpy(P).cuda(), K, bad_count=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == invalid
    assert np.array_equal(packed_to_numpy(Wp), wp_ref)


def test_repack_t5_full_size_then_decode_call(tl):
    """gate+up 5120 x 34816 stored as base-3 bytes: repacked bit-exact, then
    the T = 1 call on the repacked weights against the oracle evaluated on the
    base-3 bytes themselves (sampled outputs)."""
    import torch
    c = synth.config_decode("gu")
    K, N = c.K, c.N
    P, _ = oracle.pack_t5(c.W)
    wp_ref, _ = oracle.pack(c.W)
    Wp = tl.tern_repack_t5(torch.from_numpy(P).cuda(), K)
    torch.cuda.synchronize()
    assert np.array_equal(packed_to_numpy(Wp), wp_ref)
    _, s, x = to_device(c)
    y = tl.tern_linear(Wp, s, x).cpu().numpy()
    assert tl.tern_device_status() == 0
    ti, ni = sample_indices(1, N, 4096, seed=K)
    y_ref, m = oracle.linear_f64_sampled(P, c.scales, c.x, K, N, ti, ni)
    assert_bf16_parity(y[ti, ni], y_ref, m, "gate+up T=1 from base-3 bytes")


# ---------------------------------------------------------------- rotation

def _rotation_bound(xb, exact):
    T, K = exact.shape
    absx = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)).reshape(T, K // 1024, 1024)
    acc = np.repeat(10 * 2.0 ** -24 * absx.sum(-1) / 32, 1024, axis=1).reshape(T, K)
    # half a bf16 step at |exact| + acc: the step is 2^(e-8) for a value in
    # [2^(e-1), 2^e), and 2^-133 for subnormals
    _, e = np.frexp(np.abs(exact) + acc)
    return np.exp2(np.maximum(e - 9, -134).astype(np.float64)) + acc


def _check_rotation(xr_bits, xb, exact, what):
    g = synth.bf16_bits_to_f32(xr_bits).astype(np.float64)
    err = np.abs(g - exact)
    bound = _rotation_bound(xb, exact)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; worst at "
                             f"{i}: got {g[i]!r}, exact {exact[i]!r}, bound {bound[i]!r}")


@pytest.mark.parametrize("T,K", [(1, 1024), (5, 3072), (37, 5120), (3, 17408)])
def test_rotate_bf16_parity(tl, T, K):
    import torch
    xb = synth.activations(T, K, seed=T * 7 + K, outlier_frac=0.01)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    xr = tl.tern_rotate_bf16(x)
    torch.cuda.synchronize()
    got = xr.view(torch.int16).cpu().numpy().view(np.uint16)
    exact, ref_bits = oracle.rotate(xb, T, K)
    _check_rotation(got, xb, exact, f"rotate T={T} K={K}")
    # almost every output is the exact value's own bf16 rounding
    assert np.mean(got == ref_bits) > 0.99


def test_rotate_bf16_in_place_and_zeros(tl):
    import torch
    T, K = 4, 2048
    xb = synth.activations(T, K, seed=5, outlier_frac=0.01)
    xb[1] = 0  # an all-zero token
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    out_of_place = tl.tern_rotate_bf16(x)
    tl.tern_rotate_bf16(x, x)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), out_of_place.view(torch.int16))
    got = x.view(torch.int16).cpu().numpy().view(np.uint16)
    assert not got[1].any()
    exact, _ = oracle.rotate(xb, T, K)
    _check_rotation(got, xb, exact, "rotate in place")


def test_rotate_bf16_full_size_sampled_tokens(tl):
    """T = 2048 tokens of the down projection's width (17408 = 17 blocks):
    the whole rotation on the GPU, eight sampled tokens against the oracle."""
    import torch
    T, K = 2048, 17408
    xb = synth.activations(T, K, seed=11, outlier_frac=0.01)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    xr = tl.tern_rotate_bf16(x)
    torch.cuda.synchronize()
    got = xr.view(torch.int16).cpu().numpy().view(np.uint16)
    ti = np.array([0, 1, 511, 1024, 1500, 2000, 2046, 2047])
    exact, _ = oracle.rotate(np.ascontiguousarray(xb[ti]), len(ti), K)
    _check_rotation(got[ti], xb[ti], exact, "rotate T=2048 K=17408 (sampled tokens)")
