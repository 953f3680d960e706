"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every rung is forced on every token band (each rung must be right for every
T), on shapes that span several row blocks, several k stages and ragged tails
in N, K and T; then the workload families at full size, on sampled outputs.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from helpers import (assert_bf16_parity, assert_s8_parity, packed_to_numpy, sample_indices,
                     to_device)

pytestmark = pytest.mark.gpu

RUNGS = ("gemv", "small_t", "small_t_tiled", "s8", "bf16")


@pytest.fixture(scope="module")
def tl():
    import torch
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    torch.cuda.init()
    return tl


class forced_rung:
    def __init__(self, tl, rung):
        self.tl, self.rung = tl, rung

    def __enter__(self):
        self.old = os.environ.get("TERN_RUNG")
        if self.rung is None:
            os.environ.pop("TERN_RUNG", None)
        else:
            os.environ["TERN_RUNG"] = self.rung
        self.tl.tern_reload_env()

    def __exit__(self, *a):
        if self.old is None:
            os.environ.pop("TERN_RUNG", None)
        else:
            os.environ["TERN_RUNG"] = self.old
        self.tl.tern_reload_env()


def _run(tl, case, rung=None):
    import torch
    W, s, x = to_device(case)
    Wp = tl.tern_pack(W)
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, s, x)
        ran = tl.tern_last_rung()
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    return Wp, y.cpu().numpy(), ran


def _check_case(tl, case, rung=None, full=True, samples=4096):
    Wp, y, ran = _run(tl, case, rung)
    wp_ref, bad = oracle.pack(case.W)
    assert bad == 0
    assert np.array_equal(packed_to_numpy(Wp), wp_ref), "tern_pack differs from the oracle"
    T, K, N = case.T, case.K, case.N
    if ran == "s8":
        q_ref, xs_ref = oracle.quant_s8(case.x, T, K)
        if full:
            y_ref, m, _ = oracle.linear_s8(wp_ref, case.scales, q_ref, xs_ref, T, K, N)
            assert_s8_parity(y, y_ref, m, f"{case.name} T={T} rung={ran}")
        else:
            ti, ni = sample_indices(T, N, samples, seed=K)
            y_ref, m, _ = oracle.linear_s8_sampled(wp_ref, case.scales, q_ref, xs_ref, K, N, ti, ni)
            assert_s8_parity(y[ti, ni], y_ref, m, f"{case.name} T={T} rung={ran}")
    else:
        if full:
            y_ref, m = oracle.linear_f64(wp_ref, case.scales, case.x, T, K, N)
            assert_bf16_parity(y, y_ref, m, f"{case.name} T={T} rung={ran}")
        else:
            ti, ni = sample_indices(T, N, samples, seed=K)
            y_ref, m = oracle.linear_f64_sampled(wp_ref, case.scales, case.x, K, N, ti, ni)
            assert_bf16_parity(y[ti, ni], y_ref, m, f"{case.name} T={T} rung={ran}")
    return ran


# ---------------------------------------------------------------- pack / quant

def test_pack_bit_exact_and_bad_count(tl):
    import torch
    W = synth.ternary_weights(300, 640, 0.4, seed=3)
    W[5, 7] = 2
    W[299, 639] = -3
    Wd = torch.from_numpy(W).cuda()
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wp = tl.tern_pack(Wd, bad_count=bad)
    ref, nbad = oracle.pack(W)
    assert int(bad.item()) == nbad == 2
    assert np.array_equal(packed_to_numpy(Wp), ref)


@pytest.mark.parametrize("rung,T", [("gemv", 1), ("small_t", 5), ("small_t_tiled", 13), ("s8", 37)])
def test_invalid_pairs_decode_as_zero(tl, rung, T):
    """The header documents that the linear kernels read the invalid pair
    (nz = 0, neg = 1) as weight 0; so does the oracle.  A quarter of the
    nonzero weights are turned into that pair in the packed words."""
    import torch
    K, N = 1280, 300
    case = synth.case("invalid", T, K=K, N=N, seed=81)
    wp, _ = oracle.pack(case.W)
    rng = np.random.default_rng(82)
    nz = np.argwhere(case.W != 0)
    pick = nz[rng.choice(len(nz), size=len(nz) // 4, replace=False)]
    bit = 8 * ((pick[:, 1] % 16) // 4) + np.array([0, 1, 4, 5])[pick[:, 1] % 4]
    words = wp[pick[:, 0], pick[:, 1] // 16]
    np.bitwise_and.at(wp, (pick[:, 0], pick[:, 1] // 16),
                      ~(np.uint32(1) << bit.astype(np.uint32)))
    np.bitwise_or.at(wp, (pick[:, 0], pick[:, 1] // 16),
                     np.uint32(1) << (bit + 2).astype(np.uint32))
    assert not np.array_equal(wp[pick[:, 0], pick[:, 1] // 16], words)
    Wz, bad = oracle.unpack(wp, K)
    assert bad == len(pick)
    assert np.array_equal(Wz, np.where(np.isin(np.arange(N * K).reshape(N, K),
                                                pick[:, 0] * K + pick[:, 1]), 0, case.W))
    _, s, x = to_device(case)
    Wp = torch.from_numpy(wp.view(np.int32)).cuda()
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, s, x)
        assert tl.tern_last_rung() == rung
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    y = y.cpu().numpy()
    if rung == "s8":
        q_ref, xs_ref = oracle.quant_s8(case.x, T, K)
        y_ref, m, _ = oracle.linear_s8(wp, case.scales, q_ref, xs_ref, T, K, N)
        assert_s8_parity(y, y_ref, m, f"invalid pairs rung={rung}")
    else:
        y_ref, m = oracle.linear_f64(wp, case.scales, case.x, T, K, N)
        assert_bf16_parity(y, y_ref, m, f"invalid pairs rung={rung}")


@pytest.mark.parametrize("T,K", [(1, 128), (17, 5120), (508, 6144), (3, 16)])
def test_quant_s8_bit_exact(tl, T, K):
    import torch
    xb = synth.activations(T, K, seed=T, outlier_frac=0.01)
    xb[0, :4] = 0  # a few exact zeros
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    q, xs = tl.tern_quant_act_s8(x)
    q_ref, xs_ref = oracle.quant_s8(xb, T, K)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))


def test_quant_s8_golden_ties_and_zero_row(tl):
    import torch
    rows = [[127, 0.5, 1.5, 2.5, 3.5, 4.5, 126.5, 0] + [0] * 8,
            [-127, -0.5, -1.5, -2.5, -3.5, -4.5, -126.5, 0] + [0] * 8,
            [0.0] * 16]
    x32 = np.array(rows, dtype=np.float32)
    xb = (x32.view(np.uint32) >> 16).astype(np.uint16)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    q, xs = tl.tern_quant_act_s8(x)
    q = q.cpu().numpy()
    assert list(q[0, :8]) == [127, 0, 2, 2, 4, 4, 126, 0]
    assert list(q[1, :8]) == [-127, 0, -2, -2, -4, -4, -126, 0]
    assert not q[2].any() and float(xs[2].item()) == 0.0
    assert float(xs[0].item()) == 1.0


def _every_bf16_up_to(absmax_values, K, seed):
    """bf16 bits [len(absmax_values), K]: row t holds every finite bf16
    magnitude <= a_t (a_t itself first), random signs, zeros after."""
    rng = np.random.default_rng(seed)
    codes = np.arange(0, 0x7F80, dtype=np.uint32)          # every finite bf16 >= 0
    mags = (codes << 16).view(np.float32)
    rows = np.zeros((len(absmax_values), K), dtype=np.uint16)
    for t, a in enumerate(absmax_values):
        a_bits = np.uint16(np.array([a], dtype=np.float32).view(np.uint32)[0] >> 16)
        a_bf = float((np.uint32(a_bits) << 16).view(np.float32))
        sel = codes[(mags <= a_bf) & (codes != a_bits)].astype(np.uint16)
        assert 1 + len(sel) <= K
        sign = rng.integers(0, 2, size=len(sel)).astype(np.uint16) << 15
        rows[t, 0] = a_bits
        rows[t, 1:1 + len(sel)] = sel | sign
    return rows


# absmax values whose scale a / 127 is normal (the product-and-check path)
# or below 2^-126 (every element divides), including a bf16 subnormal
_EVERY_A = [127.0, 100.0, 3.3, 1e-3, 6.0e4, 3.0e38, 2e-36, 1e-36, 1e-39]


def test_quant_s8_every_bf16_value(tl):
    # every finite bf16 magnitude up to each absmax, both signs: the codes
    # equal rint(x / scale) with the quotient rounded as an IEEE division
    import torch
    K = 32768
    xb = _every_bf16_up_to(_EVERY_A, K, seed=3)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    q, xs = tl.tern_quant_act_s8(x)
    q_ref, xs_ref = oracle.quant_s8(xb, len(_EVERY_A), K)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_s8_pieces_every_bf16_value(tl):
    # The same rows through the s8 rung, whose own quantiser splits the codes
    # into two fp8 pieces: with unit scales the integer sums are exact (|acc|
    # < 2^24), so y = fl(x_scale * acc) bit for bit.
    K, N = 32768, 128
    xb = _every_bf16_up_to(_EVERY_A, K, seed=4)
    T = len(_EVERY_A)
    W = synth.ternary_weights(N, K, 0.4, seed=7)
    s = np.ones((N, K // 128), dtype=np.float16)
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, "s8"):
        y = tl.tern_linear(Wp, sd, xd).cpu().numpy()
    q_ref, xs_ref = oracle.quant_s8(xb, T, K)
    acc = q_ref.astype(np.int64) @ W.astype(np.int64).T
    assert np.abs(acc).max() < 2 ** 24
    expect = xs_ref.astype(np.float32)[:, None] * acc.astype(np.float32)
    assert np.array_equal(y.view(np.uint32), expect.view(np.uint32))


# ---------------------------------------------------------------- every rung, every band

@pytest.mark.parametrize("rung", RUNGS)
@pytest.mark.parametrize("T", [1, 3, 8, 9, 16, 17, 40])
def test_forced_rung_ragged(tl, rung, T):
    # K = 640: one full 512-wide stage plus a 128 tail; N = 300: ragged row block.
    case = synth.case("ragged", T, K=640, N=300, seed=T, p_zero=0.4, outliers=True)
    ran = _check_case(tl, case, rung)
    assert ran == rung


@pytest.mark.parametrize("T,expect", [(1, "gemv"), (2, "small_t"), (8, "small_t"),
                                      (9, "small_t_tiled"), (16, "small_t_tiled"), (17, "s8"),
                                      (130, "s8")])
def test_default_dispatch(tl, T, expect):
    case = synth.case("disp", T, K=1024, N=256, seed=T)
    assert _check_case(tl, case, None) == expect


@pytest.mark.parametrize("K,N", [(24576, 300), (25088, 300), (16384, 34816), (17408, 34816)])
def test_gemv_k_limit_of_the_one_token_tile(tl, K, N):
    # The one-token kernel keeps the activation blocks of every k stage a CTA
    # visits resident, at most 16: a CTA of K = 16384 x N = 34816 visits all
    # 16 stages; K = 17408 x N = 34816 would need 17 and runs on the
    # four-token tile; with N = 300 (3 row blocks) each CTA visits one or two
    # stages at any K, and most row blocks are cut between CTAs.
    _check_case(tl, synth.case("bigk", 1, K=K, N=N, seed=K), full=N < 1000)


def test_workspace_reused_across_calls(tl):
    import torch
    cases = [synth.case("ws_a", 1, K=1152, N=700, seed=5),
             synth.case("ws_b", 12, K=17408, N=300, seed=6),
             synth.case("ws_c", 3, K=640, N=1000, seed=7)]
    need = max(tl.tern_linear_workspace_bytes(c.T, c.K, c.N) for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for c in cases:
            W, s, x = to_device(c)
            y = tl.tern_linear(tl.tern_pack(W), s, x, workspace=ws)
            torch.cuda.synchronize()
            assert tl.tern_device_status() == 0
            wp_ref, _ = oracle.pack(c.W)
            y_ref, m = oracle.linear_f64(wp_ref, c.scales, c.x, c.T, c.K, c.N)
            assert_bf16_parity(y.cpu().numpy(), y_ref, m, f"{c.name} pass {rep}")
    # every call leaves the ticket counters of the synchronisation area zeroed
    assert not ws[:tl.SYNC_BYTES].cpu().numpy().any()


@pytest.mark.parametrize("K,N", [(128, 1), (128, 17), (256, 129), (1152, 520), (2048, 4096)])
def test_shapes_bf16(tl, K, N):
    for T in (1, 5, 13):
        _check_case(tl, synth.case("shape", T, K=K, N=N, seed=K + N + T))


@pytest.mark.parametrize("K,N,T", [(128, 1, 17), (256, 129, 33), (1152, 520, 200), (2048, 300, 129),
                                   (1024, 77, 32), (3072, 1001, 31)])
def test_shapes_s8(tl, K, N, T):
    _check_case(tl, synth.case("shape", T, K=K, N=N, seed=K + N + T))


def test_s8_deep_ring_ragged(tl):
    # The s8 kernel's deeper stage ring, taken when the activation pieces
    # (2 T K bytes) exceed half the L2: a ragged token tile (2100 = 16 x 128 +
    # 52), an odd group count (K = 16512, 129 groups) and a partial row block
    # (N = 333), on sampled outputs.
    import torch
    props = torch.cuda.get_device_properties(0)
    T, K, N = 2100, 16512, 333
    assert 2 * T * K > props.L2_cache_size // 2
    assert _check_case(tl, synth.case("deep", T, K=K, N=N, seed=11, outliers=True), full=False,
                       samples=8192) == "s8"


@pytest.mark.parametrize("K,N,T", [(1024, 64, 3000), (40960, 64, 40), (65664, 16, 20)])
def test_s8_quantiser_row_modes(tl, K, N, T):
    # The s8 rung's activation quantiser keeps a token's row in shared memory:
    # two buffers per CTA with many tokens per CTA (K = 1024, T = 3000), one
    # buffer (K = 40960), or none, reading global memory (K = 65664).
    assert _check_case(tl, synth.case("qmode", T, K=K, N=N, seed=K + T, outliers=True), "s8") == "s8"


@pytest.mark.parametrize("K,N,T", [(128, 1, 17), (256, 129, 33), (1152, 521, 200), (2048, 300, 129)])
def test_shapes_bf16_rung(tl, K, N, T):
    # the exact bf16 prefill rung on ragged shapes (N % 4 != 0: y stored directly)
    assert _check_case(tl, synth.case("shape", T, K=K, N=N, seed=K + N + T + 1), "bf16") == "bf16"


# ---------------------------------------------------------------- degenerate inputs

def _dev_case(W, s, xb):
    import torch
    return (torch.from_numpy(W).cuda(),
            torch.from_numpy(s.view(np.uint16)).view(torch.float16).cuda(),
            torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda())


@pytest.mark.parametrize("rung", RUNGS)
def test_zero_weights_give_zero(tl, rung):
    T, K, N = 20, 640, 200
    W = np.zeros((N, K), dtype=np.int8)
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=1)
    xb = synth.activations(T, K, seed=2, outlier_frac=0.01)
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, sd, xd).cpu().numpy()
    assert np.all(np.abs(y) <= 1e-6)


@pytest.mark.parametrize("rung", RUNGS)
def test_one_hot_x_picks_scaled_weight(tl, rung):
    T, K, N = 4, 512, 300
    W = synth.ternary_weights(N, K, 1.0 / 3.0, seed=9)
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=10)
    cols = [0, 200, 333, 511]
    x32 = np.zeros((T, K), dtype=np.float32)
    for t, k in enumerate(cols):
        x32[t, k] = 1.0
    xb = (x32.view(np.uint32) >> 16).astype(np.uint16)
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, sd, xd).cpu().numpy()
    for t, k in enumerate(cols):
        expect = s[:, k // 128].astype(np.float64) * W[:, k]
        if rung == "s8":
            # x_scale = 1/127 in fp32, q = 127: exact up to that one rounding
            np.testing.assert_allclose(y[t].astype(np.float64), expect, rtol=1e-6, atol=0)
        else:
            np.testing.assert_array_equal(y[t].astype(np.float64), expect)


def test_s8_integer_accumulators_bit_exact(tl):
    # scales = 1 and integer rows holding +-127: q = x and x_scale = 1, so the
    # fp32 output equals the exact integer dot product (all partial sums < 2^24).
    T, K, N = 64, 17408, 256
    W = synth.ternary_weights(N, K, 0.4, seed=5)
    s = np.ones((N, K // 128), dtype=np.float16)
    rng = np.random.default_rng(6)
    x32 = rng.integers(-127, 128, size=(T, K)).astype(np.float32)
    x32[:, 3] = 127.0
    x32[1] = 127.0  # every product at its extreme
    xb = (x32.view(np.uint32) >> 16).astype(np.uint16)
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, "s8"):
        y = tl.tern_linear(Wp, sd, xd).cpu().numpy()
    exact = x32.astype(np.int64) @ W.astype(np.int64).T
    assert np.array_equal(y.astype(np.int64), exact)
    assert np.array_equal(y, exact.astype(np.float32))


# ---------------------------------------------------------------- adversarial activations
# Inputs real activations can have and the N(0,1) families do not: a group's
# absmax on a weight that is zero in every row, a wide dynamic range inside
# a group, bf16 subnormals, values spread over more binades than the
# activation pieces cover (the kernels' exact leftover path), and one
# outlier channel far above the rest.  Every rung is forced on each.

def _adversarial_x(kind, T, K, seed, zero_cols=None):
    """bf16 bits [T, K] of one adversarial kind (see the section comment)."""
    rng = np.random.default_rng([seed, T, K])
    sign = rng.choice([-1.0, 1.0], size=(T, K))
    if kind == "absmax_on_zero_weight":
        x = np.full((T, K), 0.01) * sign
        x[:, zero_cols] = 80.0 * sign[:, zero_cols]
    elif kind == "absmax_huge_on_zero_weight":
        x = rng.standard_normal((T, K)) * 1e-3
        x[:, zero_cols] = 2.0 ** 40 * sign[:, zero_cols]
    elif kind == "range_2e-20":
        x = np.exp2(-rng.uniform(0, 20, (T, K))) * sign
    elif kind == "range_2e-60":
        # several clusters per group: spans far beyond the pieces' 21 binades
        x = np.exp2(rng.choice([40.0, 10.0, -15.0, -45.0], size=(T, K)) +
                    rng.uniform(0, 4, (T, K))) * sign
    elif kind == "subnormal":
        # bf16 subnormals (below 2^-126) next to normal values, and whole
        # groups of subnormals only
        x = rng.standard_normal((T, K))
        x[:, 1::3] = rng.integers(1, 128, size=(T, len(range(1, K, 3)))) * 2.0 ** -133
        x[:, :128] = rng.integers(1, 128, size=(T, 128)) * 2.0 ** -133 * sign[:, :128]
    elif kind == "outlier_x1000":
        x = rng.standard_normal((T, K))
        ch = rng.choice(K, size=max(1, K // 100), replace=False)
        x[:, ch] *= 1000.0
    else:
        raise ValueError(kind)
    return synth.f32_to_bf16_bits(x.astype(np.float32))


ADVERSARIAL = ("absmax_on_zero_weight", "absmax_huge_on_zero_weight", "range_2e-20",
               "range_2e-60", "subnormal", "outlier_x1000")


@pytest.mark.parametrize("kind", ADVERSARIAL)
@pytest.mark.parametrize("rung,T", [("gemv", 1), ("small_t", 3), ("small_t", 8),
                                    ("small_t_tiled", 13), ("s8", 20), ("bf16", 20)])
def test_adversarial_activations(tl, kind, rung, T):
    import torch
    K, N = 1280, 300
    W = synth.ternary_weights(N, K, 0.4, seed=31)
    zero_cols = np.arange(5, K, 128)  # one per group, zero in every row
    W[:, zero_cols] = 0
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=32)
    xb = _adversarial_x(kind, T, K, seed=33, zero_cols=zero_cols)
    x64 = synth.bf16_bits_to_f32(xb).astype(np.float64)
    assert np.isfinite(x64).all()
    if kind == "subnormal":
        assert ((np.abs(x64) < 2.0 ** -126) & (x64 != 0)).any()
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, sd, xd)
        assert tl.tern_last_rung() == rung
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    y = y.cpu().numpy()
    wp_ref, _ = oracle.pack(W)
    what = f"{kind} rung={rung} T={T}"
    if rung == "s8":
        q_ref, xs_ref = oracle.quant_s8(xb, T, K)
        y_ref, m, _ = oracle.linear_s8(wp_ref, s, q_ref, xs_ref, T, K, N)
        assert_s8_parity(y, y_ref, m, what)
    else:
        y_ref, m = oracle.linear_f64(wp_ref, s, xb, T, K, N)
        assert_bf16_parity(y, y_ref, m, what)


@pytest.mark.parametrize("rung,T", [("gemv", 1), ("small_t", 4), ("small_t_tiled", 16)])
def test_leftovers_alone_carry_the_output(tl, rung, T):
    """Only the leftovers have nonzero weights: a group's absmax 2^50 sits on
    a zero weight and everything else lies 30+ binades below it, so y comes
    entirely from the kernels' exact leftover path."""
    import torch
    K, N = 1024, 200
    W = synth.ternary_weights(N, K, 1.0 / 3.0, seed=41)
    big = np.arange(0, K, 128) + 7
    W[:, big] = 0
    s = synth.scales_lognormal(N, K, -3.5, 0.3, seed=42)
    rng = np.random.default_rng(43)
    x = rng.standard_normal((T, K)) * 2.0 ** 10
    x[:, big] = 2.0 ** 50
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    Wd, sd, xd = _dev_case(W, s, xb)
    Wp = tl.tern_pack(Wd)
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, sd, xd)
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    wp_ref, _ = oracle.pack(W)
    y_ref, m = oracle.linear_f64(wp_ref, s, xb, T, K, N)
    assert np.abs(y_ref).max() > 1.0
    assert_bf16_parity(y.cpu().numpy(), y_ref, m, f"leftovers only rung={rung}")


def test_decode_gate_up_outlier_x1000_sampled(tl):
    """The full-size gate+up projection at T = 1 with 1% outlier channels
    scaled x1000 instead of x20."""
    import torch
    c = synth.config_decode("gu")
    xb = synth.activations(1, c.K, seed=0, outlier_frac=0.01, outlier_gain=1000.0)
    W, s, _ = to_device(c)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    Wp = tl.tern_pack(W)
    del W
    y = tl.tern_linear(Wp, s, x)
    assert tl.tern_last_rung() == "gemv"
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    wp_ref, _ = oracle.pack(c.W)
    y_ref, m = oracle.linear_f64(wp_ref, c.scales, xb, 1, c.K, c.N)
    assert_bf16_parity(y.cpu().numpy(), y_ref, m, "gate+up T=1 outliers x1000")


def test_split_row_blocks_are_deterministic(tl):
    """Row blocks split between CTAs are reduced in CTA order: repeated calls
    give identical bits."""
    import torch
    # (the T = 1 down and attention-sized layers run in cluster mode)
    for proj, T in (("dn", 1), ("gu", 1), ("ai", 1), ("ao", 1), ("dn", 4), ("ao", 12)):
        c = synth.case(proj, T, seed=51)
        W, s, x = to_device(c)
        Wp = tl.tern_pack(W)
        del W
        ys = [tl.tern_linear(Wp, s, x).clone() for _ in range(4)]
        torch.cuda.synchronize()
        assert tl.tern_device_status() == 0
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32)), proj


# ---------------------------------------------------------------- workload families

def test_tiny_config_full(tl):
    _check_case(tl, synth.config_tiny(), full=True)


@pytest.mark.parametrize("proj", ["gu", "dn"])
def test_decode_config_full(tl, proj):
    _check_case(tl, synth.config_decode(proj), full=True)


@pytest.mark.parametrize("proj", ["gu", "dn"])
@pytest.mark.parametrize("T", synth.VERIFY_T)
def test_verify_config_sampled(tl, proj, T):
    ran = _check_case(tl, synth.config_verify(proj, T), full=False)
    assert ran == ("small_t" if T <= 8 else "small_t_tiled")


@pytest.mark.parametrize("proj", ["gu", "dn", "ai", "ao"])
@pytest.mark.parametrize("T", synth.PREFILL_T)
def test_prefill_config_sampled(tl, proj, T):
    assert _check_case(tl, synth.config_prefill(proj, T), full=False) == "s8"


class prefill_bf16:
    """TERN_PREFILL=bf16 for the duration of a block: the s8 band runs on
    the bf16 rung."""

    def __init__(self, tl):
        self.tl = tl

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in ("TERN_PREFILL", "TERN_RUNG")}
        os.environ["TERN_PREFILL"] = "bf16"
        os.environ.pop("TERN_RUNG", None)
        self.tl.tern_reload_env()

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        self.tl.tern_reload_env()


@pytest.mark.parametrize("proj", ["gu", "dn", "ai", "ao"])
@pytest.mark.parametrize("T", synth.PREFILL_T)
def test_prefill_config_sampled_bf16_rung(tl, proj, T):
    # the prefill configs on the exact bf16 rung: the bf16 bar, no quantisation
    with prefill_bf16(tl):
        assert tl.tern_select_rung(T) == 4
        assert _check_case(tl, synth.config_prefill(proj, T), full=False) == "bf16"


def test_prefill_switch_dispatch(tl):
    with prefill_bf16(tl):
        assert [tl.tern_rung_name(tl.tern_select_rung(T)) for T in (1, 16, 17, 2048)] == \
            ["gemv", "small_t_tiled", "bf16", "bf16"]
    assert tl.tern_rung_name(tl.tern_select_rung(17)) == "s8"


@pytest.mark.parametrize("p_zero", synth.STACK_P_ZERO)
@pytest.mark.parametrize("seed", synth.STACK_SEEDS)
def test_stack_sweep_sampled(tl, p_zero, seed):
    """The layer-stack family: every projection of a layer with P(0) in
    {0.2, 0.4, 0.6} and seeds 1-3, each layer's weights packed once and run at
    T = 1 (gemv), 4 (small_t) and 2048 (s8), checked on sampled outputs."""
    import torch
    for proj in synth.STACK_PROJ:
        base = synth.case(proj, 1, seed=seed, p_zero=p_zero, outliers=True)
        K, N = base.K, base.N
        wp_ref, bad = oracle.pack(base.W)
        assert bad == 0
        Wd, sd, _ = to_device(base)
        Wp = tl.tern_pack(Wd)
        del Wd
        assert np.array_equal(packed_to_numpy(Wp), wp_ref), f"{proj}: tern_pack differs"
        for T, want in ((1, "gemv"), (4, "small_t"), (2048, "s8")):
            xb = synth.activations(T, K, seed, outlier_frac=0.01 if T != 4 else 0.0)
            xd = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
            y = tl.tern_linear(Wp, sd, xd)
            ran = tl.tern_last_rung()
            torch.cuda.synchronize()
            assert tl.tern_device_status() == 0
            assert ran == want
            y = y.cpu().numpy()
            ti, ni = sample_indices(T, N, 2048, seed=K + T)
            what = f"{proj} p0={p_zero} seed={seed} T={T}"
            if ran == "s8":
                q_ref, xs_ref = oracle.quant_s8(xb, T, K)
                y_ref, m, _ = oracle.linear_s8_sampled(wp_ref, base.scales, q_ref, xs_ref, K, N,
                                                       ti, ni)
                assert_s8_parity(y[ti, ni], y_ref, m, what)
            else:
                y_ref, m = oracle.linear_f64_sampled(wp_ref, base.scales, xb, K, N, ti, ni)
                assert_bf16_parity(y[ti, ni], y_ref, m, what)


def test_chained_calls_in_a_cuda_graph(tl):
    """Back-to-back calls chained by programmatic dependent launch, captured
    once in a CUDA graph and replayed: every rung, several shapes, one shared
    workspace.  Each replay must leave the device status clean and every
    output equal to the oracle's (sampled)."""
    import torch
    specs = [("gu", 1, 21), ("dn", 1, 22), ("ai", 4, 23), ("ao", 8, 24), ("ai", 12, 25),
             ("gu", 1, 26), ("ao", 40, 27), ("dn", 1, 28)]
    calls = []
    ws_bytes = 0
    for proj, T, seed in specs:
        c = synth.case(proj, T, seed=seed, outliers=(T == 1 or T > 16))
        W, s, x = to_device(c)
        Wp = tl.tern_pack(W)
        del W
        y = torch.empty(T, c.N, dtype=torch.float32, device="cuda")
        calls.append((c, Wp, s, x, y))
        ws_bytes = max(ws_bytes, tl.tern_linear_workspace_bytes(T, c.K, c.N))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        for c, Wp, s, x, y in calls:  # library set-up outside the capture
            tl.tern_linear(Wp, s, x, y, ws)
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for c, Wp, s, x, y in calls:
                tl.tern_linear(Wp, s, x, y, ws)
    for _ in range(5):
        for _, _, _, _, y in calls:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert tl.tern_device_status() == 0
    for c, Wp, s, x, y in calls:
        yh = y.cpu().numpy()
        wp_ref, _ = oracle.pack(c.W)
        ti, ni = sample_indices(c.T, c.N, 1024, seed=c.K + c.T)
        what = f"{c.name} T={c.T} (graph replay)"
        if c.T >= 17:
            q_ref, xs_ref = oracle.quant_s8(c.x, c.T, c.K)
            y_ref, m, _ = oracle.linear_s8_sampled(wp_ref, c.scales, q_ref, xs_ref, c.K, c.N, ti, ni)
            assert_s8_parity(yh[ti, ni], y_ref, m, what)
        else:
            y_ref, m = oracle.linear_f64_sampled(wp_ref, c.scales, c.x, c.K, c.N, ti, ni)
            assert_bf16_parity(yh[ti, ni], y_ref, m, what)


# ---------------------------------------------------------------- probe

def test_debug_probe_reports_each_rung(tl):
    import subprocess
    import sys
    code = r"""
import numpy as np, torch, synth, ternary_weight_linear_gb300 as tl
from helpers import to_device
for T in (1, 4, 12, 20):
    c = synth.case("p", T, K=256, N=64, seed=T)
    W, s, x = to_device(c)
    tl.tern_linear(tl.tern_pack(W), s, x)
torch.cuda.synchronize()
"""
    env = dict(os.environ, TERN_DEBUG="1", TERN_DEBUG_MIN_T="1", TERN_DEBUG_BUDGET="3")
    env.pop("TERN_RUNG", None)
    here = os.path.dirname(os.path.abspath(__file__))
    env["PYTHONPATH"] = os.pathsep.join([here, os.path.dirname(here), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stderr.splitlines() if l.startswith("tern: rung=")]
    # budget 3: the fourth call is not reported
    assert [l.split()[1] for l in lines] == ["rung=gemv", "rung=small_t", "rung=small_t_tiled"]


# ---------------------------------------------------------------- launch counts

@pytest.mark.parametrize("K,N,T,rung,expect", [
    (5120, 34816, 1, "gemv", 2),     # nine units per CTA: prep kernel + main kernel
    (1024, 34816, 1, "gemv", 1),     # two units per CTA: the main kernel builds x itself
    (17408, 5120, 1, "gemv", 2),     # cluster mode (few row blocks): prep kernel + main kernel
    (5120, 34816, 4, "small_t", 2),
    (5120, 6144, 20, "small_t_tiled", 4),   # two token tiles (16 + 4)
    (5120, 6144, 37, "s8", 2),
    (5120, 6144, 37, "bf16", 2),    # x reordered for the MMA, then the GEMM
])
def test_launch_count_probe(tl, K, N, T, rung, expect):
    import torch
    W = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    Wp = tl.tern_pack(W)
    s = torch.ones((N, K // 128), dtype=torch.float16, device="cuda")
    x = torch.ones((T, K), dtype=torch.bfloat16, device="cuda")
    with forced_rung(tl, rung):
        y = tl.tern_linear(Wp, s, x)
        assert tl.tern_last_rung() == rung
        assert tl.tern_last_launches() == expect
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0
    assert float(y.abs().max().item()) == 0.0
