"""tern_linear_small_t_noalloc: the workspace-free, allocation-free T <= 16 call.

Some callers cannot allocate device memory or hand over a workspace (plug-in
interfaces that see only their inputs and outputs, engines that reserve all
device memory at start-up, code where a cudaMalloc would synchronise the
device); this call uses the library's fixed device scratch instead.  The GPU
test calls it twice in a row through the C ABI, with different shapes and
token counts so that the second call runs over the first call's scratch
contents, and checks each output against the CPU oracle element by element
and against tern_linear on the same inputs, within the bf16 rungs' bar.
This file is collected last so that it also runs after every other test has
used the library in the same process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import BF16_ABS, BF16_REL, assert_bf16_parity, to_device


@pytest.fixture(scope="module")
def tl():
    import ternary_weight_linear_gb300 as tl
    tl.build()
    tl.load()
    return tl


def _noalloc_raw(tl, T, K, N):
    """Call the entry point with placeholder (never dereferenced) pointers:
    only for argument combinations the host rejects before any device work."""
    fake = ctypes.c_void_p(1 << 12)
    return tl.load().tern_linear_small_t_noalloc(fake, fake, fake, fake, T, K, N, None)


def test_noalloc_rejects_sizes_beyond_its_scratch(tl):
    assert tl.NOALLOC_SCRATCH_BYTES == 8 << 20
    # T outside 1..16
    assert _noalloc_raw(tl, 17, 512, 64) == -1
    assert _noalloc_raw(tl, 0, 512, 64) == -1
    # K whose scratch exceeds the 8 MiB: the largest K that fits is 479232
    # for T <= 4, 219136 for T = 5..8 and 118784 for T = 9..16
    for T, kmax in ((1, 479232), (4, 479232), (5, 219136), (8, 219136), (9, 118784),
                    (16, 118784)):
        assert _noalloc_raw(tl, T, kmax + 128, 64) == -3, (T, kmax)
    assert "workspace" in tl.tern_status_string(-3)


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_and_tern_linear_on_two_calls_in_a_row(tl):
    import torch
    torch.cuda.init()
    cases = [
        # larger K first, so the second call reads over stale scratch bytes
        synth.case("noalloc_a", 12, seed=11, K=17408, N=700),
        synth.case("noalloc_b", 3, seed=12, K=640, N=300),
    ]
    prepared = []
    for c in cases:
        W, s, x = to_device(c)
        Wp = tl.tern_pack(W)
        y_ws = tl.tern_linear(Wp, s, x)
        prepared.append((c, Wp, s, x, y_ws))
    torch.cuda.synchronize()

    outs = []
    for c, Wp, s, x, _ in prepared:  # two calls in a row, same stream
        y = torch.full((c.T, c.N), float("nan"), dtype=torch.float32, device="cuda")
        tl.tern_linear_small_t_noalloc(Wp, s, x, y)
        outs.append(y)
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0

    for (c, Wp, s, x, y_ws), y in zip(prepared, outs):
        wp_ref, _ = oracle.pack(c.W)
        y_ref, m = oracle.linear_f64(wp_ref, c.scales, c.x, c.T, c.K, c.N)
        a = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all(), c.name
        assert_bf16_parity(a, y_ref, m, f"{c.name} (no-alloc call)")
        b = y_ws.cpu().numpy().astype(np.float64)
        err = np.abs(a - b)
        bound = BF16_REL * m + BF16_ABS
        assert (err <= bound).all(), (
            f"{c.name}: {int((err > bound).sum())} outputs differ from tern_linear; "
            f"worst {float((err - bound).max())}")
