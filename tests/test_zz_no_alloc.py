"""tern_linear_small_t_noalloc: the workspace-free, allocation-free T <= 16 call.

It uses the library's fixed device scratch instead of a caller workspace.
The GPU test calls it twice in a row through the C ABI, with different shapes
and token counts so that the second call runs over the first call's scratch
contents, and checks each output against tern_linear on the same inputs.
This file is collected last so that it also runs after every other test has
used the library in the same process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import BF16_ABS, BF16_REL, to_device


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
    assert tl.NOALLOC_SCRATCH_BYTES == 4 << 20
    # T outside 1..16
    assert _noalloc_raw(tl, 17, 512, 64) == -1
    assert _noalloc_raw(tl, 0, 512, 64) == -1
    # K whose activation blocks exceed the 4 MiB scratch (the largest K that
    # fits is 257024 for T <= 8 and 128000 for T <= 16)
    assert _noalloc_raw(tl, 1, 257152, 64) == -3
    assert _noalloc_raw(tl, 8, 257152, 64) == -3
    assert _noalloc_raw(tl, 9, 128128, 64) == -3
    assert _noalloc_raw(tl, 16, 128128, 64) == -3
    assert _noalloc_raw(tl, 16, 257152, 64) == -3
    assert "workspace" in tl.tern_status_string(-3)


@pytest.mark.gpu
def test_noalloc_matches_tern_linear_on_two_calls_in_a_row(tl):
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
        y_ref_gpu = tl.tern_linear(Wp, s, x)
        prepared.append((c, Wp, s, x, y_ref_gpu))
    torch.cuda.synchronize()

    outs = []
    for c, Wp, s, x, _ in prepared:  # two calls in a row, same stream
        y = torch.full((c.T, c.N), float("nan"), dtype=torch.float32, device="cuda")
        tl.tern_linear_small_t_noalloc(Wp, s, x, y)
        outs.append(y)
    torch.cuda.synchronize()
    assert tl.tern_device_status() == 0

    for (c, Wp, s, x, y_ref_gpu), y in zip(prepared, outs):
        wp_ref, _ = oracle.pack(c.W)
        _, m = oracle.linear_f64(wp_ref, c.scales, c.x, c.T, c.K, c.N)
        a = y.cpu().numpy().astype(np.float64)
        b = y_ref_gpu.cpu().numpy().astype(np.float64)
        bound = BF16_REL * m + BF16_ABS
        err = np.abs(a - b)
        assert np.isfinite(a).all(), c.name
        assert (err <= bound).all(), (
            f"{c.name}: {int((err > bound).sum())} outputs differ from tern_linear; "
            f"worst {float((err - bound).max())}")
