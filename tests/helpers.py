"""Shared test helpers: moving synthetic cases to the GPU and the parity bars."""
from __future__ import annotations

import numpy as np

# Parity bars.
#  bf16 rungs: |y - y_ref| <= 1e-3 * sum|s w x| + 1e-6
#  s8 rung:    int8 codes and x_scale bit-exact; y within 1e-5 relative, read
#              as |y - y_ref| <= 1e-5 * xs * sum_g |s * acc| + 1e-30 (a literal
#              1e-5 * |y_ref| cannot hold where the groups cancel).
BF16_REL = 1e-3
BF16_ABS = 1e-6
S8_REL = 1e-5
S8_ABS = 1e-30


def to_device(case):
    import torch
    W = torch.from_numpy(case.W).cuda()
    s = torch.from_numpy(case.scales.view(np.uint16)).view(torch.float16).cuda()
    x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).cuda()
    return W, s, x


def packed_to_numpy(Wp):
    return Wp.cpu().numpy().view(np.uint32)


def assert_bf16_parity(y, y_ref, m, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = BF16_REL * m + BF16_ABS
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside 1e-3*sum|swx|+1e-6; "
            f"worst at {i}: y={y[i]!r} ref={y_ref[i]!r} bound={bound[i]!r}")


def assert_s8_parity(y, y_ref, m, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = S8_REL * m + S8_ABS
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside 1e-5 relative; "
            f"worst at {i}: y={y[i]!r} ref={y_ref[i]!r} bound={bound[i]!r}")


def sample_indices(T, N, count, seed):
    """Seeded sample of (t, n) outputs that always includes the corners."""
    rng = np.random.default_rng([seed, T, N])
    t = rng.integers(0, T, size=count).astype(np.int32)
    n = rng.integers(0, N, size=count).astype(np.int32)
    t[:4] = [0, 0, T - 1, T - 1]
    n[:4] = [0, N - 1, 0, N - 1]
    return t, n
