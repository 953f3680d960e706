"""CPU oracle for the ternary-weight linear layer.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never
imports it and never falls back to it.

The arithmetic lives in ``tern_oracle.c`` (plain C11, fp64 / exact integers).
This module compiles it with gcc on first use (or from ``build()``) and exposes
numpy-friendly wrappers.  See the header of ``tern_oracle.c`` for what each
function computes and which page section it follows.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (hand-written packed words, brute force on tiny
inputs, closed forms, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tern_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = [
    "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
    "-ffp-contract=off", "-fno-fast-math",
]


def build(force: bool = False) -> str:
    """Compile tern_oracle.c into _build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        i64 = ctypes.c_long
        lib.tern_oracle_pack.argtypes = [P, i32, i32, P]
        lib.tern_oracle_pack.restype = i64
        lib.tern_oracle_unpack.argtypes = [P, i32, i32, P]
        lib.tern_oracle_unpack.restype = i64
        lib.tern_oracle_linear_f64.argtypes = [P, P, P, i32, i32, i32, P, P]
        lib.tern_oracle_linear_f64.restype = None
        lib.tern_oracle_linear_f64_sampled.argtypes = [P, P, P, i32, i32, P, P, i64, P, P]
        lib.tern_oracle_linear_f64_sampled.restype = None
        lib.tern_oracle_quant_s8.argtypes = [P, i32, i32, P, P]
        lib.tern_oracle_quant_s8.restype = None
        lib.tern_oracle_linear_s8.argtypes = [P, P, P, P, i32, i32, i32, P, P, P]
        lib.tern_oracle_linear_s8.restype = None
        lib.tern_oracle_linear_s8_sampled.argtypes = [P, P, P, P, i32, i32, P, P, i64, P, P, P]
        lib.tern_oracle_linear_s8_sampled.restype = None
        lib.tern_oracle_num_threads.argtypes = []
        lib.tern_oracle_num_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a: np.ndarray) -> np.ndarray:
    """bf16 / fp16 payloads travel as raw uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def num_threads() -> int:
    return int(_load().tern_oracle_num_threads())


def pack(W: np.ndarray) -> tuple[np.ndarray, int]:
    """W int8 [N, K] -> (packed uint32 [N, K/16], count of values not in {-1,0,1})."""
    W = np.ascontiguousarray(W, dtype=np.int8)
    N, K = W.shape
    assert K % 16 == 0
    wp = np.empty((N, K // 16), dtype=np.uint32)
    bad = _load().tern_oracle_pack(_ptr(W), K, N, _ptr(wp))
    return wp, int(bad)


def unpack(wp: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """packed uint32 [N, K/16] -> (W int8 [N, K], count of invalid codes)."""
    wp = np.ascontiguousarray(wp, dtype=np.uint32)
    N = wp.shape[0]
    assert wp.shape[1] * 16 == K
    W = np.empty((N, K), dtype=np.int8)
    bad = _load().tern_oracle_unpack(_ptr(wp), K, N, _ptr(W))
    return W, int(bad)


def linear_f64(wp, scales_f16, x_bf16, T: int, K: int, N: int):
    """bf16-rung definition in fp64.  Returns (y [T, N], m [T, N]) where
    m = sum |s w x| is the tolerance scale."""
    wp = np.ascontiguousarray(wp, dtype=np.uint32)
    s = _u16(scales_f16)
    x = _u16(x_bf16)
    assert wp.size == N * (K // 16) and s.size == N * (K // 128) and x.size == T * K
    y = np.empty((T, N), dtype=np.float64)
    m = np.empty((T, N), dtype=np.float64)
    _load().tern_oracle_linear_f64(_ptr(wp), _ptr(s), _ptr(x), T, K, N, _ptr(y), _ptr(m))
    return y, m


def linear_f64_sampled(wp, scales_f16, x_bf16, K: int, N: int, t_idx, n_idx):
    """The bf16-rung definition at the listed (t, n) outputs only."""
    wp = np.ascontiguousarray(wp, dtype=np.uint32)
    s = _u16(scales_f16)
    x = _u16(x_bf16)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int32)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int32)
    cnt = t_idx.size
    y = np.empty(cnt, dtype=np.float64)
    m = np.empty(cnt, dtype=np.float64)
    _load().tern_oracle_linear_f64_sampled(_ptr(wp), _ptr(s), _ptr(x), K, N, _ptr(t_idx),
                                           _ptr(n_idx), cnt, _ptr(y), _ptr(m))
    return y, m


def quant_s8(x_bf16, T: int, K: int):
    """Per-token absmax/127 int8 quantisation (fp32, RNE).  Returns (q int8 [T, K], xs f32 [T])."""
    x = _u16(x_bf16)
    assert x.size == T * K
    q = np.empty((T, K), dtype=np.int8)
    xs = np.empty(T, dtype=np.float32)
    _load().tern_oracle_quant_s8(_ptr(x), T, K, _ptr(q), _ptr(xs))
    return q, xs


def linear_s8(wp, scales_f16, q, xs, T: int, K: int, N: int, want_acc: bool = False):
    """s8-rung definition.  Returns (y [T, N] fp64, m [T, N], acc int64 [T, N, G] or None)."""
    wp = np.ascontiguousarray(wp, dtype=np.uint32)
    s = _u16(scales_f16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    G = K // 128
    y = np.empty((T, N), dtype=np.float64)
    m = np.empty((T, N), dtype=np.float64)
    acc = np.empty((T, N, G), dtype=np.int64) if want_acc else None
    _load().tern_oracle_linear_s8(_ptr(wp), _ptr(s), _ptr(q), _ptr(xs), T, K, N, _ptr(acc),
                                  _ptr(y), _ptr(m))
    return y, m, acc


def linear_s8_sampled(wp, scales_f16, q, xs, K: int, N: int, t_idx, n_idx,
                      want_acc: bool = False):
    """s8-rung definition at the listed (t, n) outputs.  Returns (y, m, acc [cnt, G] or None)."""
    wp = np.ascontiguousarray(wp, dtype=np.uint32)
    s = _u16(scales_f16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int32)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int32)
    cnt = t_idx.size
    G = K // 128
    y = np.empty(cnt, dtype=np.float64)
    m = np.empty(cnt, dtype=np.float64)
    acc = np.empty((cnt, G), dtype=np.int64) if want_acc else None
    _load().tern_oracle_linear_s8_sampled(_ptr(wp), _ptr(s), _ptr(q), _ptr(xs), K, N,
                                          _ptr(t_idx), _ptr(n_idx), cnt, _ptr(acc), _ptr(y),
                                          _ptr(m))
    return y, m, acc
