"""CPU oracle for the ternary-weight linear layer.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never
imports it and never falls back to it.

The arithmetic lives in ``tern_oracle.c`` (plain C11, fp64 / exact integers).
This module compiles it with gcc on first use (or from ``build()``) and exposes
numpy-friendly wrappers.  See the header of ``tern_oracle.c`` for what each
function computes and which page section it follows.

Two packed weight formats are understood: the 2-bit code (uint32 words
[N, K/16]) and the base-3 code, five weights per byte (uint8 [N, K/128*26]).
The linear definitions take either and pick the format from the dtype.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (hand-written packed words and bytes, brute force
on tiny inputs, closed forms, numpy's base conversion, invariants); none is
"parity unpinned".
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
        lib.tern_oracle_pack_t5.argtypes = [P, i32, i32, P]
        lib.tern_oracle_pack_t5.restype = i64
        lib.tern_oracle_unpack_t5.argtypes = [P, i32, i32, P]
        lib.tern_oracle_unpack_t5.restype = i64
        lib.tern_oracle_linear_t5_f64.argtypes = [P, P, P, i32, i32, i32, P, P]
        lib.tern_oracle_linear_t5_f64.restype = None
        lib.tern_oracle_linear_t5_f64_sampled.argtypes = [P, P, P, i32, i32, P, P, i64, P, P]
        lib.tern_oracle_linear_t5_f64_sampled.restype = None
        lib.tern_oracle_linear_t5_s8.argtypes = [P, P, P, P, i32, i32, i32, P, P, P]
        lib.tern_oracle_linear_t5_s8.restype = None
        lib.tern_oracle_linear_t5_s8_sampled.argtypes = [P, P, P, P, i32, i32, P, P, i64, P, P, P]
        lib.tern_oracle_linear_t5_s8_sampled.restype = None
        lib.tern_oracle_f64_to_bf16.argtypes = [P, i64, P]
        lib.tern_oracle_f64_to_bf16.restype = None
        lib.tern_oracle_rotate.argtypes = [P, i32, i32, i32, P, P]
        lib.tern_oracle_rotate.restype = None
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


T5_GROUP_BYTES = 26  # ceil(128 / 5) base-3 bytes per 128-weight group


def _packed(wp, K: int, N: int):
    """The packed weights and their format: uint32 words [N, K/16] are the
    2-bit code ("2bit"), uint8 bytes [N, K/128*26] the base-3 code ("t5")."""
    wp = np.ascontiguousarray(wp)
    if wp.dtype == np.uint32:
        assert wp.size == N * (K // 16), (wp.shape, K, N)
        return wp, "2bit"
    assert wp.dtype == np.uint8, wp.dtype
    assert wp.size == N * (K // 128) * T5_GROUP_BYTES, (wp.shape, K, N)
    return wp, "t5"


def _fn(name: str, fmt: str):
    """The C entry point of a definition ("linear_f64", "linear_s8_sampled", ...)
    for a weight format."""
    if fmt == "t5":
        name = name.replace("linear_", "linear_t5_", 1)
    return getattr(_load(), "tern_oracle_" + name)


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


def pack_t5(W: np.ndarray) -> tuple[np.ndarray, int]:
    """W int8 [N, K] -> (base-3 bytes uint8 [N, K/128*26], count of values not
    in {-1,0,1}).  Five weights per byte, 26 bytes per 128-weight group."""
    W = np.ascontiguousarray(W, dtype=np.int8)
    N, K = W.shape
    assert K % 128 == 0
    p = np.empty((N, K // 128 * T5_GROUP_BYTES), dtype=np.uint8)
    bad = _load().tern_oracle_pack_t5(_ptr(W), K, N, _ptr(p))
    return p, int(bad)


def unpack_t5(p: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """base-3 bytes [N, K/128*26] -> (W int8 [N, K], count of invalid bytes)."""
    p = np.ascontiguousarray(p, dtype=np.uint8)
    N = p.shape[0]
    assert p.shape[1] == K // 128 * T5_GROUP_BYTES
    W = np.empty((N, K), dtype=np.int8)
    bad = _load().tern_oracle_unpack_t5(_ptr(p), K, N, _ptr(W))
    return W, int(bad)


def linear_f64(wp, scales_f16, x_bf16, T: int, K: int, N: int):
    """bf16-rung definition in fp64.  Returns (y [T, N], m [T, N]) where
    m = sum |s w x| is the tolerance scale.  wp is either packed format."""
    wp, fmt = _packed(wp, K, N)
    s = _u16(scales_f16)
    x = _u16(x_bf16)
    assert s.size == N * (K // 128) and x.size == T * K
    y = np.empty((T, N), dtype=np.float64)
    m = np.empty((T, N), dtype=np.float64)
    _fn("linear_f64", fmt)(_ptr(wp), _ptr(s), _ptr(x), T, K, N, _ptr(y), _ptr(m))
    return y, m


def linear_f64_sampled(wp, scales_f16, x_bf16, K: int, N: int, t_idx, n_idx):
    """The bf16-rung definition at the listed (t, n) outputs only."""
    wp, fmt = _packed(wp, K, N)
    s = _u16(scales_f16)
    x = _u16(x_bf16)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int32)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int32)
    cnt = t_idx.size
    y = np.empty(cnt, dtype=np.float64)
    m = np.empty(cnt, dtype=np.float64)
    _fn("linear_f64_sampled", fmt)(_ptr(wp), _ptr(s), _ptr(x), K, N, _ptr(t_idx),
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
    wp, fmt = _packed(wp, K, N)
    s = _u16(scales_f16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    G = K // 128
    y = np.empty((T, N), dtype=np.float64)
    m = np.empty((T, N), dtype=np.float64)
    acc = np.empty((T, N, G), dtype=np.int64) if want_acc else None
    _fn("linear_s8", fmt)(_ptr(wp), _ptr(s), _ptr(q), _ptr(xs), T, K, N, _ptr(acc),
                          _ptr(y), _ptr(m))
    return y, m, acc


def linear_s8_sampled(wp, scales_f16, q, xs, K: int, N: int, t_idx, n_idx,
                      want_acc: bool = False):
    """s8-rung definition at the listed (t, n) outputs.  Returns (y, m, acc [cnt, G] or None)."""
    wp, fmt = _packed(wp, K, N)
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
    _fn("linear_s8_sampled", fmt)(_ptr(wp), _ptr(s), _ptr(q), _ptr(xs), K, N,
                                  _ptr(t_idx), _ptr(n_idx), cnt, _ptr(acc), _ptr(y),
                                  _ptr(m))
    return y, m, acc


def f64_to_bf16(v) -> np.ndarray:
    """fp64 values -> bf16 bits (uint16), round to nearest even in one step."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().tern_oracle_f64_to_bf16(_ptr(v), v.size, _ptr(out))
    return out


def rotate(x_bf16, T: int, K: int, block: int = 1024):
    """Blockwise Hadamard rotation of bf16 activations [T, K]: returns
    (exact fp64 [T, K], bf16 bits [T, K]).  block is a power of two dividing K."""
    x = _u16(x_bf16)
    assert x.size == T * K and block > 0 and block & (block - 1) == 0 and K % block == 0
    exact = np.empty((T, K), dtype=np.float64)
    xr = np.empty((T, K), dtype=np.uint16)
    _load().tern_oracle_rotate(_ptr(x), T, K, block, _ptr(exact), _ptr(xr))
    return exact, xr
