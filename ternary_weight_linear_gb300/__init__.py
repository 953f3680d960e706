"""Ternary-weight linear layer for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/tern.h`` (``libtern.so``,
built in-tree by ``ternary_weight_linear_gb300.build``).  The functions here
only marshal arguments: they check dtypes, shapes and devices of torch
tensors, pass raw device pointers and the current CUDA stream, and raise on a
non-zero status.  Every step of the layer runs in the library's CUDA kernels;
there is no CPU path.  If the library has not been built, importing works but
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH, build  # noqa: F401  (re-exported for convenience)

__all__ = [
    "tern_pack", "tern_quant_act_s8", "tern_linear", "tern_linear_workspace_bytes",
    "tern_select_rung", "tern_rung_name", "tern_last_rung", "tern_last_rung_id",
    "tern_last_launches",
    "tern_reload_env", "tern_device_status", "tern_status_string", "TernError", "load",
    "tern_linear_small_t_noalloc", "tern_repack_t5", "tern_rotate_bf16",
    "tern_selftest_wait_timeout", "RUNGS",
    "EXPORTED_SYMBOLS", "NOALLOC_SCRATCH_BYTES", "SYNC_BYTES", "T5_GROUP_BYTES", "ROTATION_BLOCK",
]

RUNGS = {0: "gemv", 1: "small_t", 2: "small_t_tiled", 3: "s8", 4: "bf16"}

# Every symbol include/tern.h declares.
EXPORTED_SYMBOLS = (
    "tern_pack", "tern_quant_act_s8", "tern_linear_workspace_bytes", "tern_linear",
    "tern_select_rung", "tern_rung_name", "tern_last_rung_id", "tern_last_rung",
    "tern_last_launches", "tern_status_string", "tern_reload_env", "tern_device_status",
    "tern_linear_small_t_noalloc", "tern_repack_t5", "tern_rotate_bf16",
    "tern_selftest_wait_timeout",
)

# Size of the library's fixed scratch for tern_linear_small_t_noalloc.
NOALLOC_SCRATCH_BYTES = 8 << 20
# Leading bytes of every workspace owned by the library (TERN_SYNC_BYTES):
# zero before first use, then left alone.
SYNC_BYTES = 4096
# Base-3 bytes per 128-weight group (five weights per byte, rounded up).
T5_GROUP_BYTES = 26
# Width of the Hadamard rotation's blocks along K.
ROTATION_BLOCK = 1024

_lock = threading.Lock()
_lib = None


class TernError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {status_text(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libtern.so.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (or ternary_weight_linear_gb300.build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.tern_pack.argtypes = [P, P, I, I, P, P]
        lib.tern_pack.restype = I
        lib.tern_quant_act_s8.argtypes = [P, P, P, I, I, P]
        lib.tern_quant_act_s8.restype = I
        lib.tern_linear_workspace_bytes.argtypes = [I, I, I]
        lib.tern_linear_workspace_bytes.restype = Z
        lib.tern_linear.argtypes = [P, P, P, P, I, I, I, P, Z, P]
        lib.tern_linear.restype = I
        lib.tern_select_rung.argtypes = [I]
        lib.tern_select_rung.restype = I
        lib.tern_rung_name.argtypes = [I]
        lib.tern_rung_name.restype = ctypes.c_char_p
        lib.tern_last_rung_id.argtypes = []
        lib.tern_last_rung_id.restype = I
        lib.tern_last_rung.argtypes = []
        lib.tern_last_rung.restype = ctypes.c_char_p
        lib.tern_last_launches.argtypes = []
        lib.tern_last_launches.restype = I
        lib.tern_status_string.argtypes = [I]
        lib.tern_status_string.restype = ctypes.c_char_p
        lib.tern_reload_env.argtypes = []
        lib.tern_reload_env.restype = None
        lib.tern_device_status.argtypes = [P]
        lib.tern_device_status.restype = I
        lib.tern_linear_small_t_noalloc.argtypes = [P, P, P, P, I, I, I, P]
        lib.tern_linear_small_t_noalloc.restype = I
        lib.tern_repack_t5.argtypes = [P, P, I, I, P, P]
        lib.tern_repack_t5.restype = I
        lib.tern_rotate_bf16.argtypes = [P, P, I, I, P]
        lib.tern_rotate_bf16.restype = I
        lib.tern_selftest_wait_timeout.argtypes = [I, P]
        lib.tern_selftest_wait_timeout.restype = I
        _lib = lib
        return lib


def status_text(status: int) -> str:
    try:
        return load().tern_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return "status"


def tern_status_string(status: int) -> str:
    return load().tern_status_string(int(status)).decode()


def _check(func: str, rc: int) -> None:
    if rc != 0:
        raise TernError(func, rc)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype, shape=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------ entry points

def tern_pack(W: torch.Tensor, Wpacked: torch.Tensor | None = None,
              bad_count: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int8 [N, K] ternary weights -> packed int32 [N, K/16] (uint32 bit patterns)."""
    N, K = W.shape
    if Wpacked is None:
        Wpacked = torch.empty((N, K // 16), dtype=torch.int32, device=W.device)
    pw = _dev(W, "W", torch.int8)
    pp = _dev(Wpacked, "Wpacked", torch.int32, (N, K // 16))
    pb = _dev(bad_count, "bad_count", torch.int32) if bad_count is not None else None
    _check("tern_pack", load().tern_pack(pw, pp, K, N, pb, _stream(stream)))
    return Wpacked


def tern_repack_t5(Pt5: torch.Tensor, K: int, Wpacked: torch.Tensor | None = None,
                   bad_count: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """base-3 packed weights uint8 [N, K/128*26] (five weights per byte) ->
    packed int32 [N, K/16] (uint32 bit patterns of the 2-bit layout)."""
    N = Pt5.shape[0]
    if Wpacked is None:
        Wpacked = torch.empty((N, K // 16), dtype=torch.int32, device=Pt5.device)
    pp = _dev(Pt5, "Pt5", torch.uint8, (N, K // 128 * T5_GROUP_BYTES))
    pw = _dev(Wpacked, "Wpacked", torch.int32, (N, K // 16))
    pb = _dev(bad_count, "bad_count", torch.int32) if bad_count is not None else None
    _check("tern_repack_t5", load().tern_repack_t5(pp, pw, int(K), N, pb, _stream(stream)))
    return Wpacked


def tern_rotate_bf16(x: torch.Tensor, xr: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Blockwise (1024) Hadamard rotation of bf16 activations [T, K]; xr may be x."""
    T, K = x.shape
    if xr is None:
        xr = torch.empty_like(x)
    _check("tern_rotate_bf16", load().tern_rotate_bf16(
        _dev(x, "x", torch.bfloat16), _dev(xr, "xr", torch.bfloat16, (T, K)), T, K,
        _stream(stream)))
    return xr


def tern_quant_act_s8(x: torch.Tensor, q: torch.Tensor | None = None,
                      x_scale: torch.Tensor | None = None, stream=None):
    """bf16 [T, K] -> (int8 codes [T, K], fp32 x_scale [T])."""
    T, K = x.shape
    if q is None:
        q = torch.empty((T, K), dtype=torch.int8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty((T,), dtype=torch.float32, device=x.device)
    _check("tern_quant_act_s8", load().tern_quant_act_s8(
        _dev(x, "x", torch.bfloat16), _dev(q, "q", torch.int8, (T, K)),
        _dev(x_scale, "x_scale", torch.float32, (T,)), T, K, _stream(stream)))
    return q, x_scale


def tern_linear_workspace_bytes(T: int, K: int, N: int) -> int:
    return int(load().tern_linear_workspace_bytes(int(T), int(K), int(N)))


def tern_linear(Wpacked: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """y [T, N] fp32 = ternary linear of bf16 x [T, K] with packed weights [N, K/16]
    and fp16 group scales [N, K/128].

    `workspace` (uint8, at least tern_linear_workspace_bytes(T, K, N) bytes) is
    allocated zeroed per call when omitted.  A workspace kept across calls
    must start with SYNC_BYTES zero bytes before its first use and then be
    left alone (the library keeps that area valid); zero it again after
    tern_device_status reports a timeout."""
    T, K = x.shape
    N = Wpacked.shape[0]
    if y is None:
        y = torch.empty((T, N), dtype=torch.float32, device=x.device)
    need = tern_linear_workspace_bytes(T, K, N)
    if workspace is None and need:
        # zeros: the leading synchronisation area must start zeroed
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    pws = _dev(workspace, "workspace", torch.uint8) if workspace is not None else None
    nws = workspace.numel() if workspace is not None else 0
    rc = load().tern_linear(
        _dev(Wpacked, "Wpacked", torch.int32, (N, K // 16)),
        _dev(scales, "scales", torch.float16, (N, K // 128)),
        _dev(x, "x", torch.bfloat16), _dev(y, "y", torch.float32, (T, N)),
        T, K, N, pws, nws, _stream(stream))
    _check("tern_linear", rc)
    return y


def tern_linear_small_t_noalloc(Wpacked: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                                y: torch.Tensor, stream=None) -> torch.Tensor:
    """tern_linear for T = 1..16 that takes no workspace and allocates nothing.

    For callers that cannot allocate device memory (plug-in interfaces that
    pass only inputs and outputs, engines that forbid allocation after
    start-up, latency-critical code where cudaMalloc/cudaFree would
    synchronise the device).  The library's fixed 4 MiB device scratch is
    shared by every call on a device, so calls must not overlap on the GPU.
    The first call on a device does per-device set-up and should come before
    any stream capture.  `y` must be given (fp32 [T, N])."""
    T, K = x.shape
    N = Wpacked.shape[0]
    rc = load().tern_linear_small_t_noalloc(
        _dev(Wpacked, "Wpacked", torch.int32, (N, K // 16)),
        _dev(scales, "scales", torch.float16, (N, K // 128)),
        _dev(x, "x", torch.bfloat16), _dev(y, "y", torch.float32, (T, N)),
        T, K, N, _stream(stream))
    _check("tern_linear_small_t_noalloc", rc)
    return y


def tern_select_rung(T: int) -> int:
    return int(load().tern_select_rung(int(T)))


def tern_rung_name(rung: int) -> str:
    return load().tern_rung_name(int(rung)).decode()


def tern_last_rung() -> str:
    return load().tern_last_rung().decode()


def tern_last_rung_id() -> int:
    return int(load().tern_last_rung_id())


def tern_last_launches() -> int:
    """Kernels this thread's last successful tern_linear launched."""
    return int(load().tern_last_launches())


def tern_reload_env() -> None:
    load().tern_reload_env()


def tern_selftest_wait_timeout(which: int, stream=None) -> None:
    """Launch the failure-path diagnostic: a kernel whose bounded wait (0: an
    mbarrier, 1: a device counter) runs out after 2 s and records the timeout;
    tern_device_status then returns TERN_ETIMEOUT (-6)."""
    _check("tern_selftest_wait_timeout",
           load().tern_selftest_wait_timeout(int(which), _stream(stream)))


def tern_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(load().tern_device_status(_stream(stream)))
