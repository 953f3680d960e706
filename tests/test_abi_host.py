"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every symbol include/tern.h declares; the dispatcher's bands and env
overrides; workspace sizing; argument validation before any device work."""
import os
import re

import pytest

import ternary_weight_linear_gb300 as tl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    tl.build()
    tl.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tern.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(tern_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(tl.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    import ctypes
    lib = ctypes.CDLL(tl.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


class env:
    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        for k, v in self.kv.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = str(v)
        tl.tern_reload_env()

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        tl.tern_reload_env()


def test_default_bands():
    with env(TERN_RUNG=None, TERN_SMALL_T_MAX=None, TERN_TILED_MAX=None, TERN_S8_MIN_T=None):
        got = {T: tl.tern_rung_name(tl.tern_select_rung(T)) for T in (1, 2, 8, 9, 16, 17, 2048)}
    assert got == {1: "gemv", 2: "small_t", 8: "small_t", 9: "small_t_tiled",
                   16: "small_t_tiled", 17: "s8", 2048: "s8"}


def test_env_thresholds_and_force():
    with env(TERN_S8_MIN_T=33, TERN_SMALL_T_MAX=4):
        assert tl.tern_rung_name(tl.tern_select_rung(5)) == "small_t_tiled"
        assert tl.tern_rung_name(tl.tern_select_rung(20)) == "small_t_tiled"  # gap below s8
        assert tl.tern_rung_name(tl.tern_select_rung(33)) == "s8"
    for name in ("gemv", "small_t", "small_t_tiled", "s8"):
        with env(TERN_RUNG=name):
            assert all(tl.tern_rung_name(tl.tern_select_rung(T)) == name for T in (1, 7, 16, 500))
    with env(TERN_RUNG="no_such_rung"):
        assert tl.tern_rung_name(tl.tern_select_rung(1)) == "gemv"


def test_env_is_read_once_until_reload():
    with env(TERN_RUNG=None):
        os.environ["TERN_RUNG"] = "s8"
        try:
            assert tl.tern_rung_name(tl.tern_select_rung(1)) == "gemv"  # not re-read
            tl.tern_reload_env()
            assert tl.tern_rung_name(tl.tern_select_rung(1)) == "s8"
        finally:
            os.environ.pop("TERN_RUNG", None)


def test_workspace_bytes():
    assert tl.tern_linear_workspace_bytes(2048, 5120, 34816) >= 2048 * 5120 + 4 * 2048
    assert tl.tern_linear_workspace_bytes(1, 512, 1024) >= 512 + 4
    assert tl.tern_linear_workspace_bytes(0, 512, 1024) == 0


def test_status_strings_and_rung_names():
    assert tl.tern_status_string(0) == "ok"
    assert "workspace" in tl.tern_status_string(-3)
    assert [tl.tern_rung_name(i) for i in range(4)] == ["gemv", "small_t", "small_t_tiled", "s8"]
    assert tl.tern_rung_name(9) == "?"
    assert tl.tern_select_rung(0) == -1


def test_invalid_arguments_are_rejected_before_device_work():
    lib = tl.load()
    p = 4096  # a 16-byte aligned fake address; never dereferenced
    # null pointers / bad sizes -> TERN_EINVAL (-1)
    assert lib.tern_linear(None, p, p, p, 1, 128, 8, None, 0, None) == -1
    assert lib.tern_linear(p, p, p, p, 0, 128, 8, None, 0, None) == -1
    assert lib.tern_linear(p, p, p, p, 1, 100, 8, None, 0, None) == -1   # K % 128
    assert lib.tern_linear(p, p, p, p, 1, 128, 0, None, 0, None) == -1
    assert lib.tern_pack(p, p, 24, 4, None, None) == -1                  # K % 16
    assert lib.tern_quant_act_s8(p, p, p, 0, 16, None) == -1
    # misaligned pointers -> TERN_EALIGN (-2)
    assert lib.tern_linear(p + 2, p, p, p, 1, 128, 8, None, 0, None) == -2
    assert lib.tern_pack(p, p + 4, 16, 4, None, None) == -2
    assert lib.tern_quant_act_s8(p, p, p + 8, 1, 16, None) == -2
    # base-3 repack: K % 128, null, misaligned
    assert lib.tern_repack_t5(p, p, 64, 4, None, None) == -1
    assert lib.tern_repack_t5(None, p, 128, 4, None, None) == -1
    assert lib.tern_repack_t5(p + 2, p, 128, 4, None, None) == -2
    # rotation: K % 1024, partial overlap of x and xr, misaligned
    assert lib.tern_rotate_bf16(p, 1 << 20, 1, 512, None) == -1
    assert lib.tern_rotate_bf16(p, p + 1024, 2, 1024, None) == -1
    assert lib.tern_rotate_bf16(p, (1 << 20) + 8, 1, 1024, None) == -2
    # failure-path diagnostic: only which = 0 or 1
    assert lib.tern_selftest_wait_timeout(2, None) == -1
    assert lib.tern_selftest_wait_timeout(-1, None) == -1


def test_rotation_switch_rejects_unrotatable_k(monkeypatch):
    lib = tl.load()
    p = 4096
    monkeypatch.setenv("TERN_ROTATE", "1")
    tl.tern_reload_env()
    try:
        # whole 1024-wide rotation blocks only, and K <= 65536
        assert lib.tern_linear(p, p, p, p, 1, 512, 8, None, 0, None) == -1
        assert lib.tern_linear(p, p, p, p, 1, 66560, 8, None, 0, None) == -1
        assert lib.tern_linear_small_t_noalloc(p, p, p, p, 1, 1536, 8, None) == -1
    finally:
        monkeypatch.delenv("TERN_ROTATE")
        tl.tern_reload_env()


def test_int8_decode_has_no_rotated_form(monkeypatch):
    lib = tl.load()
    p = 4096
    monkeypatch.setenv("TERN_ROTATE", "1")
    monkeypatch.setenv("TERN_DECODE_ACT", "int8")
    tl.tern_reload_env()
    try:
        assert lib.tern_linear(p, p, p, p, 1, 1024, 8, None, 0, None) == -1
        assert lib.tern_linear_small_t_noalloc(p, p, p, p, 4, 1024, 8, None) == -1
    finally:
        monkeypatch.delenv("TERN_ROTATE")
        monkeypatch.delenv("TERN_DECODE_ACT")
        tl.tern_reload_env()


def test_no_gpu_gives_enodev():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    lib = tl.load()
    p = 4096
    assert lib.tern_linear(p, p, p, p, 1, 128, 8, None, 0, None) == -4
    assert lib.tern_device_status(None) == -4
