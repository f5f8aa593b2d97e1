"""The C-ABI library builds, loads without a GPU and exports every symbol that
include/moe.h declares; host-side argument checks answer without touching the
device."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_expert_ffn_gb300 import build
    build.build()
    import moe_expert_ffn_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree(lib):
    assert _declared() == sorted(lib.ABI_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name


def test_sizes_and_host_checks(lib):
    cfg = lib.make_config(128, 7168, 2048, 256, 8)
    ws, wb = lib.workspace_bytes(cfg), lib.weight_bytes(cfg)
    assert wb >= 256 * 3 * 7168 * 2048
    assert ws >= 128 * 8 * (2048 + 2 * 7168)
    bad = lib.make_config(128, 7168 + 64, 2048, 256, 8)     # H not a multiple of 128
    assert lib.workspace_bytes(bad) == 0 and lib.weight_bytes(bad) == 0
    assert lib.workspace_bytes(lib.make_config(0, 256, 128, 8, 2)) == 0
    assert lib.workspace_bytes(lib.make_config(4, 256, 128, 8, 2, act_clamp=math.nan)) == 0
    L = lib.lib()
    ctx = ctypes.c_void_p()
    assert L.moe_create(ctypes.byref(ctx), ctypes.byref(cfg), None, None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, 1, None, None, None, None, None, None, None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_device_status(None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_test_arm_timeout(None, 1, 1000) == lib.MOE_ERR_INVALID_ARG
    assert lib.strerror(lib.MOE_ERR_BAD_EXPERT).startswith("topk_idx")
    L.moe_destroy(None)
