"""CPU oracle of the MegaMoE expert layer (ctypes wrapper around moe_oracle.c).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The CUDA product path
never imports it and shares no code with it.

The C source states what is computed and which passage of the pages each step
follows (MegaMoE SM90 Implementation Design (Final), §3.3, §10.1, §11, §15, §20;
PR357 Green-Context Split MegaMoE code review, §1, §3.2, §6).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
EINVAL = -1
EBADEXPERT = -5


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (gcc, OpenMP, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class OrcCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("wfmt", ctypes.c_int),
                ("act_clamp", ctypes.c_float)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, u8 = ctypes.c_void_p, ctypes.c_uint8
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [u8]
            L.orc_e4m3_encode.restype = u8
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_bf16_encode.restype = ctypes.c_uint16
            L.orc_bf16_encode.argtypes = [ctypes.c_float]
            L.orc_bf16_decode.restype = ctypes.c_float
            L.orc_bf16_decode.argtypes = [ctypes.c_uint16]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [u8]
            L.orc_e2m1_encode.restype = u8
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_ue8m0_decode.restype = ctypes.c_double
            L.orc_ue8m0_decode.argtypes = [u8]
            L.orc_ue8m0_for_amax.restype = u8
            L.orc_ue8m0_for_amax.argtypes = [ctypes.c_float, ctypes.c_float]
            L.orc_quant_fp8_group.restype = ctypes.c_float
            L.orc_quant_fp8_group.argtypes = [vp, ctypes.c_int, vp]
            L.orc_quant_fp8_ue8m0_group.restype = u8
            L.orc_quant_fp8_ue8m0_group.argtypes = [vp, ctypes.c_int, vp]
            L.orc_dispatch.restype = ctypes.c_int
            L.orc_dispatch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
            L.orc_forward.restype = ctypes.c_int
            L.orc_forward.argtypes = [ctypes.POINTER(OrcCfg), vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_int, vp, vp]
            L.orc_pair.restype = ctypes.c_int
            L.orc_pair.argtypes = [ctypes.POINTER(OrcCfg), vp, vp, vp, vp, vp, vp,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                   vp, vp, vp, vp, vp]
            L.orc_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(a):
    """numpy view of a CPU tensor or array (no copy for contiguous inputs)."""
    if hasattr(a, "detach"):
        a = a.detach()
        if a.device.type != "cpu":
            a = a.cpu()
        a = a.contiguous()
        import torch
        if a.dtype in (torch.float8_e4m3fn, torch.float8_e8m0fnu):
            a = a.view(torch.uint8)
        elif a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        return a.numpy()
    return np.ascontiguousarray(a)


# ---- scalar codecs -------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def bf16_encode(v: float) -> int:
    return lib().orc_bf16_encode(float(v))


def bf16_decode(h: int) -> float:
    return lib().orc_bf16_decode(int(h) & 0xFFFF)


def e2m1_decode(nib: int) -> float:
    return lib().orc_e2m1_decode(int(nib))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def ue8m0_decode(code: int) -> float:
    return lib().orc_ue8m0_decode(int(code))


def ue8m0_for_amax(amax: float, qmax: float) -> int:
    return lib().orc_ue8m0_for_amax(float(amax), float(qmax))


def quant_fp8_group(a) -> tuple[float, np.ndarray]:
    a = np.ascontiguousarray(a, dtype=np.float32)
    q = np.zeros(a.shape[0], dtype=np.uint8)
    sf = lib().orc_quant_fp8_group(_ptr(a), a.shape[0], _ptr(q))
    return sf, q


def quant_fp8_ue8m0_group(a) -> tuple[int, np.ndarray]:
    a = np.ascontiguousarray(a, dtype=np.float32)
    q = np.zeros(a.shape[0], dtype=np.uint8)
    code = lib().orc_quant_fp8_ue8m0_group(_ptr(a), a.shape[0], _ptr(q))
    return code, q


# ---- dispatch and the layer ---------------------------------------------
def dispatch(topk_idx, num_experts: int):
    """Returns (status, count[E], offset[E+1], gather[P_active])."""
    idx = np.ascontiguousarray(_np(topk_idx), dtype=np.int32)
    T, k = idx.shape
    count = np.zeros(num_experts, dtype=np.int32)
    offset = np.zeros(num_experts + 1, dtype=np.int32)
    gather = np.full(max(T * k, 1), -1, dtype=np.int32)
    st = lib().orc_dispatch(T, k, num_experts, _ptr(idx), _ptr(count), _ptr(offset), _ptr(gather))
    return st, count, offset, gather[: int(offset[-1])]


def _cfg(T, H, I, E, k, wfmt, act_clamp):
    return OrcCfg(T, H, I, E, k, wfmt, act_clamp)


def forward(inp: dict, tokens=None, wfmt: int = 0, act_clamp: float = float("inf")):
    """y rows (BF16 bits as uint16) of ``tokens`` (default: all tokens).

    ``inp`` holds x, x_sf, topk_idx, topk_weights, w1, w1_sf, w2, w2_sf as CPU
    tensors or numpy arrays in the canonical layouts of the C-ABI.
    """
    x = _np(inp["x"]); x_sf = _np(inp["x_sf"])
    idx = np.ascontiguousarray(_np(inp["topk_idx"]), dtype=np.int32)
    tw = np.ascontiguousarray(_np(inp["topk_weights"]), dtype=np.float32)
    w1 = _np(inp["w1"]); w1_sf = _np(inp["w1_sf"]); w2 = _np(inp["w2"]); w2_sf = _np(inp["w2_sf"])
    T, H = x.shape
    k = idx.shape[1]
    E = w1.shape[0]
    I = w2.shape[2] * (2 if wfmt == 1 else 1)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    sel = np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.zeros((sel.shape[0], H), dtype=np.uint16)
    cfg = _cfg(T, H, I, E, k, wfmt, act_clamp)
    st = lib().orc_forward(ctypes.byref(cfg), _ptr(x), _ptr(x_sf), _ptr(idx), _ptr(tw),
                           _ptr(w1), _ptr(w1_sf), _ptr(w2), _ptr(w2_sf), sel.shape[0], _ptr(sel), _ptr(y))
    if st not in (OK, EBADEXPERT):
        raise ValueError(f"oracle forward failed: {st}")
    return y


def pair(inp: dict, t: int, e: int, w: float, wfmt: int = 0, act_clamp: float = float("inf")):
    """Intermediates of one (token, expert) pair: a, q, sf, o, ob."""
    x = _np(inp["x"]); x_sf = _np(inp["x_sf"])
    w1 = _np(inp["w1"]); w1_sf = _np(inp["w1_sf"]); w2 = _np(inp["w2"]); w2_sf = _np(inp["w2_sf"])
    T, H = x.shape
    E = w1.shape[0]
    I = w2.shape[2] * (2 if wfmt == 1 else 1)
    a = np.zeros(I, dtype=np.float32)
    q = np.zeros(I, dtype=np.uint8)
    sf = np.zeros(I // 32, dtype=np.float32)
    o = np.zeros(H, dtype=np.float64)
    ob = np.zeros(H, dtype=np.uint16)
    cfg = _cfg(T, H, I, E, 1, wfmt, act_clamp)
    st = lib().orc_pair(ctypes.byref(cfg), _ptr(x), _ptr(x_sf), _ptr(w1), _ptr(w1_sf), _ptr(w2),
                        _ptr(w2_sf), int(t), int(e), float(w), _ptr(a), _ptr(q), _ptr(sf), _ptr(o), _ptr(ob))
    if st != OK:
        raise ValueError(f"oracle pair failed: {st}")
    ng = I // 64 if wfmt == 0 else I // 32
    return {"a": a, "q": q, "sf": sf[:ng], "o": o, "ob": ob}


def num_threads() -> int:
    return lib().orc_num_threads()
