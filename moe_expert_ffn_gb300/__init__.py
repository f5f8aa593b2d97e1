"""GB300 (sm_103a) MegaMoE expert layer: thin Python binding of libmoe_gb300.so.

Everything the layer computes runs in the CUDA library behind the C ABI of
``include/moe.h``; this module only allocates device memory through PyTorch,
marshals pointers and sizes, and turns error codes into exceptions.  If the
library has not been built the import of ``lib()`` raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_DEVICE_TIMEOUT = -4
MOE_ERR_BAD_EXPERT = -5
MOE_ERR_NOT_READY = -6

MOE_W_FP8_BLK128 = 0
MOE_W_FP4_E2M1_UE8M0_32 = 1

# every symbol include/moe.h declares
ABI_SYMBOLS = (
    "moe_workspace_bytes", "moe_weight_bytes", "moe_create", "moe_transform_weights",
    "moe_forward", "moe_forward_host", "moe_get_dispatch", "moe_get_intermediates",
    "moe_dispatch_noalloc", "moe_profile_begin", "moe_profile_end", "moe_test_arm_timeout",
    "moe_device_status", "moe_strerror", "moe_destroy",
)


class MoEConfig(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
                ("num_experts", ctypes.c_int), ("topk", ctypes.c_int), ("wfmt", ctypes.c_int),
                ("act_clamp", ctypes.c_float), ("fast_math", ctypes.c_int)]


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded C-ABI library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            cfgp = ctypes.POINTER(MoEConfig)
            L.moe_workspace_bytes.restype = sz
            L.moe_workspace_bytes.argtypes = [cfgp]
            L.moe_weight_bytes.restype = sz
            L.moe_weight_bytes.argtypes = [cfgp]
            L.moe_create.restype = i32
            L.moe_create.argtypes = [ctypes.POINTER(vp), cfgp, vp, vp]
            L.moe_transform_weights.restype = i32
            L.moe_transform_weights.argtypes = [vp, vp, vp, vp, vp, vp]
            L.moe_forward.restype = i32
            L.moe_forward.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
            L.moe_forward_host.restype = i32
            L.moe_forward_host.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
            L.moe_get_dispatch.restype = i32
            L.moe_get_dispatch.argtypes = [vp, vp, vp, vp, vp]
            L.moe_get_intermediates.restype = i32
            L.moe_get_intermediates.argtypes = [vp, vp, vp, vp, vp]
            L.moe_profile_begin.restype = i32
            L.moe_profile_begin.argtypes = [vp, i32]
            L.moe_profile_end.restype = i32
            L.moe_profile_end.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
            L.moe_test_arm_timeout.restype = i32
            L.moe_test_arm_timeout.argtypes = [vp, i32, i32]
            L.moe_device_status.restype = i32
            L.moe_device_status.argtypes = [vp]
            L.moe_strerror.restype = ctypes.c_char_p
            L.moe_strerror.argtypes = [i32]
            L.moe_destroy.restype = None
            L.moe_destroy.argtypes = [vp]
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_strerror(int(code)).decode()


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoEError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(max_tokens, hidden, inter, num_experts, topk, wfmt=MOE_W_FP8_BLK128,
                act_clamp=math.inf, fast_math=False) -> MoEConfig:
    return MoEConfig(int(max_tokens), int(hidden), int(inter), int(num_experts), int(topk),
                     int(wfmt), float(act_clamp), int(bool(fast_math)))


def workspace_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg)))


def weight_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_weight_bytes(ctypes.byref(cfg)))


class MoELayer:
    """One expert layer bound to a CUDA device: owns (through PyTorch) the
    workspace and the transformed-weight store, and a C-ABI context."""

    def __init__(self, max_tokens, hidden, inter, num_experts, topk, wfmt=MOE_W_FP8_BLK128,
                 act_clamp=math.inf, fast_math=False, device=None):
        self.cfg = make_config(max_tokens, hidden, inter, num_experts, topk, wfmt, act_clamp, fast_math)
        self.device = torch.device(device if device is not None else "cuda")
        ws, wb = workspace_bytes(self.cfg), weight_bytes(self.cfg)
        if ws == 0 or wb == 0:
            raise MoEError(MOE_ERR_INVALID_ARG, "moe config")
        with torch.cuda.device(self.device):
            self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
            self.weights = torch.empty(wb, dtype=torch.uint8, device=self.device)
            ctx = ctypes.c_void_p()
            _check(lib().moe_create(ctypes.byref(ctx), ctypes.byref(self.cfg), _ptr(self.workspace),
                                    _ptr(self.weights)), "moe_create")
        self._ctx = ctx

    # -- properties
    H = property(lambda s: s.cfg.hidden)
    I = property(lambda s: s.cfg.inter)
    E = property(lambda s: s.cfg.num_experts)
    k = property(lambda s: s.cfg.topk)

    def _cuda(self, t, dtype, shape, name):
        if t.device != self.device or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor on {self.device}")
        if t.dtype != dtype and not (dtype == torch.uint8 and t.dtype == torch.float8_e4m3fn):
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        return t

    @property
    def fp4(self) -> bool:
        return self.cfg.wfmt == MOE_W_FP4_E2M1_UE8M0_32

    def transform_weights(self, w1, w1_sf, w2, w2_sf, stream=None):
        E, H, I = self.E, self.H, self.I
        if self.fp4:
            self._cuda(w1, torch.uint8, (E, 2 * I, H // 2), "w1")
            self._cuda(w1_sf, torch.uint8, (E, 2 * I, H // 32), "w1_sf")
            self._cuda(w2, torch.uint8, (E, H, I // 2), "w2")
            self._cuda(w2_sf, torch.uint8, (E, H, I // 32), "w2_sf")
        else:
            self._cuda(w1, torch.uint8, (E, 2 * I, H), "w1")
            self._cuda(w1_sf, torch.float32, (E, 2 * I // 128, H // 128), "w1_sf")
            self._cuda(w2, torch.uint8, (E, H, I), "w2")
            self._cuda(w2_sf, torch.float32, (E, H // 128, I // 128), "w2_sf")
        _check(lib().moe_transform_weights(self._ctx, _ptr(w1), _ptr(w1_sf), _ptr(w2), _ptr(w2_sf),
                                           _stream(stream)), "moe_transform_weights")

    def forward(self, x, x_sf, topk_idx, topk_weights, y=None, stats=None, stream=None):
        T = x.shape[0]
        H, k = self.H, self.k
        self._cuda(x, torch.uint8, (T, H), "x")
        if self.fp4:
            self._cuda(x_sf, torch.uint8, (T, H // 32), "x_sf")
        else:
            self._cuda(x_sf, torch.float32, (T, H // 128), "x_sf")
        self._cuda(topk_idx, torch.int32, (T, k), "topk_idx")
        self._cuda(topk_weights, torch.float32, (T, k), "topk_weights")
        if y is None:
            y = torch.empty(T, H, dtype=torch.bfloat16, device=self.device)
        self._cuda(y, torch.bfloat16, (T, H), "y")
        if stats is not None:
            self._cuda(stats, torch.int32, (self.E,), "stats")
        _check(lib().moe_forward(self._ctx, T, _ptr(x), _ptr(x_sf), _ptr(topk_idx), _ptr(topk_weights),
                                 _ptr(y), _ptr(stats), _stream(stream)), "moe_forward")
        return y

    def forward_host(self, x, x_sf, topk_idx, topk_weights, y=None, stream=None):
        """Host (CPU) tensors in and out; copies happen inside the library call."""
        T = x.shape[0]
        for t, n in ((x, "x"), (x_sf, "x_sf"), (topk_idx, "topk_idx"), (topk_weights, "topk_weights")):
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError(f"{n} must be a contiguous CPU tensor")
        if y is None:
            y = torch.empty(T, self.H, dtype=torch.bfloat16, pin_memory=x.is_pinned())
        _check(lib().moe_forward_host(self._ctx, T, _ptr(x), _ptr(x_sf), _ptr(topk_idx),
                                      _ptr(topk_weights), _ptr(y), _stream(stream)), "moe_forward_host")
        return y

    def get_dispatch(self, num_tokens, stream=None):
        P = num_tokens * self.k
        counts = torch.empty(self.E, dtype=torch.int32, device=self.device)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=self.device)
        gather = torch.empty(max(P, 1), dtype=torch.int32, device=self.device)
        _check(lib().moe_get_dispatch(self._ctx, _ptr(counts), _ptr(offsets), _ptr(gather),
                                      _stream(stream)), "moe_get_dispatch")
        return counts, offsets, gather[:P]

    def get_intermediates(self, num_tokens, stream=None):
        P = max(num_tokens * self.k, 1)
        acts = torch.empty(P, self.I, dtype=torch.uint8, device=self.device)
        if self.fp4:
            sf = torch.empty(P, self.I // 32, dtype=torch.uint8, device=self.device)
        else:
            sf = torch.empty(P, self.I // 64, dtype=torch.float32, device=self.device)
        out = torch.empty(P, self.H, dtype=torch.bfloat16, device=self.device)
        _check(lib().moe_get_intermediates(self._ctx, _ptr(acts), _ptr(sf), _ptr(out), _stream(stream)),
               "moe_get_intermediates")
        return acts, sf, out

    def profile_begin(self, max_forwards: int):
        _check(lib().moe_profile_begin(self._ctx, int(max_forwards)), "moe_profile_begin")

    def profile_end(self):
        """Summed milliseconds per stage (dispatch, l1, l2, combine) and the forward count."""
        ms = (ctypes.c_float * 4)()
        n = ctypes.c_int()
        _check(lib().moe_profile_end(self._ctx, ms, ctypes.byref(n)), "moe_profile_end")
        return {"dispatch": ms[0], "l1": ms[1], "l2": ms[2], "combine": ms[3]}, n.value

    def device_status(self) -> int:
        return int(lib().moe_device_status(self._ctx))

    def arm_timeout_test(self, which: int, wait_limit_us: int):
        """Make the next forward time out on purpose after `wait_limit_us`
        (a test of the failure path): in GEMM `which` (1 = L1, 2 = L2), or at
        the multi-CTA dispatch's barrier (3, batches of 8192 pairs or more)."""
        _check(lib().moe_test_arm_timeout(self._ctx, int(which), int(wait_limit_us)), "moe_test_arm_timeout")

    def close(self):
        if getattr(self, "_ctx", None):
            lib().moe_destroy(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
