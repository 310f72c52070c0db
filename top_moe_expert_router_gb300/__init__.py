"""Python binding of libmoe.so: one top-k Mixture-of-Experts layer on one
GB300 (sm_103a).

Argument marshalling only. Every step of the layer runs in the CUDA kernels
behind the C ABI declared in ``include/moe.h``; PyTorch supplies device
memory and streams. There is no fallback: if ``libmoe.so`` is missing or no
GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import _build

_lib = None
_lock = threading.Lock()
HEADER = os.path.join(_build.ROOT, "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE, MOE_ERR_TIMEOUT = range(6)
MOE_W_BF16, MOE_W_NVFP4 = 0, 1
MOE_DECODE_AUTO, MOE_DECODE_CUDA_CORES, MOE_DECODE_TENSOR_CORES = 0, 1, 2


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("E", ctypes.c_int), ("top_k", ctypes.c_int), ("I", ctypes.c_int),
        ("max_tokens", ctypes.c_int), ("fmt", ctypes.c_int),
        ("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
        ("q_gate", ctypes.c_void_p), ("q_up", ctypes.c_void_p), ("q_down", ctypes.c_void_p),
        ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
        ("g_gate", ctypes.c_void_p), ("g_up", ctypes.c_void_p), ("g_down", ctypes.c_void_p),
        ("expert_out_norm", ctypes.c_int),
        ("gate_up_interleaved", ctypes.c_int),
    ]


def header_functions() -> list[str]:
    """Names of the functions include/moe.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status|int|const char\s*\*)\s*(moe_\w+)\s*\(", text, flags=re.M)))


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load(path: str | None = None):
    """Load libmoe.so (building it when stale) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.build()
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        st = ctypes.c_int
        sig = {
            "moe_workspace_size": ([ctypes.POINTER(MoeLayerDesc), ctypes.POINTER(ctypes.c_size_t)], st),
            "moe_layer_create": ([ctypes.POINTER(MoeLayerDesc), vp, ctypes.c_size_t, ctypes.POINTER(vp)], st),
            "moe_route": ([vp, vp, i, vp, vp, vp, vp, vp, vp, vp], st),
            "moe_forward": ([vp, vp, vp, i, vp], st),
            "moe_forward_residual": ([vp, vp, vp, vp, i, vp], st),
            "moe_forward_host": ([vp, vp, vp, i, vp], st),
            "moe_debug_expert_outputs": ([vp, vp, i, vp], st),
            "moe_debug_route_records": ([vp, i, vp, vp, vp, vp, vp, vp, vp], st),
            "moe_debug_hold_grid_barrier": ([vp, i, vp], st),
            "moe_set_decode_path": ([vp, i], st),
            "moe_rmsnorm": ([vp, vp, i, i, f, vp], st),
            "moe_quantize_nvfp4": ([vp, i, i, i, vp, vp, vp, vp], st),
            "moe_get_device_status": ([vp, vp], st),
            "moe_last_launch_count": ([vp], i),
            "moe_profile_begin": ([vp, i], st),
            "moe_profile_end": ([vp, vp, i, ctypes.POINTER(i), ctypes.POINTER(i)], st),
            "moe_layer_destroy": ([vp], st),
            "moe_forward_static_scratch": ([ctypes.POINTER(MoeLayerDesc), vp, vp, i, vp], st),
            "moe_stack_create": ([ctypes.POINTER(vp), i, ctypes.POINTER(vp)], st),
            "moe_stack_forward": ([vp, vp, vp, i, f, vp, vp], st),
            "moe_stack_forward_host": ([vp, vp, vp, i, f, vp], st),
            "moe_stack_destroy": ([vp], st),
            "moe_status_string": ([st], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(s: int) -> str:
    return load().moe_status_string(s).decode()


def _check(s: int, what: str):
    if s != MOE_OK:
        raise MoeError(s, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("device tensors must be contiguous CUDA tensors")


class MoeLayer:
    """One MoE layer over caller-owned device weights (torch CUDA tensors).

    bf16 experts: ``w_gate``/``w_up`` [E, I, d], ``w_down`` [E, d, I] (torch.bfloat16).
    NVFP4 experts: ``nvfp4`` dict with q_gate/q_up [E, I, d/2], q_down [E, d, I/2],
    s_gate/s_up [E, I, d/16], s_down [E, d, I/16] (uint8) and g_gate/g_up/g_down [E] (fp32).
    The workspace is allocated here with torch; the library allocates nothing.
    """

    def __init__(self, w_router, *, w_gate=None, w_up=None, w_down=None, nvfp4=None, w_gate_up=None,
                 router_bias=None, top_k=8, max_tokens=16, expert_out_norm=False):
        lib = load()
        E, d = w_router.shape
        self.d, self.E, self.k, self.max_tokens = d, E, top_k, max_tokens
        desc = MoeLayerDesc()
        desc.d, desc.E, desc.top_k, desc.max_tokens = d, E, top_k, max_tokens
        desc.expert_out_norm = 1 if expert_out_norm else 0
        self._keep = [w_router, router_bias]
        desc.w_router = _ptr(w_router)
        desc.router_bias = _ptr(router_bias)
        if w_gate_up is not None:
            # [E, I, 2, d]: gate row i then up row i of each expert
            _require_cuda(w_router, w_gate_up, w_down, router_bias)
            self.I = w_gate_up.shape[1]
            desc.fmt = MOE_W_BF16
            desc.gate_up_interleaved = 1
            desc.w_gate, desc.w_up, desc.w_down = _ptr(w_gate_up), None, _ptr(w_down)
            self._keep += [w_gate_up, w_down]
        elif nvfp4 is None:
            _require_cuda(w_router, w_gate, w_up, w_down, router_bias)
            self.I = w_gate.shape[1]
            desc.fmt = MOE_W_BF16
            desc.w_gate, desc.w_up, desc.w_down = _ptr(w_gate), _ptr(w_up), _ptr(w_down)
            self._keep += [w_gate, w_up, w_down]
        else:
            _require_cuda(w_router, router_bias, *nvfp4.values())
            self.I = nvfp4["q_gate"].shape[1]
            desc.fmt = MOE_W_NVFP4
            for key, v in nvfp4.items():
                setattr(desc, key, _ptr(v))
            self._keep += list(nvfp4.values())
        desc.I = self.I
        self.fmt = desc.fmt
        size = ctypes.c_size_t(0)
        _check(lib.moe_workspace_size(ctypes.byref(desc), ctypes.byref(size)), "moe_workspace_size")
        self.workspace = torch.empty(size.value, dtype=torch.uint8, device=w_router.device)
        h = ctypes.c_void_p()
        _check(lib.moe_layer_create(ctypes.byref(desc), _ptr(self.workspace), size.value, ctypes.byref(h)),
               "moe_layer_create")
        self._h = h
        self._desc = desc

    # -- calls ----------------------------------------------------------------
    _RECORDS = ("ids", "w", "counts", "offsets", "perm", "pos")

    def _records(self, T, dev):
        return {
            "ids": torch.empty((T, self.k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, self.k), dtype=torch.float32, device=dev),
            "counts": torch.empty(self.E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(self.E + 1, dtype=torch.int32, device=dev),
            "perm": torch.empty(T * self.k, dtype=torch.int32, device=dev),
            "pos": torch.empty((T, self.k), dtype=torch.int32, device=dev),
        }

    def route(self, x, stream=None):
        _require_cuda(x)
        T = x.shape[0]
        out = self._records(T, x.device)
        _check(load().moe_route(self._h, _ptr(x), T, *(_ptr(out[n]) for n in self._RECORDS), _stream(stream)),
               "moe_route")
        return out

    def route_records(self, T, stream=None):
        """The routing records the last forward (or route) of T tokens left in
        the workspace, as that path's own kernels computed them."""
        out = self._records(T, self.workspace.device)
        _check(load().moe_debug_route_records(self._h, T, *(_ptr(out[n]) for n in self._RECORDS),
                                              _stream(stream)), "moe_debug_route_records")
        return out

    def set_decode_path(self, path: int):
        """MOE_DECODE_AUTO, MOE_DECODE_CUDA_CORES or MOE_DECODE_TENSOR_CORES (T <= 16)."""
        _check(load().moe_set_decode_path(self._h, int(path)), "moe_set_decode_path")

    def hold_grid_barrier(self, hold: bool, stream=None):
        """Test hook: make the decode kernel's grid barriers wait for an arrival
        that never comes (its bounded wait then runs out), or restore them."""
        _check(load().moe_debug_hold_grid_barrier(self._h, 1 if hold else 0, _stream(stream)),
               "moe_debug_hold_grid_barrier")

    def forward(self, x, out=None, res=None, stream=None):
        _require_cuda(x, out, res)
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.bfloat16, device=x.device)
        if res is None:
            _check(load().moe_forward(self._h, _ptr(x), _ptr(out), T, _stream(stream)), "moe_forward")
        else:
            _check(load().moe_forward_residual(self._h, _ptr(x), _ptr(res), _ptr(out), T, _stream(stream)),
                   "moe_forward_residual")
        return out

    def forward_host(self, x_host, out_host, stream=None):
        """x_host, out_host: CPU tensors [T, d] bf16 (pinned for async copies)."""
        T = x_host.shape[0]
        _check(load().moe_forward_host(self._h, _ptr(x_host), _ptr(out_host), T, _stream(stream)),
               "moe_forward_host")
        return out_host

    def expert_outputs(self, T, stream=None):
        Y = torch.empty((T * self.k, self.d), dtype=torch.float32, device=self.workspace.device)
        _check(load().moe_debug_expert_outputs(self._h, _ptr(Y), T, _stream(stream)), "moe_debug_expert_outputs")
        return Y

    def device_status(self, stream=None) -> int:
        return load().moe_get_device_status(self._h, _stream(stream))

    def last_launch_count(self) -> int:
        return load().moe_last_launch_count(self._h)

    def profile_begin(self, max_forwards: int):
        _check(load().moe_profile_begin(self._h, max_forwards), "moe_profile_begin")
        self._prof_max = max_forwards

    def profile_end(self, max_kernels: int = 8):
        """-> float32 array [recorded forwards, kernels] of kernel durations in ms."""
        import numpy as np
        nf, nk = ctypes.c_int(), ctypes.c_int()
        buf = np.zeros((getattr(self, "_prof_max", 1), max_kernels), np.float32)
        _check(load().moe_profile_end(self._h, buf.ctypes.data, max_kernels, ctypes.byref(nf), ctypes.byref(nk)),
               "moe_profile_end")
        return buf[:nf.value, :nk.value]

    def close(self):
        if getattr(self, "_h", None):
            load().moe_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoeStack:
    """Layers of equal shape run in one launch: x <- x + MoE_l(RMSNorm(x)) for
    each layer in order (moe_stack_forward). The stack runs on the first
    layer's workspace; keep the layers alive while the stack is used."""

    def __init__(self, layers):
        self.layers = list(layers)
        handles = (ctypes.c_void_p * len(self.layers))(*[ly._h.value for ly in self.layers])
        h = ctypes.c_void_p()
        _check(load().moe_stack_create(handles, len(self.layers), ctypes.byref(h)), "moe_stack_create")
        self._h = h
        self.d = self.layers[0].d

    def forward(self, x, out=None, eps=1e-6, layer_out=None, stream=None):
        _require_cuda(x, out, layer_out)
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.bfloat16, device=x.device)
        _check(load().moe_stack_forward(self._h, _ptr(x), _ptr(out), T, float(eps), _ptr(layer_out),
                                        _stream(stream)), "moe_stack_forward")
        return out

    def forward_host(self, x_host, out_host, eps=1e-6, stream=None):
        """x_host, out_host: CPU tensors [T, d] bf16 (pinned for async copies)."""
        T = x_host.shape[0]
        _check(load().moe_stack_forward_host(self._h, _ptr(x_host), _ptr(out_host), T, float(eps),
                                             _stream(stream)), "moe_stack_forward_host")
        return out_host

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().moe_stack_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rmsnorm(x, eps=1e-6, out=None, stream=None):
    _require_cuda(x, out)
    T, d = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(load().moe_rmsnorm(_ptr(x), _ptr(out), T, d, eps, _stream(stream)), "moe_rmsnorm")
    return out


def quantize_nvfp4(W, stream=None):
    """W [n, rows, K] bf16 on the GPU -> (q [n, rows, K/2] u8, s [n, rows, K/16] u8, g [n] fp32)."""
    _require_cuda(W)
    n, rows, K = W.shape
    q = torch.empty((n, rows, K // 2), dtype=torch.uint8, device=W.device)
    s = torch.empty((n, rows, K // 16), dtype=torch.uint8, device=W.device)
    g = torch.empty(n, dtype=torch.float32, device=W.device)
    _check(load().moe_quantize_nvfp4(_ptr(W), n, rows, K, _ptr(q), _ptr(s), _ptr(g), _stream(stream)),
           "moe_quantize_nvfp4")
    return q, s, g
