"""CPU oracle for one top-k Mixture-of-Experts layer — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library and its Python binding
never import it, and the oracle never imports them.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
independent tokens/slots); this module compiles it with the host gcc on first
use and wraps it with numpy. Every function cites, in ``oracle.c``, the
passage of the pages it follows and the reading taken where the pages are
silent. All functions are pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place. -ffp-contract=off keeps every product and
    sum separately rounded, as written in the C source."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class OrcLayer(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
        ("fmt", ctypes.c_int),
        ("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
        ("q_gate", ctypes.c_void_p), ("q_up", ctypes.c_void_p), ("q_down", ctypes.c_void_p),
        ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
        ("g_gate", ctypes.c_void_p), ("g_up", ctypes.c_void_p), ("g_down", ctypes.c_void_p),
        ("expert_norm", ctypes.c_int),
    ]


def _lib_get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = d
            lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_decode.restype = ctypes.c_float
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = ctypes.c_float
            lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
            lib.orc_e2m1_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_quantize_nvfp4.argtypes = [vp, i, i, vp, vp, vp]
            lib.orc_dequant_nvfp4_row.argtypes = [vp, vp, ctypes.c_float, i, vp]
            lib.orc_router_logits.argtypes = [vp, vp, vp, i, i, i, vp]
            lib.orc_select_topk.argtypes = [vp, i, i, i, vp, vp, vp]
            lib.orc_weights_for_ids.argtypes = [vp, i, i, i, vp, vp]
            lib.orc_permute.argtypes = [vp, i, i, i, vp, vp, vp, vp]
            lib.orc_expert_ffn.argtypes = [ctypes.POINTER(OrcLayer), i, vp, vp, vp]
            lib.orc_forward.argtypes = [ctypes.POINTER(OrcLayer), vp, i, vp, i, vp, vp, vp, vp, vp, vp]
            lib.orc_rmsnorm.argtypes = [vp, i, i, d, vp]
            lib.orc_residual_add.argtypes = [vp, vp, ctypes.c_longlong, vp]
            lib.orc_max_threads.restype = i
            lib.orc_set_threads.argtypes = [i]
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return float(_lib_get().orc_e2m1_decode(code))


def e4m3_decode(code: int) -> float:
    return float(_lib_get().orc_e4m3_decode(code))


def e2m1_encode(v: float) -> int:
    return int(_lib_get().orc_e2m1_encode(v))


def e4m3_encode(v: float) -> int:
    return int(_lib_get().orc_e4m3_encode(v))


def quantize_nvfp4(W: np.ndarray):
    """One tensor W[rows, K] (bf16 bits) -> (q [rows, K/2] u8, s [rows, K/16] u8, g fp32)."""
    W = _c(W, np.uint16)
    rows, K = W.shape
    assert K % 16 == 0
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 16), np.uint8)
    g = np.zeros(1, np.float32)
    _lib_get().orc_quantize_nvfp4(_p(W), rows, K, _p(q), _p(s), _p(g))
    return q, s, float(g[0])


def dequant_nvfp4(q: np.ndarray, s: np.ndarray, g: float) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    rows = q.shape[0]
    K = q.shape[1] * 2
    out = np.empty((rows, K), np.float32)
    lib = _lib_get()
    for r in range(rows):
        lib.orc_dequant_nvfp4_row(q[r].ctypes.data, s[r].ctypes.data, ctypes.c_float(g), K,
                                  out[r].ctypes.data)
    return out


# ---------------------------------------------------------------------------
# routing and permutation
# ---------------------------------------------------------------------------

def router_logits(x, w_router, bias=None):
    x, w_router = _c(x, np.uint16), _c(w_router, np.uint16)
    bias = _c(bias, np.float32)
    T, d = x.shape
    E = w_router.shape[0]
    out = np.empty((T, E), np.float32)
    _lib_get().orc_router_logits(_p(x), _p(w_router), _p(bias), T, d, E, _p(out))
    return out


def select_topk(logits, k):
    """-> ids [T,k] int32, w [T,k] float64, gap [T] float64."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    gap = np.empty(T, np.float64)
    _lib_get().orc_select_topk(_p(logits), T, E, k, _p(ids), _p(w), _p(gap))
    return ids, w, gap


def weights_for_ids(logits, ids):
    logits, ids = _c(logits, np.float32), _c(ids, np.int32)
    T, E = logits.shape
    k = ids.shape[1]
    w = np.empty((T, k), np.float64)
    _lib_get().orc_weights_for_ids(_p(logits), T, E, k, _p(ids), _p(w))
    return w


def permute(ids, E):
    """-> counts [E], offsets [E+1], perm [T*k], pos [T,k] (int32)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pos = np.empty((T, k), np.int32)
    _lib_get().orc_permute(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(pos))
    return counts, offsets, perm, pos


# ---------------------------------------------------------------------------
# layer
# ---------------------------------------------------------------------------

class Layer:
    """Host copies of one layer's parameters for the oracle.

    bf16 experts: ``gate``/``up`` [E, I, d] and ``down`` [E, d, I] as uint16 bits.
    nvfp4 experts: ``nvfp4`` = dict with q_gate/q_up [E, I, d/2], q_down [E, d, I/2],
    s_gate/s_up [E, I, d/16], s_down [E, d, I/16] (uint8) and g_gate/g_up/g_down [E] fp32.
    """

    def __init__(self, w_router, gate=None, up=None, down=None, router_bias=None, k=8, nvfp4=None,
                 expert_norm=False):
        self.w_router = _c(w_router, np.uint16)
        self.router_bias = _c(router_bias, np.float32)
        self.E, self.d = self.w_router.shape
        self.k = k
        self._keep = []
        s = OrcLayer()
        s.d, s.E, s.k = self.d, self.E, k
        s.w_router = _p(self.w_router)
        s.router_bias = _p(self.router_bias)
        if nvfp4 is None:
            self.gate, self.up, self.down = (_c(a, np.uint16) for a in (gate, up, down))
            self.I = self.gate.shape[1]
            s.fmt = 0
            s.w_gate, s.w_up, s.w_down = _p(self.gate), _p(self.up), _p(self.down)
        else:
            f = {key: _c(v, np.float32 if key.startswith("g_") else np.uint8) for key, v in nvfp4.items()}
            self.nvfp4 = f
            self.I = f["q_gate"].shape[1]
            s.fmt = 1
            for key, v in f.items():
                setattr(s, key, _p(v))
        s.I = self.I
        s.expert_norm = 1 if expert_norm else 0
        self._s = s

    def forward(self, x, tokens=None, forced_ids=None, want_Y=False):
        """Oracle layer output for the listed tokens (all when None).

        Returns dict: ids [n,k], w [n,k], gap [n], y [n,d] (float64), Y [n,k,d] if want_Y.
        """
        x = _c(x, np.uint16)
        T = x.shape[0]
        tok = None if tokens is None else _c(tokens, np.int32)
        n = T if tok is None else tok.shape[0]
        forced = _c(forced_ids, np.int32)
        ids = np.empty((n, self.k), np.int32)
        w = np.empty((n, self.k), np.float64)
        gap = np.empty(n, np.float64)
        Y = np.empty((n, self.k, self.d), np.float64) if want_Y else None
        y = np.empty((n, self.d), np.float64)
        _lib_get().orc_forward(ctypes.byref(self._s), _p(x), T, _p(tok), n, _p(forced),
                               _p(ids), _p(w), _p(gap), _p(Y), _p(y))
        out = {"ids": ids, "w": w, "gap": gap, "y": y}
        if want_Y:
            out["Y"] = Y
        return out

    def expert(self, e, x_row):
        """(h [I], Y [d]) of expert e on one bf16 token row."""
        x_row = _c(x_row, np.uint16)
        h = np.empty(self.I, np.float64)
        Y = np.empty(self.d, np.float64)
        _lib_get().orc_expert_ffn(ctypes.byref(self._s), int(e), _p(x_row), _p(h), _p(Y))
        return h, Y


def rmsnorm(x, eps=1e-6):
    x = _c(x, np.uint16)
    T, d = x.shape
    u = np.empty_like(x)
    _lib_get().orc_rmsnorm(_p(x), T, d, float(eps), _p(u))
    return u


def residual_add(x, y):
    x = _c(x, np.uint16)
    y = _c(y, np.float64)
    out = np.empty_like(x)
    _lib_get().orc_residual_add(_p(x), _p(y), x.size, _p(out))
    return out


def max_threads() -> int:
    return int(_lib_get().orc_max_threads())


def set_threads(n: int) -> None:
    _lib_get().orc_set_threads(int(n))
