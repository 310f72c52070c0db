"""Seeded synthetic inputs for the MoE layer.

This package draws numbers and nothing else: it holds no step of the MoE
method (no routing, no FFN, no quantisation). Both the CPU oracle and the
CUDA path consume the arrays it returns, so the two sides always see the same
bytes. The C generator (``datagen.c``) is compiled on first use with the host
gcc; it is portable C (no architecture intrinsics).

Workload recipes follow the five MoE-layer workloads the layer is measured on
(tiny correctness case, T=1 decode, T=4/16 batched decode, T=4096 prefill with
a skewed router bias, 8 stacked NVFP4 layers). Bf16 arrays are returned as
``numpy.uint16`` holding the raw bf16 bits.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "datagen.c")
_LIB = os.path.join(_HERE, "libdatagen.so")
_lock = threading.Lock()
_lib = None

# Stream tags; each layer adds 16 * layer so layers draw independent streams.
TAG_ROUTER, TAG_GATE, TAG_UP, TAG_DOWN, TAG_X, TAG_BIAS_PERM = 0, 1, 2, 3, 4, 5
WEIGHT_SIGMA = 0.02


def build(force: bool = False) -> str:
    """Compile libdatagen.so in place (gcc, OpenMP). Returns the path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32p = ctypes.c_uint64, ctypes.POINTER(ctypes.c_int32)
            lib.dg_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_void_p]
            lib.dg_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_void_p]
            lib.dg_uniform_f64.argtypes = [u64, u64, u64, u64, ctypes.c_void_p]
            lib.dg_permutation.argtypes = [u64, u64, ctypes.c_int, i32p]
            lib.dg_raw.argtypes = [u64, u64, u64]
            lib.dg_raw.restype = u64
            _lib = lib
    return _lib


def normal_bf16(seed: int, tag: int, shape, sigma: float, start: int = 0, out=None) -> np.ndarray:
    """bf16 bits of sigma * N(0,1), elements [start, start+n) of stream (seed, tag)."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _get().dg_normal_bf16(seed, tag, start, n, float(sigma), out.ctypes.data)
    return out


def normal_f32(seed: int, tag: int, shape, sigma: float, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(shape, dtype=np.float32)
    _get().dg_normal_f32(seed, tag, start, n, float(sigma), out.ctypes.data)
    return out


def uniform_f64(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _get().dg_uniform_f64(seed, tag, start, n, out.ctypes.data)
    return out


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _get().dg_permutation(seed, tag, n, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return out


def raw_u64(seed: int, tag: int, i: int) -> int:
    return int(_get().dg_raw(seed, tag, i))


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bits (NaN kept quiet)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = (u & 0x7F800000) == 0x7F800000
    nan &= (u & 0x007FFFFF) != 0
    if nan.any():
        r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

# Router weight multiplier for the d=4096 workloads: W_r = bf16(s * N(0, 0.02^2)).
# With s = ROUTER_SCALE_D4096 about 5% of N(0,1) tokens have a gap below 0.05
# between their 8th and 9th largest fp32 logit (seed 0, 16384 tokens). The value
# was found by bisection with oracle/calibrate_inputs.py and is re-checked on a
# smaller sample by the test suite.
ROUTER_SCALE_D4096 = 12.8
# Skew of the prefill router bias: b_e = alpha * (-1.1 * ln r_e), r a seeded
# permutation of 1..E. alpha puts max/mean expert load near 4 at T=4096 (seed 0);
# found with oracle/calibrate_inputs.py.
ZIPF_ALPHA = 2.34
ZIPF_EXPONENT = 1.1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    fmt: str = "bf16"           # expert weight format: "bf16" or "nvfp4"
    router_scale: float = 1.0
    zipf_alpha: float = 0.0      # 0: no router bias
    layers: int = 1
    seed: int = 0

    @property
    def expert_bytes_bf16(self) -> int:
        return 3 * self.d * self.I * 2

    @property
    def expert_bytes_nvfp4(self) -> int:
        # packed E2M1 (4 bit) + one E4M3 byte per 16 elements, three matrices
        return 3 * self.d * self.I // 2 + 3 * self.d * self.I // 16


WORKLOADS = {
    "tiny": Workload("tiny", T=8, d=256, E=256, k=8, I=128),
    "decode_t1": Workload("decode_t1", T=1, d=4096, E=256, k=8, I=1536,
                          router_scale=ROUTER_SCALE_D4096),
    "decode_t4": Workload("decode_t4", T=4, d=4096, E=256, k=8, I=1536,
                          router_scale=ROUTER_SCALE_D4096),
    "decode_t8": Workload("decode_t8", T=8, d=4096, E=256, k=8, I=1536,
                          router_scale=ROUTER_SCALE_D4096),
    "decode_t16": Workload("decode_t16", T=16, d=4096, E=256, k=8, I=1536,
                           router_scale=ROUTER_SCALE_D4096),
    "prefill_t4096": Workload("prefill_t4096", T=4096, d=4096, E=256, k=8, I=1536,
                              router_scale=ROUTER_SCALE_D4096, zipf_alpha=ZIPF_ALPHA),
    "nvfp4_stack_t4": Workload("nvfp4_stack_t4", T=4, d=4096, E=256, k=8, I=1536,
                               fmt="nvfp4", router_scale=ROUTER_SCALE_D4096, layers=8),
    # the prefill layer (same seeded weights and router bias) with its experts in NVFP4
    "nvfp4_prefill_t4096": Workload("nvfp4_prefill_t4096", T=4096, d=4096, E=256, k=8, I=1536, fmt="nvfp4",
                                    router_scale=ROUTER_SCALE_D4096, zipf_alpha=ZIPF_ALPHA),
}


def tag(base: int, layer: int) -> int:
    return base + 16 * layer


def router_weights(w: Workload, layer: int = 0, seed: int | None = None) -> np.ndarray:
    seed = w.seed if seed is None else seed
    return normal_bf16(seed, tag(TAG_ROUTER, layer), (w.E, w.d), WEIGHT_SIGMA * w.router_scale)


def router_bias(w: Workload, layer: int = 0, seed: int | None = None, alpha: float | None = None):
    """fp32 per-expert bias, alpha * (-1.1 ln r_e) with r a seeded permutation of 1..E."""
    seed = w.seed if seed is None else seed
    alpha = w.zipf_alpha if alpha is None else alpha
    if alpha == 0.0:
        return None
    ranks = permutation(seed, tag(TAG_BIAS_PERM, layer), w.E).astype(np.float64) + 1.0
    return (alpha * (-ZIPF_EXPONENT * np.log(ranks))).astype(np.float32)


def expert_weights(w: Workload, layer: int = 0, seed: int | None = None, experts=None):
    """bf16 expert stacks: gate, up [E, I, d]; down [E, d, I].

    ``experts``: optional list of expert ids; then only those slices are drawn
    (the others are left zero) and the arrays still have the full [E, ...] shape.
    """
    seed = w.seed if seed is None else seed
    gate = np.zeros((w.E, w.I, w.d), dtype=np.uint16) if experts is not None else np.empty((w.E, w.I, w.d), np.uint16)
    up = np.zeros_like(gate) if experts is not None else np.empty_like(gate)
    down = np.zeros((w.E, w.d, w.I), dtype=np.uint16) if experts is not None else np.empty((w.E, w.d, w.I), np.uint16)
    per = w.I * w.d
    if experts is None:
        normal_bf16(seed, tag(TAG_GATE, layer), gate.shape, WEIGHT_SIGMA, out=gate)
        normal_bf16(seed, tag(TAG_UP, layer), up.shape, WEIGHT_SIGMA, out=up)
        normal_bf16(seed, tag(TAG_DOWN, layer), down.shape, WEIGHT_SIGMA, out=down)
    else:
        for e in sorted(set(int(e) for e in experts)):
            normal_bf16(seed, tag(TAG_GATE, layer), (w.I, w.d), WEIGHT_SIGMA, start=e * per, out=gate[e])
            normal_bf16(seed, tag(TAG_UP, layer), (w.I, w.d), WEIGHT_SIGMA, start=e * per, out=up[e])
            normal_bf16(seed, tag(TAG_DOWN, layer), (w.d, w.I), WEIGHT_SIGMA, start=e * per, out=down[e])
    return gate, up, down


def tokens(w: Workload, n: int, layer: int = 0, seed: int | None = None, start_row: int = 0) -> np.ndarray:
    """n rows of x ~ N(0, 1) in bf16, rows [start_row, start_row + n) of the token stream."""
    seed = w.seed if seed is None else seed
    return normal_bf16(seed, tag(TAG_X, layer), (n, w.d), 1.0, start=start_row * w.d)
