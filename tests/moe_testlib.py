"""Shared helpers of the parity tests: build one layer's inputs with the seeded
generator, hand the same bytes to the CUDA layer and to the CPU oracle, and
compare the two the way the parity bar states it."""
from __future__ import annotations

import numpy as np
import torch

import datagen
import oracle

BF16_TOL = 2e-2      # layer output, bf16 expert weights: max normwise relative error
NVFP4_TOL = 5e-2     # layer output, NVFP4 expert weights
NEAR_TIE = 1e-3      # fp32 logit gap between the k-th and (k+1)-th expert
# Renormalised weights: w_j = exp(l_j - l_max) / sum_sel exp(l_i - l_max), so
# their relative error is about twice the absolute error of the fp32 logits.
# An fp32 dot product over d = 4096 terms of size ~0.3 (logits of size ~20)
# carries errors of order sqrt(d) * 2^-24 * 20 ~ 1e-4, up to a few 1e-4 on
# unlucky rows: hence 1e-3.
W_RTOL = 1e-3


def to_dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class HostLayer:
    """Host arrays of one layer, drawn from the seeded generator."""

    def __init__(self, w: datagen.Workload, layer: int = 0, experts=None, with_bias=None):
        self.w = w
        self.wr = datagen.router_weights(w, layer)
        self.bias = datagen.router_bias(w, layer) if (with_bias is None or with_bias) else None
        self.gate, self.up, self.down = datagen.expert_weights(w, layer, experts=experts)

    def oracle(self, bias=True):
        return oracle.Layer(self.wr, self.gate, self.up, self.down,
                            router_bias=self.bias if bias else None, k=self.w.k)


def normwise_rel_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    """Per row: max_c |y_gpu - y_ref| / max_c |y_ref|."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = np.maximum(np.abs(y_ref).max(axis=-1), 1e-30)
    return np.abs(y_gpu - y_ref).max(axis=-1) / den


def check_route(r_gpu: dict, ref_ids: np.ndarray, ref_w: np.ndarray, gap: np.ndarray, E: int, tokens=None):
    """Routing parity. ids bit-exact where the oracle's gap exceeds NEAR_TIE;
    the permutation bit-exact against the oracle's permutation of the GPU ids
    (which equals the oracle's own wherever ids agree). Returns near-tie count."""
    ids = r_gpu["ids"].cpu().numpy()
    w = r_gpu["w"].cpu().numpy()
    sel = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    clear = gap > NEAR_TIE
    np.testing.assert_array_equal(ids[sel][clear], ref_ids[clear])
    np.testing.assert_allclose(w[sel][clear], ref_w[clear], rtol=W_RTOL, atol=1e-6)
    # every GPU row is a valid top-k selection: k distinct experts, weights sum to 1, descending
    assert all(len(set(row.tolist())) == ids.shape[1] for row in ids)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-5)
    assert (np.diff(w, axis=1) <= 1e-7).all()
    counts, offsets, perm, pos = oracle.permute(ids, E)
    np.testing.assert_array_equal(r_gpu["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(r_gpu["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(r_gpu["perm"].cpu().numpy(), perm)
    np.testing.assert_array_equal(r_gpu["pos"].cpu().numpy(), pos)
    return int((~clear).sum())
