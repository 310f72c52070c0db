"""Stacked layers in one launch (moe_stack_forward): every layer's output is
bit-identical to running the layers one by one (moe_rmsnorm, then
moe_forward_residual), which the other parity tests check against the
oracle; and the last layer is checked against the oracle directly."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from moe_testlib import BF16_TOL, NVFP4_TOL, bf16_host, normwise_rel_err, to_dev_bf16

pytestmark = pytest.mark.gpu


def _per_layer(moe, layers, x, eps):
    """Reference on the GPU: one rmsnorm and one residual forward per layer."""
    cur = x.clone()
    outs = []
    for gl in layers:
        u = moe.rmsnorm(cur, eps)
        cur = gl.forward(u, res=cur)
        outs.append(cur.clone())
    return outs


def _bf16_layers(moe, w, n):
    layers, host = [], []
    for li in range(n):
        wr = datagen.router_weights(w, li)
        g, u, d = datagen.expert_weights(w, li)
        layers.append(moe.MoeLayer(to_dev_bf16(wr), w_gate=to_dev_bf16(g), w_up=to_dev_bf16(u),
                                   w_down=to_dev_bf16(d), top_k=w.k, max_tokens=16))
        host.append((wr, g, u, d))
    return layers, host


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_stack_bf16_matches_layer_by_layer(gpu_lib, T, path):
    """path 1: the CUDA-core kernel, 2: the tensor-core kernel, for the stack
    and for the layer-by-layer reference alike."""
    w = datagen.WORKLOADS["tiny"]
    layers, host = _bf16_layers(gpu_lib, w, 3)
    for gl in layers:
        gl.set_decode_path(path)
    x = to_dev_bf16(datagen.tokens(w, T, start_row=40))
    stack = gpu_lib.MoeStack(layers)
    lo = torch.empty((3, T, w.d), dtype=torch.bfloat16, device="cuda")
    y = stack.forward(x, eps=1e-6, layer_out=lo)
    assert layers[0].last_launch_count() == 1
    ref = _per_layer(gpu_lib, layers, x, 1e-6)
    torch.cuda.synchronize()
    assert layers[0].device_status() == 0
    for li in range(3):
        assert torch.equal(lo[li].view(torch.int16), ref[li].view(torch.int16)), f"layer {li}"
    assert torch.equal(y.view(torch.int16), ref[-1].view(torch.int16))
    # the last layer against the oracle, given the GPU's input to it
    wr, g, u, d = host[2]
    xin = bf16_host(lo[1])
    L = oracle.Layer(wr, g, u, d, k=w.k)
    uin = oracle.rmsnorm(xin, 1e-6)
    ref_y = L.forward(uin)["y"]
    want = datagen.bf16_to_f32(xin) + ref_y
    got = datagen.bf16_to_f32(bf16_host(lo[2]))
    bound = np.abs(want) * 2 ** -7 + BF16_TOL * np.abs(ref_y).max(1, keepdims=True)
    assert (np.abs(got - want) <= bound).all()


@pytest.mark.parametrize("path", [1, 2])
def test_stack_nvfp4_matches_layer_by_layer(gpu_lib, path):
    """4 NVFP4 layers of the full width (d=4096, I=1536), 32 experts each, T=4
    (path 1: CUDA-core kernel, 2: tensor-core kernel)."""
    w = datagen.Workload("fp4stack", T=4, d=4096, E=32, k=8, I=1536, fmt="nvfp4",
                         router_scale=datagen.ROUTER_SCALE_D4096)
    layers = []
    for li in range(4):
        wr = datagen.router_weights(w, li)
        g, u, d = datagen.expert_weights(w, li)
        packs = {}
        for name, arr in (("gate", g), ("up", u), ("down", d)):
            q, s, gs = gpu_lib.quantize_nvfp4(to_dev_bf16(arr))
            packs["q_" + name], packs["s_" + name], packs["g_" + name] = q, s, gs
        layers.append(gpu_lib.MoeLayer(to_dev_bf16(wr), nvfp4=packs, top_k=8, max_tokens=16))
        layers[-1].set_decode_path(path)
    x = to_dev_bf16(datagen.tokens(w, 4, start_row=8))
    stack = gpu_lib.MoeStack(layers)
    lo = torch.empty((4, 4, w.d), dtype=torch.bfloat16, device="cuda")
    y = stack.forward(x, eps=1e-6, layer_out=lo)
    ref = _per_layer(gpu_lib, layers, x, 1e-6)
    torch.cuda.synchronize()
    assert layers[0].device_status() == 0
    for li in range(4):
        assert torch.equal(lo[li].view(torch.int16), ref[li].view(torch.int16)), f"layer {li}"
    assert torch.equal(y.view(torch.int16), ref[-1].view(torch.int16))
    # and the stack output moved: every layer added something
    for li in range(1, 4):
        assert not torch.equal(lo[li], lo[li - 1])


def test_stack_arguments(gpu_lib):
    w = datagen.WORKLOADS["tiny"]
    layers, _ = _bf16_layers(gpu_lib, w, 2)
    stack = gpu_lib.MoeStack(layers)
    x = to_dev_bf16(datagen.tokens(w, 9))
    with pytest.raises(gpu_lib.MoeError):
        stack.forward(x)                     # T > 8
    assert layers[0].device_status() == 0
