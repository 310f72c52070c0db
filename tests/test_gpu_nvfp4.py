"""NVFP4 experts on the GPU: the quantiser is bit-exact with the oracle's, and
the streaming expert stage with dequantisation fused into the weight stream
matches the oracle run on its own quantisation of the same weights; the
8-layer stacked decode (RMSNorm, MoE, residual) matches layer by layer."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from moe_testlib import NVFP4_TOL, bf16_host, check_route, normwise_rel_err, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _quant_host(arr, experts):
    """Oracle quantisation of the listed experts of one [E, rows, K] stack."""
    E, rows, K = arr.shape
    q = np.zeros((E, rows, K // 2), np.uint8)
    s = np.zeros((E, rows, K // 16), np.uint8)
    g = np.ones(E, np.float32)
    for e in experts:
        q[e], s[e], g[e] = oracle.quantize_nvfp4(arr[e])
    return q, s, g


def test_quantizer_bit_exact(gpu_lib):
    W = datagen.normal_bf16(11, 70, (3, 64, 512), 0.02)
    W[1, 5, :16] = 0                                  # an all-zero block
    W[2] = datagen.f32_to_bf16(np.full((64, 512), -0.001, np.float32))
    q, s, g = gpu_lib.quantize_nvfp4(to_dev_bf16(W))
    torch.cuda.synchronize()
    for n in range(3):
        qr, sr, gr = oracle.quantize_nvfp4(W[n])
        np.testing.assert_array_equal(q[n].cpu().numpy(), qr)
        np.testing.assert_array_equal(s[n].cpu().numpy(), sr)
        assert g[n].item() == gr
    qz, sz, gz = gpu_lib.quantize_nvfp4(torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda"))
    assert gz.item() == 1.0 and not qz.any() and not sz.any()


def _nvfp4_gpu_layer(moe, wr, bias, packs_dev, k, max_tokens):
    return moe.MoeLayer(to_dev_bf16(wr), nvfp4=packs_dev, router_bias=None if bias is None else to_dev(bias),
                        top_k=k, max_tokens=max_tokens)


def _quantize_on_gpu(moe, g, u, d):
    packs = {}
    for name, arr in (("gate", g), ("up", u), ("down", d)):
        dev = to_dev_bf16(arr)
        q, s, gs = moe.quantize_nvfp4(dev)
        del dev
        packs["q_" + name], packs["s_" + name], packs["g_" + name] = q, s, gs
    return packs


@pytest.mark.parametrize("T,path", [(1, 1), (4, 1), (16, 1), (1, 2), (4, 2), (16, 2), (17, 0), (40, 0), (300, 0)])
def test_small_nvfp4_layer(gpu_lib, T, path):
    """T <= 16: the single-launch decode kernels (path 1: CUDA cores, 2:
    tensor cores with the codes widened into tensor memory); T > 16: the
    NVFP4 grouped GEMMs (several 128-row tiles per expert and ragged tails at
    T = 300)."""
    w = datagen.Workload("fp4small", T=T, d=512, E=64, k=8, I=256, fmt="nvfp4", router_scale=4.0)
    wr = datagen.router_weights(w)
    g, u, d = datagen.expert_weights(w)
    packs = _quantize_on_gpu(gpu_lib, g, u, d)
    host = {}
    for name, arr in (("gate", g), ("up", u), ("down", d)):
        q, s, gs = _quant_host(arr, range(w.E))
        np.testing.assert_array_equal(packs["q_" + name].cpu().numpy(), q)
        np.testing.assert_array_equal(packs["s_" + name].cpu().numpy(), s)
        np.testing.assert_array_equal(packs["g_" + name].cpu().numpy(), gs)
        host["q_" + name], host["s_" + name], host["g_" + name] = q, s, gs
    gl = _nvfp4_gpu_layer(gpu_lib, wr, None, packs, w.k, 512)
    gl.set_decode_path(path)
    L = oracle.Layer(wr, k=w.k, nvfp4=host)
    x = datagen.tokens(w, T, start_row=3)
    xd = to_dev_bf16(x)
    r = gl.route(xd)
    y = gl.forward(xd)
    rec = gl.route_records(T)          # the records the forward's own kernels computed
    Y = gl.expert_outputs(T)
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    assert gl.last_launch_count() == (1 if T <= 16 else 7)
    ref = L.forward(x, forced_ids=r["ids"].cpu().numpy(), want_Y=True)
    own = L.forward(x)
    check_route(r, own["ids"], own["w"], own["gap"], w.E)
    check_route(rec, own["ids"], own["w"], own["gap"], w.E)
    err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y)), ref["y"])
    assert err.max() <= NVFP4_TOL
    # the kernels add only fp32 (decode) or bf16 h / bf16 expert-output (GEMM)
    # rounding to the shared quantisation
    assert err.max() < 1e-2
    pos = r["pos"].cpu().numpy()
    eY = normwise_rel_err(Y.cpu().numpy()[pos], ref["Y"])
    assert eY.max() < 1e-2


def test_nvfp4_prefill_full_size(gpu_lib):
    """T=4096 prefill with NVFP4 experts at full size (d=4096, E=256, I=1536,
    the skewed router bias of the bf16 prefill workload): routing bit-exact on
    all 4096 tokens off near-ties (the route call and the forward's own
    records), the layer output and all 8 slots of a seeded 256-token sample
    within the NVFP4 tolerance of the oracle run on its own quantisation."""
    w = datagen.WORKLOADS["nvfp4_prefill_t4096"]
    T = w.T
    wr = datagen.router_weights(w)
    bias = datagen.router_bias(w)
    g, u, d = datagen.expert_weights(w)
    packs = _quantize_on_gpu(gpu_lib, g, u, d)
    gl = _nvfp4_gpu_layer(gpu_lib, wr, bias, packs, w.k, T)
    x = datagen.tokens(w, T)
    xd = to_dev_bf16(x)
    r = gl.route(xd)
    y = gl.forward(xd)
    rec = gl.route_records(T)
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    lg = oracle.router_logits(x, wr, bias)
    ids, wts, gap = oracle.select_topk(lg, w.k)
    check_route(r, ids, wts, gap, w.E)
    check_route(rec, ids, wts, gap, w.E)
    sample = np.sort(np.random.default_rng(1).choice(T, 256, replace=False))
    gpu_ids = r["ids"].cpu().numpy()
    need = np.unique(gpu_ids[sample])
    host = {}
    for name, arr in (("gate", g), ("up", u), ("down", d)):
        q, s, gs = _quant_host(arr, need)
        np.testing.assert_array_equal(packs["q_" + name][need].cpu().numpy(), q[need])
        np.testing.assert_array_equal(packs["s_" + name][need].cpu().numpy(), s[need])
        np.testing.assert_array_equal(packs["g_" + name][need].cpu().numpy(), gs[need])
        host["q_" + name], host["s_" + name], host["g_" + name] = q, s, gs
    del g, u, d
    L = oracle.Layer(wr, k=w.k, nvfp4=host, router_bias=bias)
    ref = L.forward(x, tokens=sample, forced_ids=gpu_ids, want_Y=True)
    err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y))[sample], ref["y"])
    assert err.max() <= NVFP4_TOL and err.max() < 1e-2
    Y = gl.expert_outputs(T)
    pos = r["pos"].cpu().numpy()[sample]
    Yg = Y[torch.from_numpy(pos.reshape(-1)).to(Y.device)].cpu().numpy().reshape(len(sample), w.k, -1)
    del Y
    assert normwise_rel_err(Yg, ref["Y"]).max() <= NVFP4_TOL


def test_stacked_nvfp4_decode_full_size(gpu_lib):
    """8 layers x (RMSNorm, NVFP4 MoE, residual) at T=4, d=4096, E=256, I=1536.
    Each layer is checked with the GPU's own layer input (teacher forcing)."""
    w = datagen.WORKLOADS["nvfp4_stack_t4"]
    x = datagen.tokens(w, w.T)
    xg = to_dev_bf16(x)
    worst = 0.0
    for layer in range(w.layers):
        wr = datagen.router_weights(w, layer)
        g, u, d = datagen.expert_weights(w, layer)
        packs = _quantize_on_gpu(gpu_lib, g, u, d)
        gl = _nvfp4_gpu_layer(gpu_lib, wr, None, packs, w.k, 16)
        ug = gpu_lib.rmsnorm(xg, 1e-6)
        r = gl.route(ug)
        y = gl.forward(ug)
        xn = gl.forward(ug, res=xg)
        torch.cuda.synchronize()
        assert gl.device_status() == 0
        x_host, u_host = bf16_host(xg), bf16_host(ug)
        # RMSNorm within one bf16 ulp of the oracle
        np.testing.assert_allclose(datagen.bf16_to_f32(u_host), datagen.bf16_to_f32(oracle.rmsnorm(x_host)),
                                   rtol=2 ** -7, atol=0)
        lg = oracle.router_logits(u_host, wr)
        ids_o, w_o, gap_o = oracle.select_topk(lg, w.k)
        gids = r["ids"].cpu().numpy()
        need = np.union1d(np.unique(ids_o), np.unique(gids))
        host = {}
        for name, arr in (("gate", g), ("up", u), ("down", d)):
            q, s, gs = _quant_host(arr, need)
            # quantiser parity on every expert the step touches
            np.testing.assert_array_equal(packs["q_" + name][need].cpu().numpy(), q[need])
            np.testing.assert_array_equal(packs["s_" + name][need].cpu().numpy(), s[need])
            np.testing.assert_array_equal(packs["g_" + name][need].cpu().numpy(), gs[need])
            host["q_" + name], host["s_" + name], host["g_" + name] = q, s, gs
        check_route(r, ids_o, w_o, gap_o, w.E)
        L = oracle.Layer(wr, k=w.k, nvfp4=host)
        ref = L.forward(u_host, forced_ids=gids)
        err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y)), ref["y"])
        assert err.max() <= NVFP4_TOL, f"layer {layer}: {err.max():.3g}"
        worst = max(worst, float(err.max()))
        want = datagen.bf16_to_f32(oracle.residual_add(x_host, ref["y"]))
        got = datagen.bf16_to_f32(bf16_host(xn))
        bound = np.abs(want) * 2 ** -7 + NVFP4_TOL * np.abs(ref["y"]).max(1, keepdims=True)
        assert (np.abs(got - want) <= bound).all()
        xg = xn
        del gl, packs
        torch.cuda.empty_cache()
    assert worst < 1e-2
