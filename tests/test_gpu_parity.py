"""Parity of the CUDA layer (through the C ABI) with the CPU oracle on the
same seeded inputs: routing and permutation bit-exact off near-ties, layer
output and every expert slot within the stated tolerance."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from moe_testlib import (BF16_TOL, NEAR_TIE, HostLayer, bf16_host, check_route, normwise_rel_err, to_dev,
                         to_dev_bf16)

pytestmark = pytest.mark.gpu

W = datagen.WORKLOADS
D4096 = W["decode_t1"]


def _gpu_layer(moe, host: HostLayer, max_tokens: int, bias=True):
    w = host.w
    return moe.MoeLayer(to_dev_bf16(host.wr), w_gate=to_dev_bf16(host.gate), w_up=to_dev_bf16(host.up),
                        w_down=to_dev_bf16(host.down),
                        router_bias=to_dev(host.bias) if (bias and host.bias is not None) else None,
                        top_k=w.k, max_tokens=max_tokens)


def _parity(gl, L: oracle.Layer, x: np.ndarray, E: int, tol: float, tokens=None, check_Y=True, check_records=True):
    """Forward x through the GPU layer and the oracle; assert parity. Returns stats."""
    T = x.shape[0]
    xd = to_dev_bf16(x)
    r = gl.route(xd)
    y = gl.forward(xd)
    rec = gl.route_records(T)           # the records the forward's own kernels computed
    Y = gl.expert_outputs(T) if check_Y else None
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    ref = L.forward(x, tokens=tokens, want_Y=check_Y)
    n_near = check_route(r, ref["ids"], ref["w"], ref["gap"], E, tokens)
    if tokens is None and check_records:
        check_route(rec, ref["ids"], ref["w"], ref["gap"], E)
        # where no token is a near-tie both routing paths are unique: identical ids
        if (ref["gap"] > NEAR_TIE).all():
            assert torch.equal(rec["ids"], r["ids"])
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    gpu_ids = r["ids"].cpu().numpy()
    near = ref["gap"] <= NEAR_TIE
    if near.any():
        forced = L.forward(x, tokens=sel[near], forced_ids=gpu_ids, want_Y=check_Y)
        for key in ("y", "Y") if check_Y else ("y",):
            ref[key][near] = forced[key]
    y_gpu = datagen.bf16_to_f32(bf16_host(y))[sel]
    err = normwise_rel_err(y_gpu, ref["y"])
    assert err.max() <= tol, f"layer output error {err.max():.3g} > {tol}"
    if check_Y:
        pos = r["pos"].cpu().numpy()[sel]
        Yg = Y.cpu().numpy()[pos]              # [n, k, d]
        eY = normwise_rel_err(Yg, ref["Y"])
        assert eY.max() <= tol, f"expert output error {eY.max():.3g} > {tol}"
    return {"err": float(err.max()), "near": n_near}


# --------------------------------------------------------------------------
# fixtures
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(gpu_lib):
    host = HostLayer(W["tiny"])
    gl = _gpu_layer(gpu_lib, host, max_tokens=64)
    return host, gl


@pytest.fixture(scope="module")
def full_layer(gpu_lib):
    """The d=4096, E=256, I=1536 bf16 layer (9.66 GB of expert weights)."""
    host = HostLayer(W["prefill_t4096"])       # same weights as the decode workloads, plus the skew bias
    dev = {"wr": to_dev_bf16(host.wr), "gate": to_dev_bf16(host.gate), "up": to_dev_bf16(host.up),
           "down": to_dev_bf16(host.down), "bias": to_dev(host.bias)}
    return host, dev


def _full_gpu_layer(moe, dev, max_tokens, bias):
    return moe.MoeLayer(dev["wr"], w_gate=dev["gate"], w_up=dev["up"], w_down=dev["down"],
                        router_bias=dev["bias"] if bias else None, top_k=8, max_tokens=max_tokens)


# --------------------------------------------------------------------------
# tiny layer: every token, several batch sizes, ragged chunks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T", [8, 1, 2, 3, 5, 16, 17, 40])
def test_tiny_every_token(tiny, T):
    host, gl = tiny
    x = datagen.tokens(host.w, T, start_row=100 if T != 8 else 0)
    st = _parity(gl, host.oracle(), x, host.w.E, BF16_TOL, check_Y=T <= 16)
    assert st["err"] < 5e-3


@pytest.mark.parametrize("path", ["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("T", [1, 2, 5, 16])
def test_tiny_both_decode_kernels(gpu_lib, T, path):
    """The two single-launch small-batch kernels (experts on CUDA cores, or
    on the tensor cores with the tokens as the N = 16 operand), each against
    the oracle on every token and every expert slot."""
    host = HostLayer(W["tiny"])
    gl = _gpu_layer(gpu_lib, host, max_tokens=16)
    gl.set_decode_path(gpu_lib.MOE_DECODE_CUDA_CORES if path == "cuda_cores" else gpu_lib.MOE_DECODE_TENSOR_CORES)
    x = datagen.tokens(host.w, T, start_row=700 + T)
    st = _parity(gl, host.oracle(), x, host.w.E, BF16_TOL)
    assert gl.last_launch_count() == 1
    assert st["err"] < 5e-3
    gl.close()


def test_chunked_path_for_shapes_the_gemms_do_not_take(gpu_lib):
    """A bf16 layer whose hidden size is not a multiple of 256 (d = 320) runs
    batches above 16 tokens in chunks of 16 through the split streaming
    kernels (route, gate/up, down, combine per chunk)."""
    w = datagen.Workload("d320", T=40, d=320, E=64, k=8, I=192, router_scale=3.0)
    host = HostLayer(w)
    gl = _gpu_layer(gpu_lib, host, max_tokens=64)
    x = datagen.tokens(w, 40, start_row=11)
    # (each chunk overwrites the routing records and expert outputs of the one before)
    st = _parity(gl, host.oracle(), x, w.E, BF16_TOL, check_Y=False, check_records=False)
    assert gl.last_launch_count() == 3 * 4          # three chunks of four launches
    assert st["err"] < 5e-3


@pytest.mark.parametrize("path", ["cuda_cores", "tensor_cores"])
def test_alternating_inputs_read_nothing_stale(gpu_lib, path):
    """Successive forwards on one layer with different tokens and token
    counts (one token among them: its own routing path): every result matches
    the oracle. The workspace then always holds the previous call's logits,
    token rows, h and expert outputs, so a hand-off that read them before the
    current call rewrote them (a missing wait, a logit word taken with a stale
    tag) shows up as a wrong token."""
    host = HostLayer(W["tiny"])
    gl = _gpu_layer(gpu_lib, host, max_tokens=16)
    gl.set_decode_path(gpu_lib.MOE_DECODE_CUDA_CORES if path == "cuda_cores" else gpu_lib.MOE_DECODE_TENSOR_CORES)
    L = host.oracle()
    for i, T in enumerate([16, 16, 5, 1, 16, 3, 1, 1, 16, 9, 2, 16]):
        x = datagen.tokens(host.w, T, start_row=3000 + 41 * i)
        y = gl.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y)), L.forward(x)["y"])
        assert err.max() < 1e-2, f"call {i} (T={T}): {err.max():.3g}"
    assert gl.device_status() == 0
    gl.close()


@pytest.mark.parametrize("T,path", [(1, 1), (5, 1), (16, 1), (5, 2), (16, 2), (40, 0)])
def test_interleaved_gate_up_layout(gpu_lib, T, path):
    """gate/up weights as one [E, I, 2, d] tensor interleaved by row (gate row
    i, then up row i): the small-batch kernels (path 1: CUDA cores, 2: tensor
    cores) and the prefill GEMMs (T = 40) against the oracle, which keeps the
    two matrices separate."""
    host = HostLayer(W["tiny"])
    gu = np.ascontiguousarray(np.stack([host.gate, host.up], axis=2))      # [E, I, 2, d]
    gl = gpu_lib.MoeLayer(to_dev_bf16(host.wr), w_gate_up=to_dev_bf16(gu), w_down=to_dev_bf16(host.down),
                          top_k=host.w.k, max_tokens=64)
    gl.set_decode_path(path)
    x = datagen.tokens(host.w, T, start_row=4000 + T)
    st = _parity(gl, host.oracle(), x, host.w.E, BF16_TOL)
    # beside the 2e-2 bar: well inside it on every path (the prefill GEMMs round
    # h and the expert outputs to bf16, ~5e-3 here)
    assert st["err"] < 1e-2
    gl.close()


def test_tiny_route_large_batch(tiny):
    """The multi-kernel routing path (T > 32): router GEMM, top-k, permutation."""
    host, gl = tiny
    x = datagen.tokens(host.w, 64, start_row=500)
    r = gl.route(to_dev_bf16(x))
    torch.cuda.synchronize()
    ref = host.oracle().forward(x)
    check_route(r, ref["ids"], ref["w"], ref["gap"], host.w.E)


def test_all_tokens_identical_fill_one_expert_set(tiny):
    """16 identical tokens: 8 experts receive all 16 tokens, the rest none."""
    host, gl = tiny
    x = np.repeat(datagen.tokens(host.w, 1, start_row=7), 16, axis=0)
    st = _parity(gl, host.oracle(), x, host.w.E, BF16_TOL)
    r = gl.route(to_dev_bf16(x))
    counts = r["counts"].cpu().numpy()
    assert sorted(counts[counts > 0].tolist()) == [16] * 8
    assert st["err"] < 5e-3


def test_deterministic_and_launch_count(tiny):
    host, gl = tiny
    xd = to_dev_bf16(datagen.tokens(host.w, 5, start_row=900))
    a = gl.forward(xd).clone()
    assert gl.last_launch_count() == 1        # the whole small-batch layer is one persistent kernel
    b = gl.forward(xd)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_host_matches_forward(tiny):
    host, gl = tiny
    x = datagen.tokens(host.w, 4, start_row=321)
    xd = to_dev_bf16(x)
    y = bf16_host(gl.forward(xd))
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    gl.forward_host(xh, oh)
    np.testing.assert_array_equal(oh.view(torch.int16).numpy().view(np.uint16), y)


def test_residual_forward(tiny):
    host, gl = tiny
    x = datagen.tokens(host.w, 6, start_row=50)
    res = datagen.tokens(host.w, 6, start_row=60)
    xd, rd = to_dev_bf16(x), to_dev_bf16(res)
    out = gl.forward(xd, res=rd)
    torch.cuda.synchronize()
    ref = host.oracle().forward(x)
    want = datagen.bf16_to_f32(oracle.residual_add(res, ref["y"]))
    got = datagen.bf16_to_f32(bf16_host(out))
    # within one bf16 spacing of the sum (the MoE part, within its tolerance, may
    # move the sum across a rounding boundary; a spacing is at most 2^-7 of the
    # value) plus the layer tolerance on the MoE part
    bound = np.abs(want) * 2 ** -7 + BF16_TOL * np.abs(ref["y"]).max(1, keepdims=True)
    assert (np.abs(got - want) <= bound).all()


def test_argument_errors(tiny, gpu_lib):
    host, gl = tiny
    xd = to_dev_bf16(datagen.tokens(host.w, 65))
    with pytest.raises(gpu_lib.MoeError) as ei:
        gl.forward(xd)                       # T > max_tokens
    assert ei.value.status == gpu_lib.MOE_ERR_INVALID_ARG
    assert gl.device_status() == 0


def test_rmsnorm_matches_oracle(gpu_lib):
    x = datagen.normal_bf16(2, 40, (5, 4096), 2.0)
    u = gpu_lib.rmsnorm(to_dev_bf16(x), 1e-6)
    ref = datagen.bf16_to_f32(oracle.rmsnorm(x, 1e-6))
    got = datagen.bf16_to_f32(bf16_host(u))
    # at most one bf16 ulp apart (fp32 vs double before the final rounding)
    np.testing.assert_allclose(got, ref, rtol=2 ** -7, atol=0)
    assert (got != ref).mean() < 0.01


# --------------------------------------------------------------------------
# full-size layer d=4096, E=256, I=1536
# --------------------------------------------------------------------------

@pytest.mark.parametrize("path", ["auto", "cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("T,start", [(4, 100), (16, 200)])
def test_decode_full_size_every_token(gpu_lib, full_layer, T, start, path):
    host, dev = full_layer
    gl = _full_gpu_layer(gpu_lib, dev, max_tokens=16, bias=False)
    gl.set_decode_path({"auto": gpu_lib.MOE_DECODE_AUTO, "cuda_cores": gpu_lib.MOE_DECODE_CUDA_CORES,
                        "tensor_cores": gpu_lib.MOE_DECODE_TENSOR_CORES}[path])
    x = datagen.tokens(D4096, T, start_row=start)
    st = _parity(gl, host.oracle(bias=False), x, 256, BF16_TOL)
    assert st["err"] < 1e-2


def test_decode_t1_every_pool_token(gpu_lib, full_layer):
    """Single-token decode over the 64 seeded tokens the T=1 measurement
    rotates through (rows 0..63 of the token stream), one forward each:
    routing records of each launch bit-exact off near-ties, the layer output
    and all 8 expert slots within the bf16 tolerance."""
    host, dev = full_layer
    gl = _full_gpu_layer(gpu_lib, dev, max_tokens=16, bias=False)
    n = 64
    x = datagen.tokens(D4096, n, start_row=0)
    ys, Ys, recs = [], [], []
    for t in range(n):
        y = gl.forward(to_dev_bf16(x[t:t + 1]))
        recs.append({key: v.cpu() for key, v in gl.route_records(1).items()})
        Ys.append(gl.expert_outputs(1).cpu().numpy())
        ys.append(bf16_host(y)[0])
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    L = host.oracle(bias=False)
    ref = L.forward(x, want_Y=True)
    near = ref["gap"] <= NEAR_TIE
    gpu_ids = np.stack([r["ids"].numpy()[0] for r in recs])
    if near.any():
        forced = L.forward(x, tokens=np.flatnonzero(near), forced_ids=gpu_ids, want_Y=True)
        ref["y"][near], ref["Y"][near] = forced["y"], forced["Y"]
    for t in range(n):
        check_route(recs[t], ref["ids"][t:t + 1], ref["w"][t:t + 1], ref["gap"][t:t + 1], 256)
    err = normwise_rel_err(datagen.bf16_to_f32(np.stack(ys)), ref["y"])
    assert err.max() <= BF16_TOL and err.max() < 1e-2
    Yg = np.stack([Ys[t][recs[t]["pos"].numpy()[0]] for t in range(n)])     # [n, k, d]
    assert normwise_rel_err(Yg, ref["Y"]).max() <= BF16_TOL


def test_decode_full_size_skewed_routing(gpu_lib, full_layer):
    """16 tokens under the skewed router bias: a few experts take many of the
    tokens, so the stage shares are cut by cost, not by count."""
    host, dev = full_layer
    gl = _full_gpu_layer(gpu_lib, dev, max_tokens=16, bias=True)
    x = datagen.tokens(D4096, 16, start_row=300)
    r = gl.route(to_dev_bf16(x))
    counts = r["counts"].cpu().numpy()
    assert counts.max() >= 3                       # multi-token experts present
    st = _parity(gl, host.oracle(bias=True), x, 256, BF16_TOL)
    assert st["err"] < 1e-2


def test_prefill_full_size_routing_all_and_output_sample(gpu_lib, full_layer):
    host, dev = full_layer
    T = 4096
    gl = _full_gpu_layer(gpu_lib, dev, max_tokens=T, bias=True)
    x = datagen.tokens(D4096, T)
    xd = to_dev_bf16(x)
    r = gl.route(xd)
    y = gl.forward(xd)
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    L = host.oracle(bias=True)
    lg = oracle.router_logits(x, host.wr, host.bias)
    ids, w, gap = oracle.select_topk(lg, 8)
    check_route(r, ids, w, gap, 256)
    counts = r["counts"].cpu().numpy()
    assert 3.0 < counts.max() / counts.mean() < 5.0       # the skewed load the workload asks for
    sample = np.sort(np.random.default_rng(1).choice(T, 256, replace=False))
    gpu_ids = r["ids"].cpu().numpy()
    ref = L.forward(x, tokens=sample, forced_ids=gpu_ids, want_Y=True)
    ref_ids_own = ids[sample]
    assert (ref["ids"] == gpu_ids[sample]).all()
    near = gap[sample] <= 1e-3
    assert ((ref_ids_own == gpu_ids[sample]).all(1) | near).all()
    err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y))[sample], ref["y"])
    assert err.max() <= BF16_TOL
    # every slot of the sample: the grouped GEMMs' expert outputs (kept in bf16)
    Y = gl.expert_outputs(T)
    pos = r["pos"].cpu().numpy()[sample]
    Yg = Y[torch.from_numpy(pos.reshape(-1)).to(Y.device)].cpu().numpy().reshape(len(sample), 8, -1)
    del Y
    assert normwise_rel_err(Yg, ref["Y"]).max() <= BF16_TOL
