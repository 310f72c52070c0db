"""Pins of the CPU oracle against facts other than the oracle itself.

Each test fixes one part of the oracle with a closed form, a brute-force
enumeration, an invariant, an independent library routine (torch / numpy in
float64) or a published number-format table, so that a plausible slip in
``oracle/oracle.c`` (a dropped bias, a wrong sign in SiLU, a transposed
W_down, a wrong tie rule, an off-by-one in the permutation) fails here.
"""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle

TINY = datagen.WORKLOADS["tiny"]


def _tiny_layer(seed=0, k=8, bias=None):
    wr = datagen.router_weights(TINY, seed=seed)
    g, u, d = datagen.expert_weights(TINY, seed=seed)
    return oracle.Layer(wr, g, u, d, router_bias=bias, k=k), (wr, g, u, d)


def _f32(a):
    return datagen.bf16_to_f32(a).astype(np.float64)


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def test_router_logits_match_torch_float64():
    wr = datagen.router_weights(TINY)
    x = datagen.tokens(TINY, 64)
    bias = datagen.normal_f32(3, 99, (TINY.E,), 0.5)
    got = oracle.router_logits(x, wr, bias)
    ref = (torch.from_numpy(_f32(x)) @ torch.from_numpy(_f32(wr)).T).to(torch.float32)
    ref = (ref + torch.from_numpy(bias)).numpy()
    # different summation order in double; after the single fp32 rounding the
    # two agree to within one fp32 ulp
    np.testing.assert_allclose(got, ref, rtol=2 ** -23, atol=1e-30)
    # the bias enters with its sign: dropping or negating it is caught
    nob = oracle.router_logits(x, wr, None)
    assert np.abs((got - nob) - bias[None, :]).max() < 1e-5


def test_topk_matches_bruteforce_sort_and_torch_topk():
    rng = np.random.default_rng(0)
    for trial in range(200):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, E + 1))
        T = 50
        # coarse integer grid makes exact ties common
        lg = rng.integers(-4, 5, size=(T, E)).astype(np.float32) * 0.5
        ids, w, gap = oracle.select_topk(lg, k)
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))
            assert list(ids[t]) == order[:k]
            p = np.exp(lg[t].astype(np.float64) - lg[t].max())
            p /= p.sum()
            np.testing.assert_allclose(w[t], p[order[:k]] / p[order[:k]].sum(), rtol=1e-12)
            if k < E:
                assert gap[t] == float(lg[t, order[k - 1]]) - float(lg[t, order[k]])
        # values (not order of equal keys) agree with torch.topk in float64
        tv, _ = torch.topk(torch.from_numpy(lg.astype(np.float64)), k, dim=1)
        np.testing.assert_array_equal(np.take_along_axis(lg, ids, 1).astype(np.float64), tv.numpy())


def test_topk_tie_rule_and_closed_form_weights():
    # all equal: the k lowest ids, equal weights
    lg = np.zeros((1, 16), np.float32)
    ids, w, _ = oracle.select_topk(lg, 8)
    assert list(ids[0]) == list(range(8))
    np.testing.assert_allclose(w[0], np.full(8, 1 / 8), rtol=1e-15)
    # a tie straddling the cut keeps the lower id
    lg = np.array([[0.0, 3.0, 1.0, 3.0, 1.0]], np.float32)
    ids, w, gap = oracle.select_topk(lg, 3)
    assert list(ids[0]) == [1, 3, 2]
    assert gap[0] == 0.0
    # closed form: logits (2, 0, 1, 0), k = 2 -> ids (0, 2), w = (e/(e+1), 1/(e+1))
    lg = np.array([[2.0, 0.0, 1.0, 0.0]], np.float32)
    ids, w, gap = oracle.select_topk(lg, 2)
    assert list(ids[0]) == [0, 2]
    np.testing.assert_allclose(w[0], [math.e / (math.e + 1), 1 / (math.e + 1)], rtol=1e-14)
    assert gap[0] == 1.0


def test_renormalised_weights_sum_to_one_and_descend():
    L, _ = _tiny_layer()
    x = datagen.tokens(TINY, 32)
    r = L.forward(x)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, atol=1e-12)
    assert (np.diff(r["w"], axis=1) <= 0).all()
    assert all(len(set(row)) == TINY.k for row in r["ids"])


def test_weights_for_forced_ids():
    lg = np.array([[2.0, 0.0, 1.0, 0.0]], np.float32)
    w = oracle.weights_for_ids(lg, np.array([[3, 1]], np.int32))
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=1e-15)


# --------------------------------------------------------------------------
# permutation
# --------------------------------------------------------------------------

def test_permute_hand_enumerated_example():
    # E = 4, k = 2, T = 3. Tokens route to (2,0), (0,3), (2,3).
    # expert 0 holds tokens 0,1; expert 1 none; expert 2 tokens 0,2; expert 3 tokens 1,2.
    ids = np.array([[2, 0], [0, 3], [2, 3]], np.int32)
    counts, offsets, perm, pos = oracle.permute(ids, 4)
    assert counts.tolist() == [2, 0, 2, 2]
    assert offsets.tolist() == [0, 2, 2, 4, 6]
    assert perm.tolist() == [0, 1, 0, 2, 1, 2]
    assert pos.tolist() == [[2, 0], [1, 4], [3, 5]]


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (37, 16, 4), (500, 256, 8), (64, 8, 8)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, pos = oracle.permute(ids, E)
    assert counts.sum() == T * k
    np.testing.assert_array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and (np.diff(offsets) == counts).all()
    np.testing.assert_array_equal(np.bincount(perm, minlength=T), np.full(T, k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()               # ascending, each token once
        assert set(seg.tolist()) == set(np.nonzero((ids == e).any(1))[0].tolist())
    for t in range(T):
        for j in range(k):
            r = pos[t, j]
            assert perm[r] == t and offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]


# --------------------------------------------------------------------------
# expert FFN and combine
# --------------------------------------------------------------------------

def _torch_ffn(x, g, u, d):
    """Independent float64 SwiGLU with torch: down(silu(gate x) * up x)."""
    xt = torch.from_numpy(_f32(x))
    gt = torch.from_numpy(_f32(g))
    ut = torch.from_numpy(_f32(u))
    dt = torch.from_numpy(_f32(d))
    return (dt @ (torch.nn.functional.silu(gt @ xt) * (ut @ xt))).numpy()


def test_swiglu_closed_form_two_dims():
    # d = 2, I = 1, E = 2, k = 1: x = (1, 0), Wg = ((1, 0)), Wu = ((2, 0)), Wd = ((1), (-1))
    # g = 1, u = 2, h = 2 / (1 + e^-1), y = (h, -h). Expert 1 is never chosen.
    bf = lambda v: datagen.f32_to_bf16(np.array(v, np.float32))
    wr = bf([[1.0, 0.0], [-1.0, 0.0]])
    g = bf([[[1.0, 0.0]], [[0.0, 0.0]]])
    u = bf([[[2.0, 0.0]], [[0.0, 0.0]]])
    dn = bf([[[1.0], [-1.0]], [[0.0], [0.0]]])
    L = oracle.Layer(wr, g, u, dn, k=1)
    r = L.forward(bf([[1.0, 0.0]]))
    h = 2.0 / (1.0 + math.exp(-1.0))
    assert r["ids"][0, 0] == 0 and r["w"][0, 0] == 1.0
    np.testing.assert_allclose(r["y"][0], [h, -h], rtol=1e-15)


def test_identical_experts_give_one_ffn_regardless_of_routing():
    wr = datagen.router_weights(TINY)
    g1, u1, d1 = (a[:1] for a in datagen.expert_weights(TINY, experts=[0]))
    g = np.repeat(g1, TINY.E, 0)
    u = np.repeat(u1, TINY.E, 0)
    d = np.repeat(d1, TINY.E, 0)
    L = oracle.Layer(wr, g, u, d, k=8)
    x = datagen.tokens(TINY, 8)
    r = L.forward(x)
    for t in range(8):
        ref = _torch_ffn(x[t], g1[0], u1[0], d1[0])
        np.testing.assert_allclose(r["y"][t], ref, rtol=1e-10, atol=1e-14)


def test_forward_matches_torch_float64_on_tiny_workload():
    L, (wr, g, u, d) = _tiny_layer()
    x = datagen.tokens(TINY, TINY.T)
    r = L.forward(x, want_Y=True)
    logits = (torch.from_numpy(_f32(x)) @ torch.from_numpy(_f32(wr)).T).to(torch.float32).double()
    p = torch.softmax(logits, dim=1)
    for t in range(TINY.T):
        order = sorted(range(TINY.E), key=lambda e: (-float(p[t, e]), e))[:TINY.k]
        assert list(r["ids"][t]) == order
        w = p[t, order] / p[t, order].sum()
        np.testing.assert_allclose(r["w"][t], w.numpy(), rtol=1e-12)
        y = np.zeros(TINY.d)
        for j, e in enumerate(order):
            Y = _torch_ffn(x[t], g[e], u[e], d[e])
            np.testing.assert_allclose(r["Y"][t, j], Y, rtol=1e-10, atol=1e-14)
            y += float(w[j]) * Y
        np.testing.assert_allclose(r["y"][t], y, rtol=1e-10, atol=1e-14)


def test_k_equals_E_is_the_dense_softmax_mixture():
    E, d, I = 6, 32, 16
    w = datagen.Workload("dense", T=4, d=d, E=E, k=E, I=I)
    wr = datagen.router_weights(w)
    g, u, dn = datagen.expert_weights(w)
    L = oracle.Layer(wr, g, u, dn, k=E)
    x = datagen.tokens(w, 4)
    r = L.forward(x)
    logits = (torch.from_numpy(_f32(x)) @ torch.from_numpy(_f32(wr)).T).to(torch.float32).double()
    p = torch.softmax(logits, 1).numpy()
    for t in range(4):
        ref = sum(p[t, e] * _torch_ffn(x[t], g[e], u[e], dn[e]) for e in range(E))
        np.testing.assert_allclose(r["y"][t], ref, rtol=1e-10, atol=1e-14)
        assert np.isinf(r["gap"][t])


def test_k_equals_1_is_the_argmax_expert():
    L, (wr, g, u, d) = _tiny_layer(k=1)
    x = datagen.tokens(TINY, 8)
    r = L.forward(x)
    lg = oracle.router_logits(x, wr)
    for t in range(8):
        e = int(np.argmax(lg[t]))
        assert r["ids"][t, 0] == e and r["w"][t, 0] == 1.0
        np.testing.assert_allclose(r["y"][t], _torch_ffn(x[t], g[e], u[e], d[e]), rtol=1e-10, atol=1e-14)


def test_linearity_in_w_down():
    L, (wr, g, u, d) = _tiny_layer()
    d2 = datagen.f32_to_bf16(datagen.bf16_to_f32(d) * 2.0)   # exact in bf16
    L2 = oracle.Layer(wr, g, u, d2, k=8)
    x = datagen.tokens(TINY, 8)
    np.testing.assert_allclose(L2.forward(x)["y"], 2.0 * L.forward(x)["y"], rtol=1e-14, atol=0)


def test_token_permutation_equivariance():
    L, _ = _tiny_layer()
    x = datagen.tokens(TINY, 16)
    sh = np.random.default_rng(1).permutation(16)
    a = L.forward(x)
    b = L.forward(x[sh])
    np.testing.assert_array_equal(b["ids"], a["ids"][sh])
    np.testing.assert_allclose(b["y"], a["y"][sh], rtol=1e-15, atol=0)


def test_expert_relabelling_invariance():
    L, (wr, g, u, d) = _tiny_layer()
    x = datagen.tokens(TINY, 16)
    a = L.forward(x)
    lab = np.random.default_rng(2).permutation(TINY.E)       # new expert i is old lab[i]
    L2 = oracle.Layer(wr[lab], g[lab], u[lab], d[lab], k=8)
    b = L2.forward(x)
    clear = a["gap"] > 1e-3
    assert clear.sum() >= 8                     # the check below covers most tokens
    for t in np.flatnonzero(clear):
        np.testing.assert_array_equal(lab[b["ids"][t]], a["ids"][t])
        np.testing.assert_allclose(b["y"][t], a["y"][t], rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------
# NVFP4 number formats and quantiser
# --------------------------------------------------------------------------

# OCP Microscaling Formats (MX) v1.0, FP4 E2M1 element values by code 0..7.
E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    for c in range(16):
        v = E2M1_SPEC[c & 7] * (-1.0 if c & 8 else 1.0)
        assert oracle.e2m1_decode(c) == v


def test_e4m3_decode_all_codes_against_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_against_torch_rne():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(447.9), 20000)),
        # exact midpoints between neighbouring codes, where the tie rule decides
        [(oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2 for c in range(0, 0x7E)],
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    np.testing.assert_array_equal(got, ref)
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0


def test_e2m1_encode_nearest_ties_even_saturating():
    # midpoints go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2.0,
    # 2.5->2.0, 3.5->4.0, 5->4.0; beyond 6 saturates to 6
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             7.0: 6.0, 100.0: 6.0, 0.3: 0.5, 2.6: 3.0, 4.9: 4.0, 5.1: 6.0}
    for v, want in cases.items():
        assert oracle.e2m1_decode(oracle.e2m1_encode(v)) == want, v
        assert oracle.e2m1_decode(oracle.e2m1_encode(-v)) == -want, v
    for c in range(8):   # every magnitude encodes to itself
        assert oracle.e2m1_encode(E2M1_SPEC[c]) == c
    assert oracle.e2m1_encode(-0.1) == 8   # sign kept on a value that rounds to zero


def test_quantizer_properties():
    W = datagen.normal_bf16(5, 77, (64, 256), 0.02)
    q, s, g = oracle.quantize_nvfp4(W)
    wf = datagen.bf16_to_f32(W)
    amax = np.abs(wf).max()
    assert g == np.float32(amax) / np.float32(2688.0)
    scales = np.array([oracle.e4m3_decode(c) for c in s.ravel()]).reshape(s.shape)
    assert (scales <= 448).all() and (s != 0x7F).all()
    deq = oracle.dequant_nvfp4(q, s, g)
    # error bound: at most half of the widest E2M1 step (6 - 4 = 2) times the scale
    blk_scale = np.repeat(scales, 16, axis=1) * g
    assert (np.abs(deq - wf) <= blk_scale * 1.0 + 1e-12).all()
    # the block maximum lands on code 6 or just below; quantisation keeps sign
    assert (np.sign(deq) * np.sign(wf) >= 0).all()
    # an all-equal tensor: every block maps to one scale and one code
    W2 = datagen.f32_to_bf16(np.full((4, 32), 0.375, np.float32))
    q2, s2, g2 = oracle.quantize_nvfp4(W2)
    assert len(set(q2.ravel().tolist())) == 1 and len(set(s2.ravel().tolist())) == 1
    np.testing.assert_allclose(oracle.dequant_nvfp4(q2, s2, g2), 0.375, rtol=2 ** -3)
    # all zero: scale 1, codes 0
    q3, s3, g3 = oracle.quantize_nvfp4(np.zeros((2, 32), np.uint16))
    assert g3 == 1.0 and not q3.any() and not s3.any()


def test_quantize_roundtrip_of_representable_tensor():
    # A tensor already on the NVFP4 grid with tensor scale exactly 2^-10: every
    # block holds a +6 code, one block has scale 448, so amax = 6 * 448 * 2^-10
    # and s_t = amax / 2688 = 2^-10 exactly. Quantising must return the same
    # codes and block scales bit for bit.
    rng = np.random.default_rng(4)
    rows, K = 8, 64
    codes = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    codes[:, ::16] = 7
    sc = rng.integers(0x08, 0x7E, size=(rows, K // 16)).astype(np.uint8)
    sc[0, 0] = 0x7E
    st = 2.0 ** -10
    vals = np.array([[oracle.e2m1_decode(codes[r, c]) * oracle.e4m3_decode(sc[r, c // 16]) * st
                      for c in range(K)] for r in range(rows)], np.float32)
    W = datagen.f32_to_bf16(vals)
    assert (datagen.bf16_to_f32(W) == vals).all()     # representable in bf16
    q, s, g = oracle.quantize_nvfp4(W)
    assert g == st
    np.testing.assert_array_equal(s, sc)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    np.testing.assert_array_equal(q, packed)
    np.testing.assert_array_equal(oracle.dequant_nvfp4(q, s, g), vals)


def test_nvfp4_layer_uses_dequantised_weights():
    w = datagen.Workload("q", T=4, d=64, E=4, k=2, I=32)
    wr = datagen.router_weights(w)
    g, u, d = datagen.expert_weights(w)
    packs = {}
    for name, arr in (("gate", g), ("up", u), ("down", d)):
        qs, ss, gs = zip(*(oracle.quantize_nvfp4(arr[e]) for e in range(w.E)))
        packs["q_" + name] = np.stack(qs)
        packs["s_" + name] = np.stack(ss)
        packs["g_" + name] = np.array(gs, np.float32)
    Lq = oracle.Layer(wr, router_bias=None, k=2, nvfp4=packs)
    deq = {n: np.stack([datagen.f32_to_bf16(oracle.dequant_nvfp4(packs["q_" + n][e], packs["s_" + n][e],
                                                                 packs["g_" + n][e])) for e in range(w.E)])
           for n in ("gate", "up", "down")}
    # dequantised values are representable in bf16 only approximately; compare with tolerance
    Lb = oracle.Layer(wr, deq["gate"], deq["up"], deq["down"], k=2)
    x = datagen.tokens(w, 4)
    a, b = Lq.forward(x), Lb.forward(x)
    np.testing.assert_array_equal(a["ids"], b["ids"])
    np.testing.assert_allclose(a["y"], b["y"], rtol=2e-2, atol=2e-3)


# --------------------------------------------------------------------------
# RMSNorm and residual
# --------------------------------------------------------------------------

def test_rmsnorm_against_torch_and_properties():
    x = datagen.normal_bf16(1, 50, (6, 4096), 3.0)
    u = oracle.rmsnorm(x, 1e-6)
    xf = torch.from_numpy(_f32(x))
    ref = (xf / torch.sqrt((xf * xf).mean(1, keepdim=True) + 1e-6)).float().numpy()
    uf = datagen.bf16_to_f32(u)
    np.testing.assert_allclose(uf, ref, rtol=2 ** -8, atol=0)
    assert np.allclose(np.sqrt((uf.astype(np.float64) ** 2).mean(1)), 1.0, atol=1e-2)
    z = oracle.rmsnorm(np.zeros((2, 64), np.uint16))
    assert not z.any()


def test_residual_add():
    x = datagen.f32_to_bf16(np.array([1.0, -2.0, 0.5], np.float32))
    out = oracle.residual_add(x, np.array([0.25, 0.5, -0.5]))
    assert datagen.bf16_to_f32(out).tolist() == [1.25, -1.5, 0.0]


# --------------------------------------------------------------------------
# per-expert output normalisation before the combine (optional variant)
# --------------------------------------------------------------------------

def test_expert_norm_identical_experts_closed_form():
    wr = datagen.router_weights(TINY)
    g1, u1, d1 = (a[:1] for a in datagen.expert_weights(TINY, experts=[0]))
    rep = lambda a: np.repeat(a, TINY.E, 0)
    L = oracle.Layer(wr, rep(g1), rep(u1), rep(d1), k=8, expert_norm=True)
    x = datagen.tokens(TINY, 4)
    r = L.forward(x)
    for t in range(4):
        f = _torch_ffn(x[t], g1[0], u1[0], d1[0])
        ref = f / np.sqrt(np.mean(f * f) + 1e-6)
        np.testing.assert_allclose(r["y"][t], ref, rtol=1e-10, atol=1e-14)


def test_expert_norm_is_scale_invariant_and_bounded():
    L, (wr, g, u, d) = _tiny_layer()
    Ln = oracle.Layer(wr, g, u, d, k=8, expert_norm=True)
    # W_down scaled by 2^8 and 2^9 (exact in bf16): mean(Y^2) then dwarfs eps
    big = [oracle.Layer(wr, g, u, datagen.f32_to_bf16(datagen.bf16_to_f32(d) * s), k=8, expert_norm=True)
           for s in (256.0, 512.0)]
    x = datagen.tokens(TINY, 8)
    a = Ln.forward(x, want_Y=True)
    b1, b2 = (L_.forward(x)["y"] for L_ in big)
    # RMS normalisation removes the scale of W_down
    np.testing.assert_allclose(b2, b1, rtol=1e-6, atol=1e-7)
    assert np.abs(b1).max() > 1e-3               # the invariance is not that of an all-zero output
    # each slot contributes unit RMS: the combined RMS is at most sum(w) = 1
    assert (np.sqrt((a["y"] ** 2).mean(1)) <= 1.0 + 1e-9).all()
    # the raw expert outputs are the same as without the normalisation
    np.testing.assert_allclose(a["Y"], L.forward(x, want_Y=True)["Y"], rtol=0, atol=0)
