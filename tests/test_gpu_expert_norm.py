"""The per-expert output normalisation variant (each expert output RMS-
normalised before the weighted sum) against the oracle with the same flag, on
the decode path and on the large-batch path."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from moe_testlib import BF16_TOL, NEAR_TIE, bf16_host, normwise_rel_err, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,T", [("tiny", 8), ("tiny", 40), ("d4096", 4), ("d4096", 16)])
def test_expert_norm_matches_oracle(gpu_lib, shape, T):
    if shape == "tiny":
        w = datagen.WORKLOADS["tiny"]
    else:
        w = datagen.Workload("d4096_e16", T=T, d=4096, E=16, k=8, I=1536, router_scale=datagen.ROUTER_SCALE_D4096)
    wr = datagen.router_weights(w)
    g, u, d = datagen.expert_weights(w)
    gl = gpu_lib.MoeLayer(to_dev_bf16(wr), w_gate=to_dev_bf16(g), w_up=to_dev_bf16(u), w_down=to_dev_bf16(d),
                          top_k=w.k, max_tokens=64, expert_out_norm=True)
    x = datagen.tokens(w, T, start_row=77)
    xd = to_dev_bf16(x)
    r = gl.route(xd)
    y = gl.forward(xd)
    torch.cuda.synchronize()
    assert gl.device_status() == 0
    L = oracle.Layer(wr, g, u, d, k=w.k, expert_norm=True)
    ids = r["ids"].cpu().numpy()
    ref = L.forward(x, forced_ids=ids)
    own = L.forward(x)
    clear = own["gap"] > NEAR_TIE
    np.testing.assert_array_equal(ids[clear], own["ids"][clear])
    err = normwise_rel_err(datagen.bf16_to_f32(bf16_host(y)), ref["y"])
    assert err.max() <= BF16_TOL
    # the normalisation really is applied: the plain sum differs
    plain = oracle.Layer(wr, g, u, d, k=w.k).forward(x, forced_ids=ids)["y"]
    assert normwise_rel_err(plain, ref["y"]).max() > 10 * BF16_TOL
    gl.close()
