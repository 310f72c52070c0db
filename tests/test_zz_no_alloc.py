"""The forward for callers that cannot allocate device memory.

moe_forward_static_scratch() serves callers that cannot call cudaMalloc (a
plugin that only receives input and output buffers from its host
application, or a loop that may not allocate after start-up): it keeps its
scratch in a static device array instead of a caller workspace. This test
calls it through the C ABI twice in a row and checks each result against
moe_forward on the same layer and tokens, at the layer-output tolerance of
the other parity tests. The file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import datagen
from moe_testlib import BF16_TOL, bf16_host, normwise_rel_err, to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(moe, w):
    wr = datagen.router_weights(w)
    g, u, d = datagen.expert_weights(w)
    return moe.MoeLayer(to_dev_bf16(wr), w_gate=to_dev_bf16(g), w_up=to_dev_bf16(u), w_down=to_dev_bf16(d),
                        top_k=w.k, max_tokens=16)


@pytest.mark.parametrize("shape", ["tiny", "d4096"])
def test_static_scratch_forward_matches_forward(gpu_lib, shape):
    if shape == "tiny":
        w = datagen.WORKLOADS["tiny"]
    else:   # full hidden and expert widths, fewer experts to keep the layer small
        w = datagen.Workload("d4096_e16", T=16, d=4096, E=16, k=8, I=1536, router_scale=datagen.ROUTER_SCALE_D4096)
    layer = _layer(gpu_lib, w)
    # the no-alloc call runs the CUDA-core small-batch kernel: compare with the same kernel
    layer.set_decode_path(gpu_lib.MOE_DECODE_CUDA_CORES)
    lib = gpu_lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the call ignores max_tokens: the second call passes a copy with 0 there
    desc0 = gpu_lib.MoeLayerDesc.from_buffer_copy(layer._desc)
    desc0.max_tokens = 0
    for call, T in enumerate((5, 16)):          # two calls in a row, different token batches
        x = to_dev_bf16(datagen.tokens(w, T, start_row=1000 + 100 * call))
        ref = layer.forward(x)
        out = torch.empty_like(ref)
        desc = layer._desc if call == 0 else desc0
        s = lib.moe_forward_static_scratch(ctypes.byref(desc), ctypes.c_void_p(x.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), T, stream)
        assert s == gpu_lib.MOE_OK, gpu_lib.status_string(s)
        torch.cuda.synchronize()
        a = datagen.bf16_to_f32(bf16_host(out))
        b = datagen.bf16_to_f32(bf16_host(ref))
        assert normwise_rel_err(a, b).max() <= BF16_TOL
        np.testing.assert_array_equal(a, b)        # same kernels, same order: identical bits
    layer.close()


def test_static_scratch_rejects_oversize(gpu_lib):
    w = datagen.WORKLOADS["tiny"]
    layer = _layer(gpu_lib, w)
    lib = gpu_lib.load()
    x = to_dev_bf16(datagen.tokens(w, 17))
    out = torch.empty_like(x)
    s = lib.moe_forward_static_scratch(ctypes.byref(layer._desc), ctypes.c_void_p(x.data_ptr()),
                                       ctypes.c_void_p(out.data_ptr()), 17, None)
    assert s == gpu_lib.MOE_ERR_INVALID_ARG
    layer.close()
