"""Device-side failure detection, exercised without a fault: a test hook
makes the decode kernel's grid barriers wait for an arrival that never comes,
so its bounded wait (1.5 s) runs out. The launch must unwind on its own, the
host must read MOE_ERR_TIMEOUT from the layer's error word, and the next
forward must be correct again (the counters the aborted launch used are
reset on its way out). No trap, no bad address, no unbounded wait."""
import pytest
import torch

import datagen
from moe_testlib import HostLayer, to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(moe, host):
    return moe.MoeLayer(to_dev_bf16(host.wr), w_gate=to_dev_bf16(host.gate), w_up=to_dev_bf16(host.up),
                        w_down=to_dev_bf16(host.down), top_k=host.w.k, max_tokens=16)


@pytest.mark.parametrize("T", [1, 5])
def test_barrier_timeout_is_reported_and_the_next_call_recovers(gpu_lib, T):
    host = HostLayer(datagen.WORKLOADS["tiny"])
    gl = _layer(gpu_lib, host)
    x = to_dev_bf16(datagen.tokens(host.w, T, start_row=77))
    good = gl.forward(x).clone()
    assert gl.device_status() == gpu_lib.MOE_OK
    gl.hold_grid_barrier(True)
    gl.forward(x)                                   # gives up after the wait limit
    assert gl.device_status() == gpu_lib.MOE_ERR_TIMEOUT
    assert gl.device_status() == gpu_lib.MOE_OK     # reading the status cleared it
    gl.hold_grid_barrier(False)
    for _ in range(3):                              # counters, barriers and combine blocks all reset
        again = gl.forward(x)
        torch.cuda.synchronize()
        assert gl.device_status() == gpu_lib.MOE_OK
        assert torch.equal(again.view(torch.int16), good.view(torch.int16))
    gl.close()


def test_stack_barrier_timeout_recovers(gpu_lib):
    w = datagen.WORKLOADS["tiny"]
    layers = []
    for li in range(2):
        h = HostLayer(w, layer=li)
        layers.append(_layer(gpu_lib, h))
    stack = gpu_lib.MoeStack(layers)
    x = to_dev_bf16(datagen.tokens(w, 3, start_row=5))
    good = stack.forward(x).clone()
    assert layers[0].device_status() == gpu_lib.MOE_OK
    layers[0].hold_grid_barrier(True)
    stack.forward(x)
    assert layers[0].device_status() == gpu_lib.MOE_ERR_TIMEOUT
    layers[0].hold_grid_barrier(False)
    again = stack.forward(x)
    torch.cuda.synchronize()
    assert layers[0].device_status() == gpu_lib.MOE_OK
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
