"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/moe.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes

import pytest

import top_moe_expert_router_gb300 as moe


@pytest.fixture(scope="module")
def lib():
    return moe.load()


def test_exports_every_declared_function(lib):
    names = moe.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    d = moe.MoeLayerDesc()
    d.d, d.E, d.top_k, d.I, d.max_tokens, d.fmt = 4096, 256, 8, 1536, 16, moe.MOE_W_BF16
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_workspace_size_and_shape_checks(lib):
    size = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(_desc()), ctypes.byref(size)) == moe.MOE_OK
    small = size.value
    assert lib.moe_workspace_size(ctypes.byref(_desc(max_tokens=4096)), ctypes.byref(size)) == moe.MOE_OK
    assert size.value > small
    bad = [dict(top_k=9), dict(E=300), dict(top_k=0), dict(d=4000), dict(I=100), dict(max_tokens=0),
           dict(fmt=7), dict(fmt=moe.MOE_W_NVFP4, I=1600)]
    for kw in bad:
        s = lib.moe_workspace_size(ctypes.byref(_desc(**kw)), ctypes.byref(size))
        assert s in (moe.MOE_ERR_INVALID_ARG, moe.MOE_ERR_UNSUPPORTED), kw
    assert lib.moe_workspace_size(None, ctypes.byref(size)) == moe.MOE_ERR_INVALID_ARG


def test_create_rejects_missing_or_misaligned_pointers(lib):
    h = ctypes.c_void_p()
    # no weights
    assert lib.moe_layer_create(ctypes.byref(_desc()), ctypes.c_void_p(4096), 1 << 40,
                                ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    # misaligned router pointer
    d = _desc(w_router=4100, w_gate=8192, w_up=8192, w_down=8192)
    assert lib.moe_layer_create(ctypes.byref(d), ctypes.c_void_p(4096), 1 << 40,
                                ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    # workspace not 256-byte aligned
    d = _desc(w_router=4096, w_gate=8192, w_up=8192, w_down=8192)
    assert lib.moe_layer_create(ctypes.byref(d), ctypes.c_void_p(4096 + 16), 1 << 40,
                                ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert lib.moe_layer_create(ctypes.byref(d), ctypes.c_void_p(4096), 100,
                                ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    # nvfp4 without its scale tensors
    d = _desc(fmt=moe.MOE_W_NVFP4, w_router=4096, q_gate=8192, q_up=8192, q_down=8192)
    assert lib.moe_layer_create(ctypes.byref(d), ctypes.c_void_p(4096), 1 << 40,
                                ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG


def test_calls_reject_null_layer_and_bad_sizes(lib):
    assert lib.moe_forward(None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), 1, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, ctypes.c_void_p(4096), 1, None, None, None, None, None, None,
                         None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_rmsnorm(ctypes.c_void_p(4096), ctypes.c_void_p(8192), 0, 64, 1e-6,
                           None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_nvfp4(ctypes.c_void_p(4096), 1, 4, 48, ctypes.c_void_p(8192), ctypes.c_void_p(8192),
                                  ctypes.c_void_p(8192), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_last_launch_count(None) == 0
    assert moe.status_string(moe.MOE_ERR_TIMEOUT) == "kernel wait timed out"


def test_stack_calls_reject_bad_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.moe_stack_create(None, 2, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    handles = (ctypes.c_void_p * 2)(None, None)
    assert lib.moe_stack_create(handles, 0, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_create(handles, 65, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_create(handles, 2, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG   # null layers
    assert lib.moe_stack_forward(None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), 1, 1e-6, None,
                                 None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_destroy(None) == moe.MOE_OK


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        ctypes.CDLL(str(tmp_path / "libmoe.so"))


def test_debug_and_host_stack_calls_reject_null_handles(lib):
    assert lib.moe_debug_route_records(None, 1, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_hold_grid_barrier(None, 1, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_forward_host(None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), 1, 1e-6,
                                      None) == moe.MOE_ERR_INVALID_ARG


def _fake_weights(d):
    """Aligned, non-null pointer values: every case below is rejected on the
    host before the pointers could be used."""
    for name in ("w_router", "w_gate", "w_up", "w_down"):
        setattr(d, name, 1 << 20)
    return d


@pytest.mark.parametrize("kw,T,want", [
    (dict(), 17, moe.MOE_ERR_INVALID_ARG),                        # more tokens than the decode path takes
    (dict(), 0, moe.MOE_ERR_INVALID_ARG),
    (dict(d=8192, I=4096), 16, moe.MOE_ERR_UNSUPPORTED),          # scratch above MOE_STATIC_SCRATCH_BYTES
    (dict(d=8192, I=1536), 8, moe.MOE_ERR_UNSUPPORTED),           # tokens do not fit in shared memory
    (dict(top_k=9), 4, moe.MOE_ERR_UNSUPPORTED),
])
def test_static_scratch_rejects_before_gpu_work(lib, kw, T, want):
    d = _fake_weights(_desc(**kw))
    s = lib.moe_forward_static_scratch(ctypes.byref(d), ctypes.c_void_p(1 << 21), ctypes.c_void_p(1 << 22), T, None)
    assert s == want
    assert lib.moe_forward_static_scratch(None, ctypes.c_void_p(1 << 21), ctypes.c_void_p(1 << 22), 1,
                                          None) == moe.MOE_ERR_INVALID_ARG
