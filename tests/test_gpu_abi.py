"""With a GPU present, the C ABI refuses memory that is not device memory of
the current device (LMOE_ERR_DEVICE, -8) before it launches anything: pinned
and pageable host memory, and (with two or more GPUs visible) a tensor on
another GPU passed by raw address past the binding's own device check."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()


def _layer_args(d, dev):
    from tests.gpu_util import weights_to_device
    w = weights_to_device(W.layer_weights(d, 0))
    x = torch.zeros((d.T, d.hidden), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((d.T, d.num_experts), dtype=torch.float32, device=dev)
    out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
    return w, x, lg, out, ws


@pytest.mark.parametrize("where", ["pinned", "pageable"])
def test_host_memory_is_refused(where):
    from tests.gpu_util import DEV
    d = W.TINY
    w, x, lg, out, ws = _layer_args(d, DEV)
    if where == "pinned":
        host = torch.zeros((d.T, d.hidden), dtype=torch.int16).pin_memory()
        addr, keep = host.data_ptr(), host
    else:
        keep = np.zeros(d.T * d.hidden + 64, dtype=np.int16)
        addr = keep.ctypes.data + (-keep.ctypes.data) % 256
    lib = lm.load_library()
    dd, ww = lm.make_dims(d), lm.make_weights(w, d)
    stream = torch.cuda.current_stream().cuda_stream
    # host memory as the hidden states, then as the output
    for args in ((addr, lg.data_ptr(), out.data_ptr()), (x.data_ptr(), lg.data_ptr(), addr)):
        st = lib.latent_moe_forward(ctypes.byref(dd), ctypes.byref(ww), *args, ws.data_ptr(),
                                    ws.numel(), None, stream)
        assert st == -8, st
    # host memory as a weight
    ww2 = lm.make_weights(dict(w, w_up=addr))
    st = lib.latent_moe_forward(ctypes.byref(dd), ctypes.byref(ww2), x.data_ptr(), lg.data_ptr(),
                                out.data_ptr(), ws.data_ptr(), ws.numel(), None, stream)
    assert st == -8
    assert lib.situ_and_mul(addr, out.data_ptr(), 4, 16, 4.0, 8.0, stream) == -8
    assert lib.lmoe_linear(x.data_ptr(), addr, None, out.data_ptr(), 8, 128, 64, stream) == -8
    torch.cuda.synchronize()
    assert keep is not None
    assert lm.lmoe_device_error() == 0


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two visible GPUs")
def test_other_device_memory_is_refused():
    # a tensor on cuda:1 handed by address to a call made with cuda:0 current:
    # refused before any tensor map is made (launches nothing)
    from tests.gpu_util import DEV
    d = W.TINY
    w, x, lg, out, ws = _layer_args(d, DEV)
    other = torch.zeros((d.T, d.hidden), dtype=torch.bfloat16, device="cuda:1")
    lib = lm.load_library()
    dd, ww = lm.make_dims(d), lm.make_weights(w, d)
    with torch.cuda.device(0):
        st = lib.latent_moe_forward(ctypes.byref(dd), ctypes.byref(ww), other.data_ptr(),
                                    lg.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                    None, torch.cuda.current_stream().cuda_stream)
    assert st == -8
