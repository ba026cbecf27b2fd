"""The layer forward called from two host threads at once, each on its own
stream and workspace, one of them capturing its call into a CUDA graph and
replaying it while the other runs eagerly: both outputs are bit-identical to
a call made alone, which matches the oracle.  Each caller stream gets its own
second stream for the shared expert, so neither call is ordered behind the
other's work nor drawn into the other's capture."""
import dataclasses
import threading

import numpy as np
import pytest
import torch

import workloads as W
from oracle import lmoe_oracle as O

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()


@pytest.mark.parametrize("T", [8, 300])
def test_two_threads_one_capturing(T):
    from tests.gpu_util import (DEV, weights_to_device, dev_bf16, dev_f32, host_bits,
                                assert_layer_close, addend_scale)
    d = dataclasses.replace(W.TINY, T=T)
    wts = W.layer_weights(d, 4)
    wdev = weights_to_device(wts)
    xb, lgh = W.hidden_states(d, 4), W.router_logits(d.T, d.num_experts, 4)
    x, lg = dev_bf16(xb), dev_f32(lgh)
    nbytes = lm.latent_moe_workspace_bytes(d)

    def buffers():
        return (torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV),
                torch.empty(nbytes, dtype=torch.uint8, device=DEV))

    # a call made alone, on a stream of its own
    ref, ws0 = buffers()
    s0 = torch.cuda.Stream()
    with torch.cuda.stream(s0):
        lm.latent_moe_forward(d, wdev, x, lg, ref, ws0, stream=s0)
    torch.cuda.synchronize()
    ref_bits = host_bits(ref)

    outs, errors = {}, []
    start = threading.Barrier(2)
    reps = 20

    def eager():
        try:
            out, ws = buffers()
            s = torch.cuda.Stream()
            start.wait()
            for _ in range(reps):
                with torch.cuda.stream(s):
                    lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)
            s.synchronize()
            outs["eager"] = host_bits(out)
        except Exception as e:   # reported by the main thread
            errors.append(e)

    def captured():
        try:
            out, ws = buffers()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):   # the first call on s makes its second stream
                lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)
            s.synchronize()
            out.zero_()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            start.wait()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)
            for _ in range(reps):
                with torch.cuda.stream(s):
                    g.replay()
            s.synchronize()
            outs["graph"] = host_bits(out)
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=eager), threading.Thread(target=captured)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert np.array_equal(outs["eager"], ref_bits)
    assert np.array_equal(outs["graph"], ref_bits)
    ref_o, mid = O.latent_moe_forward(d, wts, xb, lgh, intermediates=True)
    r = O.bf16_to_f64(ref_o)
    assert_layer_close(O.bf16_to_f64(ref_bits), r, 2e-2, scale=addend_scale(r, mid, wts["w_up"]))
    assert lm.lmoe_device_error() == 0
