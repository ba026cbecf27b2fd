"""The Python binding refuses, before calling the library, tensors that the
kernels could not access as the C ABI describes (host memory, wrong dtype,
too few elements, not contiguous).  Runs without a GPU."""
import dataclasses

import pytest
import torch

import workloads as W

lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from latent_mixture_experts_sigmoid_gb300 import build
    build.build()
    lm.load_library()


def test_host_tensors_are_refused():
    d = W.TINY
    x = torch.zeros((d.T, d.hidden), dtype=torch.bfloat16)
    lg = torch.zeros((d.T, d.num_experts))
    ids = torch.zeros((d.T, d.topk), dtype=torch.int32)
    w = torch.zeros((d.T, d.topk))
    with pytest.raises(ValueError, match="CUDA"):
        lm.moe_route(lg, None, d.topk, 2.5, ids, w)
    with pytest.raises(ValueError, match="CUDA"):
        lm.situ_and_mul(torch.zeros((4, 16), dtype=torch.bfloat16),
                        torch.zeros((4, 8), dtype=torch.bfloat16), 4.0, 8.0)
    with pytest.raises(ValueError, match="CUDA"):
        lm.latent_moe_forward(d, lm.make_weights({}), x, lg, x, torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        lm.latent_moe_forward_routed(d, lm.make_weights({}), x, ids, w, x,
                                     torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        lm.lmoe_linear(x, torch.zeros((128, d.hidden), dtype=torch.bfloat16),
                       torch.zeros((d.T, 128), dtype=torch.bfloat16))


def test_weight_sizes_follow_the_dims():
    d = W.TINY
    w = W.layer_weights(d, 0)
    t = {k: (torch.from_numpy(v.view("int16")) if v is not None and v.dtype.kind == "u"
             else (torch.from_numpy(v) if v is not None else None)) for k, v in w.items()}
    # host tensors of the right sizes: refused for being on the host, by name
    with pytest.raises(ValueError, match="w_down.*CUDA"):
        lm.make_weights(t, d)
    # without dims nothing is checked (addresses are passed through)
    lm.make_weights(t)
    assert lm.make_weights({"w_down": 4096}, d).w_down == 4096
    small = dataclasses.replace(d, inter=64)
    with pytest.raises(ValueError):
        lm.make_weights({"w13": torch.zeros(3, dtype=torch.bfloat16)}, small)
