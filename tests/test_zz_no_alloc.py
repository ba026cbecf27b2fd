"""latent_moe_forward_noalloc: the layer forward for callers that cannot
allocate device memory (a runtime plugin handed only its input and output
buffers, host code without an allocator, a path where cudaMalloc's implicit
synchronisation is not allowed).  It must give the same output as
latent_moe_forward with a caller workspace, call after call, although every
call reuses the library's one static scratch array.

This file is collected last on purpose: it passes alone in a fresh process and
after every other test."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import lmoe_oracle as O

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")

# the 896-expert model's shapes with 64 experts (weights stay small), decode T=8
MID = dataclasses.replace(W.DECODE, num_experts=64)


def _inputs(d, seed):
    from tests.gpu_util import dev_bf16, dev_f32
    x = dev_bf16(W.hidden_states(d, seed))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, seed))
    return x, lg


def _workspace_forward(d, w, x, lg):
    from tests.gpu_util import DEV
    out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    lm.latent_moe_forward(d, w, x, lg, out, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d", [W.TINY, MID], ids=["tiny", "mid64"])
def test_noalloc_matches_workspace_forward_on_two_calls(cuda_ok, d):
    from tests.gpu_util import DEV, weights_to_device, device_layer_weights, host_bits, \
        assert_layer_close
    lm.load_library()
    w = weights_to_device(W.layer_weights(d, 0)) if d is W.TINY else device_layer_weights(d, 0)
    # two calls in a row on different inputs: the second runs on the scratch
    # contents the first left behind
    for seed in (0, 1):
        x, lg = _inputs(d, seed)
        ref = _workspace_forward(d, w, x, lg)
        out = torch.full((d.T, d.hidden), float("nan"), dtype=torch.bfloat16, device=DEV)
        lm.latent_moe_forward_noalloc(d, w, x, lg, out)
        torch.cuda.synchronize()
        got, want = O.bf16_to_f64(host_bits(out)), O.bf16_to_f64(host_bits(ref))
        assert_layer_close(got, want, 2e-2)
        assert np.array_equal(host_bits(out), host_bits(ref))   # same kernels, same bits
    assert lm.lmoe_device_error() == 0


def test_noalloc_rejects_calls_beyond_its_scratch(cuda_ok):
    from tests.gpu_util import DEV
    lm.load_library()
    d = dataclasses.replace(W.DECODE, T=64)          # needs ~134 MiB of scratch
    assert lm.latent_moe_workspace_bytes(d) > 32 * 2 ** 20
    x = torch.zeros((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    lg = torch.zeros((d.T, d.num_experts), device=DEV)
    # placeholder weights, unchecked by the binding: the library refuses first
    w = lm.make_weights({k: x for k in ("w_down", "w13", "w2", "w_up")})
    with pytest.raises(lm.LmoeError) as e:
        lm.latent_moe_forward_noalloc(d, w, x, lg, x)
    assert e.value.status == -5
