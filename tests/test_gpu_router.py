"""GPU parity of the router GEMM (lmoe_router_logits) and of the layer forward
built on it (latent_moe_forward_router) against the oracle.

Logits: every element within the fp32 accumulation bound
(H/16 + 32) * 2^-23 * sum_h |x_h w_h| of the oracle's float64 product rounded
to fp32 (one rounding per K = 16 tensor-core step and per split, each at most
one fp32 step of the running sum, doubled for truncating accumulation).
Routing from those logits: ids bit-exact and weights within 1e-6 of the
oracle's routing of the GPU's own logits (the routing stage fed identical
inputs), and against the oracle's own logits wherever the k-th and (k+1)-th
selection keys are further apart than the logit bound can move them.  Layer
output: the layer tolerance of tests/gpu_util against the oracle's layer on
the GPU's logits; the literal 2e-2 figure at the tiny layer."""
import dataclasses

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


def logit_bound(x_bits, wr_bits):
    X = np.abs(O.bf16_to_f64(x_bits))
    Wr = np.abs(O.bf16_to_f64(wr_bits))
    H = X.shape[1]
    return (H / 16 + 32) * 2.0 ** -23 * (X @ Wr.T) + 1e-30


def check_logits(got, x_bits, wr_bits):
    ref = O.router_gemm(x_bits, wr_bits).astype(np.float64)
    bound = logit_bound(x_bits, wr_bits)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound), (float((err / bound).max()), np.argwhere(err > bound)[:5])
    return ref, bound


@pytest.mark.parametrize("T", [1, 8, 128, 129, 300])
@pytest.mark.parametrize("E,H", [(64, 256), (100, 512), (896, 7168)])
def test_router_logits(T, E, H):
    from tests.gpu_util import DEV, dev_bf16
    d = dataclasses.replace(W.TINY, T=T, num_experts=E, hidden=H)
    x = W.hidden_states(d, T + E)
    wr = W.w_router(d, T + E)
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(lm.lmoe_router_logits_workspace_bytes(T, E, H), dtype=torch.uint8, device=DEV)
    lm.lmoe_router_logits(dev_bf16(x), dev_bf16(wr), logits, ws)
    torch.cuda.synchronize()
    check_logits(logits.cpu().numpy(), x, wr)
    assert lm.lmoe_device_error() == 0


def selection_margin(logits, bias, k):
    """Gap between the k-th and (k+1)-th largest selection keys of each row."""
    key = np.sort(O.sigmoid_f32(logits).astype(np.float64) + bias[None, :], axis=1)[:, ::-1]
    return key[:, k - 1] - key[:, k]


def router_layer_case(d, wdev, wor, wr_bits, seed, literal=None):
    from tests.gpu_util import (DEV, dev_bf16, host_bits, assert_layer_close, addend_scale,
                                assert_layer_literal, record_literal, workspace_view)
    from tests.test_gpu_layer import check_routing_and_permutation
    T, k, E = d.T, d.topk, d.num_experts
    x = W.hidden_states(d, seed)
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    dbg = dict(topk_ids=torch.empty((T, k), dtype=torch.int32, device=DEV),
               topk_weights=torch.empty((T, k), dtype=torch.float32, device=DEV),
               expert_num_tokens=torch.empty(E, dtype=torch.int32, device=DEV),
               expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
               row_of=torch.empty((T, k), dtype=torch.int32, device=DEV))
    lm.latent_moe_forward_router(d, wdev, dev_bf16(wr_bits), dev_bf16(x), out, ws, debug=dbg)
    torch.cuda.synchronize()
    dbg = {n: v.cpu().numpy() for n, v in dbg.items()}
    off = lm.latent_moe_workspace_offsets(d)["logits"]
    Ep = (E + 127) // 128 * 128
    lg = ws[off:off + T * Ep * 4].cpu().numpy().view(np.float32).reshape(T, Ep)[:, :E].copy()
    ref_lg, bound = check_logits(lg, x, wr_bits)
    # routing and permutation bit-exact on the GPU's logits
    check_routing_and_permutation(d, dbg, lg, wor["bias"])
    # against the oracle's own logits: equal ids unless the selection is a near tie
    oids, _ = O.route(ref_lg.astype(np.float32), wor["bias"], k, d.routed_scaling_factor,
                      d.renormalize)
    differ = ~(np.sort(oids, 1) == np.sort(dbg["topk_ids"], 1)).all(1)
    margin = selection_margin(ref_lg.astype(np.float32), wor["bias"], k)
    slack = 0.5 * bound.max(axis=1) + 2.0 ** -22      # |d sigmoid| <= |d logit| / 4, both ends
    assert np.all(margin[differ] <= slack[differ]), (np.nonzero(differ), margin[differ])
    # the layer on the GPU's logits
    ref_bits, mid = O.latent_moe_forward(d, wor, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, 2e-2, scale=addend_scale(ref, mid, wor["w_up"]))
    if literal:
        assert_layer_literal(got, ref, literal)
    else:
        record_literal(got, ref, f"router-GEMM layer T={T}, E={E}")
    assert lm.lmoe_device_error() == 0
    return lg


@pytest.mark.parametrize("T", [8, 300])
def test_router_layer_tiny(T):
    from tests.gpu_util import weights_to_device
    d = dataclasses.replace(W.TINY, T=T)
    wts = W.layer_weights(d, 41)
    router_layer_case(d, weights_to_device(wts), wts, W.w_router(d, 41), 41,
                      literal=f"router-GEMM tiny layer T={T}")


def test_router_layer_decode_full():
    from tests.gpu_util import device_layer_weights, oracle_layer_weights
    d = W.DECODE
    router_layer_case(d, device_layer_weights(d, 0), oracle_layer_weights(d, 0),
                      W.w_router(d, 0), 0)


def test_router_layer_matches_routing_from_the_router_op():
    # at T > 128 the router GEMM is the same launch lmoe_router_logits makes
    # (tokens on M, no split), so the layer's routing equals moe_route on
    # lmoe_router_logits' output bit for bit
    from tests.gpu_util import DEV, dev_bf16, weights_to_device
    d = dataclasses.replace(W.TINY, T=300)
    wts = W.layer_weights(d, 42)
    wdev = weights_to_device(wts)
    x = dev_bf16(W.hidden_states(d, 42))
    wr = dev_bf16(W.w_router(d, 42))
    lg = torch.empty((d.T, d.num_experts), dtype=torch.float32, device=DEV)
    rws = torch.empty(lm.lmoe_router_logits_workspace_bytes(d.T, d.num_experts, d.hidden),
                      dtype=torch.uint8, device=DEV)
    lm.lmoe_router_logits(x, wr, lg, rws)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    a = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    lm.latent_moe_forward(d, wdev, x, lg, a, ws)
    lm.latent_moe_forward_router(d, wdev, wr, x, b, torch.empty_like(ws))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert lm.lmoe_device_error() == 0
