"""GPU parity of latent_moe_forward against the oracle.

Layer outputs: everywhere, every element within max(2e-2 * rms(oracle), 2 bf16
steps at the largest addend of the final sum) (tests/gpu_util.assert_layer_close).
The literal bound max |gpu - oracle| / rms(oracle) <= 2e-2 is asserted at the
tiny layer and the pre-routed tiny layers; at the decode layer (every output)
and the prefill layer (256 seeded tokens, the first and last, and the first
token of every used expert) the literal figure is recorded and every element
beyond it is explained one by one (tests/gpu_util.explain_layer_outliers): the
last stage recomputed from the GPU's own N and shared-expert activations
reproduces the GPU's value, and the shared-expert output differs from the
oracle's by at most one bf16 step.  Expert ids, expert_num_tokens, offsets and
the permuted row of every (token, slot): bit-exact.  Routing weights: 1e-6
relative.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import lmoe_oracle as O

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()


def check_routing_and_permutation(d, dbg, logits, bias):
    ids, w = O.route(logits, bias, d.topk, d.routed_scaling_factor, d.renormalize)
    assert np.array_equal(dbg["topk_ids"], ids)
    assert np.all(np.abs(dbg["topk_weights"] - w) <= 1e-6 * np.abs(w))
    counts, offsets, row_of, _ = O.permute(ids, d.num_experts)
    assert np.array_equal(dbg["expert_num_tokens"], counts)
    assert np.array_equal(dbg["expert_offsets"], offsets)
    assert np.array_equal(dbg["row_of"], row_of)


def tiny_case(d, seed=0, gamma_noise=False, shared=True, zipf=False, defaults=False,
              literal=None):
    from tests.gpu_util import (weights_to_device, run_layer, host_bits, assert_layer_close,
                                addend_scale, assert_layer_literal)
    wts = W.layer_weights(d, seed, gamma_noise)
    if not shared:
        wts["ws13"] = wts["ws2"] = None
    if defaults:
        # the optional weights left out: gamma = ones, selection bias = zeros
        wts["norm_w"] = wts["bias"] = None
    x = W.hidden_states(d, seed)
    lg = W.router_logits(d.T, d.num_experts, seed, zipf=zipf)
    out, dbg = run_layer(lm, d, weights_to_device(wts), x, lg)
    ref_bits, mid = O.latent_moe_forward(d, wts, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wts["w_up"]))
    if literal:
        assert_layer_literal(got, ref, literal, TOL)
    check_routing_and_permutation(d, dbg, lg, wts["bias"])
    assert lm.lmoe_device_error() == 0


def test_tiny_layer():
    tiny_case(W.TINY, literal="tiny layer T=8")


@pytest.mark.parametrize("T", [1, 3, 17, 100, 128, 129, 300, 1000])
def test_tiny_layer_token_counts(T):
    # decode regime up to 128 tokens, prefill regime above; ragged tails
    tiny_case(dataclasses.replace(W.TINY, T=T), seed=T)


@pytest.mark.parametrize("variant", ["no_shared", "linear_beta_unset", "gamma_noise", "top1",
                                     "no_renorm", "zipf_prefill", "wide", "pairs",
                                     "no_gamma_no_bias", "no_gamma_no_bias_prefill"])
def test_tiny_layer_variants(variant):
    d = W.TINY
    kw = {}
    if variant == "no_shared":
        kw["shared"] = False
    elif variant == "linear_beta_unset":
        d = dataclasses.replace(d, linear_beta=0.0)
    elif variant == "gamma_noise":
        kw["gamma_noise"] = True
    elif variant == "top1":
        d = dataclasses.replace(d, topk=1)
    elif variant == "no_renorm":
        d = dataclasses.replace(d, renormalize=0, routed_scaling_factor=1.0)
    elif variant == "zipf_prefill":
        d = dataclasses.replace(d, T=700)
        kw["zipf"] = True
    elif variant == "wide":
        d = dataclasses.replace(d, T=200, hidden=384, latent=256, inter=192, shared_inter=320,
                                num_experts=40, topk=8)
    elif variant == "no_gamma_no_bias":
        kw["defaults"] = True
    elif variant == "no_gamma_no_bias_prefill":
        d = dataclasses.replace(d, T=300)
        kw["defaults"] = True
    elif variant == "pairs":
        # every GEMM in CTA pairs: even weight-tile counts everywhere, 5 token
        # tiles (the dense GEMMs' odd last tile is shared by two weight tiles)
        d = dataclasses.replace(d, T=600, hidden=512, latent=512, inter=256, shared_inter=256)
    tiny_case(d, seed=11, **kw)


@pytest.mark.parametrize("T", [8, 300])
def test_tiny_layer_max_experts_and_topk(T):
    # the largest expert count and top-k the library accepts (1024, 32), in the
    # decode (fused permutation + scatter) and prefill regimes
    tiny_case(dataclasses.replace(W.TINY, T=T, num_experts=1024, topk=32), seed=5)


def test_zero_tokens_is_a_no_op():
    from tests.gpu_util import DEV, weights_to_device
    d = dataclasses.replace(W.TINY, T=0)
    assert lm.latent_moe_launch_count(d) == 0
    wdev = weights_to_device(W.layer_weights(W.TINY, 0))
    x = torch.empty((0, d.hidden), dtype=torch.bfloat16, device=DEV)
    lg = torch.empty((0, d.num_experts), dtype=torch.float32, device=DEV)
    out = torch.empty((0, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(max(256, lm.latent_moe_workspace_bytes(d)), dtype=torch.uint8, device=DEV)
    lm.latent_moe_forward(d, wdev, x, lg, out, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_error() == 0


def _routed_case(T, seed=3):
    from tests.gpu_util import DEV, weights_to_device, dev_bf16, dev_f32
    d = dataclasses.replace(W.TINY, T=T)
    wdev = weights_to_device(W.layer_weights(d, seed))
    x = dev_bf16(W.hidden_states(d, seed))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, seed))
    ids = torch.empty((T, d.topk), dtype=torch.int32, device=DEV)
    w = torch.empty((T, d.topk), dtype=torch.float32, device=DEV)
    return d, wdev, x, lg, ids, w


@pytest.mark.parametrize("T", [8, 300])
def test_pre_routed_forward_is_bit_identical(T):
    # TensorRT-LLM PR #20541, commit 1: the routing runs as its own op on
    # another stream and the MoE op consumes its outputs after an event join;
    # the output is bit-identical to the op routing itself
    from tests.gpu_util import DEV
    d, wdev, x, lg, ids, w = _routed_case(T)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    ref = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    lm.latent_moe_forward(d, wdev, x, lg, ref, ws)
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    routed = torch.cuda.Event()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        lm.moe_route(lg, wdev["bias"], d.topk, d.routed_scaling_factor, ids, w,
                     renormalize=d.renormalize, stream=side)
        routed.record(side)
    out = torch.empty_like(ref)
    ws2 = torch.empty_like(ws)
    main.wait_event(routed)
    with torch.cuda.stream(main):
        lm.latent_moe_forward_routed(d, wdev, x, ids, w, out, ws2, stream=main)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert lm.lmoe_device_error() == 0


@pytest.mark.parametrize("T", [8, 300])
def test_pre_routed_forward_matches_the_oracle(T):
    # the pre-routed forward against the oracle itself on the same inputs
    # (routing by moe_route on its own stream, as TensorRT-LLM PR #20541,
    # commit 1 runs it), not only against the layer routing itself
    from tests.gpu_util import (host_bits, assert_layer_close, assert_layer_literal,
                                addend_scale, DEV)
    d, wdev, x, lg, ids, w = _routed_case(T)
    side = torch.cuda.Stream()
    routed = torch.cuda.Event()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        lm.moe_route(lg, wdev["bias"], d.topk, d.routed_scaling_factor, ids, w,
                     renormalize=d.renormalize, stream=side)
        routed.record(side)
    torch.cuda.current_stream().wait_event(routed)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    lm.latent_moe_forward_routed(d, wdev, x, ids, w, out, ws)
    torch.cuda.synchronize()
    wts = W.layer_weights(d, 3)
    ref_bits, mid = O.latent_moe_forward(d, wts, W.hidden_states(d, 3),
                                         W.router_logits(d.T, d.num_experts, 3),
                                         intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wts["w_up"]))
    assert_layer_literal(got, ref, f"pre-routed tiny layer T={T}", TOL)
    oids, ow = O.route(W.router_logits(d.T, d.num_experts, 3), wts["bias"], d.topk,
                       d.routed_scaling_factor, d.renormalize)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert np.all(np.abs(w.cpu().numpy() - ow) <= 1e-6 * np.abs(ow))
    assert lm.lmoe_device_error() == 0


@pytest.mark.parametrize("T", [8, 300])
def test_pre_routed_out_of_range_id_is_recorded(T):
    # an expert id outside [0, E) is read as expert 0 (no access outside the
    # buffers) and recorded as code 7 in the device error word
    from tests.gpu_util import DEV
    d, wdev, x, lg, ids, w = _routed_case(T)
    lm.moe_route(lg, wdev["bias"], d.topk, d.routed_scaling_factor, ids, w,
                 renormalize=d.renormalize)
    ids[T // 2, 1] = d.num_experts + 5
    ids[T - 1, 0] = -1
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    assert lm.lmoe_device_error(clear=True) == 0
    lm.latent_moe_forward_routed(d, wdev, x, ids, w, out, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_error(clear=True) == 7
    assert lm.lmoe_device_error() == 0


@pytest.fixture(scope="module")
def big_weights():
    from tests.gpu_util import device_layer_weights, oracle_layer_weights
    d = W.DECODE
    return device_layer_weights(d, 0), oracle_layer_weights(d, 0)


def test_decode_layer_full(big_weights):
    from tests.gpu_util import (run_layer, host_bits, assert_layer_close, addend_scale,
                                record_literal, explain_layer_outliers, workspace_view)
    d = W.DECODE
    wdev, wor = big_weights
    x = W.hidden_states(d, 0)
    lg = W.router_logits(d.T, d.num_experts, 0)
    out, dbg, ws = run_layer(lm, d, wdev, x, lg, keep_ws=True)
    check_routing_and_permutation(d, dbg, lg, wor["bias"])
    ref_bits, mid = O.latent_moe_forward(d, wor, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    stats = assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wor["w_up"]))
    assert stats["frac_differing"] < 0.5
    record_literal(got, ref, "decode layer T=8 (every output)", TOL)
    explain_layer_outliers(got, ref, np.arange(d.T), mid, workspace_view(lm, d, ws), x, wor, d,
                           "decode layer T=8", TOL)
    assert lm.lmoe_device_error() == 0


def test_prefill_layer_zipf_sampled(big_weights):
    from tests.gpu_util import (run_layer, host_bits, assert_layer_close, addend_scale,
                                record_literal, explain_layer_outliers, workspace_view)
    d = W.PREFILL
    wdev, wor = big_weights
    x = W.hidden_states(d, 0)
    lg = W.router_logits(d.T, d.num_experts, 0, zipf=True)
    out, dbg, ws = run_layer(lm, d, wdev, x, lg, keep_ws=True)
    check_routing_and_permutation(d, dbg, lg, wor["bias"])
    counts = dbg["expert_num_tokens"]
    assert counts.max() > 500 and (counts == 0).sum() > 100     # the skew is real
    # a seeded sample of 256 tokens, the first and the last token, and for every
    # expert that receives tokens its first token (so that each used expert's
    # weights meet the oracle at least once)
    ids = dbg["topk_ids"]
    first_of_expert = [int(np.argmax((ids == e).any(axis=1))) for e in np.unique(ids)]
    toks = np.unique(np.concatenate([[0, d.T - 1], first_of_expert,
                                     np.random.default_rng(3).choice(d.T, 256, replace=False)]))
    ref_bits, mid = O.latent_moe_forward(d, wor, x[toks], lg[toks], intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))[toks]
    stats = assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wor["w_up"]))
    assert stats["frac_differing"] < 0.5
    case = f"prefill layer T=4096 Zipf ({len(toks)} sampled tokens)"
    record_literal(got, ref, case, TOL)
    explain_layer_outliers(got, ref, toks, mid, workspace_view(lm, d, ws), x, wor, d, case, TOL)
    # every output finite
    assert torch.isfinite(out.float()).all()
    assert lm.lmoe_device_error() == 0


def test_graph_replay_and_determinism():
    from tests.gpu_util import weights_to_device, dev_bf16, dev_f32, DEV
    d = dataclasses.replace(W.TINY, T=64)
    wts = weights_to_device(W.layer_weights(d, 2))
    x = dev_bf16(W.hidden_states(d, 2))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, 2))
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    a = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    c = torch.zeros_like(a)
    lm.latent_moe_forward(d, wts, x, lg, a, ws)
    lm.latent_moe_forward(d, wts, x, lg, b, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lm.latent_moe_forward(d, wts, x, lg, c, ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("T", [1, 128])
def test_decode_layer_graph_replays_are_bit_identical(big_weights, T):
    # the 896-expert layer at decode sizes (GEMM1 + SituGLU with its two MMA
    # issuers at 16 and 128 token columns, the shared expert forked onto the
    # second stream after GEMM1): 20 graph replays, each bit-identical to the
    # eager forward, and no device error
    from tests.gpu_util import dev_bf16, dev_f32, DEV
    d = dataclasses.replace(W.DECODE, T=T)
    wdev, _ = big_weights
    x = dev_bf16(W.hidden_states(d, 5))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, 5))
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    ref = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lm.latent_moe_forward(d, wdev, x, lg, ref, ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)
    for _ in range(20):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert lm.lmoe_device_error() == 0


def test_invalid_arguments_are_rejected():
    from tests.gpu_util import DEV
    d = W.TINY
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    x = torch.zeros((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    lg = torch.zeros((d.T, d.num_experts), device=DEV)
    # placeholder weights, unchecked by the binding: the library refuses first
    pw = lm.make_weights({"w_down": x, "w13": x, "w2": x, "w_up": x})
    with pytest.raises(lm.LmoeError) as e:
        lm.latent_moe_forward(d, pw, x, lg, x, ws)
    assert e.value.status == -5   # workspace too small
    # the binding refuses tensors the kernels could not use as the ABI says
    wts = {"w_down": x, "w13": x, "w2": x, "w_up": x}
    with pytest.raises(ValueError, match="w_down"):
        lm.latent_moe_forward(d, wts, x, lg, x, ws)
    full = lm.make_weights({})   # no weights at all: the library reports the missing ones
    with pytest.raises(ValueError, match="router_logits"):
        lm.latent_moe_forward(d, full, x, lg.double(), x, ws)
    with pytest.raises(ValueError, match="contiguous"):
        lm.latent_moe_forward(d, full, x.t(), lg, x, ws)
    with pytest.raises(ValueError, match="workspace"):
        lm.latent_moe_forward(d, full, x, lg, x, ws, workspace_bytes=1 << 20)
    for bad, st in [(dict(beta=0.0), -4), (dict(n_group=4), -3), (dict(hidden=200), -2),
                    (dict(topk=65), -2)]:
        with pytest.raises(lm.LmoeError) as e:
            lm.latent_moe_forward(dataclasses.replace(d, **bad), {}, x, lg, x, ws)
        assert e.value.status == st
