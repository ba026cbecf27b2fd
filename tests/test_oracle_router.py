"""Pins of the oracle's router GEMM (CPU only): fp32 logits = X W_router^T.

One-hot router rows pick one hidden feature each (scaled by a power of two):
the logits are those features exactly, which fixes the operand orientation
and every index.  Two-hot rows add two features: the sum of two bf16 values
is exact in float32 but usually not in bf16, which fixes the precision of the
stored logits.  The layer built on the router GEMM routes on its logits."""
import dataclasses

import numpy as np

import workloads as W
from oracle import lmoe_oracle as O
from tests.test_oracle_route import brute_force_route

D = W.TINY


def _bits(x):
    return O.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def check_one_hot_router_rows_pick_features():
    g = np.random.default_rng(31)
    E, H, T = 24, 40, 6
    x = W.hidden_states(dataclasses.replace(D, T=T, hidden=H), 31)
    j = g.integers(0, H, E)
    a = g.integers(-3, 4, E)
    wr = np.zeros((E, H))
    wr[np.arange(E), j] = 2.0 ** a
    logits = O.router_gemm(x, _bits(wr))
    assert logits.dtype == np.float32 and logits.shape == (T, E)
    X = O.bf16_to_f64(x)
    assert np.array_equal(logits.astype(np.float64), X[:, j] * 2.0 ** a)


def test_one_hot_router_rows_pick_features():
    check_one_hot_router_rows_pick_features()


def check_two_hot_router_rows_sum_in_fp32():
    g = np.random.default_rng(32)
    E, H, T = 16, 24, 8
    x = W.hidden_states(dataclasses.replace(D, T=T, hidden=H), 32)
    i = g.integers(0, H, E)
    j = (i + 1 + g.integers(0, H - 1, E)) % H
    wr = np.zeros((E, H))
    wr[np.arange(E), i] = 1.0
    wr[np.arange(E), j] = 1.0
    logits = O.router_gemm(x, _bits(wr)).astype(np.float64)
    X = O.bf16_to_f64(x)
    want = X[:, i] + X[:, j]                      # exact in float64 and in float32
    assert np.array_equal(want.astype(np.float32).astype(np.float64), want)
    assert np.array_equal(logits, want)
    # most such sums are not bf16 values: stored logits keep float32 precision
    assert (O.round_bf16(want) != want).mean() > 0.5


def test_two_hot_router_rows_sum_in_fp32():
    check_two_hot_router_rows_sum_in_fp32()


def test_zero_router_leaves_the_bias_to_decide():
    d = dataclasses.replace(D, T=5)
    x = W.hidden_states(d, 33)
    wr = np.zeros((d.num_experts, d.hidden), dtype=np.uint16)
    lg = O.router_gemm(x, wr)
    assert np.all(lg == 0)
    bias = W.score_bias(d.num_experts, 33)
    ids, w = O.route(lg, bias, d.topk, d.routed_scaling_factor)
    bids, bw = brute_force_route(lg, bias, d.topk, d.routed_scaling_factor)
    assert np.array_equal(ids, bids) and np.allclose(w, bw, rtol=1e-12)
    # sigmoid(0) = 1/2 for every pick: equal weights rsf / k
    assert np.allclose(w, d.routed_scaling_factor / d.topk, rtol=1e-12)


def test_layer_on_the_router_gemm_routes_on_its_logits():
    d = dataclasses.replace(D, T=6)
    wts = W.layer_weights(d, 34)
    x = W.hidden_states(d, 34)
    wr = W.w_router(d, 34)
    out, mid = O.latent_moe_forward_router(d, wts, x, wr, intermediates=True)
    assert np.array_equal(mid["logits"], O.router_gemm(x, wr))
    bids, _ = brute_force_route(mid["logits"], wts["bias"], d.topk, d.routed_scaling_factor)
    assert np.array_equal(mid["ids"], bids)
    assert np.array_equal(out, O.latent_moe_forward(d, wts, x, mid["logits"]))


def test_router_weight_gives_unit_scale_logits():
    d = W.DECODE
    lg = O.router_gemm(W.hidden_states(d, 0), W.w_router(d, 0))
    assert 0.8 < float(np.std(lg)) < 1.2
