"""Pins of the oracle's MXFP4 (block-scaled E2M1) weight format.

The format (vLLM PR #50088, commits 4-5 and TensorRT-LLM PR #20541 run this
layer's routed experts on the TRTLLM-Gen MXFP4 backend; the encoding is the
OCP microscaling one): 4-bit E2M1 elements (1 sign, 2 exponent bits with bias
1, 1 mantissa bit; exponent 0 subnormal), two per byte with element 2i in the
low nibble, and one E8M0 power of two per 32 consecutive elements.

Pinned against: the E2M1 value set (largest normal 1.5 * 2^2 = 6, smallest
normal 1, the one subnormal 0.5), sign symmetry, PyTorch's own E8M0 decoding
(torch.float8_e8m0fnu), hand-packed bytes whose element order is known, and
block-boundary placement of the scales.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import lmoe_oracle as O


def test_e2m1_positive_value_set():
    # codes 0..7 in increasing order: 0, the subnormal 0.5, then 1, 1.5 (e=1),
    # 2, 3 (e=2), 4, 6 (e=3)
    assert O.e2m1_value(np.arange(8)).tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_sign_bit_negates():
    v = O.e2m1_value(np.arange(16))
    assert np.array_equal(v[8:], -v[:8])
    assert np.signbit(v[8]) and v[8] == 0.0   # code 8 is negative zero


def test_e8m0_matches_torch_decoding():
    s = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(s).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = O.e8m0_value(s)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got[255])
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127


def check_nibble_order():
    # byte 0x21: element 0 = code 1 (0.5), element 1 = code 2 (1.0); byte 0xF7:
    # element 2 = code 7 (6.0), element 3 = code 15 (-6.0); the rest zero
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0], packed[0, 1] = 0x21, 0xF7
    w = O.dequant_mxfp4(packed, np.full((1, 1), 127, dtype=np.uint8))
    assert w[0, :4].tolist() == [0.5, 1.0, 6.0, -6.0]
    assert not w[0, 4:].any()


def test_nibble_order():
    check_nibble_order()


def check_scale_blocks():
    # K = 96: three scale blocks of 32 elements, every code 2 (1.0); scales
    # 2^0, 2^1, 2^-1 placed block by block, and a second row with 2^-127, 2^10
    # and NaN
    packed = np.full((2, 48), 0x22, dtype=np.uint8)
    scales = np.array([[127, 128, 126], [0, 137, 255]], dtype=np.uint8)
    w = O.dequant_mxfp4(packed, scales)
    assert np.array_equal(w[0], np.repeat([1.0, 2.0, 0.5], 32))
    assert np.array_equal(w[1, :64], np.repeat([2.0 ** -127, 1024.0], 32))
    assert np.isnan(w[1, 64:]).all()


def test_scale_blocks():
    check_scale_blocks()


def test_bf16_bits_exact_over_the_supported_scale_range():
    g = np.random.default_rng(0)
    packed = g.integers(0, 256, size=(64, 128), dtype=np.uint8)
    scales = g.integers(2, 253, size=(64, 8), dtype=np.uint8)
    bits = O.mxfp4_as_bf16_bits(packed, scales)
    assert np.array_equal(O.bf16_to_f64(bits), O.dequant_mxfp4(packed, scales))
    # the extremes of the range: 6 * 2^125 and 0.5 * 2^-125
    hi = O.mxfp4_as_bf16_bits(np.full((1, 16), 0x77, np.uint8), np.full((1, 1), 252, np.uint8))
    lo = O.mxfp4_as_bf16_bits(np.full((1, 16), 0x11, np.uint8), np.full((1, 1), 2, np.uint8))
    assert O.bf16_to_f64(hi)[0, 0] == 6.0 * 2.0 ** 125
    assert O.bf16_to_f64(lo)[0, 0] == 0.5 * 2.0 ** -125


def test_generator_draws_every_code_and_the_stated_scales():
    q, s = W.mxfp4_w13_expert(W.TINY, 3)
    assert q.shape == (2 * W.TINY.inter, W.TINY.latent // 2)
    assert s.shape == (2 * W.TINY.inter, W.TINY.latent // 32)
    assert set(np.unique(O.unpack_e2m1(q)).tolist()) == set(range(16))
    assert s.min() >= W.MXFP4_SCALE_LO and s.max() <= W.MXFP4_SCALE_HI


def test_mxfp4_layer_is_the_layer_on_the_dequantized_weights():
    # the MXFP4 forward changes only where the expert weights come from
    d = dataclasses.replace(W.TINY, T=5)
    wts = W.layer_weights(d, 2)
    Q = W.mxfp4_experts(d, 2)
    x = W.hidden_states(d, 2)
    lg = W.router_logits(d.T, d.num_experts, 2)
    got = O.latent_moe_forward_mxfp4(d, wts, Q, x, lg)
    deq = dict(wts, w13=np.stack([O.mxfp4_as_bf16_bits(Q["w13_q"][e], Q["w13_s"][e])
                                  for e in range(d.num_experts)]),
               w2=np.stack([O.mxfp4_as_bf16_bits(Q["w2_q"][e], Q["w2_s"][e])
                            for e in range(d.num_experts)]))
    assert np.array_equal(got, O.latent_moe_forward(d, deq, x, lg))


def check_gate_and_up_halves():
    # the MXFP4 w13 keeps the bf16 row order (gate rows 0..d-1, up rows d..2d-1):
    # with every up weight zero the expert output is SituGLU(g, 0) = 0, and with
    # every gate weight zero it is 0 too (tanh(0) = 0); only the pair with both
    # halves nonzero gives a nonzero latent output
    d = dataclasses.replace(W.TINY, T=2, topk=1, shared_inter=0)
    wts = W.layer_weights(d, 1)
    wts["ws13"] = wts["ws2"] = None
    Q = W.mxfp4_experts(d, 1)
    x = W.hidden_states(d, 1)
    lg = W.router_logits(d.T, d.num_experts, 1)
    _, mid = O.latent_moe_forward_mxfp4(d, wts, Q, x, lg, intermediates=True)
    assert np.abs(mid["C"]).max() > 0
    for half in (0, 1):
        Qz = dict(Q, w13_q=Q["w13_q"].copy())
        Qz["w13_q"][:, half * d.inter:(half + 1) * d.inter] = 0
        _, mz = O.latent_moe_forward_mxfp4(d, wts, Qz, x, lg, intermediates=True)
        assert not mz["C"].any()


def test_mxfp4_gate_and_up_halves():
    check_gate_and_up_halves()
