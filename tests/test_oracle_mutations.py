"""Planted mistakes: each plausible bug, put into the oracle on the CPU, must be
caught by one of the pins.  This shows the pins bite."""
import numpy as np
import pytest

import workloads as W
from oracle import lmoe_oracle as O
import tests.test_oracle_numerics as N
import tests.test_oracle_route as R
import tests.test_oracle_layer as L
import tests.test_oracle_router as RG
import tests.test_oracle_mxfp4 as MX

_route = O.route
_situ = O.situ
_permute = O.permute
_router_gemm = O.router_gemm
_e2m1_value = O.e2m1_value
_dequant_mxfp4 = O.dequant_mxfp4


def _situ_no_sigmoid(g, u, beta, lb):
    up = lb * np.tanh(u / lb) if lb > 0 else u
    return beta * np.tanh(g / beta) * up


def _situ_and_mul_swapped(x_bits, beta, lb):
    x = O.bf16_to_f64(x_bits)
    d = x.shape[-1] // 2
    return O.f64_to_bf16_bits(_situ(x[..., d:], x[..., :d], beta, lb))


def _route_no_bias(logits, bias, *a, **k):
    return _route(logits, None, *a, **k)


def _route_weights_from_keys(logits, bias, topk, rsf, *a, **k):
    ids, _ = _route(logits, bias, topk, rsf, *a, **k)
    key = (O.sigmoid_f32(logits) + (0 if bias is None else bias)).astype(np.float64)
    w = np.take_along_axis(key, ids.astype(np.int64), 1)
    return ids, w / w.sum(1, keepdims=True) * rsf


def _route_not_renormalised(logits, bias, topk, rsf, renormalize=1, *a, **k):
    return _route(logits, bias, topk, rsf, 0, *a, **k)


def _route_weights_reversed(*a, **k):
    ids, w = _route(*a, **k)
    return ids, w[:, ::-1].copy()


def _rms_norm_over_tokens(x, gamma, eps):
    return x / np.sqrt(np.mean(x * x, axis=0, keepdims=True) + eps) * gamma


def _rms_norm_gamma_dropped(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rms_norm_gamma_divided(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) / gamma


def _rms_norm_eps_outside_root(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * gamma


def _router_gemm_bf16_logits(x_bits, w_bits):
    return O.round_bf16(_router_gemm(x_bits, w_bits)).astype(np.float32)


def _router_gemm_rows_reversed(x_bits, w_bits):
    return _router_gemm(x_bits, w_bits[::-1].copy())


def _router_gemm_features_reversed(x_bits, w_bits):
    return _router_gemm(x_bits[:, ::-1].copy(), w_bits)


def _e2m1_no_subnormal(code):
    # exponent field 0 read like the others: 2^(e-1) * (1 + m/2)
    code = np.asarray(code).astype(np.int64)
    e, m = (code >> 1) & 3, code & 1
    return np.where(code & 8, -1.0, 1.0) * np.ldexp(1.0 + m * 0.5, e - 1)


def _dequant_nibbles_swapped(packed, scales):
    p = np.asarray(packed, dtype=np.uint8)
    return _dequant_mxfp4(((p & 15) << 4 | (p >> 4)).astype(np.uint8), scales)


def _dequant_scale_bias_128(packed, scales):
    return _dequant_mxfp4(packed, scales) * 0.5


def _dequant_blocks_of_16(packed, scales):
    codes = O.unpack_e2m1(packed)
    sc = np.repeat(np.ldexp(1.0, np.asarray(scales, np.int64) - 127), 16, axis=-1)
    sc = np.concatenate([sc, sc], axis=-1)[..., :codes.shape[-1]]
    return O.e2m1_value(codes) * sc


def _dequant_up_from_gate_rows(packed, scales):
    # a w13 read with its gate rows standing in for the up rows too
    w = _dequant_mxfp4(packed, scales)
    if w.shape[0] != 2 * W.TINY.inter:
        return w
    h = w.shape[0] // 2
    return np.concatenate([w[:h], w[:h]])


def _permute_descending(ids, E):
    counts, offsets, row_of, tok_of_row = _permute(ids[::-1].copy(), E)
    return counts, offsets, row_of[::-1].copy(), (ids.shape[0] - 1 - tok_of_row).astype(np.int32)


MUTATIONS = [
    ("situ", _situ_no_sigmoid, N.test_situ_large_beta_is_silu_gated_and_up_passes_through),
    ("situ_and_mul", _situ_and_mul_swapped, N.test_situ_and_mul_gate_is_first_half),
    ("route", _route_no_bias, R.check_equal_logits_bias_decides),
    ("route", _route_weights_from_keys, R.check_equal_logits_bias_decides),
    ("route", _route_not_renormalised, L.check_identical_experts_reduce_to_dense_mlp),
    ("route", _route_weights_reversed, L.check_power_of_two_scaled_experts),
    ("rms_norm", _rms_norm_over_tokens, L.check_token_independence),
    ("rms_norm", _rms_norm_gamma_dropped, L.check_rms_norm_gamma_scales_each_feature_exactly),
    ("rms_norm", _rms_norm_gamma_dropped, L.check_layer_gamma_power_of_two_scales_the_norm_output),
    ("rms_norm", _rms_norm_gamma_divided, L.check_rms_norm_gamma_multiplies),
    ("rms_norm", _rms_norm_gamma_divided, L.check_layer_gamma_power_of_two_scales_the_norm_output),
    ("rms_norm", _rms_norm_eps_outside_root, L.check_rms_norm_constant_row_closed_form),
    ("router_gemm", _router_gemm_bf16_logits, RG.check_two_hot_router_rows_sum_in_fp32),
    ("router_gemm", _router_gemm_rows_reversed, RG.check_one_hot_router_rows_pick_features),
    ("router_gemm", _router_gemm_features_reversed, RG.check_one_hot_router_rows_pick_features),
    ("e2m1_value", _e2m1_no_subnormal, MX.test_e2m1_positive_value_set),
    ("dequant_mxfp4", _dequant_nibbles_swapped, MX.check_nibble_order),
    ("dequant_mxfp4", _dequant_scale_bias_128, MX.check_scale_blocks),
    ("dequant_mxfp4", _dequant_blocks_of_16, MX.check_scale_blocks),
    ("dequant_mxfp4", _dequant_up_from_gate_rows, MX.check_gate_and_up_halves),
    ("permute", _permute_descending, lambda: R.check_permute(
        np.stack([np.random.default_rng(t).permutation(16)[:3] for t in range(20)]).astype(np.int32), 16)),
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check()
