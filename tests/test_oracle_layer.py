"""Pins of the oracle's layer composition (CPU only).

Closed-form reductions of the layer (identical experts, power-of-two scaled
experts, zero expert outputs, identity shared expert), brute force for the GEMM
stage, and structural invariants (token independence, expert relabelling).
"""
import dataclasses

import numpy as np

import workloads as W
from oracle import lmoe_oracle as O
from tests.test_oracle_route import brute_force_route

D = W.TINY


def tiny(seed=0, gamma_noise=False):
    wts = W.layer_weights(D, seed, gamma_noise)
    x = W.hidden_states(D, seed)
    lg = W.router_logits(D.T, D.num_experts, seed)
    return wts, x, lg


def test_linear_stage_matches_triple_loop():
    g = np.random.default_rng(0)
    x = g.standard_normal((3, 5))
    wb = O.f64_to_bf16_bits(g.standard_normal((4, 5)))
    wf = O.bf16_to_f64(wb)
    ref = np.zeros((3, 4))
    for i in range(3):
        for o in range(4):
            acc = 0.0
            for c in range(5):
                acc += x[i, c] * wf[o, c]
            ref[i, o] = acc
    assert np.allclose(O.linear_bf16(x, wb), O.round_bf16(ref), rtol=0, atol=1e-12)


def test_rms_norm_rows_have_unit_rms_and_are_scale_free():
    g = np.random.default_rng(1)
    x = g.standard_normal((6, 128)) * 7
    n = O.rms_norm(x, np.ones(128), 0.0)
    assert np.allclose(np.sqrt(np.mean(n * n, axis=1)), 1.0, rtol=1e-12)
    assert np.allclose(O.rms_norm(3 * x, np.ones(128), 0.0), n, rtol=1e-12)


def check_token_independence():
    wts, x, lg = tiny(1)
    full = O.latent_moe_forward(D, wts, x, lg)
    for sub in ([0], [3, 5], [7, 1, 2]):
        part = O.latent_moe_forward(D, wts, x[sub], lg[sub])
        assert np.array_equal(part, full[sub])


def test_token_independence():
    check_token_independence()


def check_identical_experts_reduce_to_dense_mlp():
    wts, x, lg = tiny(2)
    wts["w13"] = np.broadcast_to(wts["w13"][0], wts["w13"].shape)
    wts["w2"] = np.broadcast_to(wts["w2"][0], wts["w2"].shape)
    out, mid = O.latent_moe_forward(D, wts, x, lg, intermediates=True)
    Z = mid["Z"]
    G = O.linear_bf16(Z, wts["w13"][0])
    act = O.round_bf16(O.situ(G[:, :D.inter], G[:, D.inter:], D.beta, D.linear_beta))
    Yd = O.linear_bf16(act, wts["w2"][0])
    # sum_j w_j = rsf, so the routed sum is rsf times the dense expert output
    assert np.allclose(mid["C"], D.routed_scaling_factor * Yd, rtol=1e-12, atol=1e-15)


def test_identical_experts_reduce_to_dense_mlp():
    check_identical_experts_reduce_to_dense_mlp()


def check_power_of_two_scaled_experts():
    # W2_e = 2^a_e * W2_0 and W13_e = W13_0 give Y_e = 2^a_e * Y_0 exactly in
    # bf16, so C[t] = (sum_j w[t,j] 2^a_{ids[t,j]}) * Y_0[t]: each weight must
    # meet its own expert's output.
    wts, x, lg = tiny(3)
    a = np.random.default_rng(9).integers(-3, 4, D.num_experts)
    w2_0 = O.bf16_to_f64(wts["w2"][0])
    wts["w13"] = np.broadcast_to(wts["w13"][0], wts["w13"].shape)
    wts["w2"] = np.stack([O.f64_to_bf16_bits(w2_0 * 2.0 ** int(a[e])) for e in range(D.num_experts)])
    _, mid = O.latent_moe_forward(D, wts, x, lg, intermediates=True)
    # ids and weights from the brute-force selection, not from the oracle's route
    ids, w = brute_force_route(lg, wts["bias"], D.topk, D.routed_scaling_factor)
    Y0 = mid["Y"][:, 0] / (2.0 ** a[ids[:, 0]])[:, None]
    scale = (w * 2.0 ** a[ids]).sum(1)
    assert np.allclose(mid["C"], scale[:, None] * Y0, rtol=1e-12, atol=1e-15)


def test_power_of_two_scaled_experts():
    check_power_of_two_scaled_experts()


def test_zero_expert_outputs_leave_the_shared_expert():
    wts, x, lg = tiny(4)
    wts["w2"] = np.zeros_like(wts["w2"])
    out, mid = O.latent_moe_forward(D, wts, x, lg, intermediates=True)
    assert np.all(mid["N"] == 0)
    assert np.array_equal(O.bf16_to_f64(out), mid["Sh"])


def test_identity_shared_expert_is_elementwise_situ():
    # hidden == shared_inter, Ws13 = [a*I; b*I], Ws2 = I: Sh = bf16(situ(bf16(aX), bf16(bX)))
    d = dataclasses.replace(D, shared_inter=D.hidden)
    wts, x, lg = tiny(5)
    eye = np.eye(D.hidden)
    a, b = 0.5, 2.0
    wts["ws13"] = O.f64_to_bf16_bits(np.concatenate([a * eye, b * eye]))
    wts["ws2"] = O.f64_to_bf16_bits(eye)
    wts["w2"] = np.zeros_like(wts["w2"])
    out = O.latent_moe_forward(d, wts, x, lg)
    X = O.bf16_to_f64(x)
    expect = O.round_bf16(O.situ(O.round_bf16(a * X), O.round_bf16(b * X), d.beta, d.linear_beta))
    assert np.array_equal(O.bf16_to_f64(out), expect)


def test_no_shared_expert_and_identity_up_projection_gives_the_norm():
    # latent == hidden, W_up = I, no shared expert, gamma = 1, eps = 0: out = N
    # and the rows of N have unit RMS up to bf16 rounding.
    d = dataclasses.replace(D, hidden=D.latent, T=8, rms_eps=0.0)
    wts, _, lg = tiny(6)
    wts = dict(wts, ws13=None, ws2=None, w_up=O.f64_to_bf16_bits(np.eye(d.latent)),
               w_down=O.f64_to_bf16_bits(np.eye(d.latent)))
    x = W.hidden_states(d, 6)
    out, mid = O.latent_moe_forward(d, wts, x, lg, intermediates=True)
    assert np.array_equal(O.bf16_to_f64(out), mid["N"])
    rms = np.sqrt(np.mean(mid["N"] ** 2, axis=1))
    assert np.allclose(rms, 1.0, rtol=4e-3)


def check_expert_relabelling_invariance():
    wts, x, lg = tiny(7)
    perm = np.random.default_rng(11).permutation(D.num_experts)
    wts2 = dict(wts, w13=wts["w13"][perm], w2=wts["w2"][perm], bias=wts["bias"][perm])
    a = O.latent_moe_forward(D, wts, x, lg)
    b = O.latent_moe_forward(D, wts2, x, np.ascontiguousarray(lg[:, perm]))
    assert np.array_equal(a, b)


def test_expert_relabelling_invariance():
    check_expert_relabelling_invariance()


def test_lazy_expert_weights_match_stacked():
    wts, x, lg = tiny(8)
    lazy = dict(wts, w13=lambda e: W.w13_expert(D, e, 8), w2=lambda e: W.w2_expert(D, e, 8))
    assert np.array_equal(O.latent_moe_forward(D, wts, x, lg), O.latent_moe_forward(D, lazy, x, lg))


# --- RMSNorm gamma and epsilon (vLLM latent_moe_runner page,
# _shard_up_proj_tail: transform.norm of the reduced latent; vLLM PR #50088,
# commit 7: the routed sum is complete before the norm) ----------------------

def check_rms_norm_gamma_scales_each_feature_exactly():
    # gamma = 2^a per feature multiplies column f by exactly 2^a_f (a power of
    # two changes no rounding), whatever x and eps are
    g = np.random.default_rng(21)
    x = g.standard_normal((5, 64)) * 3
    a = g.integers(-4, 5, 64)
    for eps in (0.0, 1e-6, 0.5):
        base = O.rms_norm(x, np.ones(64), eps)
        scaled = O.rms_norm(x, 2.0 ** a, eps)
        assert np.array_equal(scaled, base * 2.0 ** a)


def test_rms_norm_gamma_scales_each_feature_exactly():
    check_rms_norm_gamma_scales_each_feature_exactly()


def check_rms_norm_constant_row_closed_form():
    # a row of one value c has mean(x^2) = c^2, so the norm is c / sqrt(c^2 + eps):
    # with eps of the order of c^2 this separates eps inside the root from
    # eps added to the root (c / (|c| + eps))
    for c, eps in ((0.5, 0.25), (-2.0, 4.0), (3.0, 1e-6), (1e-3, 1e-6)):
        got = O.rms_norm(np.full((1, 32), c), np.ones(32), eps)
        assert np.allclose(got, c / np.sqrt(c * c + eps), rtol=1e-14, atol=0)
    # eps = 0: every row has unit RMS, sign kept
    got = O.rms_norm(np.full((1, 8), -7.0), np.ones(8), 0.0)
    assert np.array_equal(got, np.full((1, 8), -1.0))


def test_rms_norm_constant_row_closed_form():
    check_rms_norm_constant_row_closed_form()


def check_rms_norm_gamma_multiplies():
    # the gamma != 1 output divided by the gamma = 1 output is gamma itself
    # (not 1/gamma, not 1): one row with every entry nonzero
    g = np.random.default_rng(22)
    x = g.standard_normal((3, 48)) + 4.0
    gamma = 1.0 + g.random(48)
    ratio = O.rms_norm(x, gamma, 1e-6) / O.rms_norm(x, np.ones(48), 1e-6)
    assert np.allclose(ratio, np.broadcast_to(gamma, ratio.shape), rtol=1e-14, atol=0)


def test_rms_norm_gamma_multiplies():
    check_rms_norm_gamma_multiplies()


def check_layer_gamma_power_of_two_scales_the_norm_output():
    # the layer applies gamma to the normalised routed sum: with W_up = I, no
    # shared expert and gamma = 2^a per feature the output is the gamma = 1
    # output times 2^a exactly (bf16 rounding commutes with powers of two)
    d = dataclasses.replace(D, hidden=D.latent, T=8)
    wts, _, lg = tiny(6)
    wts = dict(wts, ws13=None, ws2=None, w_up=O.f64_to_bf16_bits(np.eye(d.latent)),
               w_down=O.f64_to_bf16_bits(np.eye(d.latent)))
    x = W.hidden_states(d, 6)
    a = np.random.default_rng(23).integers(-3, 4, d.latent)
    one = O.bf16_to_f64(O.latent_moe_forward(d, dict(wts, norm_w=None), x, lg))
    two = O.bf16_to_f64(O.latent_moe_forward(
        d, dict(wts, norm_w=O.f64_to_bf16_bits(2.0 ** a)), x, lg))
    assert np.array_equal(two, one * 2.0 ** a)


def test_layer_gamma_power_of_two_scales_the_norm_output():
    check_layer_gamma_power_of_two_scales_the_norm_output()
