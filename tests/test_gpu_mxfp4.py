"""GPU parity of the MXFP4 (block-scaled E2M1) routed-expert path against the
oracle.

Dequantization: bit-exact (every MXFP4 weight with a scale exponent in 2..252
is a bf16 value; exponent 0 too for these magnitudes; 255 gives NaN).
Expert stages (4-bit weights read directly; experts with more than 16 tokens
on the tensor-core GEMMs from a compact bf16 copy): each stage fed the GPU's
own inputs against the oracle's stage on the dequantized weights, to the
stage bounds the bf16 path meets (tests/gpu_util.assert_stage_close,
assert_gemm_situ_close).  Layer: within max(2e-2 rms, 2 bf16 steps at the
largest addend of the final sum) everywhere, the literal 2e-2 rms bound
asserted on the tiny layers.  With inter % 128 != 0 above 128 tokens the
MXFP4 forward runs the bf16 kernels on weights it dequantizes, so its output
is bit-identical to latent_moe_forward on lmoe_dequant_mxfp4's weights.
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


def dev_u8(a: np.ndarray) -> torch.Tensor:
    from tests.gpu_util import DEV
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def device_mxfp4(Q: dict) -> dict:
    return {k: dev_u8(v) for k, v in Q.items()}


def _dequant_gpu(packed, scales):
    from tests.gpu_util import DEV, host_bits
    rows, K = packed.shape[0], packed.shape[1] * 2
    out = torch.empty((rows, K), dtype=torch.bfloat16, device=DEV)
    lm.lmoe_dequant_mxfp4(dev_u8(packed), dev_u8(scales), out)
    torch.cuda.synchronize()
    return host_bits(out)


@pytest.mark.parametrize("rows,K", [(1, 32), (37, 96), (1000, 2048), (4096, 512),
                                    (3, 32 * 700), (5, 32 * 1031)])
def test_dequant_bit_exact(rows, K):
    g = np.random.default_rng(rows + K)
    packed = g.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = g.integers(2, 253, size=(rows, K // 32), dtype=np.uint8)
    got = _dequant_gpu(packed, scales)
    assert np.array_equal(got, O.mxfp4_as_bf16_bits(packed, scales))


def test_dequant_special_scales():
    # exponent 0 (2^-127: the products are bf16 subnormals, still exact),
    # 127 (1.0) and 255 (NaN), every code in every block
    codes = np.arange(32, dtype=np.uint8) % 16
    packed = np.tile((codes[0::2] | (codes[1::2] << 4)).astype(np.uint8), (3, 1))
    scales = np.array([[0], [127], [255]], dtype=np.uint8)
    got = O.bf16_to_f64(_dequant_gpu(packed, scales))
    ref = O.dequant_mxfp4(packed, scales)
    assert np.array_equal(got[:2], ref[:2])
    assert np.isnan(got[2]).all()


def test_dequant_full_size_experts():
    # the decode layer's expert matrices, 64 experts of each
    d = W.DECODE
    for fn in (W.mxfp4_w13_expert, W.mxfp4_w2_expert):
        parts = [fn(d, e) for e in range(0, d.num_experts, 14)]
        packed = np.concatenate([p[0] for p in parts])
        scales = np.concatenate([p[1] for p in parts])
        assert np.array_equal(_dequant_gpu(packed, scales), O.mxfp4_as_bf16_bits(packed, scales))


def run_mxfp4(d, wdev, qdev, x_bits, logits, keep_ws=False):
    from tests.gpu_util import DEV, dev_bf16, dev_f32
    out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes_mxfp4(d), dtype=torch.uint8, device=DEV)
    lm.latent_moe_forward_mxfp4(d, wdev, qdev, dev_bf16(x_bits), dev_f32(logits), out, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_error() == 0
    return (out, ws) if keep_ws else out


def check_expert_stages(d, Qfn, toks, ws, logits, bias):
    """GEMM1 + SituGLU and GEMM2 of the (token, slot) rows of `toks`, each from
    the GPU's own stage inputs (A, act) against the oracle on the dequantized
    weights."""
    from tests.gpu_util import workspace_view, assert_gemm_situ_close, assert_stage_close
    f = O.bf16_to_f64
    v = workspace_view(lm, d, ws)
    ids, _ = O.route(logits[toks], bias, d.topk, d.routed_scaling_factor, d.renormalize)
    rr = v["row_of"][toks].ravel()
    deq = {}

    def w(name, e):
        if (name, e) not in deq:
            q, s = Qfn(name, int(e))
            deq[(name, e)] = O.mxfp4_as_bf16_bits(q, s)
        return deq[(name, e)]

    Gref = np.stack([O.linear_bf16(f(v["A"][r:r + 1]), w("w13", e))[0]
                     for r, e in zip(rr, ids.ravel())])
    act = f(v["act"][rr])
    res = [assert_gemm_situ_close(act, Gref, d.beta, d.linear_beta, "fp4 gemm1+situ")]
    Yref = np.stack([O.linear_bf16(act[i:i + 1], w("w2", e))[0]
                     for i, e in enumerate(ids.ravel())])
    res.append(assert_stage_close(f(v["Y"][rr]), Yref, "fp4 gemm2"))
    return res


def _tiny(d, seed):
    from tests.gpu_util import weights_to_device
    wts = W.layer_weights(d, seed)
    Q = W.mxfp4_experts(d, seed)
    wdev = weights_to_device(dict(wts, w13=None, w2=None))
    return wts, Q, wdev, device_mxfp4(Q)


def tiny_case(d, seed=0, literal=None, zipf=False):
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale, assert_layer_literal
    wts, Q, wdev, qdev = _tiny(d, seed)
    x = W.hidden_states(d, seed)
    lg = W.router_logits(d.T, d.num_experts, seed, zipf=zipf)
    out, ws = run_mxfp4(d, wdev, qdev, x, lg, keep_ws=True)
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wts, Q, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wts["w_up"]))
    if literal:
        assert_layer_literal(got, ref, literal, TOL)
    toks = list(range(min(d.T, 24))) + [d.T - 1]
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]), toks, ws, lg,
                        wts["bias"])


def test_mxfp4_tiny_layer():
    tiny_case(W.TINY, literal="MXFP4 tiny layer T=8")


@pytest.mark.parametrize("T", [1, 3, 17, 100, 128, 129, 200, 256, 257, 300])
def test_mxfp4_tiny_layer_token_counts(T):
    # the 4-bit kernels (heavy experts split off to the tensor-core GEMMs
    # above 16 tokens; the decode-sized dense GEMMs up to 128, the one-block
    # permutation up to 256, three passes above)
    tiny_case(dataclasses.replace(W.TINY, T=T), seed=T)


@pytest.mark.parametrize("variant", ["ragged", "crowded", "all_heavy", "wide_k1", "wide_k2",
                                     "max_experts"])
def test_mxfp4_layer_shapes(variant):
    d = W.TINY
    if variant == "ragged":
        # latent 384 (192-byte code rows: 64-byte swizzle), inter 192 (96-byte
        # rows: 32-byte swizzle, 6 scale blocks), 40 experts
        d = dataclasses.replace(d, T=5, hidden=384, latent=384, inter=192, shared_inter=320,
                                num_experts=40, topk=6)
    elif variant == "crowded":
        # 128 tokens over 16 experts: ~32 rows an expert, several passes of up
        # to 8 tokens over the same strip; the experts with more than 16 run
        # on the tensor-core GEMMs, the others on the 4-bit kernels
        d = dataclasses.replace(d, T=128, num_experts=16, topk=4)
    elif variant == "all_heavy":
        # 64 rows for each of 4 experts: all on the tensor-core GEMMs, the
        # 4-bit kernels get no expert
        d = dataclasses.replace(d, T=128, num_experts=4, topk=2)
    elif variant == "wide_k1":
        # GEMM1 over latent 4096 (the largest the MXFP4 forward takes): one
        # token a stage, two stages
        d = dataclasses.replace(d, T=4, latent=4096, inter=256, num_experts=4, topk=2)
    elif variant == "wide_k2":
        # GEMM2 over inter 4096
        d = dataclasses.replace(d, T=4, latent=128, inter=4096, num_experts=4, topk=2)
    elif variant == "max_experts":
        d = dataclasses.replace(d, T=8, num_experts=1024, topk=32)
    tiny_case(d, seed=7)


@pytest.mark.parametrize("log2_scale", [-60, 40])
def test_mxfp4_decode_input_scale_extremes(log2_scale):
    # the 4-bit decode kernels scale each token's input rows by a power of two
    # into the f16 range; hidden states scaled by 2^-60 or 2^40 (exact in
    # bf16) move the expert inputs far outside it, with the stages still
    # matching the oracle fed the GPU's own inputs
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale
    d = dataclasses.replace(W.TINY, T=6)
    wts, Q, wdev, qdev = _tiny(d, 9)
    x = O.f64_to_bf16_bits(O.bf16_to_f64(W.hidden_states(d, 9)) * 2.0 ** log2_scale)
    lg = W.router_logits(d.T, d.num_experts, 9)
    out, ws = run_mxfp4(d, wdev, qdev, x, lg, keep_ws=True)
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wts, Q, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert np.isfinite(got).all()
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wts["w_up"]))
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]), list(range(d.T)), ws,
                        lg, wts["bias"])


@pytest.mark.parametrize("T", [8, 300])
def test_mxfp4_zero_scale_blocks(T):
    # scale exponent 0 (2^-127: the weights of the block are bf16/fp32
    # subnormals) on a seeded 5% of the blocks: the 4-bit decode kernels take
    # their exact scale path for such items, the prefill path dequantizes them
    # exactly; both against the oracle
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale
    d = dataclasses.replace(W.TINY, T=T)
    wts = W.layer_weights(d, 12)
    Q = W.mxfp4_experts(d, 12)
    g = np.random.default_rng(12)
    for name in ("w13_s", "w2_s"):
        Q[name] = Q[name].copy()
        Q[name][g.random(Q[name].shape) < 0.05] = 0
    from tests.gpu_util import weights_to_device
    wdev = weights_to_device(dict(wts, w13=None, w2=None))
    x = W.hidden_states(d, 12)
    lg = W.router_logits(d.T, d.num_experts, 12)
    out, ws = run_mxfp4(d, wdev, device_mxfp4(Q), x, lg, keep_ws=True)
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wts, Q, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wts["w_up"]))
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]), list(range(min(T, 24))),
                        ws, lg, wts["bias"])


def test_mxfp4_prefill_is_the_bf16_forward_on_dequantized_weights():
    # inter % 128 != 0 above 128 tokens: the same kernels as
    # latent_moe_forward once the weights are dequantized, so bit-identical
    # outputs
    from tests.gpu_util import DEV, dev_bf16, dev_f32
    d = dataclasses.replace(W.TINY, T=300, inter=192)
    wts, Q, wdev, qdev = _tiny(d, 4)
    x = W.hidden_states(d, 4)
    lg = W.router_logits(d.T, d.num_experts, 4)
    out = run_mxfp4(d, wdev, qdev, x, lg)
    w13 = torch.empty((d.num_experts, 2 * d.inter, d.latent), dtype=torch.bfloat16, device=DEV)
    w2 = torch.empty((d.num_experts, d.latent, d.inter), dtype=torch.bfloat16, device=DEV)
    lm.lmoe_dequant_mxfp4(qdev["w13_q"], qdev["w13_s"], w13)
    lm.lmoe_dequant_mxfp4(qdev["w2_q"], qdev["w2_s"], w2)
    ref = torch.empty_like(out)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    lm.latent_moe_forward(d, dict(wdev, w13=w13, w2=w2), dev_bf16(x), dev_f32(lg), ref, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.fixture(scope="module")
def decode_full():
    """The decode layer (T=8, 896 experts, top-16) with MXFP4 experts."""
    from tests.gpu_util import device_layer_weights, oracle_layer_weights
    d = W.DECODE
    wdev = device_layer_weights(d, 0)
    wdev["w13"] = wdev["w2"] = None
    Q = W.mxfp4_experts(d, 0)
    return d, wdev, device_mxfp4(Q), oracle_layer_weights(d, 0), Q


def test_mxfp4_decode_full_size(decode_full):
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale, record_literal
    d, wdev, qdev, wor, Q = decode_full
    x = W.hidden_states(d, 0)
    lg = W.router_logits(d.T, d.num_experts, 0)
    out, ws = run_mxfp4(d, wdev, qdev, x, lg, keep_ws=True)
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wor, Q, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wor["w_up"]))
    record_literal(got, ref, "MXFP4 decode layer T=8", TOL)
    # every (token, slot) row of both expert stages
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]), list(range(d.T)), ws,
                        lg, wor["bias"])


def test_mxfp4_decode_skewed_full_size(decode_full):
    # 64 tokens of the 896-expert layer with Zipf-skewed routing: the experts
    # most tokens choose get more than 16 rows and run on the tensor-core
    # GEMMs from a compact bf16 copy, the rest on the 4-bit kernels
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale, record_literal
    d, wdev, qdev, wor, Q = decode_full
    d = dataclasses.replace(d, T=64)
    x = W.hidden_states(d, 5)
    lg = W.router_logits(d.T, d.num_experts, 5, zipf=True)
    ids, _ = O.route(lg, wor["bias"], d.topk, d.routed_scaling_factor, d.renormalize)
    counts = np.bincount(ids.ravel(), minlength=d.num_experts)
    assert (counts > 16).sum() >= 4 and ((counts > 0) & (counts <= 16)).sum() >= 4
    out, ws = run_mxfp4(d, wdev, qdev, x, lg, keep_ws=True)
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wor, Q, x, lg, intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wor["w_up"]))
    record_literal(got, ref, "MXFP4 decode layer T=64 Zipf", TOL)
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]),
                        list(range(12)) + [d.T - 1], ws, lg, wor["bias"])


def test_mxfp4_prefill_zipf_sampled(decode_full):
    # the prefill workload (T = 4096, Zipf-skewed routing) with MXFP4 experts:
    # the experts with more than 16 tokens on the tensor-core GEMMs from their
    # bf16 copies, the others on the 4-bit kernels; a seeded sample of tokens
    # plus the first token of every used expert against the oracle, and the
    # expert stages of the first token of every used expert (both paths)
    from tests.gpu_util import host_bits, assert_layer_close, addend_scale, record_literal
    d, wdev, qdev, wor, Q = decode_full
    d = dataclasses.replace(d, T=4096)
    x = W.hidden_states(d, 0)
    lg = W.router_logits(d.T, d.num_experts, 0, zipf=True)
    ids, _ = O.route(lg, wor["bias"], d.topk, d.routed_scaling_factor, d.renormalize)
    counts = np.bincount(ids.ravel(), minlength=d.num_experts)
    assert (counts > 16).sum() >= 4 and ((counts > 0) & (counts <= 16)).sum() >= 4
    out, ws = run_mxfp4(d, wdev, qdev, x, lg, keep_ws=True)
    first_of_expert = [int(np.argmax((ids == e).any(axis=1))) for e in np.unique(ids)]
    toks = np.unique(np.concatenate([[0, d.T - 1], first_of_expert,
                                     np.random.default_rng(4).choice(d.T, 96, replace=False)]))
    ref_bits, mid = O.latent_moe_forward_mxfp4(d, wor, Q, x[toks], lg[toks], intermediates=True)
    ref = O.bf16_to_f64(ref_bits)
    got = O.bf16_to_f64(host_bits(out))[toks]
    assert_layer_close(got, ref, TOL, scale=addend_scale(ref, mid, wor["w_up"]))
    record_literal(got, ref, f"MXFP4 prefill layer T=4096 Zipf ({len(toks)} sampled tokens)", TOL)
    check_expert_stages(d, lambda n, e: (Q[n + "_q"][e], Q[n + "_s"][e]),
                        sorted(set(first_of_expert)), ws, lg, wor["bias"])
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("T,zipf", [(8, False), (64, True)])
def test_mxfp4_decode_graph_replay(decode_full, T, zipf):
    # the decode forward captured in a CUDA graph reproduces the eager output
    # bit for bit (no host state decides anything at replay; at T = 64 the
    # device splits the experts between the two expert paths)
    from tests.gpu_util import DEV, dev_bf16, dev_f32
    d, wdev, qdev, _, _ = decode_full
    d = dataclasses.replace(d, T=T)
    x = dev_bf16(W.hidden_states(d, 0))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, 0, zipf=zipf))
    out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes_mxfp4(d), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lm.latent_moe_forward_mxfp4(d, wdev, qdev, x, lg, out, ws, stream=s)
    s.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lm.latent_moe_forward_mxfp4(d, wdev, qdev, x, lg, out, ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
