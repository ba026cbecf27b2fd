"""Seeded synthetic inputs for the latent-MoE layer forward and its kernels.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no sigmoid, no top-k, no GEMM, no SituGLU).  It is the one
module that both the CPU oracle and the CUDA path consume.

Recipe (every tensor is reproducible on its own, so a caller can regenerate one
token's logits, one expert's weights or one row block of a dense matrix without
drawing the rest):

* every draw comes from ``numpy.random.default_rng(SeedSequence([seed, stream,
  index]))`` (PCG64), where ``stream`` names the tensor (constants below) and
  ``index`` is a token, an expert or a 64-row block;
* floats are drawn as float32 ``standard_normal`` and scaled; bf16 tensors are
  the round-to-nearest-even bf16 of those float32 draws (torch's conversion),
  carried as raw ``uint16`` bits;
* weights are N(0, 0.02^2) (the router weight N(0, 1/hidden), so that its
  logits are about N(0, 1)), hidden states N(0, 1), router logits N(0, 1), the
  selection bias N(0, 0.1^2) in float32, RMSNorm gamma = 1 (or 1 + N(0, 0.02^2)
  when ``gamma_noise`` is set);
* the routing-alone workload makes every 64th token (t % 64 == 0) a row of
  exactly tied logits (one N(0,1) value repeated E times);
* the skewed (Zipf s=1.1) prefill adds ``-1.1 * ln(r_e)`` to every token's logit
  for expert e, with r a seeded random permutation of 1..E, so a few experts get
  most tokens and many get none;
* the SituGLU workloads draw N(0, 3^2) and set 1% of entries (mask
  ``u < 0.01``) to +-40 to reach tanh saturation; the masked workload draws
  ``expert_num_tokens`` uniform in [0, T_max] and fills padded rows (input and
  output) with the sentinel bf16 pattern 0xDEAD.

Shapes follow the layer described on the pages (vLLM PR #50088, "[MoE]
Latent-MoE runner, fused MoE tail, SituGLU activation and single-group top-k
routing"; TensorRT-LLM PR #20541 "Kimi K3 MoE decode"): hidden 7168, latent
2048, 896 experts, top-16, expert intermediate 512, shared intermediate 4096.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

# --- stream identifiers (one per tensor) -----------------------------------
S_LOGITS, S_BIAS, S_ZIPF, S_W_DOWN, S_W13, S_W2 = 1, 2, 3, 4, 5, 6
S_WS13, S_WS2, S_NORM, S_W_UP, S_HIDDEN = 7, 8, 9, 10, 11
S_SITU, S_SITU_MASK, S_SITU_SIGN, S_COUNTS = 12, 13, 14, 15
S_W_ROUTER = 16
S_FP4_W13, S_FP4_W2 = 17, 18

ROW_BLOCK = 64          # rows per independent stream in dense matrices
SENTINEL = 0xDEAD       # bf16 bit pattern for padded rows
WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class LayerDims:
    """Dimensions and scalars of one latent-MoE layer call."""
    T: int
    hidden: int
    latent: int
    num_experts: int
    topk: int
    inter: int
    shared_inter: int
    n_group: int = 1
    topk_group: int = 1
    renormalize: int = 1
    routed_scaling_factor: float = 2.5
    beta: float = 4.0
    linear_beta: float = 8.0
    rms_eps: float = 1e-6


# The tiny layer (T=8, hidden 256, latent 128, 64 experts, top-4, d=128).
TINY = LayerDims(T=8, hidden=256, latent=128, num_experts=64, topk=4,
                 inter=128, shared_inter=128)
# The decode layer (T=8) and the prefill layer (T=4096) of the 896-expert model.
DECODE = LayerDims(T=8, hidden=7168, latent=2048, num_experts=896, topk=16,
                   inter=512, shared_inter=4096)
PREFILL = dataclasses.replace(DECODE, T=4096)

ROUTE_TOKENS = (1, 8, 16, 256, 4096, 16384)
ROUTE_E, ROUTE_K, ROUTE_RSF = 896, 16, 2.5


def _rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, stream, index]))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> raw bf16 bits (uint16), round to nearest even (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal_rows(seed: int, stream: int, rows: int, cols: int, std: float,
                 first_block: int = 0) -> np.ndarray:
    """[rows, cols] bf16 bits, one stream per 64-row block, drawn in parallel."""
    out = np.empty((rows, cols), dtype=np.uint16)
    nblk = (rows + ROW_BLOCK - 1) // ROW_BLOCK

    def fill(b: int) -> None:
        r0, r1 = b * ROW_BLOCK, min(rows, (b + 1) * ROW_BLOCK)
        g = _rng(seed, stream, first_block + b)
        x = g.standard_normal((r1 - r0, cols), dtype=np.float32) * np.float32(std)
        out[r0:r1] = to_bf16_bits(x)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(nblk)))
    return out


# --- layer weights -----------------------------------------------------------
def w_down(d: LayerDims, seed: int = 0) -> np.ndarray:
    """Latent down-projection weight, bf16 bits [latent, hidden]."""
    return _normal_rows(seed, S_W_DOWN, d.latent, d.hidden, WEIGHT_STD)


def w_up(d: LayerDims, seed: int = 0) -> np.ndarray:
    """Latent up-projection weight, bf16 bits [hidden, latent]."""
    return _normal_rows(seed, S_W_UP, d.hidden, d.latent, WEIGHT_STD)


def ws13(d: LayerDims, seed: int = 0) -> np.ndarray:
    """Shared expert gate|up weight, bf16 bits [2*shared_inter, hidden]."""
    return _normal_rows(seed, S_WS13, 2 * d.shared_inter, d.hidden, WEIGHT_STD)


def ws2(d: LayerDims, seed: int = 0) -> np.ndarray:
    """Shared expert down weight, bf16 bits [hidden, shared_inter]."""
    return _normal_rows(seed, S_WS2, d.hidden, d.shared_inter, WEIGHT_STD)


def w13_expert(d: LayerDims, e: int, seed: int = 0) -> np.ndarray:
    """Expert e gate|up weight, bf16 bits [2*inter, latent] (gate rows first)."""
    g = _rng(seed, S_W13, e)
    x = g.standard_normal((2 * d.inter, d.latent), dtype=np.float32)
    return to_bf16_bits(x * np.float32(WEIGHT_STD))


def w2_expert(d: LayerDims, e: int, seed: int = 0) -> np.ndarray:
    """Expert e down weight, bf16 bits [latent, inter]."""
    g = _rng(seed, S_W2, e)
    x = g.standard_normal((d.latent, d.inter), dtype=np.float32)
    return to_bf16_bits(x * np.float32(WEIGHT_STD))


def _stack_experts(d: LayerDims, fn, seed: int) -> np.ndarray:
    with ThreadPoolExecutor(_threads()) as ex:
        parts = list(ex.map(lambda e: fn(d, e, seed), range(d.num_experts)))
    return np.stack(parts)


def w13_all(d: LayerDims, seed: int = 0) -> np.ndarray:
    """All experts' gate|up weights, bf16 bits [E, 2*inter, latent]."""
    return _stack_experts(d, w13_expert, seed)


def w2_all(d: LayerDims, seed: int = 0) -> np.ndarray:
    """All experts' down weights, bf16 bits [E, latent, inter]."""
    return _stack_experts(d, w2_expert, seed)


def w_router(d: LayerDims, seed: int = 0) -> np.ndarray:
    """Router weight, bf16 bits [num_experts, hidden], N(0, 1/hidden): with N(0,1)
    hidden states the router logits are about N(0,1), like the logits of the
    routing workloads."""
    return _normal_rows(seed, S_W_ROUTER, d.num_experts, d.hidden, float(d.hidden) ** -0.5)


def norm_weight(d: LayerDims, seed: int = 0, gamma_noise: bool = False) -> np.ndarray:
    """RMSNorm gamma, bf16 bits [latent]; ones unless gamma_noise."""
    if not gamma_noise:
        return to_bf16_bits(np.ones(d.latent, dtype=np.float32))
    g = _rng(seed, S_NORM)
    x = 1.0 + g.standard_normal(d.latent, dtype=np.float32) * np.float32(WEIGHT_STD)
    return to_bf16_bits(x.astype(np.float32))


def score_bias(E: int, seed: int = 0) -> np.ndarray:
    """Selection-only correction bias, float32 [E], N(0, 0.1^2)."""
    g = _rng(seed, S_BIAS)
    return (g.standard_normal(E, dtype=np.float32) * np.float32(0.1)).astype(np.float32)


# --- activations and logits ---------------------------------------------------
def hidden_rows(d: LayerDims, tokens, seed: int = 0) -> np.ndarray:
    """Hidden states of the given token indices, bf16 bits [len(tokens), hidden]."""
    out = np.empty((len(tokens), d.hidden), dtype=np.uint16)
    for i, t in enumerate(tokens):
        g = _rng(seed, S_HIDDEN, int(t))
        out[i] = to_bf16_bits(g.standard_normal(d.hidden, dtype=np.float32))
    return out


def hidden_states(d: LayerDims, seed: int = 0) -> np.ndarray:
    """bf16 bits [T, hidden], N(0,1)."""
    with ThreadPoolExecutor(_threads()) as ex:
        chunks = np.array_split(np.arange(d.T), max(1, min(d.T, 64)))
        parts = list(ex.map(lambda c: hidden_rows(d, c, seed), chunks))
    return np.concatenate(parts, axis=0)


def zipf_offsets(E: int, seed: int = 0, s: float = 1.1) -> np.ndarray:
    """Per-expert logit offset -s*ln(r_e), r a random permutation of 1..E (float32)."""
    g = _rng(seed, S_ZIPF)
    r = g.permutation(E).astype(np.float64) + 1.0
    return (-s * np.log(r)).astype(np.float32)


def logits_rows(E: int, tokens, seed: int = 0, tie_every: int = 0,
                zipf: bool = False) -> np.ndarray:
    """Router logits of the given tokens, float32 [len(tokens), E], N(0,1).

    tie_every > 0 makes tokens with t % tie_every == 0 exactly tied rows.
    zipf adds the skew offsets (after the draw, in float32).
    """
    out = np.empty((len(tokens), E), dtype=np.float32)
    off = zipf_offsets(E, seed) if zipf else None
    for i, t in enumerate(tokens):
        g = _rng(seed, S_LOGITS, int(t))
        if tie_every and int(t) % tie_every == 0:
            out[i] = np.float32(g.standard_normal(dtype=np.float32))
        else:
            out[i] = g.standard_normal(E, dtype=np.float32)
        if off is not None:
            out[i] = (out[i] + off).astype(np.float32)
    return out


def router_logits(T: int, E: int, seed: int = 0, tie_every: int = 0,
                  zipf: bool = False) -> np.ndarray:
    """float32 [T, E]."""
    with ThreadPoolExecutor(_threads()) as ex:
        chunks = np.array_split(np.arange(T), max(1, min(T, 64)))
        parts = list(ex.map(lambda c: logits_rows(E, c, seed, tie_every, zipf), chunks))
    return np.concatenate(parts, axis=0)


def layer_weights(d: LayerDims, seed: int = 0, gamma_noise: bool = False) -> dict:
    """Every weight of the layer as bf16 bits (bias as float32), in ABI layout."""
    return dict(
        w_down=w_down(d, seed), w13=w13_all(d, seed), w2=w2_all(d, seed),
        ws13=ws13(d, seed), ws2=ws2(d, seed),
        norm_w=norm_weight(d, seed, gamma_noise), w_up=w_up(d, seed),
        bias=score_bias(d.num_experts, seed),
    )


# --- SituGLU workloads -------------------------------------------------------
def situ_input(rows: int, two_d: int, seed: int = 0, first_block: int = 0) -> np.ndarray:
    """bf16 bits [rows, two_d], N(0, 3^2) with 1% of entries set to +-40."""
    out = np.empty((rows, two_d), dtype=np.uint16)
    nblk = (rows + ROW_BLOCK - 1) // ROW_BLOCK

    def fill(b: int) -> None:
        r0, r1 = b * ROW_BLOCK, min(rows, (b + 1) * ROW_BLOCK)
        g = _rng(seed, S_SITU, first_block + b)
        x = g.standard_normal((r1 - r0, two_d), dtype=np.float32) * np.float32(3.0)
        m = g.random((r1 - r0, two_d), dtype=np.float32) < np.float32(0.01)
        sign = g.integers(0, 2, size=(r1 - r0, two_d)).astype(np.float32) * 2.0 - 1.0
        x = np.where(m, np.float32(40.0) * sign, x).astype(np.float32)
        out[r0:r1] = to_bf16_bits(x)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(nblk)))
    return out


def masked_counts(E: int, T_max: int, seed: int = 0) -> np.ndarray:
    """expert_num_tokens, int32 [E], uniform in [0, T_max]."""
    g = _rng(seed, S_COUNTS)
    return g.integers(0, T_max + 1, size=E).astype(np.int32)


def masked_situ_input(E: int, T_max: int, two_d: int, seed: int = 0):
    """(input bits [E, T_max, two_d] with sentinel padding, counts [E])."""
    counts = masked_counts(E, T_max, seed)
    x = situ_input(E * T_max, two_d, seed).reshape(E, T_max, two_d)
    for e in range(E):
        x[e, counts[e]:] = SENTINEL
    return x, counts


def sentinel_like(shape) -> np.ndarray:
    return np.full(shape, SENTINEL, dtype=np.uint16)


def expert_chunks(d: LayerDims, name: str, seed: int = 0, chunk: int = 64):
    """Yield (e0, e1, bits[e1-e0, ...]) blocks of the stacked expert weights.

    ``name`` is "w13" ([2*inter, latent] per expert) or "w2" ([latent, inter]).
    Lets a caller fill a device tensor block by block without holding every
    expert on the host.
    """
    fn = {"w13": w13_expert, "w2": w2_expert}[name]
    for e0 in range(0, d.num_experts, chunk):
        e1 = min(d.num_experts, e0 + chunk)
        with ThreadPoolExecutor(_threads()) as ex:
            parts = list(ex.map(lambda e: fn(d, e, seed), range(e0, e1)))
        yield e0, e1, np.stack(parts)


# --- block-scaled (MXFP4) expert weights ---------------------------------------
# Each expert matrix [rows, K] is stored as 4-bit codes, two per byte (element
# 2i in the low nibble of byte i, element 2i+1 in the high nibble), and one
# 8-bit power-of-two scale exponent per 32 consecutive elements of a row.  The
# generator draws the codes and the exponents directly (no quantisation of
# float weights): codes uniform over the 16 patterns, exponents uniform in
# [118, 120], so that the weights have magnitudes like the bf16 N(0, 0.02^2)
# weights (the largest code value, 6, times 2^-8 is 0.023).
MXFP4_BLOCK = 32
MXFP4_SCALE_LO, MXFP4_SCALE_HI = 118, 120


def mxfp4_matrix(seed: int, stream: int, index: int, rows: int, K: int):
    """(packed codes uint8 [rows, K/2], scale exponents uint8 [rows, K/32])."""
    g = _rng(seed, stream, index)
    codes = g.integers(0, 16, size=(rows, K), dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))).astype(np.uint8)
    scales = g.integers(MXFP4_SCALE_LO, MXFP4_SCALE_HI + 1, size=(rows, K // MXFP4_BLOCK),
                        dtype=np.uint8)
    return packed, scales


def mxfp4_w13_expert(d: LayerDims, e: int, seed: int = 0):
    """Expert e gate|up weight in MXFP4: [2*inter, latent/2] codes, [2*inter, latent/32] scales."""
    return mxfp4_matrix(seed, S_FP4_W13, e, 2 * d.inter, d.latent)


def mxfp4_w2_expert(d: LayerDims, e: int, seed: int = 0):
    """Expert e down weight in MXFP4: [latent, inter/2] codes, [latent, inter/32] scales."""
    return mxfp4_matrix(seed, S_FP4_W2, e, d.latent, d.inter)


def mxfp4_experts(d: LayerDims, seed: int = 0) -> dict:
    """Every expert's MXFP4 weights stacked: w13_q [E, 2d, L/2], w13_s [E, 2d, L/32],
    w2_q [E, L, d/2], w2_s [E, L, d/32]."""
    with ThreadPoolExecutor(_threads()) as ex:
        a = list(ex.map(lambda e: mxfp4_w13_expert(d, e, seed), range(d.num_experts)))
        b = list(ex.map(lambda e: mxfp4_w2_expert(d, e, seed), range(d.num_experts)))
    return dict(w13_q=np.stack([x[0] for x in a]), w13_s=np.stack([x[1] for x in a]),
                w2_q=np.stack([x[0] for x in b]), w2_s=np.stack([x[1] for x in b]))
