"""CPU oracle of the latent-MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 NumPy restatement of what the layer computes, written from
three pages:

* [vLLM-50088]  vLLM PR #50088, "[MoE] Latent-MoE runner, fused MoE tail,
  SituGLU activation and single-group top-k routing" (commits 1-7);
* [TRTLLM-20541] TensorRT-LLM PR #20541, "Kimi K3 MoE decode: router GEMM and
  routing kernel on a router stream" (Commit 1, Commit 2);
* [vLLM-runner] vLLM API page "vllm.models.kimi_k3.amd.latent_moe_runner"
  (ROCmLatentMoERunner: forward, _fused_forward, _shard_up_proj_tail).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its reference arm) may import this module.  The CUDA library never imports,
links or calls it, and it shares no code, constant table or helper with the
CUDA sources: the two meet only through the seeded inputs of ``workloads``.

Precision.  Floating point is float64, except where the pages fix fp32 (the
router logits and the sigmoid score that decides the top-k selection) and where
the layer's buffers are bf16: every stage output that the layer stores in bf16
(Z, G, act, Y, N, the shared expert's G and act, Sh, out) is rounded here to
bf16 with round-to-nearest-even, straight from float64.

Readings where the pages leave a step open (each is listed with its reason in
the design notes):
  R-1 gate = first d columns of the 2d-wide GEMM1 output, up = last d;
  R-2 top-k ids are ordered by descending selection key, exact ties -> lower
      expert index first;
  R-3 rows of one expert in the permuted layout are in ascending token order;
  R-4 weights = s / sum(s) (no epsilon) then * routed_scaling_factor, once;
  R-5 the fp32 sigmoid that decides the selection is the fixed sequence of
      IEEE fp32 operations in ``sigmoid_f32`` (own exp; no fused multiply-add);
  R-6 RMSNorm: x * 1/sqrt(mean(x^2) + eps) * gamma, over the latent axis;
  R-7 bf16 at stage boundaries, fp32 routing, float64 here for everything else;
  R-8 the shared expert is a SituGLU MLP on the original hidden states, with
      the same beta / linear_beta, unscaled;
  R-10 no linear biases;
  R-19 router GEMM: fp32 logits = X W_router^T from a bf16 [E, H] weight,
       rounded once to float32;
  R-20 MXFP4 experts: E2M1 codes two per byte (element 2i in the low nibble),
       one scale exponent (bias 127) per 32 elements along K;
  R-11 expert_num_tokens outside [0, T_max] is clamped.

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
(closed forms, limits, brute force, library routines in higher precision,
invariants).  None is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bf16 helpers (the layer's storage type)
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Raw bf16 bits (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even).

    bf16 keeps 8 significant bits; below 2^-126 its spacing is fixed at 2^-133.
    The value is snapped to the bf16 grid of its binade with np.rint (which
    rounds half to even).  Results past the largest bf16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
        expo = np.maximum(e - 1, -126)          # binade exponent (floor log2|x|)
        spacing = np.ldexp(1.0, expo - 7)
        y = np.rint(x / spacing) * spacing
        y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, x), y)
        y = np.where(np.isfinite(x), y, x)
    return y


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> raw bf16 bits, rounding to nearest even first."""
    y = round_bf16(x).astype(np.float32)        # exact: y is on the bf16 grid
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# R-5: the fp32 sigmoid that decides the top-k selection
# ---------------------------------------------------------------------------
# [vLLM-50088] commit 4 keeps DeepSeekV3 routing in FP32.  For expert indices to
# be exactly reproducible the fp32 value of sigmoid(x) must be fixed to the
# bit, so it is defined as this sequence of IEEE-754 fp32 operations, each
# rounded to nearest even (no fused multiply-add):
#   y   = min(max(-x, -87), 88)
#   n   = rint(y * LOG2E)                       (Cody & Waite range reduction
#   r   = (y - n*LN2_HI) - n*LN2_LO              with a 9-bit high part of ln 2)
#   p   = 1 + r(1 + r(1/2 + r(1/6 + ... + r/5040)))   (Taylor, degree 7, Horner)
#   E   = p * 2^n                                (2^n built from exponent bits)
#   s   = 1 / (1 + E)
# The constants are the float32 values nearest to log2(e), 355/512,
# ln2 - 355/512 and 1/k!; tests check each against exact arithmetic.
_F = np.float32
LOG2E = _F(float.fromhex("0x1.715476p+0"))
LN2_HI = _F(float.fromhex("0x1.63p-1"))          # 355/512, 9 significant bits
LN2_LO = _F(float.fromhex("-0x1.bd0106p-13"))    # ln2 - 355/512
INV_FACT = tuple(_F(float.fromhex(h)) for h in (
    "0x1p+0",        # 1/1!
    "0x1p-1",        # 1/2!
    "0x1.555556p-3",  # 1/3!
    "0x1.555556p-5",  # 1/4!
    "0x1.111112p-7",  # 1/5!
    "0x1.6c16c2p-10",  # 1/6!
    "0x1.a01a02p-13",  # 1/7!
))


def exp_f32(y: np.ndarray) -> np.ndarray:
    """e^y in fp32 for y in [-87, 88], by the fixed operation sequence above."""
    y = np.asarray(y, dtype=np.float32)
    n = np.rint(y * LOG2E)                        # float32, integral
    r = (y - n * LN2_HI) - n * LN2_LO
    p = INV_FACT[6]
    for c in INV_FACT[5::-1]:                     # 1/6!, 1/5!, ..., 1/1!
        p = p * r + c
    p = p * r + _F(1.0)                           # the 1/0! term
    two_n = ((n.astype(np.int32) + np.int32(127)) << np.int32(23)).view(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_f32(x: np.ndarray) -> np.ndarray:
    """sigmoid(x) = 1/(1+e^-x) in fp32, bit-for-bit as defined for R-5."""
    x = np.asarray(x, dtype=np.float32)
    y = np.minimum(np.maximum(-x, _F(-87.0)), _F(88.0))
    with np.errstate(over="ignore", under="ignore"):
        return (_F(1.0) / (_F(1.0) + exp_f32(y))).astype(np.float32)


# ---------------------------------------------------------------------------
# Step 1: single-group sigmoid top-k routing
# ---------------------------------------------------------------------------


def route(logits: np.ndarray, bias, topk: int, routed_scaling_factor: float,
          renormalize: int = 1, n_group: int = 1, topk_group: int = 1):
    """DeepSeekV3-style routing with one group.

    [vLLM-50088] commit 1: with n_group == 1 and topk_group == 1 grouped top-k is
    plain top-k over all experts.  Commit 4: the scores are sigmoid of FP32
    logits; the e_score_correction_bias is added for the selection only; the
    weights come from the unbiased scores, are renormalised and scaled by the
    routed scaling factor.  Ties in the selection key go to the lower expert
    index (R-2); the ids are returned in selection order.

    Returns (ids int32 [T, topk], weights float64 [T, topk]).
    """
    if n_group != 1 or topk_group != 1:
        raise NotImplementedError("only the single-group case is defined here")
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= topk <= E:
        raise ValueError("topk out of range")
    s = sigmoid_f32(logits)                                   # fp32 scores
    b = np.zeros(E, np.float32) if bias is None else np.asarray(bias, np.float32)
    key = (s + b[None, :]).astype(np.float32)                 # fp32 selection key
    ids = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        order = np.argsort(-key[t], kind="stable")            # desc, ties: low idx
        ids[t] = order[:topk]
    w = np.take_along_axis(s, ids.astype(np.int64), axis=1).astype(np.float64)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    w = w * float(routed_scaling_factor)
    return ids, w


# ---------------------------------------------------------------------------
# SituGLU
# ---------------------------------------------------------------------------


def situ(gate: np.ndarray, up: np.ndarray, beta: float, linear_beta: float) -> np.ndarray:
    """SituGLU, [vLLM-50088] commit 2 (and commit 3 for linear_beta <= 0):

    gate_out = beta * tanh(gate / beta) * sigmoid(gate)
    up_out   = linear_beta * tanh(up / linear_beta)  if linear_beta > 0 else up
    out      = gate_out * up_out
    """
    if not beta > 0 or not np.isfinite(beta):
        raise ValueError("beta is required and must be > 0")
    g = np.asarray(gate, dtype=np.float64)
    u = np.asarray(up, dtype=np.float64)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    gate_out = beta * np.tanh(g / beta) * sig
    up_out = linear_beta * np.tanh(u / linear_beta) if linear_beta > 0 else u
    return gate_out * up_out


def situ_and_mul(x_bits: np.ndarray, beta: float, linear_beta: float) -> np.ndarray:
    """Dense [..., 2d] -> [..., d] (bf16 bits in and out), [vLLM-50088] commit 2.

    Gate is the first half of the last axis, up the second half (R-1).
    """
    x = bf16_to_f64(x_bits)
    d = x.shape[-1] // 2
    return f64_to_bf16_bits(situ(x[..., :d], x[..., d:], beta, linear_beta))


def masked_situ_and_mul(x_bits: np.ndarray, expert_num_tokens: np.ndarray,
                        out_init_bits: np.ndarray, beta: float,
                        linear_beta: float) -> np.ndarray:
    """Batched [E, T_max, 2d] -> [E, T_max, d], [vLLM-50088] commits 2 and 3.

    Row t of expert e is computed only if t < expert_num_tokens[e] (clamped to
    [0, T_max], R-11); every other output row keeps its previous contents.
    """
    E, T_max, _ = x_bits.shape
    out = np.array(out_init_bits, dtype=np.uint16, copy=True)
    for e in range(E):
        n = int(min(max(int(expert_num_tokens[e]), 0), T_max))
        if n:
            out[e, :n] = situ_and_mul(x_bits[e, :n], beta, linear_beta)
    return out


# ---------------------------------------------------------------------------
# Step 3: token permutation into the expert-major layout
# ---------------------------------------------------------------------------


def permute(ids: np.ndarray, num_experts: int):
    """Group (token, slot) pairs by expert, tokens ascending inside an expert.

    The batched MoE layout with expert_num_tokens of [vLLM-50088] commits 2-3,
    stored compactly: expert e owns rows offsets[e] .. offsets[e+1]-1.

    Returns (expert_num_tokens int32 [E], offsets int32 [E+1],
             row_of int32 [T, k], tok_of_row int32 [T*k]).
    """
    T, k = ids.shape
    counts = np.zeros(num_experts, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[ids[t, j]] += 1
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    for e in range(num_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    nxt = offsets[:-1].copy()
    row_of = np.empty((T, k), dtype=np.int64)
    tok_of_row = np.empty(T * k, dtype=np.int64)
    for t in range(T):                       # ascending token order (R-3)
        for j in range(k):
            e = ids[t, j]
            row_of[t, j] = nxt[e]
            tok_of_row[nxt[e]] = t
            nxt[e] += 1
    return (counts.astype(np.int32), offsets.astype(np.int32),
            row_of.astype(np.int32), tok_of_row.astype(np.int32))


# ---------------------------------------------------------------------------
# GEMM stage and RMSNorm
# ---------------------------------------------------------------------------


def linear_bf16(x: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16(x @ W^T) for bf16 weight bits W [out, in]; float64 products, no bias."""
    return round_bf16(np.asarray(x, np.float64) @ bf16_to_f64(w_bits).T)


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis (R-6).

    The norm of the routed output transform, [vLLM-runner] _shard_up_proj_tail
    (``transform.norm(latent)``), applied after the routed sum per
    [vLLM-50088] commit 7.
    """
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma


def router_gemm(hidden_bits: np.ndarray, w_router_bits: np.ndarray) -> np.ndarray:
    """Router logits, float32 [T, E] = fp32(X W_router^T) for bf16 hidden states
    X [T, H] and a bf16 router weight W_router [E, H] (PyTorch Linear layout, no
    bias).

    [TRTLLM-20541] Commit 2: the router GEMM runs on the hidden states ahead of
    the routing kernel (its own stream, or fused with the latent down
    projection in the "fused router+down projection" configuration);
    [vLLM-50088] commit 4: DeepSeekV3 routing takes FP32 logits.  The product is
    formed in float64 and rounded once to float32.
    """
    X = bf16_to_f64(hidden_bits)
    Wr = bf16_to_f64(w_router_bits)
    return (X @ Wr.T).astype(np.float32)


# ---------------------------------------------------------------------------
# Block-scaled (MXFP4) expert weights
# ---------------------------------------------------------------------------
# [vLLM-50088] commits 4-5 and [TRTLLM-20541] run the routed experts of this
# layer with MXFP4 weights (the TRTLLM-Gen MXE4M3 x MXE2M1 path), with SituGLU
# acting on the dequantized gate/up.  An MXFP4 value is a 4-bit float with one
# sign bit, two exponent bits (bias 1) and one mantissa bit (E2M1), times a
# power of two shared by each block of 32 consecutive elements (an unsigned
# 8-bit exponent, bias 127).  Storage read here (R-20): two codes per byte,
# element 2i in the low nibble; scales [rows, K/32].


def e2m1_value(code: np.ndarray) -> np.ndarray:
    """float64 value of 4-bit E2M1 codes (bit 3 sign, bits 2-1 exponent, bit 0
    mantissa): exponent field 0 is subnormal (mantissa * 1/2), otherwise
    2^(e-1) * (1 + mantissa/2)."""
    code = np.asarray(code).astype(np.int64)
    sign = np.where(code & 8, -1.0, 1.0)
    e = (code >> 1) & 3
    m = code & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m * 0.5, (e - 1).astype(np.int64)))
    return sign * mag


def e8m0_value(s: np.ndarray) -> np.ndarray:
    """float64 value of unsigned 8-bit E8M0 scale exponents: 2^(s - 127), and
    NaN for 255 (the format's one non-number)."""
    s = np.asarray(s).astype(np.int64)
    return np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [rows, K/2] -> 4-bit codes [rows, K]: element 2i is the low nibble
    of byte i, element 2i+1 its high nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = packed & np.uint8(15)
    codes[..., 1::2] = packed >> np.uint8(4)
    return codes


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 [rows, K] from packed codes [rows, K/2] (uint8) and per-32
    scale exponents [rows, K/32] (uint8): E2M1 value * 2^(scale - 127), exactly."""
    codes = unpack_e2m1(packed)
    scale = e8m0_value(scales)
    return e2m1_value(codes) * np.repeat(scale, 32, axis=-1)


def mxfp4_as_bf16_bits(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The dequantized weights as bf16 bits (exact when every scale exponent
    is in 2..252, where each E2M1 value times the power of two is a bf16 value)."""
    w = dequant_mxfp4(packed, scales)
    bits = f64_to_bf16_bits(w)
    fin = np.isfinite(w)
    assert np.array_equal(bf16_to_f64(bits)[fin], w[fin]), "MXFP4 value not exact in bf16"
    return bits


def _expert(W: dict, name: str, e: int) -> np.ndarray:
    v = W[name]
    return v(int(e)) if callable(v) else v[int(e)]


# ---------------------------------------------------------------------------
# The layer
# ---------------------------------------------------------------------------


def latent_moe_forward(dims, W: dict, hidden_bits: np.ndarray, logits: np.ndarray,
                       intermediates: bool = False):
    """The latent-MoE layer forward (bf16 bits [T, hidden] out).

    Data flow of [vLLM-runner] ``_fused_forward`` / ``_shard_up_proj_tail`` on
    one device, with the routed experts of [vLLM-50088] commits 1-3 and 7 and
    the decode order of [TRTLLM-20541] Commit 2:
      1. ids, w   = route(router_logits)
      2. Z        = bf16(X W_down^T)                 routed input transform
      3. rows of the (token, slot) pairs grouped by expert
      4. per expert: G = bf16(Z W13_e^T); act = bf16(SituGLU(G)); Y = bf16(act W2_e^T)
      5. C[t]     = sum_j w[t,j] * Y[t,j]            (the routed sum, complete
                                                      before the norm)
      6. N        = bf16(RMSNorm(C) * gamma)
         Sh       = bf16(bf16(SituGLU(bf16(X Ws13^T))) Ws2^T)   shared expert on X
         out      = bf16(N W_up^T + Sh)              shared output added to the
                                                      up-projection (addmm epilogue)

    ``W`` holds bf16 bits: w_down [L,H], w13 [E,2d,L] (or a callable e ->
    [2d,L]), w2 [E,L,d] (or callable), ws13 [2ds,H] or None, ws2 [H,ds] or
    None, norm_w [L] or None (= ones), w_up [H,L]; and bias float32 [E] or None.
    Tokens are independent, so the rows of a subset of tokens can be computed
    by passing only their hidden states and logits.
    """
    X = bf16_to_f64(hidden_bits)
    T = X.shape[0]
    k, dI = dims.topk, dims.inter
    ids, w = route(logits, W.get("bias"), k, dims.routed_scaling_factor,
                   dims.renormalize, dims.n_group, dims.topk_group)
    Z = linear_bf16(X, W["w_down"])
    Y = np.zeros((T, k, dims.latent), dtype=np.float64)
    for e in np.unique(ids):
        tt, jj = np.nonzero(ids == e)
        G = linear_bf16(Z[tt], _expert(W, "w13", e))
        act = round_bf16(situ(G[:, :dI], G[:, dI:], dims.beta, dims.linear_beta))
        Y[tt, jj] = linear_bf16(act, _expert(W, "w2", e))
    C = np.zeros((T, dims.latent), dtype=np.float64)
    for j in range(k):
        C += w[:, j:j + 1] * Y[:, j]
    gamma = (np.ones(dims.latent) if W.get("norm_w") is None
             else bf16_to_f64(W["norm_w"]))
    N = round_bf16(rms_norm(C, gamma, dims.rms_eps))
    if W.get("ws13") is not None:
        ds = dims.shared_inter
        Gs = linear_bf16(X, W["ws13"])
        As = round_bf16(situ(Gs[:, :ds], Gs[:, ds:], dims.beta, dims.linear_beta))
        Sh = linear_bf16(As, W["ws2"])
    else:
        Sh = np.zeros((T, dims.hidden))
    out = round_bf16(N @ bf16_to_f64(W["w_up"]).T + Sh)
    out_bits = f64_to_bf16_bits(out)
    if not intermediates:
        return out_bits
    return out_bits, dict(ids=ids, weights=w, Z=Z, Y=Y, C=C, N=N, Sh=Sh)


def latent_moe_forward_router(dims, W: dict, hidden_bits: np.ndarray, w_router_bits: np.ndarray,
                              intermediates: bool = False):
    """The layer forward with the router GEMM in front of it: the logits are
    router_gemm(hidden, w_router) and everything else is latent_moe_forward
    ([TRTLLM-20541] Commit 2: router GEMM -> routing -> routed MoE, with the
    latent down projection on the same hidden states)."""
    logits = router_gemm(hidden_bits, w_router_bits)
    res = latent_moe_forward(dims, W, hidden_bits, logits, intermediates)
    if not intermediates:
        return res
    out, mid = res
    return out, dict(mid, logits=logits)


def latent_moe_forward_mxfp4(dims, W: dict, Q: dict, hidden_bits: np.ndarray,
                             logits: np.ndarray, intermediates: bool = False):
    """The layer forward with MXFP4 routed experts: Q holds w13_q, w13_s,
    w2_q, w2_s (stacked [E, ...] arrays, or callables e -> (codes, scales)),
    W the other weights.  The experts' GEMMs use the dequantized weights
    exactly; everything else is latent_moe_forward."""
    def expert(name):
        q, sc = Q[name + "_q"], Q[name + "_s"]
        if callable(q):
            return lambda e: mxfp4_as_bf16_bits(*q(e))
        return lambda e: mxfp4_as_bf16_bits(q[int(e)], sc[int(e)])
    return latent_moe_forward(dims, dict(W, w13=expert("w13"), w2=expert("w2")), hidden_bits,
                              logits, intermediates)
