"""Helpers shared by the GPU tests: host <-> device conversion of the seeded inputs."""
import numpy as np
import torch

DEV = torch.device("cuda:0")


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> bf16 tensor on the GPU."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bits (numpy)."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def weights_to_device(w: dict) -> dict:
    out = {}
    for k, v in w.items():
        if v is None:
            out[k] = None
        elif v.dtype == np.uint16:
            out[k] = dev_bf16(v)
        else:
            out[k] = dev_f32(v)
    return out


def rms_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / rms(ref)."""
    return float(np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2)))


def assert_situ_close(got: np.ndarray, ref: np.ndarray):
    """Elementwise |gpu - ref| <= 1e-2 |ref| + 1e-6 (SituGLU outputs in bf16)."""
    bad = np.abs(got - ref) > 1e-2 * np.abs(ref) + 1e-6
    assert not bad.any(), (f"{bad.sum()} of {bad.size} differ; first at "
                           f"{np.argwhere(bad)[0]}: {got[bad][0]} vs {ref[bad][0]}")


def device_layer_weights(d, seed=0, gamma_noise=False, shared=True) -> dict:
    """Every weight of the layer on the GPU, experts filled block by block."""
    import workloads as W
    out = {}
    E, dI, L = d.num_experts, d.inter, d.latent
    out["w13"] = torch.empty((E, 2 * dI, L), dtype=torch.bfloat16, device=DEV)
    out["w2"] = torch.empty((E, L, dI), dtype=torch.bfloat16, device=DEV)
    for name in ("w13", "w2"):
        for e0, e1, bits in W.expert_chunks(d, name, seed):
            out[name][e0:e1].copy_(dev_bf16(bits))
    out["w_down"] = dev_bf16(W.w_down(d, seed))
    out["w_up"] = dev_bf16(W.w_up(d, seed))
    out["ws13"] = dev_bf16(W.ws13(d, seed)) if shared else None
    out["ws2"] = dev_bf16(W.ws2(d, seed)) if shared else None
    out["norm_w"] = dev_bf16(W.norm_weight(d, seed, gamma_noise))
    out["bias"] = dev_f32(W.score_bias(E, seed))
    return out


def oracle_layer_weights(d, seed=0, gamma_noise=False, shared=True) -> dict:
    """The same weights for the oracle, experts generated lazily on demand."""
    import workloads as W
    return dict(
        w_down=W.w_down(d, seed), w_up=W.w_up(d, seed),
        ws13=W.ws13(d, seed) if shared else None, ws2=W.ws2(d, seed) if shared else None,
        norm_w=W.norm_weight(d, seed, gamma_noise), bias=W.score_bias(d.num_experts, seed),
        w13=lambda e: W.w13_expert(d, e, seed), w2=lambda e: W.w2_expert(d, e, seed))


def run_layer(lm, d, wdev: dict, hidden_bits, logits, debug=True, stream=None):
    """latent_moe_forward on the GPU; returns (out tensor, debug dict of numpy arrays)."""
    T, k, E = d.T, d.topk, d.num_experts
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    dbg = None
    if debug:
        dbg = dict(topk_ids=torch.empty((T, k), dtype=torch.int32, device=DEV),
                   topk_weights=torch.empty((T, k), dtype=torch.float32, device=DEV),
                   expert_num_tokens=torch.empty(E, dtype=torch.int32, device=DEV),
                   expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                   row_of=torch.empty((T, k), dtype=torch.int32, device=DEV))
    lm.latent_moe_forward(d, wdev, dev_bf16(hidden_bits), dev_f32(logits), out, ws, debug=dbg,
                          stream=stream)
    torch.cuda.synchronize()
    return out, ({k2: v.cpu().numpy() for k2, v in dbg.items()} if dbg else None)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid at |v| (2^(floor(log2|v|) - 7), at least 2^-133)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


def assert_layer_close(got: np.ndarray, ref: np.ndarray, tol: float = 2e-2) -> dict:
    """Layer parity: every element within tol * rms(ref), or within one bf16
    step of ref (the output's own quantisation: at |ref| >= 4 rms one bf16
    step is already about 2e-2 * rms, so two correct fp32/fp64 evaluations that
    round to neighbouring bf16 values would otherwise fail)."""
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = np.maximum(tol * rms, bf16_ulp(ref))
    bad = err > bound
    stats = dict(max_err_over_rms=float(err.max() / rms), frac_differing=float((err > 0).mean()),
                 max_err_in_ulps=float((err / bf16_ulp(ref)).max()))
    assert not bad.any(), (f"{bad.sum()} elements beyond max({tol}*rms, 1 bf16 step); "
                           f"first at {np.argwhere(bad)[0]}; {stats}")
    return stats
