"""Small, self-contained launches of each kernel, for profiler captures.

  python -m latent_mixture_experts_sigmoid_gb300.profile_cases CASE [--reps N]

CASE is one of
  linear   dense tcgen05 GEMM, out[8192, 8192] = x[8192, 7168] w^T (368 MB of
           operands, larger than L2; 0.96 TFLOP);
  layer    one prefill layer forward (T=4096, Zipf routing) of a 128-expert
           variant of the model (hidden 7168, latent 2048, top-16, d 512,
           shared 4096): every kernel of the path at full token count with
           ~2 GB on the device;
  decode   one decode forward (T=8) of the same 128-expert variant;
  route    routing of [16384, 896] fp32 logits, top-16;
  route8   routing of [8, 896] fp32 logits, top-16 (decode);
  situ     dense SituGLU of bf16 [16384, 8192].
Inputs are seeded (workloads/); each case runs `reps` times after one warm-up.
"""
from __future__ import annotations

import argparse
import dataclasses
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
import latent_mixture_experts_sigmoid_gb300 as lm  # noqa: E402

DEV = torch.device("cuda:0")


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def case_linear(reps):
    g = torch.Generator(device=DEV).manual_seed(0)
    x = torch.randn((8192, 7168), generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn((8192, 7168), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    out = torch.empty((8192, 8192), dtype=torch.bfloat16, device=DEV)
    for _ in range(reps + 1):
        lm.lmoe_linear(x, w, out)


def _layer(d, zipf, reps):
    w = {"w13": torch.empty((d.num_experts, 2 * d.inter, d.latent), dtype=torch.bfloat16, device=DEV),
         "w2": torch.empty((d.num_experts, d.latent, d.inter), dtype=torch.bfloat16, device=DEV)}
    for name in ("w13", "w2"):
        for e0, e1, bits in W.expert_chunks(d, name, 0):
            w[name][e0:e1].copy_(_bf16(bits))
    w.update(w_down=_bf16(W.w_down(d)), w_up=_bf16(W.w_up(d)), ws13=_bf16(W.ws13(d)),
             ws2=_bf16(W.ws2(d)), norm_w=_bf16(W.norm_weight(d)),
             bias=torch.from_numpy(W.score_bias(d.num_experts)).to(DEV))
    x = _bf16(W.hidden_states(d, 0))
    lg = torch.from_numpy(W.router_logits(d.T, d.num_experts, 0, zipf=zipf)).to(DEV)
    out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    for _ in range(reps + 1):
        lm.latent_moe_forward(d, w, x, lg, out, ws)


def case_layer(reps):
    _layer(dataclasses.replace(W.PREFILL, num_experts=128), True, reps)


def case_decode(reps):
    _layer(dataclasses.replace(W.DECODE, num_experts=128), False, reps)


def _route(T, reps):
    lg = torch.from_numpy(W.router_logits(T, 896, 0, tie_every=64)).to(DEV)
    b = torch.from_numpy(W.score_bias(896, 0)).to(DEV)
    ids = torch.empty((T, 16), dtype=torch.int32, device=DEV)
    wt = torch.empty((T, 16), dtype=torch.float32, device=DEV)
    for _ in range(reps + 1):
        lm.moe_route(lg, b, 16, 2.5, ids, wt)


def case_route(reps):
    _route(16384, reps)


def case_route8(reps):
    _route(8, reps)


def case_situ(reps):
    x = _bf16(W.situ_input(16384, 8192, 0))
    out = torch.empty((16384, 4096), dtype=torch.bfloat16, device=DEV)
    for _ in range(reps + 1):
        lm.situ_and_mul(x, out, 4.0, 8.0)


CASES = dict(linear=case_linear, layer=case_layer, decode=case_decode, route=case_route,
             route8=case_route8, situ=case_situ)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args()
    lm.load_library()
    CASES[a.case](a.reps)
    torch.cuda.synchronize()
    err = lm.lmoe_device_error()
    if err:
        raise SystemExit(f"device error word {err}")
    print(f"{a.case}: ok")


if __name__ == "__main__":
    main()
