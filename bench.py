"""Benchmark of the latent-MoE layer forward on one GB300.

Prints ONE JSON line.  The headline workload is the prefill layer: T=4096
tokens, hidden 7168, latent 2048, 896 experts, top-16, expert intermediate 512,
shared intermediate 4096, router logits skewed by a Zipf(1.1) per-expert
offset; the T=8 decode layer of the same model is measured in the same run and
reported under "decode".  A step is one latent_moe_forward call (routing,
down-projection, permutation, grouped expert GEMMs with SituGLU, combine +
RMSNorm, shared expert, up-projection with the shared add).

  python bench.py [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case linear|layer|decode|decode_mxfp4|route|route8|situ [--reps N]

Inputs are seeded synthetic tensors (workloads/), resident in HBM before the
timed region; L2 is flushed between timed steps (a 512 MiB write, then a
256 MiB read, so that no dirty line is written back inside the timed step).
--impl reference times the CPU oracle (oracle/) on a bounded sample of tokens
of the same workload on the host cores.

The layer runs on one GPU: its prefill GEMMs pair CTAs in clusters that share
operand tiles, so the library is only ever driven from a single-GPU process.
--gpus must be 1 for this arm (the reference arm, which uses no GPU, accepts
any N: only the process with RANK 0 runs and prints).

--case runs one small, self-contained launch set of a kernel for profiler
captures and prints "<case>: ok":
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
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


class _LazyWorkloads:
    """The seeded input generators, imported on first use (worker processes of
    the oracle baselines import this module and need only NumPy)."""

    def __getattr__(self, name):
        import workloads
        return getattr(workloads, name)


W = _LazyWorkloads()

METRIC = "latent-MoE layer tokens/s at T=8 and T=4096; % of HBM / bf16 TC roofline"
UNIT = "tokens/s"
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture) of
# the six GEMM launches of one prefill forward of this workload, summed; valid
# for the GEMM kernel as it was when captured, and for this workload only.  The
# capture ran on the 128-expert variant (bench.py --case layer): the dense
# GEMMs have this workload's shapes, the grouped GEMMs are scaled by the ratio
# of their algorithmic bytes (the used experts' weights and the token rows).
GEMM_SET_DRAM_BYTES = 2274500000


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sus=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# --------------------------------------------------------------------------
# algorithmic work per forward (counts only real rows: tokens actually routed)
# --------------------------------------------------------------------------
def gemm_flops(d, counts_nonzero):
    T, H, L, dI, ds, k = d.T, d.hidden, d.latent, d.inter, d.shared_inter, d.topk
    down = 2.0 * T * H * L
    experts = 2.0 * T * k * (2 * dI * L + L * dI)
    shared = 2.0 * T * (2 * ds * H + H * ds)
    up = 2.0 * T * L * H
    return dict(down=down, gemm1=2.0 * T * k * 2 * dI * L, gemm2=2.0 * T * k * L * dI,
                shared1=2.0 * T * 2 * ds * H, shared2=2.0 * T * H * ds, up=up,
                total=down + experts + shared + up)


def gemm_bytes(d, n_used):
    """Bytes a GEMM stage must move at least once (weights touched + activations)."""
    T, H, L, dI, ds, k = d.T, d.hidden, d.latent, d.inter, d.shared_inter, d.topk
    R = T * k
    return dict(
        down=2 * (L * H + T * H + T * L),
        gemm1=2 * (n_used * 2 * dI * L + R * L + R * 2 * dI),
        gemm2=2 * (n_used * L * dI + R * dI + R * L),
        shared1=2 * (2 * ds * H + T * H + T * 2 * ds),
        shared2=2 * (H * ds + T * ds + T * H),
        up=2 * (H * L + T * L + 2 * T * H))


def mxfp4_expert_bytes(d, n_used):
    """Bytes the two MXFP4 expert stages must move at least once: the used
    experts' 4-bit codes and their scales (4.25 bits a weight), the input rows
    and the bf16 outputs."""
    L, dI, R = d.latent, d.inter, d.T * d.topk
    wb = 0.5 + 1.0 / 32
    return dict(gemm1=int(n_used * 2 * dI * L * wb + 2 * (R * L + R * dI)),
                gemm2=int(n_used * L * dI * wb + 2 * (R * dI + R * L)))


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def run_ours(args):
    import torch
    import latent_mixture_experts_sigmoid_gb300 as lm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lm.load_library()
    pk = peaks()

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # weights shared by both workloads (same model)
    dD = W.DECODE
    w = {"w13": torch.empty((dD.num_experts, 2 * dD.inter, dD.latent), dtype=torch.bfloat16, device=dev),
         "w2": torch.empty((dD.num_experts, dD.latent, dD.inter), dtype=torch.bfloat16, device=dev)}
    for name in ("w13", "w2"):
        for e0, e1, bits in W.expert_chunks(dD, name, 0):
            w[name][e0:e1].copy_(dev_bf16(bits))
    w.update(w_down=dev_bf16(W.w_down(dD)), w_up=dev_bf16(W.w_up(dD)), ws13=dev_bf16(W.ws13(dD)),
             ws2=dev_bf16(W.ws2(dD)), norm_w=dev_bf16(W.norm_weight(dD)),
             bias=torch.from_numpy(W.score_bias(dD.num_experts)).to(dev))
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 * 2 ** 20, dtype=torch.float32, device=dev)   # 256 MiB
    stream = torch.cuda.Stream(device=dev)

    def flush_l2():
        # write 512 MiB (evicts everything), then read 256 MiB so that the
        # write-backs of those dirty lines happen here, outside the timed region
        flush.zero_()
        flush_rd.sum()

    def measure(d, zipf, steps, warmup):
        T = d.T
        x_bits = W.hidden_states(d, 0)
        lg = W.router_logits(T, d.num_experts, 0, zipf=zipf)
        x = dev_bf16(x_bits)
        lgd = torch.from_numpy(lg).to(dev)
        out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
        counts = torch.empty(d.num_experts, dtype=torch.int32, device=dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGES + 1)]
        dbg = {"expert_num_tokens": counts, "stage_events": evs}
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                lm.latent_moe_forward(d, w, x, lgd, out, ws, debug=dbg, stream=stream)
        torch.cuda.synchronize()
        # one forward captured in a CUDA graph (the calls are capturable): the
        # timed steps replay it, so host launch overhead is not on the clock
        if args.no_graph:
            def replay():
                lm.latent_moe_forward(d, w, x, lgd, out, ws, stream=stream)
        else:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                lm.latent_moe_forward(d, w, x, lgd, out, ws, stream=stream)
            replay = graph.replay
        for _ in range(warmup):
            with torch.cuda.stream(stream):
                replay()
        torch.cuda.synchronize()
        n_used = int((counts.cpu().numpy() > 0).sum())
        # device-timed region: K steps, one event pair around each forward
        torch.cuda.synchronize()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per_step = []
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush_l2()
                e_a.record(stream)
                replay()
                e_b.record(stream)
            stream.synchronize()
            per_step.append(e_a.elapsed_time(e_b))
        torch.cuda.synchronize()
        ms = float(sum(per_step))
        # per-stage breakdown: the library records an event after every stage
        # (the events serialise the stages, so this pass is not the headline).
        # A ~1 ms GPU spin is queued first so that the host has enqueued the
        # whole forward before the GPU reaches it: stage times exclude host gaps.
        per_stage = np.zeros(lm.NUM_STAGES)
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush_l2()
                torch.cuda._sleep(2_000_000)
                lm.latent_moe_forward(d, w, x, lgd, out, ws, debug=dbg, stream=stream)
            stream.synchronize()
            per_stage += np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(lm.NUM_STAGES)])
        # end to end through the public API with host buffers: every step copies
        # its inputs from pinned host memory and its output back.  As in a
        # serving loop, the copies of neighbouring steps overlap the forward:
        # H2D of step n+1 and D2H of step n-1 run on their own streams while
        # step n computes (two device buffer sets; events order the reuse).
        xh = torch.from_numpy(x_bits.view(np.int16)).pin_memory()
        lh = torch.from_numpy(lg).pin_memory()
        oh = [torch.empty((T, d.hidden), dtype=torch.int16).pin_memory() for _ in range(2)]
        xd, ld, od = [x, x.clone()], [lgd, lgd.clone()], [out, out.clone()]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_fw = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def pipeline(n_steps, e_start=None, e_end=None):
            if e_start is not None:
                e_start.record(s_in)
            for n in range(n_steps):
                b = n % 2
                with torch.cuda.stream(s_in):
                    if n >= 2:
                        s_in.wait_event(ev_fw[b])          # step n-2 has read xd[b], ld[b]
                    xd[b].view(torch.int16).copy_(xh, non_blocking=True)
                    ld[b].copy_(lh, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if n >= 2:
                    stream.wait_event(ev_out[b])           # step n-2's output is on the host
                lm.latent_moe_forward(d, w, xd[b], ld[b], od[b], ws, stream=stream)
                ev_fw[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_fw[b])
                    oh[b].copy_(od[b].view(torch.int16), non_blocking=True)
                    ev_out[b].record(s_out)
            if e_end is not None:
                e_end.record(s_out)

        pipeline(2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipeline(steps, e0, e1)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        # the same with nothing overlapped (copy in, forward, copy out per step)
        e2e_serial_ms = 0.0
        for _ in range(steps):
            with torch.cuda.stream(stream):
                e0.record(stream)
                x.view(torch.int16).copy_(xh, non_blocking=True)
                lgd.copy_(lh, non_blocking=True)
                lm.latent_moe_forward(d, w, x, lgd, out, ws, stream=stream)
                oh[0].copy_(out.view(torch.int16), non_blocking=True)
                e1.record(stream)
            stream.synchronize()
            e2e_serial_ms += e0.elapsed_time(e1)
        # decode with the routing done ahead (moe_route before the timed
        # region, its ids and weights fed to latent_moe_forward_routed): the
        # step without the routing on its critical path, and whether its output
        # is bit-identical to the layer routing itself
        pre = None
        if T <= 128 and not args.no_graph:
            ids = torch.empty((T, d.topk), dtype=torch.int32, device=dev)
            tw = torch.empty((T, d.topk), dtype=torch.float32, device=dev)
            out2, ws2 = torch.empty_like(out), torch.empty_like(ws)
            with torch.cuda.stream(stream):
                lm.moe_route(lgd, w["bias"], d.topk, d.routed_scaling_factor, ids, tw,
                             renormalize=d.renormalize, stream=stream)
                lm.latent_moe_forward_routed(d, w, x, ids, tw, out2, ws2, stream=stream)
            torch.cuda.synchronize()
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=stream):
                lm.latent_moe_forward_routed(d, w, x, ids, tw, out2, ws2, stream=stream)
            for _ in range(warmup):
                with torch.cuda.stream(stream):
                    g2.replay()
            torch.cuda.synchronize()
            pre_ms = 0.0
            for _ in range(steps):
                with torch.cuda.stream(stream):
                    flush_l2()
                    e_a.record(stream)
                    g2.replay()
                    e_b.record(stream)
                stream.synchronize()
                pre_ms += e_a.elapsed_time(e_b)
            pre = dict(ms=pre_ms, same=bool(torch.equal(out2.view(torch.int16),
                                                        out.view(torch.int16))))
        return dict(ms=ms, per_step=per_step, per_stage=per_stage / steps, n_used=n_used,
                    e2e_ms=e2e_ms, e2e_serial_ms=e2e_serial_ms, h2d=T * d.hidden * 2 + T * d.num_experts * 4,
                    d2h=T * d.hidden * 2, pre=pre)

    def measure_router(d, zipf, steps, warmup):
        """The layer with its router GEMM: latent_moe_forward_router (at T <= 128
        the router rows share the down-projection's launch) against the router
        GEMM as its own op (lmoe_router_logits) followed by latent_moe_forward,
        each one CUDA-graph replay per step, L2 flushed between steps."""
        T, E, H = d.T, d.num_experts, d.hidden
        x = dev_bf16(W.hidden_states(d, 0))
        wr = dev_bf16(W.w_router(d, 0))
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
        lg = torch.empty((T, E), dtype=torch.float32, device=dev)
        rws = torch.empty(lm.lmoe_router_logits_workspace_bytes(T, E, H), dtype=torch.uint8,
                          device=dev)

        def fused():
            lm.latent_moe_forward_router(d, w, wr, x, out, ws, stream=stream)

        def separate():
            lm.lmoe_router_logits(x, wr, lg, rws, stream=stream)
            lm.latent_moe_forward(d, w, x, lg, out, ws, stream=stream)

        counts = torch.empty(E, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            lm.latent_moe_forward_router(d, w, wr, x, out, ws, debug={"expert_num_tokens": counts},
                                         stream=stream)
        stream.synchronize()
        n_used = int((counts.cpu().numpy() > 0).sum())
        res = {}
        for name, fn in (("fused", fused), ("separate", separate)):
            with torch.cuda.stream(stream):
                for _ in range(warmup):
                    fn()
            torch.cuda.synchronize()
            if args.no_graph:
                replay = fn
            else:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                replay = g.replay
            for _ in range(warmup):
                with torch.cuda.stream(stream):
                    replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(steps):
                with torch.cuda.stream(stream):
                    flush_l2()
                    a.record(stream)
                    replay()
                    b.record(stream)
                stream.synchronize()
                tot += a.elapsed_time(b)
            res[name] = tot / steps * 1e3
        return {"us_per_step_fused": round(res["fused"], 2),
                "us_per_step_separate_router_op": round(res["separate"], 2),
                "tokens_per_s_fused": round(T / (res["fused"] / 1e6), 1),
                "launches_fused": lm.latent_moe_launch_count_router(d),
                "experts_used": n_used,
                "routing": "the router GEMM's logits carry no Zipf skew: tokens spread over "
                           "nearly all experts, so the grouped GEMMs read far more expert weights "
                           "than the headline workload's 118 experts",
                "what": ("latent_moe_forward_router" + (" (router rows stacked after the "
                         "down-projection's in one split-K GEMM)" if T <= 128 else
                         " (router GEMM its own launch on the second stream)") +
                         " against lmoe_router_logits + latent_moe_forward; router weight "
                         "bf16 [E, H] N(0, 1/H)")}

    def measure_mxfp4(d, zipf, steps, warmup, q):
        """latent_moe_forward_mxfp4 (routed experts in MXFP4, the rest bf16),
        one CUDA-graph replay per step, L2 flushed between steps; per-stage
        times from the library's stage events in a separate pass."""
        T = d.T
        x = dev_bf16(W.hidden_states(d, 0))
        lgd = torch.from_numpy(W.router_logits(T, d.num_experts, 0, zipf=zipf)).to(dev)
        out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(lm.latent_moe_workspace_bytes_mxfp4(d), dtype=torch.uint8, device=dev)
        counts = torch.empty(d.num_experts, dtype=torch.int32, device=dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGES + 1)]
        dbg = {"expert_num_tokens": counts, "stage_events": evs}
        wq = dict(w, w13=None, w2=None)

        def fwd():
            lm.latent_moe_forward_mxfp4(d, wq, q, x, lgd, out, ws, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                lm.latent_moe_forward_mxfp4(d, wq, q, x, lgd, out, ws, debug=dbg, stream=stream)
        torch.cuda.synchronize()
        n_used = int((counts.cpu().numpy() > 0).sum())
        if args.no_graph:
            replay = fwd
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fwd()
            replay = g.replay
        for _ in range(warmup):
            with torch.cuda.stream(stream):
                replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush_l2()
                a.record(stream)
                replay()
                b.record(stream)
            stream.synchronize()
            tot += a.elapsed_time(b)
        per_stage = np.zeros(lm.NUM_STAGES)
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush_l2()
                torch.cuda._sleep(2_000_000)
                lm.latent_moe_forward_mxfp4(d, wq, q, x, lgd, out, ws, debug=dbg, stream=stream)
            stream.synchronize()
            per_stage += np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(lm.NUM_STAGES)])
        st = dict(zip(lm.STAGE_NAMES, per_stage / steps))
        us = tot / steps * 1e3
        eb = mxfp4_expert_bytes(d, n_used)
        ex_us = (st["gemm1"] + st["situ"] + st["gemm2"]) * 1e3
        res = {"us_per_step": round(us, 2), "tokens_per_s": round(T / (us / 1e6), 1),
               "experts_used": n_used, "launches": lm.latent_moe_launch_count_mxfp4(d),
               "per_stage_ms": {n: round(v, 4) for n, v in st.items()}}
        if T <= 128:
            gb = (eb["gemm1"] + eb["gemm2"]) / (ex_us / 1e6) / 1e9
            by = gemm_bytes(d, n_used)
            layer_bytes = sum(v for k2, v in by.items() if k2 not in ("gemm1", "gemm2")) + \
                eb["gemm1"] + eb["gemm2"]
            res["expert_kernels"] = {
                "kernel": "fp4_expert_kernel (GEMM1 + SituGLU and GEMM2 on the 4-bit weights: TMA "
                          "strips, codes widened to f16 in registers, mma.sync m16n8k16)",
                "bound": "hbm", "us": round(ex_us, 2), "algorithmic_bytes": eb,
                "achieved": round(gb, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gb / pk["hbm"], 4),
                "timing": "per-stage CUDA events (stages serialised)"}
            lgb = layer_bytes / (us / 1e6) / 1e9
            res["roofline"] = {"bound": "hbm", "algorithmic_bytes": int(layer_bytes),
                               "achieved": round(lgb, 1), "peak": pk["hbm"], "unit": "GB/s",
                               "frac": round(lgb / pk["hbm"], 4)}
        res["what"] = ("latent_moe_forward_mxfp4: routed experts as MXFP4 (E2M1 codes, one E8M0 "
                       "scale per 32; codes uniform, scale exponents 118..120), every other "
                       "weight bf16 as in the bf16 lines" +
                       (": the expert stages read the 4-bit weights directly" if T <= 128 else
                        ": the experts with routed tokens dequantized to bf16 in the workspace "
                        "each call, then the tensor-core GEMMs"))
        return res

    def time_launches(fns, reps):
        """Average device time per launch of `reps` back-to-back launches.

        fns are launches on distinct input buffers, used round-robin so that no
        launch finds its inputs in L2 (each list is sized above L2); L2 is
        flushed once before the run, which also lets the host queue launches
        ahead of the device.  Mean over three runs.
        """
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            fns[0]()
        stream.synchronize()
        tot = 0.0
        for _ in range(3):
            with torch.cuda.stream(stream):
                flush_l2()
                a.record(stream)
                for i in range(reps):
                    fns[i % len(fns)]()
                b.record(stream)
            stream.synchronize()
            tot += a.elapsed_time(b) / reps
        return tot / 3

    def kernel_lines(reps):
        """The hot path's bandwidth-bound kernels alone, on their own workloads."""
        res = {"timing": "mean device time per launch over back-to-back launches; inputs above L2 "
                         "(routing rotates 8 logits buffers)"}
        Tr, Er, kr = 16384, W.ROUTE_E, W.ROUTE_K
        lg = torch.from_numpy(W.router_logits(Tr, Er, 0, tie_every=64)).to(dev)
        bias = torch.from_numpy(W.score_bias(Er, 0)).to(dev)
        ids = torch.empty((Tr, kr), dtype=torch.int32, device=dev)
        wt = torch.empty((Tr, kr), dtype=torch.float32, device=dev)
        lgs = [lg] + [lg.clone() for _ in range(7)]          # 8 x 58.7 MB rotate past L2
        ms = time_launches([lambda g=g: lm.moe_route(g, bias, kr, W.ROUTE_RSF, ids, wt, stream=stream)
                            for g in lgs], 4 * reps)
        by = 4 * Tr * Er + 4 * Er + 8 * Tr * kr
        res["route"] = {"workload": f"[{Tr}, {Er}] fp32 logits, top-{kr}", "us": round(ms * 1e3, 2),
                        "GBps": round(by / ms / 1e6, 1), "frac_hbm": round(by / ms / 1e6 / pk["hbm"], 4),
                        "tokens_per_s": round(Tr / ms * 1e3, 1)}
        del lg, lgs
        N, dd = 16384, 4096
        xs = dev_bf16(W.situ_input(N, 2 * dd, 0))
        ys = torch.empty((N, dd), dtype=torch.bfloat16, device=dev)
        for lb in (8.0, 0.0):
            ms = time_launches([lambda: lm.situ_and_mul(xs, ys, 4.0, lb, stream=stream)], reps)
            by = N * dd * 6
            res[f"situ_dense_lb{int(lb)}"] = {"workload": f"bf16 [{N}, 2*{dd}]", "us": round(ms * 1e3, 2),
                                              "GBps": round(by / ms / 1e6, 1),
                                              "frac_hbm": round(by / ms / 1e6 / pk["hbm"], 4)}
        del xs, ys
        xm, cnt = W.masked_situ_input(128, 512, 4096, 0)
        xmd = dev_bf16(xm)
        ym = torch.empty((128, 512, 2048), dtype=torch.bfloat16, device=dev)
        cd = torch.from_numpy(cnt).to(dev)
        ms = time_launches([lambda: lm.masked_situ_and_mul(xmd, ym, cd, 4.0, 8.0, stream=stream)], reps)
        by = int(cnt.sum()) * 2048 * 6
        res["situ_masked"] = {"workload": "bf16 [128, 512, 2*2048], counts U[0,512]",
                              "us": round(ms * 1e3, 2), "GBps": round(by / ms / 1e6, 1),
                              "frac_hbm": round(by / ms / 1e6 / pk["hbm"], 4)}
        del xmd, ym
        return res

    clocks = Clocks(dev.index)
    t_wall0 = time.time()
    pre = measure(W.PREFILL, True, args.steps, args.warmup)
    dec = measure(W.DECODE, False, args.steps, args.warmup)
    rtr_dec = measure_router(W.DECODE, False, args.steps, args.warmup)
    rtr_pre = measure_router(W.PREFILL, True, args.steps, args.warmup)
    # the same model with MXFP4 routed experts (bf16 experts released first)
    del w["w13"], w["w2"]
    torch.cuda.empty_cache()
    qh = W.mxfp4_experts(dD, 0)
    q4 = {k2: torch.from_numpy(v).to(dev) for k2, v in qh.items()}
    del qh
    fp4_dec = measure_mxfp4(W.DECODE, False, args.steps, args.warmup, q4)
    fp4_pre = measure_mxfp4(W.PREFILL, True, args.steps, args.warmup, q4)
    del q4
    kern = kernel_lines(max(3, args.steps))
    if not args.no_cpu_baseline:
        for name, cb in kernel_cpu_baselines().items():
            kern[name]["cpu_baseline"] = cb
    clk = clocks.stop()
    wall = time.time() - t_wall0

    pre_ms, dec_ms = pre["ms"], dec["ms"]
    pre_e2e, dec_e2e = pre["e2e_ms"], dec["e2e_ms"]
    K = args.steps
    dP, dDc = W.PREFILL, W.DECODE
    value = dP.T * K / (pre_ms / 1e3)

    # roofline of the dominant kernel (the tcgen05 GEMM, all its launches of a step)
    names = lm.STAGE_NAMES
    st = dict(zip(names, pre["per_stage"]))
    fl = gemm_flops(dP, pre["n_used"])
    gemm_stages = ["down", "gemm1", "gemm2", "shared1", "shared2", "up"]
    gemm_ms = sum(st[s] for s in gemm_stages)
    ach_tf = fl["total"] / (gemm_ms / 1e3) / 1e12
    # the step is about a millisecond at full clock, so the burst peak applies
    roof = {"kernel": "gemm_tc_kernel (all GEMM launches of one prefill forward)",
            "bound": "tensor", "achieved": round(ach_tf, 1), "peak": pk["bf16"],
            "unit": "TFLOP/s", "frac": round(ach_tf / pk["bf16"], 4),
            "peak_source": f"{pk['source']} bf16 burst",
            "traffic": GEMM_SET_DRAM_BYTES,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the six GEMM "
                              "launches of one prefill forward, captured on the 128-expert "
                              "variant and scaled to this workload (algorithmic: 2042.8 MB)",
            "flops_per_launch_set": fl["total"], "ms_per_launch_set": round(gemm_ms, 4)}
    # the grouped expert GEMMs alone (GEMM1 with SituGLU in its epilogue, GEMM2)
    ex_ms = st["gemm1"] + st["gemm2"]
    ex_fl = fl["gemm1"] + fl["gemm2"]
    ex_tf = ex_fl / (ex_ms / 1e3) / 1e12
    roof["expert_gemms"] = {
        "achieved": round(ex_tf, 1), "peak": pk["bf16"], "unit": "TFLOP/s",
        "frac": round(ex_tf / pk["bf16"], 4), "us": round(ex_ms * 1e3, 1),
        "gemm1_frac": round(fl["gemm1"] / (st["gemm1"] / 1e3) / 1e12 / pk["bf16"], 4),
        "gemm2_frac": round(fl["gemm2"] / (st["gemm2"] / 1e3) / 1e12 / pk["bf16"], 4),
        "flops": ex_fl, "what": "grouped GEMM1 (+ SituGLU epilogue) and GEMM2 of the prefill, "
                               "useful flops (routed rows only) over per-stage CUDA-event time"}
    per_stage_pre = {n: round(v, 4) for n, v in st.items()}
    per_stage_dec = {n: round(v, 4) for n, v in zip(names, dec["per_stage"])}
    # decode roofline: weight streaming of the whole layer
    by = gemm_bytes(dDc, dec["n_used"])
    dec_bytes = sum(by.values())
    dec_us = dec_ms / K * 1e3
    dec_gbs = dec_bytes / (dec_us / 1e6) / 1e9
    decode = {"workload": "decode T=8", "tokens_per_s": round(dDc.T * K / (dec_ms / 1e3), 1),
              "us_per_step": round(dec_us, 2), "experts_used": dec["n_used"],
              "algorithmic_bytes": dec_bytes,
              "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": pk["hbm"],
                           "unit": "GB/s", "frac": round(dec_gbs / pk["hbm"], 4)},
              "per_stage_ms": per_stage_dec,
              "e2e_tokens_per_s": round(dDc.T * K / (dec_e2e / 1e3), 1),
              "gpu_launches_per_step": lm.latent_moe_launch_count(dDc)}
    decode["router_gemm"] = rtr_dec
    decode["mxfp4"] = fp4_dec
    if dec["pre"] is not None:
        decode["pre_routed"] = {
            "us_per_step": round(dec["pre"]["ms"] / K * 1e3, 2),
            "what": "latent_moe_forward_routed on ids/weights from a moe_route call made before "
                    "the timed region (routing off the step's critical path)",
            "bit_identical_to_layer_routing": dec["pre"]["same"]}
    # the layer's own data-movement stages at prefill (per-stage events, algorithmic bytes)
    T, k, L = dP.T, dP.topk, dP.latent
    for name, stage, nbytes, what in (
            ("permute_scatter_prefill", "scatter", T * L * 2 + T * k * L * 2,
             "token rows into the expert-major layout: read Z [T, L], write A [T*k, L] (bf16)"),
            ("combine_norm_prefill", "combine_norm", T * k * L * 2 + T * L * 2 + T * k * 8 + L * 2,
             "top-k combine + RMSNorm: read Y [T*k, L], weights, rows; write N [T, L]"),
            ("permute_index_prefill", "permute", T * k * 4 * 3,
             "counting-sort indices (ids in, row_of and tok_of_row out): latency-bound")):
        ms_st = st[stage]
        kern[name] = {"workload": what, "us": round(ms_st * 1e3, 2),
                      "GBps": round(nbytes / ms_st / 1e6, 1),
                      "frac_hbm": round(nbytes / ms_st / 1e6 / pk["hbm"], 4),
                      "timing": "per-stage CUDA events of the prefill layer"}
    # the library's launches inside the headline's timed region (K prefill forwards)
    launches = lm.latent_moe_launch_count(dP)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(pre_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) bf16 weights)",
        "config": {"workload": "latent-MoE layer prefill T=4096, Zipf(1.1)-skewed routing",
                   "T": dP.T, "hidden": dP.hidden, "latent": dP.latent,
                   "num_experts": dP.num_experts, "topk": dP.topk, "inter": dP.inter,
                   "shared_inter": dP.shared_inter, "experts_used": pre["n_used"],
                   "l2": "flushed between timed steps (512 MiB write, then 256 MiB read, untimed)",
                   "timing": ("eager latent_moe_forward calls" if args.no_graph else
                              "CUDA-graph replay of one latent_moe_forward per step"),
                   "parallelism": "single GPU"},
        "e2e": {"value": round(dP.T * K / (pre_e2e / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": pre["h2d"], "d2h_bytes_per_step": pre["d2h"],
                "method": ("latent_moe_forward per step on host-resident inputs; H2D of step "
                           "n+1 and D2H of step n-1 overlap step n on separate streams "
                           "(timed from the first copy in to the last copy out)"),
                "serial_value": round(dP.T * K / (pre["e2e_serial_ms"] / 1e3), 1)},
        "gpu_launches": launches * K,
        "roofline": roof,
        "per_stage_ms": per_stage_pre,
        "layer_gflop": round(fl["total"] / 1e9, 1),
        "layer_tflops": round(fl["total"] / (pre_ms / K / 1e3) / 1e12, 1),
        "decode": decode,
        "prefill_router_gemm": rtr_pre,
        "prefill_mxfp4": fp4_pre,
        "kernels": kern,
        "clocks": clk,
        "wall_s": round(wall, 1),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(W.PREFILL, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------
def _cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("internal_api") in
             ("openblas", "mkl", "blis")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _oracle_sample(d, tokens, zipf):
    """Inputs of a token sample plus the weights it touches (generated up front)."""
    from oracle import lmoe_oracle as O
    x = W.hidden_rows(d, tokens, 0)
    lg = W.logits_rows(d.num_experts, tokens, 0, zipf=zipf)
    ids, _ = O.route(lg, W.score_bias(d.num_experts, 0), d.topk, d.routed_scaling_factor)
    used = sorted(set(ids.ravel().tolist()))
    w13 = {e: W.w13_expert(d, e, 0) for e in used}
    w2 = {e: W.w2_expert(d, e, 0) for e in used}
    wts = dict(w_down=W.w_down(d), w_up=W.w_up(d), ws13=W.ws13(d), ws2=W.ws2(d),
               norm_w=W.norm_weight(d), bias=W.score_bias(d.num_experts, 0),
               w13=w13.__getitem__, w2=w2.__getitem__)
    return x, lg, wts


def cpu_baseline(d, budget_s=20.0, sample=16):
    from oracle import lmoe_oracle as O
    toks = list(range(0, d.T, max(1, d.T // sample)))[:sample]
    x, lg, wts = _oracle_sample(d, toks, zipf=True)
    t0 = time.perf_counter()
    n = 0
    while True:
        O.latent_moe_forward(d, wts, x, lg)
        n += 1
        if time.perf_counter() - t0 > min(budget_s, 5.0) or n >= 3:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": round(len(toks) / dt, 2), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{len(toks)} of the {d.T} tokens of the prefill workload per call "
                      f"(float64 NumPy oracle, weights pre-generated), {n} call(s)"}


# --------------------------------------------------------------------------
# the oracle beside the kernel lines: one core, and every host core at once
# --------------------------------------------------------------------------
_BARRIER = None


def _pool_init(barrier):
    global _BARRIER
    _BARRIER = barrier
    os.environ.setdefault("OMP_NUM_THREADS", "1")


def _oracle_kernel_job(job):
    """Run one oracle call on pre-generated inputs; returns (units, seconds).

    In a pool, every worker waits at a barrier before its timed call so that
    all cores run at once."""
    from oracle import lmoe_oracle as O
    kind, inp, units = job
    if _BARRIER is not None:
        _BARRIER.wait(timeout=300)
    t0 = time.perf_counter()
    if kind == "route":
        lg, b = inp
        O.route(lg, b, W_ROUTE_K, W_ROUTE_RSF)
    elif kind == "situ":
        x, lb = inp
        O.situ_and_mul(x, 4.0, lb)
    else:
        x, cnt, init = inp
        O.masked_situ_and_mul(x, cnt, init, 4.0, 8.0)
    return units, time.perf_counter() - t0


# the routing workload's constants, for workers that do not import workloads
W_ROUTE_K, W_ROUTE_RSF = 16, 2.5


def kernel_cpu_baselines(cores=None):
    """Oracle throughput on a sample of each kernel line's workload (the same
    seeded rows the GPU line processes), on one core and on every core.
    Returns {line: cpu_baseline dict}, in the unit of the GPU line."""
    import multiprocessing as mp
    assert W.ROUTE_K == W_ROUTE_K and W.ROUTE_RSF == W_ROUTE_RSF
    cores = cores or os.cpu_count() or 1
    Er = W.ROUTE_E
    route_rows, situ_rows = 2048, 1024
    jobs = {}
    # routing: tokens of the [16384, 896] workload, one sample per worker
    jobs["route"] = [("route", (W.logits_rows(Er, range(i * route_rows, (i + 1) * route_rows), 0,
                                              tie_every=64), W.score_bias(Er, 0)), route_rows)
                     for i in range(cores)]
    for lb in (8.0, 0.0):
        x = W.situ_input(situ_rows, 8192, 0)
        jobs[f"situ_dense_lb{int(lb)}"] = [("situ", (x, lb), situ_rows * 4096)] * cores
    xm, cnt = W.masked_situ_input(128, 512, 4096, 0)
    xm, cnt = xm[:4].copy(), cnt[:4].copy()                  # 4 of the 128 experts
    init = W.sentinel_like((4, 512, 2048))
    jobs["situ_masked"] = [("masked", (xm, cnt, init), int(cnt.sum()) * 2048)] * cores
    unit_of = {"route": ("tokens/s", 1.0), "situ_dense_lb8": ("GB/s", 6e-9),
               "situ_dense_lb0": ("GB/s", 6e-9), "situ_masked": ("GB/s", 6e-9)}
    res = {}
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(cores)
    with ctx.Pool(cores, initializer=_pool_init, initargs=(barrier,)) as pool:
        for name, js in jobs.items():
            u1, t1 = _oracle_kernel_job(js[0])                # one core, this process
            out = pool.map(_oracle_kernel_job, js, chunksize=1)
            u_all = sum(u for u, _ in out)
            t_all = max(t for _, t in out)
            unit, scale = unit_of[name]
            res[name] = {"value": round(u_all / t_all * scale, 3), "unit": unit, "cores": cores,
                         "kind": "oracle", "one_core": round(u1 / t1 * scale, 3),
                         "sample": (f"{js[0][2]} units per core ("
                                    + ("tokens of the [16384, 896] logits" if name == "route" else
                                       "output elements of seeded rows of the same workload")
                                    + "), float64 NumPy oracle, all cores started together")}
    return res


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded token sample.
    Under a multi-process launcher only the process with RANK 0 runs."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from oracle import lmoe_oracle as O
    d = W.PREFILL
    sample = 8
    toks = list(range(0, d.T, d.T // sample))[:sample]
    x, lg, wts = _oracle_sample(d, toks, zipf=True)
    for _ in range(args.warmup):
        O.latent_moe_forward(d, wts, x, lg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.latent_moe_forward(d, wts, x, lg)
    dt = time.perf_counter() - t0
    value = len(toks) * args.steps / dt
    cores = _cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "latent-MoE layer prefill T=4096, Zipf(1.1)-skewed routing",
                   "sample_tokens_per_step": len(toks)},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{len(toks)} tokens of the T=4096 prefill workload per step"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# --case: small launch sets for profiler captures
# --------------------------------------------------------------------------
def run_case(name, reps):
    import dataclasses
    import torch
    import latent_mixture_experts_sigmoid_gb300 as lm

    dev = torch.device("cuda:0")
    lm.load_library()

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def layer(d, zipf):
        w = {"w13": torch.empty((d.num_experts, 2 * d.inter, d.latent), dtype=torch.bfloat16,
                                device=dev),
             "w2": torch.empty((d.num_experts, d.latent, d.inter), dtype=torch.bfloat16, device=dev)}
        for nm in ("w13", "w2"):
            for e0, e1, bits in W.expert_chunks(d, nm, 0):
                w[nm][e0:e1].copy_(bf16(bits))
        w.update(w_down=bf16(W.w_down(d)), w_up=bf16(W.w_up(d)), ws13=bf16(W.ws13(d)),
                 ws2=bf16(W.ws2(d)), norm_w=bf16(W.norm_weight(d)),
                 bias=torch.from_numpy(W.score_bias(d.num_experts)).to(dev))
        x = bf16(W.hidden_states(d, 0))
        lg = torch.from_numpy(W.router_logits(d.T, d.num_experts, 0, zipf=zipf)).to(dev)
        out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
        for _ in range(reps + 1):
            lm.latent_moe_forward(d, w, x, lg, out, ws)

    def route(T):
        lg = torch.from_numpy(W.router_logits(T, 896, 0, tie_every=64)).to(dev)
        b = torch.from_numpy(W.score_bias(896, 0)).to(dev)
        ids = torch.empty((T, 16), dtype=torch.int32, device=dev)
        wt = torch.empty((T, 16), dtype=torch.float32, device=dev)
        for _ in range(reps + 1):
            lm.moe_route(lg, b, 16, 2.5, ids, wt)

    if name == "linear":
        g = torch.Generator(device=dev).manual_seed(0)
        x = torch.randn((8192, 7168), generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn((8192, 7168), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        out = torch.empty((8192, 8192), dtype=torch.bfloat16, device=dev)
        for _ in range(reps + 1):
            lm.lmoe_linear(x, w, out)
    elif name == "layer":
        layer(dataclasses.replace(W.PREFILL, num_experts=128), True)
    elif name == "decode":
        layer(dataclasses.replace(W.DECODE, num_experts=128), False)
    elif name == "decode_mxfp4":
        d = dataclasses.replace(W.DECODE, num_experts=128)
        w = {"w_down": bf16(W.w_down(d)), "w_up": bf16(W.w_up(d)), "ws13": bf16(W.ws13(d)),
             "ws2": bf16(W.ws2(d)), "norm_w": bf16(W.norm_weight(d)),
             "bias": torch.from_numpy(W.score_bias(d.num_experts)).to(dev)}
        q = {k2: torch.from_numpy(v).to(dev) for k2, v in W.mxfp4_experts(d, 0).items()}
        x = bf16(W.hidden_states(d, 0))
        lg = torch.from_numpy(W.router_logits(d.T, d.num_experts, 0)).to(dev)
        out = torch.empty((d.T, d.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(lm.latent_moe_workspace_bytes_mxfp4(d), dtype=torch.uint8, device=dev)
        for _ in range(reps + 1):
            lm.latent_moe_forward_mxfp4(d, w, q, x, lg, out, ws)
    elif name == "route":
        route(16384)
    elif name == "route8":
        route(8)
    elif name == "situ":
        x = bf16(W.situ_input(16384, 8192, 0))
        out = torch.empty((16384, 4096), dtype=torch.bfloat16, device=dev)
        for _ in range(reps + 1):
            lm.situ_and_mul(x, out, 4.0, 8.0)
    torch.cuda.synchronize()
    err = lm.lmoe_device_error()
    if err:
        raise SystemExit(f"device error word {err}")
    print(f"{name}: ok")


CASES = ("linear", "layer", "decode", "decode_mxfp4", "route", "route8", "situ")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls instead of CUDA-graph replays (for profiler runs)")
    ap.add_argument("--case", choices=CASES,
                    help="run one small launch set of a kernel (for profiler captures) and exit")
    ap.add_argument("--reps", type=int, default=2, help="launches of --case after one warm-up")
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.reps)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.gpus != 1:
        sys.stderr.write("bench.py: the layer runs on one GPU; --gpus must be 1\n")
        raise SystemExit(2)
    run_ours(args)


if __name__ == "__main__":
    main()
