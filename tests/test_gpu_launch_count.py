"""latent_moe_launch_count (the bench's gpu_launches claim) against the kernel
nodes of a CUDA graph captured from one forward: every launch of both streams
is a kernel node, nothing else launches a kernel."""
import ctypes
import dataclasses

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")

CU_GRAPH_NODE_TYPE_KERNEL = 0


def _kernel_nodes(graph) -> int:
    cu = ctypes.CDLL("libcuda.so.1")
    g = ctypes.c_void_p(graph.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(g, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(g, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    return sum(k == CU_GRAPH_NODE_TYPE_KERNEL for k in kinds)


@pytest.mark.parametrize("T,shared", [(8, True), (300, True), (300, False), (64, False)])
def test_launch_count_matches_captured_kernels(cuda_ok, T, shared):
    if not hasattr(torch.cuda.CUDAGraph, "raw_cuda_graph"):
        pytest.skip("this PyTorch does not expose the captured graph")
    from tests.gpu_util import DEV, weights_to_device, dev_bf16, dev_f32
    lm.load_library()
    d = dataclasses.replace(W.TINY, T=T)
    wts = W.layer_weights(d, 1)
    if not shared:
        wts["ws13"] = wts["ws2"] = None
    wdev = weights_to_device(wts)
    x = dev_bf16(W.hidden_states(d, 1))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, 1))
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes(d), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)   # warm-up outside capture
    s.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this PyTorch cannot keep the captured graph")
    with torch.cuda.graph(g, stream=s):
        lm.latent_moe_forward(d, wdev, x, lg, out, ws, stream=s)
    assert _kernel_nodes(g) == lm.latent_moe_launch_count(d, shared)
    # the forward with its router GEMM
    wr = dev_bf16(W.w_router(d, 1))
    with torch.cuda.stream(s):
        lm.latent_moe_forward_router(d, wdev, wr, x, out, ws, stream=s)
    s.synchronize()
    g2 = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g2, stream=s):
        lm.latent_moe_forward_router(d, wdev, wr, x, out, ws, stream=s)
    assert _kernel_nodes(g2) == lm.latent_moe_launch_count_router(d, shared)


@pytest.mark.parametrize("T", [8, 64, 200, 300])
def test_mxfp4_launch_count_matches_captured_kernels(cuda_ok, T):
    if not hasattr(torch.cuda.CUDAGraph, "raw_cuda_graph"):
        pytest.skip("this PyTorch does not expose the captured graph")
    import numpy as np
    from tests.gpu_util import DEV, weights_to_device, dev_bf16, dev_f32
    lm.load_library()
    d = dataclasses.replace(W.TINY, T=T)
    wdev = weights_to_device(dict(W.layer_weights(d, 1), w13=None, w2=None))
    qdev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(DEV)
            for k, v in W.mxfp4_experts(d, 1).items()}
    x = dev_bf16(W.hidden_states(d, 1))
    lg = dev_f32(W.router_logits(d.T, d.num_experts, 1))
    out = torch.empty((T, d.hidden), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lm.latent_moe_workspace_bytes_mxfp4(d), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lm.latent_moe_forward_mxfp4(d, wdev, qdev, x, lg, out, ws, stream=s)
    s.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this PyTorch cannot keep the captured graph")
    with torch.cuda.graph(g, stream=s):
        lm.latent_moe_forward_mxfp4(d, wdev, qdev, x, lg, out, ws, stream=s)
    assert _kernel_nodes(g) == lm.latent_moe_launch_count_mxfp4(d)
