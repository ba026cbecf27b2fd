"""Layer parity over a seeded sample of the shapes the ABI accepts (beyond the
benchmark configs): hidden and latent multiples of 128, inter and
shared_inter multiples of 64 (so the fused and unfused SituGLU paths, 128- and
256-wide GEMM tiles and single CTAs as well as CTA pairs all occur), expert
counts that are not multiples of 4 (the routing kernels' scalar loads), top-k
up to 32, and token counts on both sides of the decode/prefill switch.  Each
case is checked against the oracle like the tiny layer (ids and permutation
bit-exact, output per the layer tolerance)."""
import dataclasses

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


def _cases(n=22, seed=20261202):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(g.choice([5, 33, 67, 130, 257, 511, 1000]))
        k = int(min(E, g.choice([1, 2, 6, 8, 16, 32])))
        T = int(g.choice([1, 7, 64, 127, 128, 129, 200, 257, 520]))
        d = W.LayerDims(T=T, hidden=int(128 * g.integers(1, 5)), latent=int(128 * g.integers(1, 4)),
                        num_experts=E, topk=k, inter=int(64 * g.integers(1, 5)),
                        shared_inter=int(64 * g.integers(0, 5)),
                        renormalize=int(g.integers(0, 2)),
                        routed_scaling_factor=float(g.choice([1.0, 2.5])),
                        beta=float(g.choice([1.0, 4.0])),
                        linear_beta=float(g.choice([0.0, 8.0])))
        out.append(d)
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()


@pytest.mark.parametrize("i", range(22))
def test_layer_shape_sample(i):
    from tests.test_gpu_layer import tiny_case
    d = _cases()[i]
    tiny_case(d, seed=100 + i, shared=d.shared_inter > 0)
