"""GPU parity of the tensor-core GEMM engine (lmoe_linear) against float64 matmul."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O

pytestmark = pytest.mark.gpu
lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()


def _bits(g, shape, std):
    return O.f64_to_bf16_bits(g.standard_normal(shape) * std)


@pytest.mark.parametrize("T,N,K", [
    (1, 128, 64), (8, 256, 128), (16, 128, 512), (37, 384, 192), (128, 256, 1024),
    (129, 256, 256), (300, 384, 128), (1024, 512, 2048), (4096, 7168, 2048),
    # CTA pairs: an odd token-tile count puts the last (ragged) tile on pairs of
    # weight tiles that share it (3 tiles x 2, 5 tiles x 4 weight tiles)
    (300, 512, 192), (600, 1024, 320)])
@pytest.mark.parametrize("with_add", [False, True])
def test_linear_matches_float64(T, N, K, with_add):
    from tests.gpu_util import dev_bf16, host_bits, DEV
    g = np.random.default_rng(T * 7 + N + K)
    x = _bits(g, (T, K), 1.0)
    w = _bits(g, (N, K), 0.02)
    add = _bits(g, (T, N), 1.0) if with_add else None
    out = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    lm.lmoe_linear(dev_bf16(x), dev_bf16(w), out, add=None if add is None else dev_bf16(add))
    torch.cuda.synchronize()
    assert lm.lmoe_device_error() == 0
    rows = np.arange(T) if T <= 1024 else np.concatenate([[0, T - 1], np.random.default_rng(0).choice(T, 200, False)])
    ref = O.bf16_to_f64(x[rows]) @ O.bf16_to_f64(w).T
    if add is not None:
        ref = ref + O.bf16_to_f64(add[rows])
    got = O.bf16_to_f64(host_bits(out))[rows]
    scale = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(err <= 8e-3 * np.abs(ref) + 2e-3 * scale), (err.max(), scale)
