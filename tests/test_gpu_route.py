"""GPU parity of moe_route against the oracle: ids bit-exact, weights to 1e-6."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import lmoe_oracle as O

pytestmark = pytest.mark.gpu

lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    lm.load_library()
    from tests.gpu_util import DEV  # noqa: F401


def run_route(logits, bias, k, rsf, renorm=1):
    from tests.gpu_util import dev_f32, DEV
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lm.moe_route(dev_f32(logits), None if bias is None else dev_f32(bias), k, rsf, ids, w,
                 renormalize=renorm)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)


def check(logits, bias, k, rsf, renorm=1):
    ids, w = run_route(logits, bias, k, rsf, renorm)
    rids, rw = O.route(logits, bias, k, rsf, renorm)
    bad = np.nonzero((ids != rids).any(1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first token {bad[0]}: {ids[bad[0]]} vs {rids[bad[0]]}"
    rel = np.abs(w - rw) / np.abs(rw)
    assert rel.max() <= 1e-6, rel.max()
    assert lm.lmoe_device_error() == 0


@pytest.mark.parametrize("T", W.ROUTE_TOKENS)
def test_route_workload_896_top16(T):
    logits = W.router_logits(T, W.ROUTE_E, seed=0, tie_every=64)
    check(logits, W.score_bias(W.ROUTE_E, 0), W.ROUTE_K, W.ROUTE_RSF)


def test_route_tie_run_zero_bias():
    # bias = 0 makes every 64th row a full tie: ids 0..15, weights rsf/16
    T = 1024
    logits = W.router_logits(T, W.ROUTE_E, seed=1, tie_every=64)
    check(logits, None, 16, 2.5)
    ids, w = run_route(logits, None, 16, 2.5)
    for t in range(0, T, 64):
        assert ids[t].tolist() == list(range(16))
        assert np.allclose(w[t], 2.5 / 16, rtol=1e-6)


@pytest.mark.parametrize("E,k", [(1, 1), (8, 3), (33, 5), (64, 4), (100, 32), (256, 8),
                                 (512, 16), (1000, 16), (1024, 1)])
def test_route_shapes(E, k):
    T = 97
    g = np.random.default_rng(E * 100 + k)
    logits = g.standard_normal((T, E)).astype(np.float32)
    bias = (g.standard_normal(E) * 0.1).astype(np.float32)
    check(logits, bias, k, 1.5)
    check(logits, bias, k, 1.5, renorm=0)


@pytest.mark.parametrize("E,k,renorm", [(600, 16, 1), (1001, 16, 1), (896, 8, 0), (130, 32, 1),
                                         (257, 3, 1)])
def test_route_warp_kernel_shapes(E, k, renorm):
    # T > 512: the warp-per-token kernel.  E = 600 leaves padded chunks (slots
    # with the logit 0 and the bias -inf), E = 1001 and 257 are not multiples of 4 (4-byte row copies),
    # k = 32 fills the candidate window, renorm = 0 keeps the raw scores
    T = 700
    g = np.random.default_rng(E * 7 + k)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[::64] = logits[::64, :1]          # every 64th row tied
    bias = (g.standard_normal(E) * 0.1).astype(np.float32)
    check(logits, bias, k, 2.5, renorm=renorm)


@pytest.mark.parametrize("T,E,k", [(700, 20, 16), (700, 40, 16), (97, 300, 16), (700, 300, 32)])
def test_route_extreme_bias(T, E, k):
    # biases of +-3e38: doubled cheap keys overflow to +-inf (threshold clamped
    # finite, fewer than k candidates -> the exact selection), tied exact keys
    # of 3e38 (the lower index first); E = 20 with k = 16 leaves fewer than k
    # lanes with an expert, so the k-th lane maximum is -inf
    g = np.random.default_rng(T + E + k)
    logits = g.standard_normal((T, E)).astype(np.float32)
    bias = (g.standard_normal(E) * 0.1).astype(np.float32)
    bias[::7] = -3e38
    bias[3::11] = 3e38
    check(logits, bias, k, 2.5)


def test_route_sigmoid_bit_exact():
    # E = 1, k = 1, no renormalisation, rsf = 1: the weight IS the fp32 sigmoid
    x = np.concatenate([np.linspace(-120, 120, 200001, dtype=np.float32),
                        np.float32([0.0, -0.0, 87.0, -87.0, 88.0, -88.0, 1e-30, -1e-30, 3.4e38,
                                    -3.4e38])])
    ids, w = run_route(x[:, None], None, 1, 1.0, renorm=0)
    got = w[:, 0].astype(np.float32)
    ref = O.sigmoid_f32(x)
    diff = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert diff.size == 0, f"{diff.size} differ, first x={x[diff[0]]}: {got[diff[0]]} vs {ref[diff[0]]}"


def test_route_many_near_ties():
    # logits on a coarse grid with a coarse bias give many equal and nearly
    # equal keys, exercising the candidate bound and the fallback
    T, E = 512, 896
    g = np.random.default_rng(7)
    logits = (g.integers(-8, 8, (T, E)) * 0.25).astype(np.float32)
    bias = (g.integers(-2, 3, E) * 1e-6).astype(np.float32)
    check(logits, bias, 16, 2.5)


def test_route_invalid_arguments_launch_nothing():
    from tests.gpu_util import DEV
    x = torch.zeros((4, 8), device=DEV)
    ids = torch.zeros((4, 2), dtype=torch.int32, device=DEV)
    w = torch.zeros((4, 2), device=DEV)
    for kw, st in [(dict(n_group=2), -3), (dict(topk_group=4), -3)]:
        with pytest.raises(lm.LmoeError) as e:
            lm.moe_route(x, None, 2, 1.0, ids, w, **kw)
        assert e.value.status == st
    # k > E: raw addresses reach the library's own check
    with pytest.raises(lm.LmoeError) as e:
        lm.moe_route(x, None, 9, 1.0, ids.data_ptr(), w.data_ptr())
    assert e.value.status == -2
    # tensors too small for k = 3, or of the wrong dtype: refused by the binding
    with pytest.raises(ValueError):
        lm.moe_route(x, None, 3, 1.0, ids, w)
    with pytest.raises(ValueError):
        lm.moe_route(x.half(), None, 2, 1.0, ids, w)


def _route_cases(n=16, seed=7):
    g = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        E = int(g.integers(1, 1025))
        k = int(g.integers(1, min(E, 32) + 1))
        T = int(g.choice([1, 3, 31, 200, 513, 700, 2049]))
        cases.append((T, E, k, int(g.integers(0, 2)), bool(g.integers(0, 2)),
                      float(g.choice([1.0, 2.5])), float(g.choice([0.1, 1.0, 4.0]))))
    return cases


@pytest.mark.parametrize("case", _route_cases())
def test_route_random_shapes(case):
    # seeded random (T, E, k, renormalise, bias present, rsf, logit scale):
    # both kernels (block per token up to 512 tokens, warp per token above),
    # every chunk count and the scalar loads of E % 4 != 0
    T, E, k, renorm, with_bias, rsf, scale = case
    g = np.random.default_rng(T * 7919 + E * 31 + k)
    logits = (g.standard_normal((T, E)) * scale).astype(np.float32)
    bias = (g.standard_normal(E) * 0.1).astype(np.float32) if with_bias else None
    check(logits, bias, k, rsf, renorm)
