"""GPU parity of situ_and_mul / masked_situ_and_mul against the oracle."""
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


def _dense(x_bits, beta, lb):
    from tests.gpu_util import dev_bf16, DEV
    N, two_d = x_bits.shape
    out = torch.empty((N, two_d // 2), dtype=torch.bfloat16, device=DEV)
    lm.situ_and_mul(dev_bf16(x_bits), out, beta, lb)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("N,d", [(1, 8), (3, 24), (257, 128), (1000, 512), (64, 4096)])
@pytest.mark.parametrize("lb", [8.0, 0.0])
def test_situ_dense_small(N, d, lb):
    from tests.gpu_util import host_bits, assert_situ_close
    x = W.situ_input(N, 2 * d, seed=N + d)
    got = O.bf16_to_f64(host_bits(_dense(x, 4.0, lb)))
    ref = O.bf16_to_f64(O.situ_and_mul(x, 4.0, lb))
    assert_situ_close(got, ref)


@pytest.mark.parametrize("lb", [8.0, 0.0])
def test_situ_dense_full_size_sampled(lb):
    # the [16384, 2*4096] workload; every output is checked on the GPU against
    # finite/bounded properties, and 96 sampled rows against the oracle
    from tests.gpu_util import host_bits, assert_situ_close
    N, d = 16384, 4096
    x = W.situ_input(N, 2 * d, seed=0)
    out = _dense(x, 4.0, lb)
    o = out.float()
    assert torch.isfinite(o).all()
    if lb > 0:
        assert (o.abs() <= 4.0 * 8.0).all()   # bf16 rounding can reach the bound
    rows = np.random.default_rng(1).choice(N, 96, replace=False)
    rows = np.concatenate([[0, N - 1], rows])
    got = O.bf16_to_f64(host_bits(out[torch.from_numpy(rows).cuda()]))
    ref = O.bf16_to_f64(O.situ_and_mul(x[rows], 4.0, lb))
    assert_situ_close(got, ref)


def _masked(x, counts, beta, lb):
    from tests.gpu_util import dev_bf16, dev_i32, DEV
    E, T_max, two_d = x.shape
    out = dev_bf16(W.sentinel_like((E, T_max, two_d // 2)))
    lm.masked_situ_and_mul(dev_bf16(x), out, dev_i32(counts), beta, lb)
    torch.cuda.synchronize()
    return out


def _check_masked(x, counts, out, lb, sample_rows=None):
    from tests.gpu_util import host_bits, assert_situ_close
    E, T_max, _ = x.shape
    bits = out.view(torch.int16)
    for e in range(E):
        n = min(max(int(counts[e]), 0), T_max)
        pad = bits[e, n:]
        assert (pad == np.int16(np.uint16(W.SENTINEL).view(np.int16))).all(), f"expert {e} padding touched"
        if n:
            rows = range(n) if sample_rows is None else sorted(set(
                [0, n - 1] + list(np.random.default_rng(e).choice(n, min(n, sample_rows), replace=False))))
            rows = list(rows)
            got = O.bf16_to_f64(host_bits(out[e, rows]))
            ref = O.bf16_to_f64(O.situ_and_mul(x[e, rows], 4.0, lb))
            assert_situ_close(got, ref)


@pytest.mark.parametrize("lb", [8.0, 0.0])
def test_masked_small_with_clamped_counts(lb):
    x, counts = W.masked_situ_input(9, 40, 2 * 64, seed=5)
    counts = counts.copy()
    counts[0], counts[1], counts[2] = -3, 1000, 0     # clamped to 0, T_max, 0
    _check_masked(x, counts, _masked(x, counts, 4.0, lb), lb)


def test_masked_full_size():
    # [E=128, T_max=512, 2*2048] with counts uniform in [0, 512]
    x, counts = W.masked_situ_input(128, 512, 2 * 2048, seed=0)
    out = _masked(x, counts, 4.0, 8.0)
    _check_masked(x, counts, out, 8.0, sample_rows=3)


def test_situ_rejects_missing_beta():
    from tests.gpu_util import DEV
    a = torch.zeros((2, 16), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((2, 8), dtype=torch.bfloat16, device=DEV)
    for beta in (0.0, -1.0, float("nan")):
        with pytest.raises(lm.LmoeError) as e:
            lm.situ_and_mul(a, b, beta, 8.0)
        assert e.value.status == -4
