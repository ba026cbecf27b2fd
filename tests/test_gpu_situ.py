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


def _pool_map(fn, items):
    """fn over items on the host's cores (NumPy releases the GIL in its loops)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        return list(ex.map(fn, items))


@pytest.mark.parametrize("lb", [8.0, 0.0])
def test_situ_dense_full_size(lb):
    # the [16384, 2*4096] workload: every one of the 67M outputs against the
    # oracle, in blocks of 512 rows
    from tests.gpu_util import host_bits, assert_situ_close
    N, d = 16384, 4096
    x = W.situ_input(N, 2 * d, seed=0)
    out = _dense(x, 4.0, lb)
    o = out.float()
    assert torch.isfinite(o).all()
    if lb > 0:
        assert (o.abs() <= 4.0 * 8.0).all()   # bf16 rounding can reach the bound
    got_all = host_bits(out)

    def block(r0):
        got = O.bf16_to_f64(got_all[r0:r0 + 512])
        ref = O.bf16_to_f64(O.situ_and_mul(x[r0:r0 + 512], 4.0, lb))
        assert_situ_close(got, ref)

    _pool_map(block, range(0, N, 512))


def _masked(x, counts, beta, lb):
    from tests.gpu_util import dev_bf16, dev_i32, DEV
    E, T_max, two_d = x.shape
    out = dev_bf16(W.sentinel_like((E, T_max, two_d // 2)))
    lm.masked_situ_and_mul(dev_bf16(x), out, dev_i32(counts), beta, lb)
    torch.cuda.synchronize()
    return out


def _check_masked(x, counts, out, lb):
    """Every padded output row bit-unchanged, every valid row against the oracle."""
    from tests.gpu_util import host_bits, assert_situ_close
    E, T_max, _ = x.shape
    got_all = host_bits(out)

    def expert(e):
        n = min(max(int(counts[e]), 0), T_max)
        assert (got_all[e, n:] == W.SENTINEL).all(), f"expert {e} padding touched"
        if n:
            got = O.bf16_to_f64(got_all[e, :n])
            ref = O.bf16_to_f64(O.situ_and_mul(x[e, :n], 4.0, lb))
            assert_situ_close(got, ref)

    _pool_map(expert, range(E))


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
    _check_masked(x, counts, out, 8.0)


def test_situ_rejects_missing_beta():
    from tests.gpu_util import DEV
    a = torch.zeros((2, 16), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((2, 8), dtype=torch.bfloat16, device=DEV)
    for beta in (0.0, -1.0, float("nan")):
        with pytest.raises(lm.LmoeError) as e:
            lm.situ_and_mul(a, b, beta, 8.0)
        assert e.value.status == -4
