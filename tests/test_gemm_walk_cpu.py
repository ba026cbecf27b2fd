"""The grouped GEMM's work-unit walk, on the CPU (the library's host copy of the
kernel's unit decoding): every output tile of every group is written by exactly
one (unit, CTA), rows and weight tiles stay inside their group, the two CTAs of
a pair share one operand, and the walk visits the groups in order."""
import numpy as np
import pytest

lm = pytest.importorskip("latent_mixture_experts_sigmoid_gb300")

BM, BN = 128, 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from latent_mixture_experts_sigmoid_gb300 import build
    build.build()
    lm.load_library()


def skewed_counts(G, seed):
    """Token counts per group: many empty, many below one tile, a few large."""
    g = np.random.default_rng(seed)
    c = np.zeros(G, dtype=np.int64)
    kind = g.integers(0, 4, size=G)
    c[kind == 1] = g.integers(1, BM + 1, size=(kind == 1).sum())
    c[kind == 2] = g.integers(BM + 1, 6 * BM, size=(kind == 2).sum())
    c[kind == 3] = g.integers(1, 40, size=(kind == 3).sum()) * 7
    return c


def check_walk(counts, nfeat, paired):
    counts = np.asarray(counts, dtype=np.int64)
    G = len(counts)
    walk = lm.gemm_unit_walk(counts, nfeat, paired)
    first = np.concatenate([[0], np.cumsum(counts)[:-1]])
    tiles = (counts + BM - 1) // BM
    M_feat = BN * nfeat
    seen = {}
    for u in range(walk.shape[0]):
        for r in range(walk.shape[1]):
            row0, nvalid, wrow0, ftile, share_a = (int(v) for v in walk[u, r])
            g, f = divmod(wrow0, M_feat)
            assert f == ftile * BN and 0 <= ftile < nfeat
            assert 0 <= g < G and tiles[g] > 0
            t_in_g, rem = divmod(row0 - int(first[g]), BM)
            assert rem == 0 and 0 <= t_in_g < tiles[g]
            assert nvalid == min(BM, counts[g] - t_in_g * BM) and nvalid > 0
            key = (g, t_in_g, ftile)
            assert key not in seen, (key, u, r, seen.get(key))
            seen[key] = (u, r)
        if paired:
            a, b = walk[u, 0], walk[u, 1]
            assert a[4] == b[4]
            if a[4]:     # shared token tile, weight tiles 2j and 2j + 1
                assert a[0] == b[0] and b[3] == a[3] + 1 and a[3] % 2 == 0
            else:        # shared weight tile, token tiles 2t and 2t + 1
                assert a[2] == b[2] and b[0] == a[0] + BM
    assert len(seen) == int(tiles.sum()) * nfeat
    return walk, tiles


@pytest.mark.parametrize("paired", [0, 1])
@pytest.mark.parametrize("nfeat", [2, 4, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_walk_covers_every_tile_once(paired, nfeat, seed):
    check_walk(skewed_counts(97, seed), nfeat, paired)


def test_walk_edge_cases():
    check_walk([0, 0, 5], 4, 1)              # only one single-tile group
    check_walk([1000, 0, 300], 4, 1)         # no single-tile group
    check_walk([1, 1, 1, 1], 8, 1)           # only single-tile groups
    check_walk([BM, BM + 1, 2 * BM, 2 * BM + 1], 2, 1)   # tile boundaries, odd tile counts
    check_walk([0] * 1023 + [4096], 8, 1)    # 1024 groups, one large
    assert lm.gemm_unit_walk([0, 0], 4, 1).shape[0] == 0
    for bad in [([], 4, 1), ([1], 3, 1), ([-1], 4, 1), ([1] * 1025, 4, 1), ([1], 0, 0)]:
        with pytest.raises(lm.LmoeError):
            lm.gemm_unit_walk(*bad)


@pytest.mark.parametrize("paired", [0, 1])
def test_walk_visits_groups_in_order(paired):
    """Consecutive units (run at the same time by neighbouring CTAs) stay in
    one group and walk its feature tiles fastest, so a group's weights and
    token tiles are shared through L2 while they are in use."""
    nfeat = 4
    counts = skewed_counts(300, 7)
    walk, tiles = check_walk(counts, nfeat, paired)
    g_of = walk[:, 0, 2] // (BN * nfeat)
    assert np.all(np.diff(g_of) >= 0)
    # inside a group: token tile (pair) changes only after all its feature tiles
    for g in np.unique(g_of):
        sel = walk[g_of == g, 0]
        rows = sel[:, 0]
        assert np.all(np.diff(rows) >= 0)
