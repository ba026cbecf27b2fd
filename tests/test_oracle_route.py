"""Pins of the oracle's routing and permutation (CPU only)."""
import numpy as np
import pytest

from oracle import lmoe_oracle as O


def brute_force_route(logits, bias, k, rsf, renormalize=1):
    """Selection by repeated 'largest key, lowest index on ties' (pure Python)."""
    s = O.sigmoid_f32(logits)
    key = (s + bias[None, :]).astype(np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k))
    for t in range(T):
        taken = set()
        for j in range(k):
            best = None
            for e in range(E):
                if e in taken:
                    continue
                if best is None or float(key[t, e]) > float(key[t, best]):
                    best = e
            taken.add(best)
            ids[t, j] = best
        tot = sum(float(s[t, e]) for e in ids[t])
        for j in range(k):
            w[t, j] = float(s[t, ids[t, j]]) / (tot if renormalize else 1.0) * rsf
    return ids, w


def check_brute_force(seed=0):
    g = np.random.default_rng(seed)
    for T, E, k in ((16, 64, 4), (9, 40, 7), (4, 8, 8), (12, 33, 1)):
        # a small value set forces many exact ties
        logits = g.choice(np.float32([-1.5, -0.25, 0.0, 0.5, 2.0]), size=(T, E)).astype(np.float32)
        bias = g.choice(np.float32([0.0, 0.125, -0.125]), size=E).astype(np.float32)
        ids, w = O.route(logits, bias, k, 2.5)
        bids, bw = brute_force_route(logits, bias, k, 2.5)
        assert np.array_equal(ids, bids)
        assert np.allclose(w, bw, rtol=1e-13, atol=0)
        logits = g.standard_normal((T, E)).astype(np.float32)
        bias = (g.standard_normal(E) * 0.1).astype(np.float32)
        ids, w = O.route(logits, bias, k, 2.5, renormalize=0)
        bids, bw = brute_force_route(logits, bias, k, 2.5, renormalize=0)
        assert np.array_equal(ids, bids)
        assert np.allclose(w, bw, rtol=1e-13, atol=0)


def test_route_matches_brute_force_with_ties():
    check_brute_force()


def check_equal_logits_bias_decides():
    # all logits equal: every score is the same, so the bias alone orders the
    # experts and the renormalised weights are exactly rsf / k.
    E, k = 50, 6
    bias = np.random.default_rng(1).permutation(E).astype(np.float32) * np.float32(0.01)
    logits = np.full((3, E), 0.3, np.float32)
    ids, w = O.route(logits, bias, k, 2.5)
    expect = np.argsort(-bias, kind="stable")[:k]
    assert np.all(ids == expect[None, :])
    assert np.allclose(w, 2.5 / k, rtol=1e-15)


def test_equal_logits_bias_decides():
    check_equal_logits_bias_decides()


def test_all_tied_row_takes_lowest_indices():
    logits = np.full((2, 896), -0.7, np.float32)
    ids, w = O.route(logits, np.zeros(896, np.float32), 16, 2.5)
    assert np.all(ids == np.arange(16)[None, :])
    assert np.allclose(w, 2.5 / 16, rtol=1e-15)


def test_zero_bias_is_argsort_of_logits():
    # sigmoid is increasing, so with no bias the selection is the top-k of the
    # logits themselves (values kept where fp32 sigmoid is strictly monotone).
    g = np.random.default_rng(4)
    logits = np.stack([g.permutation(200) for _ in range(5)]).astype(np.float32) * np.float32(0.02) - 2
    ids, _ = O.route(logits, None, 10, 1.0)
    expect = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :10]
    assert np.array_equal(ids, expect)


def test_weights_sum_to_rsf_and_keys_sorted():
    g = np.random.default_rng(5)
    logits = g.standard_normal((64, 896)).astype(np.float32)
    bias = (g.standard_normal(896) * 0.1).astype(np.float32)
    ids, w = O.route(logits, bias, 16, 2.5)
    assert np.allclose(w.sum(1), 2.5, rtol=1e-14)
    key = (O.sigmoid_f32(logits) + bias).astype(np.float32)
    for t in range(64):
        assert len(set(ids[t])) == 16
        sel = key[t, ids[t]]
        assert np.all(np.diff(sel.astype(np.float64)) <= 0)
        rest = np.setdiff1d(np.arange(896), ids[t])
        assert np.all(key[t, rest] <= sel[-1])


def test_unsupported_groups_raise():
    with pytest.raises(NotImplementedError):
        O.route(np.zeros((1, 8), np.float32), None, 2, 1.0, n_group=2)


# --- permutation -------------------------------------------------------------

def check_permute(ids, E):
    counts, offsets, row_of, tok_of_row = O.permute(ids, E)
    T, k = ids.shape
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    # naive O(T*k*E) recomputation: expert e's rows are its tokens ascending
    for e in range(E):
        toks = [t for t in range(T) if e in ids[t]]
        assert counts[e] == len(toks)
        for r, t in enumerate(toks):
            j = int(np.nonzero(ids[t] == e)[0][0])
            assert row_of[t, j] == offsets[e] + r
            assert tok_of_row[offsets[e] + r] == t
    assert sorted(row_of.ravel().tolist()) == list(range(T * k))


def test_permute_against_naive_recount():
    g = np.random.default_rng(6)
    for T, E, k in ((1, 8, 3), (37, 64, 4), (100, 20, 5)):
        ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        check_permute(ids, E)
