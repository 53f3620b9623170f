"""Pins of the oracle on rows whose sampling filter reaches past the 64 best
tokens: top_p with top_k off, top_k above 64 (alone and with top_p), ties at
the cut value, and an unfiltered target.  Each is checked against brute force
on a small row: a full stable sort in the candidate order (value descending,
then lower id), running sums in fp64, and the smallest prefix whose mass
reaches top_p (the filter order of FreeToken PR 857, "Speed": temperature ->
top_k -> renormalise -> top_p -> renormalise).  No GPU needed.
"""
import numpy as np
import torch

from dflash_draft_selection_gb300 import synth


def _order(z):
    """Token ids in candidate order: value descending, then lower id."""
    return np.lexsort((np.arange(z.shape[0]), -z))


def _brute(z, T, top_k, top_p):
    """The kept prefix (ids in candidate order) and its weights relative to the maximum.  T and
    top_p are taken as the f32 values the sampling record holds."""
    T, top_p = float(np.float32(T)), float(np.float32(top_p))
    z = np.asarray(z, np.float64)
    order = _order(z)
    w = np.exp((z[order] - z[order[0]]) / T)
    k = z.shape[0] if top_k == 0 or top_k >= z.shape[0] else top_k
    w = w[:k]
    n = k
    if top_p < 1.0:
        cum = np.cumsum(w)
        n = int(np.searchsorted(cum, top_p * cum[-1], side="left")) + 1
    return order[:n], w[:n]


def _row(seed, V, scale=1.5):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(V, generator=g) * scale).float()


def _check_topk16(ref, z, T, top_k, top_p):
    ids, w = _brute(z.numpy(), T, top_k, top_p)
    P = w.sum()
    m = float(z.max())
    T = float(np.float32(T))
    idx, U, lse, _ = ref.topk16(z[None], params=synth.make_params(1, T, top_k, top_p))
    order = _order(z.numpy().astype(np.float64))
    assert idx[0].tolist() == order[:16].tolist()
    for j in range(16):
        if j < len(ids):
            want = (float(z[order[j]]) - m) / T - np.log(P)
            assert abs(U[0, j] - want) < 1e-6, (j, U[0, j], want)
        else:
            assert np.isneginf(U[0, j])
    assert abs(lse[0] - (m / T + np.log(P))) < 1e-6
    return ids, w


def _check_target(ref, z, T, top_k, top_p):
    ids, w = _brute(z.numpy(), T, top_k, top_p)
    n, r_ids, r_pr, _ = ref.target_dist(z, T, top_k, top_p)
    assert n == len(ids)
    np.testing.assert_array_equal(r_ids, ids)
    np.testing.assert_allclose(r_pr, w / w.sum(), rtol=1e-12, atol=0)
    return n


def test_deep_top_p_with_top_k_off(ref):
    """top_p 0.9 on a flat row of 3000 tokens: the cut lies thousands of tokens deep."""
    z = _row(1, 3000)
    ids, _ = _check_topk16(ref, z, 1.0, 0, 0.9)
    assert len(ids) > 64
    assert _check_target(ref, z, 1.0, 0, 0.9) > 64
    _check_target(ref, z, 0.7, 0, 0.5)


def test_top_k_above_64(ref):
    z = _row(2, 2000)
    ids, _ = _check_topk16(ref, z, 1.0, 300, 1.0)
    assert len(ids) == 300
    assert _check_target(ref, z, 1.3, 300, 1.0) == 300


def test_top_k_above_64_then_top_p(ref):
    """top_p renormalised over the top_k kept first: the threshold is top_p of the top-500 mass."""
    z = _row(3, 4000)
    ids, w = _check_topk16(ref, z, 1.0, 500, 0.8)
    assert 64 < len(ids) < 500
    _check_target(ref, z, 1.0, 500, 0.8)


def test_ties_at_the_cut_keep_the_lowest_ids(ref):
    """50 tokens at 2.0, 200 at 1.0, the rest at -1.0 (V = 1000).  A cut inside the ties keeps
    the lowest ids among them; every tie carries the same mass, e^-1 of the maximum's."""
    rng = np.random.default_rng(4)
    V = 1000
    z = np.full(V, -1.0, np.float32)
    perm = rng.permutation(V)
    top, tie = np.sort(perm[:50]), np.sort(perm[50:250])
    z[top] = 2.0
    z[tie] = 1.0
    zt = torch.tensor(z)
    # top_k 120 keeps the 50, then the 70 lowest-id ties
    n, ids, pr, _ = ref.target_dist(zt, 1.0, 120, 1.0)
    assert n == 120
    np.testing.assert_array_equal(ids, np.r_[top, tie[:70]])
    P = 50 + 70 * np.exp(-1.0)
    np.testing.assert_allclose(pr, np.r_[np.full(50, 1 / P), np.full(70, np.exp(-1.0) / P)], rtol=1e-12)
    _check_topk16(ref, zt, 1.0, 120, 1.0)
    # top_p set so that the running mass reaches it at the 30th tie
    total = 50 + 200 * np.exp(-1.0) + 750 * np.exp(-3.0)
    tp = (50 + 29.5 * np.exp(-1.0)) / total
    n, ids, pr, _ = ref.target_dist(zt, 1.0, 0, tp)
    assert n == 80
    np.testing.assert_array_equal(ids, np.r_[top, tie[:30]])
    _check_topk16(ref, zt, 1.0, 0, tp)


def test_unfiltered_target_is_the_whole_softmax(ref):
    z = _row(5, 1500)
    n, ids, pr, _ = ref.target_dist(z, 0.8, 0, 1.0)
    assert n == 1500
    zz = z.numpy().astype(np.float64)
    np.testing.assert_array_equal(ids, _order(zz))
    sm = np.exp((zz - zz.max()) / float(np.float32(0.8)))
    np.testing.assert_allclose(pr, (sm / sm.sum())[ids], rtol=1e-12)
