"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks an oracle function against a closed form, a special case
that reduces to a library routine, brute force on tiny inputs, exact rational
arithmetic, or a Monte Carlo estimate of a known distribution.  A plausible
slip in the oracle (a dropped term, a wrong sign, index or tie rule, a
transposed operand) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
from scipy.special import expit, log_softmax, logsumexp, softmax

from dflash_draft_selection_gb300 import synth


GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_fixed_values.json")))


def bf16(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)


def f32_of(t):
    return t.float().numpy().astype(np.float64)


# ----------------------------------------------------------------- top-16 ----
@pytest.mark.parametrize("V", [16, 17, 64, 4096])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk16_matches_full_stable_sort(ref, V, dtype):
    g = torch.Generator().manual_seed(V)
    # few distinct values so that ties are everywhere
    z = (torch.randint(-6, 6, (9, V), generator=g).float() * 0.5).to(dtype)
    z[3, :] = 1.0                     # a row of all ties
    z[4, ::3] = -0.0
    z[4, 1::3] = 0.0
    idx, U, lse, _ = ref.topk16(z)
    zz = f32_of(z)
    for r in range(z.shape[0]):
        order = np.lexsort((np.arange(V), -zz[r]))  # value desc, then id asc
        assert idx[r].tolist() == order[:16].tolist()


def test_topk16_greedy_U_is_log_softmax(ref):
    g = torch.Generator().manual_seed(1)
    z = torch.randn(5, 1000, generator=g) * 3
    idx, U, lse, _ = ref.topk16(z)
    zz = f32_of(z)
    for r in range(5):
        ls = log_softmax(zz[r])
        np.testing.assert_allclose(U[r], ls[idx[r]], rtol=0, atol=1e-12)
        assert abs(math.fsum(np.exp(zz[r] - lse[r])) - 1.0) < 1e-12


def test_topk16_unfiltered_temperature(ref):
    z = torch.randn(3, 500, generator=torch.Generator().manual_seed(2))
    p = synth.make_params(3, 0.7, 0, 1.0)
    idx, U, lse, _ = ref.topk16(z, params=p)
    zz = f32_of(z)
    for r in range(3):
        ls = log_softmax(zz[r] / 0.7)
        np.testing.assert_allclose(U[r], ls[idx[r]], atol=1e-12)


def test_topk16_filter_closed_forms(ref):
    probs = np.array([0.5, 0.3, 0.15, 0.05])
    V = 64
    z = np.full(V, -np.inf)
    z[[7, 3, 40, 12]] = np.log(probs)           # rank order 7, 3, 40, 12
    z = z.astype(np.float32)
    # top_p 0.75 keeps {7, 3}: cumulative 0.5 < 0.75 <= 0.8
    p = synth.make_params(1, 1.0, 0, 0.75)
    idx, U, lse, mg = ref.topk16(torch.tensor(z)[None], params=p)
    assert idx[0, :4].tolist() == [7, 3, 40, 12]
    np.testing.assert_allclose(U[0, :2], np.log([0.5 / 0.8, 0.3 / 0.8]), atol=1e-7)
    assert np.all(np.isneginf(U[0, 2:]))
    # top_k 3 alone: renormalise over the first three
    p = synth.make_params(1, 1.0, 3, 1.0)
    idx, U, lse, _ = ref.topk16(torch.tensor(z)[None], params=p)
    np.testing.assert_allclose(U[0, :3], np.log(probs[:3] / 0.95), atol=1e-7)
    assert np.all(np.isneginf(U[0, 3:]))
    # top_k 1: the top candidate has probability 1
    p = synth.make_params(1, 1.0, 1, 1.0)
    _, U, _, _ = ref.topk16(torch.tensor(z)[None], params=p)
    assert U[0, 0] == 0.0 and np.all(np.isneginf(U[0, 1:]))
    # temperature 2 on logits 2*log(p) gives p back; then top_p 0.9 keeps three
    z2 = np.full(V, -np.inf)
    z2[[7, 3, 40, 12]] = 2 * np.log(probs)
    p = synth.make_params(1, 2.0, 0, 0.9)
    _, U, _, _ = ref.topk16(torch.tensor(z2.astype(np.float32))[None], params=p)
    np.testing.assert_allclose(U[0, :3], np.log(probs[:3] / 0.95), atol=1e-6)


def test_topk16_filter_invariants(ref):
    g = torch.Generator().manual_seed(3)
    z = torch.randn(20, 3000, generator=g) * 2
    p = synth.make_params(20, 1.3, 20, 0.9)
    idx, U, lse, _ = ref.topk16(z, params=p, rows_per_param=1)
    zz = f32_of(z)
    for r in range(20):
        fin = np.isfinite(U[r])
        k = fin.sum()
        assert 1 <= k <= 16 and np.all(fin[:k]) and not np.any(fin[k:])
        # kept log-probs differ by (z_i - z_j)/T (the softmax shape is kept)
        np.testing.assert_allclose(U[r, :k] - U[r, 0], (zz[r, idx[r, :k]] - zz[r, idx[r, 0]]) / 1.3,
                                   atol=1e-9)
        # the mass of the kept set, normalised inside the top-20, reaches 0.9 and
        # the set without its last member does not
        top20 = np.sort(zz[r])[::-1][:20] / 1.3
        pk = softmax(top20)
        if k < 16:
            assert pk[:k].sum() >= 0.9 - 1e-12 and pk[:k - 1].sum() < 0.9 + 1e-12


def test_topk16_bad_rows(ref):
    z = torch.randn(5, 100)
    z[0, 5] = float("nan")
    z[1, 9] = float("inf")
    z[2, :] = float("-inf")
    z[3, :90] = float("-inf")                 # 10 finite tokens: 6 candidates at -inf
    idx, U, lse, _ = ref.topk16(z)
    for r in range(3):
        assert np.all(idx[r] == -1) and np.all(np.isnan(U[r])) and np.isnan(lse[r])
    assert np.all(np.isfinite(U[3, :10])) and np.all(np.isneginf(U[3, 10:]))
    assert sorted(idx[3, :10].tolist()) == list(range(90, 100))
    assert np.all(np.isfinite(U[4]))
    p = synth.make_params(5, -1.0, 0, 1.0)
    idx, U, lse, _ = ref.topk16(z, params=p)
    assert np.all(idx == -1)


# ------------------------------------------------------------------- gate ----
def test_gate_special_cases(ref):
    g = torch.Generator().manual_seed(4)
    h = torch.randn(6, 64, generator=g)
    W = torch.randn(256, 64, generator=g) / 16
    np.testing.assert_allclose(ref.ctx_gate(h, torch.zeros_like(W)), 0.5, atol=0)
    np.testing.assert_allclose(ref.ctx_gate(torch.zeros_like(h), W), 0.5, atol=0)
    e = torch.zeros(1, 64)
    e[0, 13] = 1.0
    np.testing.assert_allclose(ref.ctx_gate(e, W)[0], expit(W[:, 13].double().numpy()), atol=1e-15)
    ours = ref.ctx_gate(h.bfloat16(), W.bfloat16())
    lib = expit(h.bfloat16().double().numpy() @ W.bfloat16().double().numpy().T)
    np.testing.assert_allclose(ours, lib, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- scores ----
def _chain(ref, B=2, K=3, V=48, D=32, seed=5, scale=1.0, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(B * K, V, generator=g) * 2
    idx, U, lse, _ = ref.topk16(z)
    A = (torch.randn(V, D, generator=g) * scale).to(dtype)
    Bt = (torch.randn(V, D, generator=g) * scale).to(dtype)
    gate = torch.rand(B * K, D, generator=g).double().numpy()
    last = torch.randint(0, V, (B,), generator=g, dtype=torch.int32).numpy()
    return z, idx, U, A, Bt, gate, last


def test_scores_match_einsum_and_reduce_with_zero_factors(ref):
    B, K, V, D = 2, 3, 48, 32
    z, idx, U, A, Bt, gate, last = _chain(ref, B, K, V, D)
    S = ref.pair_scores(idx, U, last, A, Bt, gate, B, K)
    Ad, Bd = A.double().numpy(), Bt.double().numpy()
    ci = idx.reshape(B, K, 16)
    Ur = U.reshape(B, K, 16)
    gr = gate.reshape(B, K, D)
    for b in range(B):
        for t in range(K):
            pred = [last[b]] if t == 0 else ci[b, t - 1]
            lib = Ur[b, t][None, :] + np.einsum("ik,k,jk->ij", Ad[pred], gr[b, t], Bd[ci[b, t]])
            np.testing.assert_allclose(S[b, t, :len(pred)], lib, rtol=1e-12, atol=1e-12)
            if t == 0:
                assert np.all(np.isneginf(S[b, 0, 1:]))
    for zeroed in ("A", "B", "g"):
        A0 = torch.zeros_like(A) if zeroed == "A" else A
        B0 = torch.zeros_like(Bt) if zeroed == "B" else Bt
        g0 = np.zeros_like(gate) if zeroed == "g" else gate
        S0 = ref.pair_scores(idx, U, last, A0, B0, g0, B, K)
        for t in range(K):
            rows = 1 if t == 0 else 16
            np.testing.assert_array_equal(S0[:, t, :rows], np.broadcast_to(Ur[:, t, None, :], (B, rows, 16)))


def test_scores_rank_one_closed_form(ref):
    V, D = 40, 8
    A = torch.zeros(V, D)
    Bt = torch.zeros(V, D)
    A[5, 2] = 3.0
    Bt[:, 2] = torch.arange(V).float()
    idx = np.tile(np.arange(16, dtype=np.int32), (1, 1))
    U = np.zeros((1, 16))
    gate = np.zeros((1, D))
    gate[0, 2] = 0.25
    S = ref.pair_scores(idx, U, np.array([5], np.int32), A, Bt, gate, 1, 1)
    np.testing.assert_array_equal(S[0, 0, 0], 3.0 * 0.25 * np.arange(16))


def test_scores_out_of_range_ids_are_nan(ref):
    z, idx, U, A, Bt, gate, last = _chain(ref, 1, 2, 48, 32)
    idx = idx.copy()
    idx[1, 4] = 48
    S = ref.pair_scores(idx, U, np.array([-3], np.int32), A, Bt, gate, 1, 2)
    assert np.all(np.isnan(S[0, 0, 0]))
    assert np.all(np.isnan(S[0, 1, :, 4])) and np.all(np.isfinite(np.delete(S[0, 1], 4, axis=1)))


# ------------------------------------------------------------------- walk ----
def test_walk_with_zero_A_is_top1_chain(ref):
    B, K = 3, 7
    z, idx, U, A, Bt, gate, last = _chain(ref, B, K, 300, 16, seed=6)
    S = ref.pair_scores(idx, U, last, torch.zeros_like(A), Bt, gate, B, K)
    pt, ps, q, _ = ref.walk(idx, S, np.zeros(B, np.float32), np.zeros((B, K), np.float32), B, K)
    zz = f32_of(z)
    top1 = np.argmax(zz, axis=1).reshape(B, K)    # first maximal id
    np.testing.assert_array_equal(pt, top1)
    assert np.all(ps == 0)
    np.testing.assert_array_equal(q[..., 0], 1.0)


def _brute_scores_row(A, Bt, g, U, a, cands):
    return np.array([U[j] + sum(A[a, k] * g[k] * Bt[c, k] for k in range(len(g)))
                     for j, c in enumerate(cands)])


@pytest.mark.parametrize("seed", [7, 8, 9])
def test_walk_greedy_exhaustive_enumeration(ref, seed):
    B, K, V, D = 2, 3, 64, 8
    z, idx, U, A, Bt, gate, last = _chain(ref, B, K, V, D, seed=seed, scale=2.0)
    S = ref.pair_scores(idx, U, last, A, Bt, gate, B, K)
    pt, ps, q, _ = ref.walk(idx, S, np.zeros(B, np.float32), np.zeros((B, K), np.float32), B, K)
    Ad, Bd = A.double().numpy(), Bt.double().numpy()
    ci, Ur, gr = idx.reshape(B, K, 16), U.reshape(B, K, 16), gate.reshape(B, K, D)
    for b in range(B):
        prev = last[b]
        for t in range(K):
            row = _brute_scores_row(Ad, Bd, gr[b, t], Ur[b, t], prev, ci[b, t])
            best = max(range(16), key=lambda j: (row[j], -j))
            assert ps[b, t] == best and pt[b, t] == ci[b, t, best]
            prev = ci[b, t, best]


def test_walk_sampled_distribution_and_no_zero_q(ref):
    B, K, V, D = 1, 2, 64, 8
    z, idx, U, A, Bt, gate, last = _chain(ref, B, K, V, D, seed=10, scale=1.0)
    U = U.copy()
    U[0, [3, 9, 15]] = -np.inf                   # filtered candidates at position 0
    U[1, [0, 5]] = -np.inf
    S = ref.pair_scores(idx, U, last, A, Bt, gate, B, K)
    R = 1_000_000
    u = torch.rand(R, B, K, generator=torch.Generator().manual_seed(11)).numpy()
    pt, ps, q, _ = ref.walk(idx, S, np.ones(B, np.float32), u, B, K, R=R)
    Ad, Bd = A.double().numpy(), Bt.double().numpy()
    gr = gate.reshape(B, K, D)
    row0 = _brute_scores_row(Ad, Bd, gr[0, 0], U[0], last[0], idx[0])
    q0 = softmax(row0)
    # never a q = 0 candidate
    assert not np.isin(ps[:, 0, 0], [3, 9, 15]).any()
    assert not np.isin(ps[:, 0, 1], [0, 5]).any()
    emp = np.bincount(ps[:, 0, 0], minlength=16) / R
    sd = np.sqrt(q0 * (1 - q0) / R)
    assert np.all(np.abs(emp - q0) <= 5 * sd + 1e-12)
    # joint law of the two steps: q0(j0) * q1(j0, j1)
    joint = np.zeros((16, 16))
    np.add.at(joint, (ps[:, 0, 0], ps[:, 0, 1]), 1.0)
    joint /= R
    expect = np.zeros((16, 16))
    for j0 in range(16):
        row1 = _brute_scores_row(Ad, Bd, gr[0, 1], U[1], idx[0, j0], idx[1])
        expect[j0] = q0[j0] * softmax(row1)
    sd = np.sqrt(expect * (1 - expect) / R)
    assert np.all(np.abs(joint - expect) <= 5 * sd + 1e-12)


def test_walk_inverse_cdf_order(ref):
    # q = softmax(log p) = p; the draw is the first slot whose cumulative mass exceeds u
    p = np.array([0.1, 0.2, 0.3, 0.4] + [0.0] * 12)
    S = np.full((1, 1, 16, 16), -np.inf)
    with np.errstate(divide="ignore"):
        S[0, 0, 0] = np.log(p)
    idx = np.arange(100, 116, dtype=np.int32)[None]
    for u, want in [(0.05, 0), (0.1 - 1e-6, 0), (0.1 + 1e-6, 1), (0.29, 1), (0.31, 2), (0.99, 3)]:
        pt, ps, q, _ = ref.walk(idx, S, np.ones(1, np.float32), np.array([[u]], np.float32), 1, 1)
        assert ps[0, 0] == want and pt[0, 0] == 100 + want
        np.testing.assert_allclose(q[0, 0], p, atol=1e-15)


def test_walk_nan_row_stops(ref):
    S = np.zeros((1, 3, 16, 16))
    S[0, 1, 0, 4] = np.nan
    idx = np.arange(48, dtype=np.int32).reshape(3, 16)
    pt, ps, q, _ = ref.walk(idx, S, np.zeros(1, np.float32), np.zeros((1, 3), np.float32), 1, 3)
    assert pt[0, 0] == 0 and ps[0, 0] == 0
    assert np.all(pt[0, 1:] == -1) and np.all(ps[0, 1:] == -1) and np.all(np.isnan(q[0, 1:]))


# ------------------------------------------------------- target / accept ----
def test_target_dist_greedy_and_sampled(ref):
    y = bf16(np.r_[np.zeros(10), 3.0, 1.0, 3.0, np.zeros(5)])
    n, ids, pr, _ = ref.target_dist(y)
    assert n == 1 and ids[0] == 10 == int(np.argmax(f32_of(y)))
    z = torch.randn(2000, generator=torch.Generator().manual_seed(12)) * 2
    n, ids, pr, _ = ref.target_dist(z, 1.0, 20, 0.95)
    assert 1 <= n <= 20 and abs(pr.sum() - 1) < 1e-12
    zz = f32_of(z)
    top = np.sort(zz)[::-1][:20]
    pk = softmax(top)
    assert pk[:n].sum() >= 0.95 - 1e-12 and (n == 20 or pk[:n - 1].sum() < 0.95)
    np.testing.assert_allclose(pr, pk[:n] / pk[:n].sum(), rtol=1e-12)


def _sparse(ids_list, p_list, cap):
    R = len(ids_list)
    I = np.full((R, cap), -1, np.int32)
    P = np.zeros((R, cap))
    N = np.zeros(R, np.int64)
    for r, (i, p) in enumerate(zip(ids_list, p_list)):
        I[r, :len(i)] = i
        P[r, :len(p)] = p
        N[r] = len(i)
    return I, P, N


def test_accept_p_equals_q_always_accepts(ref):
    K, cap = 3, 16
    cands = np.arange(K * 16, dtype=np.int32).reshape(1, K, 16) + 100
    rng = np.random.default_rng(0)
    q = rng.dirichlet(np.ones(16), size=(1, K))
    ids, ps = [], []
    for t in range(K):
        ids.append(cands[0, t])
        ps.append(q[0, t])
    ids.append(np.array([7], np.int32))
    ps.append(np.array([1.0]))
    I, P, N = _sparse(ids, ps, cap)
    slot = rng.integers(0, 16, size=(1, K)).astype(np.int32)
    path = np.take_along_axis(cands, slot[..., None], 2)[..., 0]
    R = 2000
    ua = rng.random((R, 1, K)).astype(np.float32)
    ur = rng.random((R, 1, K + 1)).astype(np.float32)
    acc, out, st = ref.accept_sparse(I[None], P[None], N[None], np.ones(1, np.float32), path, cands, q,
                                     slot, ua, ur, 1, K, R)
    assert np.all(st == 0) and np.all(acc == K) and np.all(out[:, 0, K] == 7)
    assert np.all(out[:, 0, :K] == path)


def test_accept_disjoint_supports_resample_equals_p(ref):
    K, cap = 1, 8
    cands = (np.arange(16, dtype=np.int32) + 1000).reshape(1, 1, 16)
    q = np.zeros((1, 1, 16))
    q[0, 0, 2] = 1.0
    p_ids = np.array([40, 10, 25], np.int32)        # rank order; ascending id is 10, 25, 40
    p_val = np.array([0.5, 0.3, 0.2])
    I, P, N = _sparse([p_ids, np.array([1], np.int32)], [p_val, np.array([1.0])], cap)
    path = np.array([[1002]], np.int32)
    slot = np.array([[2]], np.int32)
    # inverse CDF over ascending ids: 10 -> (0, .3], 25 -> (.3, .5], 40 -> (.5, 1]
    us = np.array([0.1, 0.29, 0.31, 0.49, 0.51, 0.99], np.float32)
    want = [10, 10, 25, 25, 40, 40]
    R = len(us)
    ua = np.zeros((R, 1, K), np.float32)            # u*q = 0 < p(d) = 0 fails: p(1002) = 0
    ur = np.zeros((R, 1, K + 1), np.float32)
    ur[:, 0, 0] = us
    acc, out, st = ref.accept_sparse(I[None], P[None], N[None], np.ones(1, np.float32), path, cands, q,
                                     slot, ua, ur, 1, K, R)
    assert np.all(acc == 0) and out[:, 0, 0].tolist() == want and np.all(out[:, 0, 1] == -1)


def test_greedy_verify_is_longest_prefix(ref):
    g = torch.Generator().manual_seed(13)
    B, K, V = 6, 5, 300
    y = torch.randn(B * (K + 1), V, generator=g).bfloat16()
    am = np.argmax(f32_of(y), axis=1).reshape(B, K + 1)
    path = am[:, :K].copy().astype(np.int32)
    for b in range(B):
        if b < K:
            path[b, b] = (path[b, b] + 1) % V      # first mismatch at position b
    cands = np.zeros((B, K, 16), np.int32)
    q = np.zeros((B, K, 16))
    slot = np.zeros((B, K), np.int32)
    acc, out, st, _ = ref.verify(y, path, cands, q, slot, None, np.zeros((B, K), np.float32),
                                 np.zeros((B, K + 1), np.float32), B, K)
    for b in range(B):
        n = 0
        while n < K and path[b, n] == am[b, n]:
            n += 1
        assert acc[b] == n and st[b] == 0
        assert out[b, :n].tolist() == path[b, :n].tolist() and out[b, n] == am[b, n]
        assert np.all(out[b, n + 1:] == -1)


def test_verify_status_rows(ref):
    B, K, V = 5, 2, 200
    y = torch.randn(B * (K + 1), V, generator=torch.Generator().manual_seed(14))
    y[0 * (K + 1) + 1, 7] = float("nan")
    cands = np.tile(np.arange(16, dtype=np.int32), (B, K, 1))
    q = np.full((B, K, 16), 1 / 16)
    q[2] *= 1.01                                     # wrong total
    q[3, 1, 4] = np.nan
    slot = np.zeros((B, K), np.int32)
    path = np.zeros((B, K), np.int32)
    p = synth.make_params(B, 1.0, 10, 1.0)
    p["top_p"][4] = 0.0                              # invalid
    ua = np.full((B, K), 0.5, np.float32)
    ur = np.full((B, K + 1), 0.5, np.float32)
    acc, out, st, _ = ref.verify(y, path, cands, q, slot, p, ua, ur, B, K)
    assert st.tolist() == [ref.ST_NAN, 0, ref.ST_BAD_Q, ref.ST_NAN, ref.ST_BAD_PARAMS]
    for b in (0, 2, 3, 4):
        assert acc[b] == 0 and np.all(out[b] == -1)
    acc2, out2, st2, _ = ref.verify(y, path, cands, q, slot, p, ua, ur, B, K, trusted=True)
    assert st2[2] == 0


def test_accept_monte_carlo_marginals_6M_rows(ref):
    """6M verify rows: committed-token marginals at each position within 5e-3 of p_t.

    FreeToken PR 857 "Accuracy" (Monte Carlo over 6M rows, marginals within
    5e-3 of the target distribution).  Each repetition redraws the path with
    a sampled walk and then runs the accept walk.  Synthetic p_t does not
    depend on the prefix, so every committed token at position t must follow
    p_t, and the acceptance rate at t = 0 must equal sum_v min(p, q).
    """
    B, K, V = 4, 3, 2048
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=21, target_noise=1.0)
    inp = synth.make_inputs(shp, with_conv=False)
    idx, U, lse, _ = ref.topk16(inp.draft_logits, params=inp.params, rows_per_param=K)
    z, _, _, A, Bt, gate, _ = _chain(ref, B, K, V, 32, seed=23, scale=0.5)
    S = ref.pair_scores(idx, U, inp.last_tok, A, Bt, gate, B, K)
    T = inp.params["temperature"]
    cap = 20
    I = np.zeros((B, K + 1, cap), np.int32)
    P = np.zeros((B, K + 1, cap))
    N = np.zeros((B, K + 1), np.int64)
    for b in range(B):
        for t in range(K + 1):
            smp = GOLDEN["recommended_sampling"]
            n, ids, pr, _ = ref.target_dist(inp.target_logits[b * (K + 1) + t], smp["temperature"], smp["top_k"],
                                            smp["top_p"])
            I[b, t, :n], P[b, t, :n], N[b, t] = ids, pr, n
    R = GOLDEN["mc_rows"] // B                      # x B = 6M rows
    tol = GOLDEN["mc_marginal_tol"]
    g = torch.Generator().manual_seed(22)
    uw = torch.rand(R, B, K, generator=g).numpy()
    ua = torch.rand(R, B, K, generator=g).numpy()
    ur = torch.rand(R, B, K + 1, generator=g).numpy()
    acc, out = ref.walk_accept_mc(idx, S, T, I, P, N, uw, ua, ur, B, K, R)
    for b in range(B):
        for t in range(K + 1):
            reached = acc[:, b] >= t
            toks = out[reached, b, t]
            assert toks.size > 10000 and np.all(toks >= 0)
            cnt = np.bincount(toks, minlength=V) / toks.size
            expect = np.zeros(V)
            expect[I[b, t, :N[b, t]]] = P[b, t, :N[b, t]]
            assert np.max(np.abs(cnt - expect)) < tol, (b, t)
        # acceptance at t = 0 is sum_v min(p, q), q the walk's law at t = 0
        q0 = softmax(S[b, 0, 0])
        pmap = dict(zip(I[b, 0, :N[b, 0]].tolist(), P[b, 0, :N[b, 0]].tolist()))
        qmap = {int(c): float(qq) for c, qq in zip(idx.reshape(B, K, 16)[b, 0], q0)}
        alpha = sum(min(pmap.get(v, 0.0), qmap.get(v, 0.0)) for v in set(pmap) | set(qmap))
        rate = np.mean(acc[:, b] >= 1)
        assert abs(rate - alpha) <= 5 * math.sqrt(alpha * (1 - alpha) / R) + 1e-9


# ------------------------------------------------------------------- conv ----
def test_conv_identity_and_shift(ref):
    g = torch.Generator().manual_seed(15)
    B, T, H = 2, 5, 24
    x = torch.randn(B, T, H, generator=g).bfloat16()
    xp = torch.randn(B, H, generator=g).bfloat16()
    one, zero = torch.ones(B, T, H).bfloat16(), torch.zeros(B, T, H).bfloat16()
    assert torch.equal(ref.conv2tap(x, one, zero, xp), x)
    y = ref.conv2tap(x, zero, one, xp)
    assert torch.equal(y[:, 0], xp) and torch.equal(y[:, 1:], x[:, :-1])
    # grouped taps: group of 4 channels shares one tap pair
    k0 = torch.randn(B, T, H // 4, generator=g).bfloat16()
    k1 = torch.zeros(B, T, H // 4).bfloat16()
    yg = ref.conv2tap(x, k0, k1, xp, group=4)
    yf = ref.conv2tap(x, k0.repeat_interleave(4, dim=2), k1.repeat_interleave(4, dim=2), xp)
    assert torch.equal(yg, yf)


def _nearest_bf16_ok(y, exact):
    """y is a bf16 value nearest to the exact rational (ties to even mantissa)."""
    yv = Fraction(float(y))
    bits = torch.tensor([float(y)]).bfloat16().view(torch.int16).item() & 0xFFFF
    up = torch.tensor([bits + 1], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item()
    dn = torch.tensor([bits - 1], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item()
    d = abs(yv - exact)
    for nb in (up, dn):
        dn_ = abs(Fraction(nb) - exact)
        if dn_ < d or (dn_ == d and (bits & 1)):
            return False
    return True


def _conv1(x, k0, k1, xp):
    t = lambda v: torch.tensor([[[v]]]).bfloat16()
    return torch.tensor([[xp]]).bfloat16(), t(x), t(k0), t(k1)


def test_conv_rounding_is_exact_nearest_even(ref):
    def y(x, k0, k1, xp):
        xp_, x_, k0_, k1_ = _conv1(x, k0, k1, xp)
        return float(ref.conv2tap(x_, k0_, k1_, xp_))
    # 1 + 2^-8 is the midpoint of 1 (even) and 1 + 2^-7 (odd): ties to even
    assert y(1.0, 1.0, 2 ** -8, 1.0) == 1.0
    # just above / below that midpoint
    assert y(1.0, 1.0, 2 ** -8, 1 + 2 ** -7) == 1 + 2 ** -7
    assert y(1.0, 1.0, 2 ** -8, 1 - 2 ** -8) == 1.0
    # 1 + 2^-7 + 2^-8 is the midpoint of 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert y(1.0, 1 + 2 ** -7, 2 ** -8, 1.0) == 1 + 2 ** -6
    # a single product on a midpoint (7/8 * 37/32 = 259/256) plus a second product
    # far below fp64 resolution: the tiny term decides the side
    assert y(37 / 32, 7 / 8, -(2 ** -30), 2 ** -30) == 1 + 2 ** -7
    assert y(37 / 32, 7 / 8, 2 ** -30, 2 ** -30) == 1 + 2 ** -6
    assert y(37 / 32, 7 / 8, 0.0, 1.0) == 1 + 2 ** -6


def test_conv_random_against_exact_rationals(ref):
    # random inputs against exact rational arithmetic
    g = torch.Generator().manual_seed(16)
    B, T, H = 2, 4, 64
    x = torch.randn(B, T, H, generator=g).bfloat16()
    k0 = (torch.rand(B, T, H, generator=g) * 2 - 1).bfloat16()
    k1 = (torch.rand(B, T, H, generator=g) * 2 - 1).bfloat16()
    xp = torch.randn(B, H, generator=g).bfloat16()
    y = ref.conv2tap(x, k0, k1, xp)
    prev = torch.cat([xp[:, None], x[:, :-1]], dim=1)
    for i in np.ndindex(B, T, H):
        ex = Fraction(float(k0[i])) * Fraction(float(x[i])) + Fraction(float(k1[i])) * Fraction(float(prev[i]))
        assert _nearest_bf16_ok(float(y[i]), ex), i


def test_conv_f32_exact_rounding(ref):
    g = torch.Generator().manual_seed(17)
    x = torch.randn(1, 3, 50, generator=g)
    k0 = torch.rand(1, 3, 50, generator=g)
    k1 = torch.rand(1, 3, 50, generator=g)
    xp = torch.randn(1, 50, generator=g)
    y = ref.conv2tap(x, k0, k1, xp)
    prev = torch.cat([xp[:, None], x[:, :-1]], dim=1)
    for i in np.ndindex(1, 3, 50):
        ex = Fraction(float(k0[i])) * Fraction(float(x[i])) + Fraction(float(k1[i])) * Fraction(float(prev[i]))
        yv = Fraction(float(y[i]))
        # nearest f32: no other f32 is closer (compare with the f32 neighbours)
        f = np.float32(y[i])
        for nb in (np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))):
            assert abs(Fraction(float(nb)) - ex) >= abs(yv - ex)


# ------------------------------------------------- decision margins ----
# Every GPU parity test excuses a decision whose oracle margin is below 1e-5
# (the pages accept near-ties: FreeToken PR 857, "Accuracy").  These pins fix
# the margins themselves to planted distances, so that a margin that came out
# too small (excusing everything) or too large fails here.
def _planted_row(V, probs_by_id):
    """f32 logits whose softmax puts `probs_by_id` on those ids and nothing elsewhere."""
    z = np.full(V, -np.inf, np.float32)
    for i, p in probs_by_id.items():
        z[i] = np.log(p) if p > 0 else -np.inf
    return z


def test_topk16_top_p_margin_is_the_planted_gap(ref):
    z = _planted_row(64, {7: 0.5, 3: 0.3, 40: 0.15, 12: 0.05})
    # top_p 0.75: cumulative 0.5 (gap 0.25) then 0.8 (gap 0.05, cut): margin 0.05
    _, _, _, mg = ref.topk16(torch.tensor(z)[None], params=synth.make_params(1, 1.0, 0, 0.75))
    assert abs(mg[0] - 0.05) < 1e-6
    # a cut planted 3e-6 away from a cumulative mass: the row is a near-tie
    _, U, _, mg = ref.topk16(torch.tensor(z)[None], params=synth.make_params(1, 1.0, 0, 0.8 + 3e-6))
    assert abs(mg[0] - 3e-6) < 5e-7
    assert np.isfinite(U[0, :3]).all() and np.isneginf(U[0, 3:]).all()
    # no top_p decision, no margin
    for p in (synth.make_params(1, 1.0, 3, 1.0), synth.make_params(1, 0.0, 0, 1.0), None):
        _, _, _, mg = ref.topk16(torch.tensor(z)[None], params=p)
        assert np.isinf(mg[0])


def test_walk_greedy_margin_is_best_minus_second(ref):
    idx = np.arange(100, 116, dtype=np.int32)[None]
    for row, want_slot, want_mg in [([1.0, 1.37, 0.5], 1, 0.37), ([2.0, 2.0, 1.0], 0, 0.0),
                                    ([0.25], 0, np.inf), ([-1.0, -1.0 + 2 ** -20, -3.0], 1, 2 ** -20)]:
        S = np.full((1, 1, 16, 16), -np.inf)
        S[0, 0, 0, :len(row)] = row
        pt, ps, q, mg = ref.walk(idx, S, np.zeros(1, np.float32), np.zeros((1, 1), np.float32), 1, 1)
        assert ps[0, 0] == want_slot and pt[0, 0] == 100 + want_slot
        assert mg[0, 0] == pytest.approx(want_mg, abs=1e-15) if np.isfinite(want_mg) else np.isinf(mg[0, 0])


def test_walk_sampled_margin_is_distance_to_nearest_cdf_step(ref):
    p = np.array([0.1, 0.2, 0.3, 0.4] + [0.0] * 12)
    S = np.full((1, 1, 16, 16), -np.inf)
    with np.errstate(divide="ignore"):
        S[0, 0, 0] = np.log(p)
    idx = np.arange(100, 116, dtype=np.int32)[None]
    # CDF steps at 0.1, 0.3, 0.6, 1.0
    for u, slot, gap in [(0.31, 2, 0.01), (0.5, 2, 0.1), (0.0999, 0, 1e-4), (0.95, 3, 0.05)]:
        _, ps, _, mg = ref.walk(idx, S, np.ones(1, np.float32), np.array([[u]], np.float32), 1, 1)
        assert ps[0, 0] == slot
        assert abs(mg[0, 0] - gap) < 1e-7        # u is an f32: |u - f32(u)| < 3e-9


def test_walk_sampled_fallback_takes_the_last_positive_slot(ref):
    """u = 1 crosses no CDF step (the running sum reaches the total exactly, never
    above it): the draw falls back to the last slot with q > 0, skipping the
    -inf slots after it."""
    p = np.array([0.1, 0.2, 0.0, 0.3, 0.4] + [0.0] * 11)
    S = np.full((1, 1, 16, 16), -np.inf)
    with np.errstate(divide="ignore"):
        S[0, 0, 0] = np.log(p)
    idx = np.arange(100, 116, dtype=np.int32)[None]
    _, ps, q, _ = ref.walk(idx, S, np.ones(1, np.float32), np.ones((1, 1), np.float32), 1, 1)
    assert ps[0, 0] == 4 and q[0, 0, 4] > 0 and np.all(q[0, 0, 5:] == 0)


def _verify_case(ref, rows, cands, qs, path, slot, u_acc, u_res, top_k=0, top_p=1.0, trusted=False, V=64):
    """One sampled request (T = 1) with planted target rows (dicts id -> p) and q rows."""
    K = len(path)
    y = np.stack([_planted_row(V, r) for r in rows])
    cand = np.zeros((1, K, 16), np.int32)
    q = np.zeros((1, K, 16))
    for t in range(K):
        c = list(cands[t]) + [x for x in range(V) if x not in cands[t]][:16 - len(cands[t])]
        cand[0, t] = c
        q[0, t, :len(qs[t])] = qs[t]
    params = synth.make_params(1, 1.0, top_k, top_p)
    return ref.verify(torch.tensor(y), np.array([path], np.int32), cand, q, np.array([slot], np.int32), params,
                      np.array([u_acc], np.float32), np.array([u_res], np.float32), 1, K, trusted=trusted)


def test_verify_margin_of_an_accept_test_and_of_a_draw(ref):
    rows = [{5: 0.6, 9: 0.4}, {3: 0.4, 12: 0.6}]
    # accept: u q = 0.7 * 0.5 = 0.35 < p = 0.4 (gap 0.05); bonus draw over ids 3, 12 at u = 0.5:
    # CDF steps 0.4 (gap 0.1) and 1.0 -> token 12
    acc, out, st, mg = _verify_case(ref, rows, [[9, 5]], [[0.5, 0.5]], [9], [0], [0.7], [0.3, 0.5], top_k=2)
    assert st[0] == 0 and acc[0] == 1 and out[0].tolist() == [9, 12]
    assert abs(mg[0] - 0.05) < 1e-6
    # reject: 0.9 * 0.5 = 0.45 >= 0.4 (gap 0.05); the residual max(0, p - q) is 0.1 on token 5 only,
    # drawn at u = 0.99: relative gap 1 - 0.99 = 0.01 binds
    acc, out, st, mg = _verify_case(ref, rows, [[9, 5]], [[0.5, 0.5]], [9], [0], [0.9], [0.99, 0.5], top_k=2)
    assert acc[0] == 0 and out[0].tolist() == [5, -1]
    assert abs(mg[0] - 0.01) < 1e-6


def test_verify_margin_ignores_rows_the_request_never_used(ref):
    """A top_p cut within 1e-8 of a cumulative mass on the bonus row must not
    excuse a request that stopped at position 0."""
    rows = [{5: 0.6, 9: 0.4}, {5: 0.6, 9: 0.4}, {2: 0.7, 8: 0.3}]
    acc, out, st, mg = _verify_case(ref, rows, [[9, 5], [5, 9]], [[0.5, 0.5], [0.5, 0.5]], [9, 5], [0, 0],
                                    [0.9, 0.1], [0.5, 0.5, 0.5], top_p=0.7)
    assert acc[0] == 0 and out[0, 0] == 5
    # used: row 0's cut (cumulative 0.6, 1.0 against 0.7: gap 0.1), the accept test (0.05), the draw
    assert abs(mg[0] - 0.05) < 1e-6
    # the same bonus row is a near-tie once the request reaches it
    acc, out, st, mg = _verify_case(ref, rows, [[9, 5], [5, 9]], [[0.5, 0.5], [0.5, 0.5]], [9, 5], [0, 0],
                                    [0.1, 0.1], [0.5, 0.5, 0.5], top_p=0.7)
    assert acc[0] == 2 and mg[0] < 1e-6


def test_verify_zero_residual_draws_from_p(ref):
    """A trusted q that is >= p on all of p's support (here q sums to 2.2) leaves a
    zero residual: the corrected token is drawn from p itself, by inverse CDF
    over ascending token ids.  p = {10: .3, 25: .2, 40: .5} has CDF steps .3,
    .5, 1; q normalised would put them at .318, .591, 1, so the two laws give
    different tokens at u = .31 and u = .55."""
    rows = [{40: 0.5, 10: 0.3, 25: 0.2}, {1: 1.0}]
    for u, want in [(0.31, 25), (0.55, 40), (0.2, 10), (0.9, 40)]:
        acc, out, st, _ = _verify_case(ref, rows, [[40, 10, 25]], [[0.9, 0.7, 0.6]], [40], [0], [0.7], [u, 0.5],
                                       top_k=3, trusted=True)
        assert st[0] == 0 and acc[0] == 0 and out[0, 0] == want, (u, out[0])


def test_verify_draw_fallback_takes_the_last_positive_token(ref):
    """u = 1 crosses no CDF step: the bonus draw falls back to the largest
    token id with positive probability."""
    rows = [{5: 0.6, 9: 0.4}, {3: 0.4, 12: 0.6, 30: 0.0}]
    acc, out, st, _ = _verify_case(ref, rows, [[9, 5]], [[0.5, 0.5]], [9], [0], [0.1], [0.5, 1.0], top_k=3)
    assert acc[0] == 1 and out[0].tolist() == [9, 12]
