"""The near-tie comparison helpers of the GPU parity tests, checked on the CPU:
identical outcomes pass with nothing excused, a valid alternative at a planted
near-tie passes and is counted, and a wrong outcome fails."""
import numpy as np
import pytest
import torch

from dflash_draft_selection_gb300 import synth
from tests import _parity


def _walk_case():
    """One sampled step whose u sits 1e-7 below the second CDF step of q = (.1, .2, .3, .4)."""
    p = np.array([0.1, 0.2, 0.3, 0.4] + [0.0] * 12)
    S = np.full((1, 2, 16, 16), -np.inf)
    with np.errstate(divide="ignore"):
        S[0, 0, 0] = np.log(p)
        S[0, 1, :, :] = np.log(np.full(16, 1 / 16))
    cand = np.arange(32, dtype=np.int32).reshape(1, 2, 16) + 100
    u = np.array([[0.3 - 1e-7, 0.5]], np.float32)
    return S, cand, u


def test_walk_compare_identical_and_near_tie(ref):
    S, cand, u = _walk_case()
    T = np.ones(1, np.float32)
    pt, ps, q, mg = ref.walk(cand, S, T, u, 1, 2)
    ex = _parity.Excused()
    _parity.walk_compare(ref, cand, S, T, u, pt, ps, q, ex)
    assert ex.excused == 0 and ex.decisions == 2
    # the other neighbour of the CDF step at 0.3: valid, excused, and the walk goes on from it
    assert ps[0, 0] == 1
    ps2, pt2 = ps.copy(), pt.copy()
    ps2[0, 0], pt2[0, 0] = 2, cand[0, 0, 2]
    r2 = ref.walk(cand[:, 1:], np.concatenate([S[:, 1:2, 2:3], S[:, 1:2, :15]], axis=2)[:, :, :16], T, u[:, 1:], 1, 1)
    ps2[0, 1], pt2[0, 1] = r2[1][0, 0], r2[0][0, 0]
    ex = _parity.Excused()
    _parity.walk_compare(ref, cand, S, T, u, pt2, ps2, q, ex)
    assert ex.excused == 1
    # a slot far from the step is not a valid draw
    ps3, pt3 = ps.copy(), pt.copy()
    ps3[0, 0], pt3[0, 0] = 3, cand[0, 0, 3]
    with pytest.raises(AssertionError):
        _parity.walk_compare(ref, cand, S, T, u, pt3, ps3, q, _parity.Excused())


def test_walk_compare_greedy_must_match(ref):
    S, cand, u = _walk_case()
    T = np.zeros(1, np.float32)
    pt, ps, q, _ = ref.walk(cand, S, T, u, 1, 2)
    ps2, pt2 = ps.copy(), pt.copy()
    ps2[0, 0] = 2
    pt2[0, 0] = cand[0, 0, 2]
    with pytest.raises(AssertionError):
        _parity.walk_compare(ref, cand, S, T, u, pt2, ps2, q, _parity.Excused())


def _row(V, probs):
    z = np.full(V, -np.inf, np.float32)
    for i, p in probs.items():
        z[i] = np.log(p)
    return z


def _verify_case(ua0):
    """One sampled request, K = 1: accept test u q vs p(d) = 0.4 with q(d) = 0.5."""
    V = 64
    tl = torch.tensor(np.stack([_row(V, {5: 0.6, 9: 0.4}), _row(V, {3: 0.4, 12: 0.6})]))
    cand = np.zeros((1, 1, 16), np.int32)
    cand[0, 0] = [9, 5] + [x for x in range(V) if x not in (9, 5)][:14]
    q = np.zeros((1, 1, 16))
    q[0, 0, :2] = 0.5
    pt = np.array([[9]], np.int32)
    ps = np.array([[0]], np.int32)
    params = synth.make_params(1, 1.0, 2, 1.0)
    ua = np.array([[ua0]], np.float32)
    ur = np.array([[0.25, 0.5]], np.float32)
    return tl, pt, cand, q, ps, params, ua, ur


def test_verify_compare_identical_and_near_tie(ref):
    # u q = 0.8 * 0.5 = 0.4 = p(d) within rounding: a near-tie accept test
    tl, pt, cand, q, ps, params, ua, ur = _verify_case(np.float32(0.8))
    acc, out, st, mg = ref.verify(tl, pt, cand, q, ps, params, ua, ur, 1, 1)
    assert mg[0] < 1e-5
    ex = _parity.Excused()
    _parity.verify_compare(ref, tl, pt, cand, q, ps, params, ua, ur, acc, out, st, ex)
    assert ex.excused == 0
    # the other side of the test: accept (then the bonus draw) instead of reject, or the reverse
    if acc[0] == 0:
        acc2 = np.array([1], np.int32)
        out2 = np.array([[9, 12]], np.int32)   # bonus at u = .5: CDF over ids 3 (.4), 12 (1.0) -> 12
    else:
        acc2 = np.array([0], np.int32)
        out2 = np.array([[5, -1]], np.int32)   # the residual (p - q)+ lives on token 5 only
    ex = _parity.Excused()
    _parity.verify_compare(ref, tl, pt, cand, q, ps, params, ua, ur, acc2, out2, st, ex)
    assert ex.excused == 1


def test_verify_compare_rejects_a_real_difference(ref):
    tl, pt, cand, q, ps, params, ua, ur = _verify_case(np.float32(0.1))   # 0.05 < 0.4: a clear accept
    acc, out, st, _ = ref.verify(tl, pt, cand, q, ps, params, ua, ur, 1, 1)
    assert acc[0] == 1
    with pytest.raises(AssertionError):
        _parity.verify_compare(ref, tl, pt, cand, q, ps, params, ua, ur, np.array([0], np.int32),
                               np.array([[5, -1]], np.int32), st, _parity.Excused())


def test_topk_compare_near_tie_cut(ref):
    # cumulative masses .5, .8 (top_p at .8 + 1e-7): the cut at 2 or 3 candidates is a near-tie
    z = torch.tensor(_row(64, {7: 0.5, 3: 0.3, 40: 0.15, 12: 0.05}))[None]
    params = synth.make_params(1, 1.0, 0, np.float32(0.8))
    idx, U, lse, mg = ref.topk16(z, params=params)
    assert mg[0] < 1e-5
    ex = _parity.Excused()
    Ug = U.astype(np.float32)
    _parity.topk_compare(z, params, idx, Ug, lse, idx, U, lse, mg, ex)
    assert ex.excused == 0          # the same outputs: nothing to excuse
    # the neighbouring cut, renormalised, is accepted and excused
    kept = int(np.isfinite(U[0]).sum())
    alt = 3 if kept == 2 else 2
    pr = np.array([0.5, 0.3, 0.15, 0.05])
    Ua = np.full((1, 16), -np.inf, np.float32)
    Ua[0, :alt] = np.log(pr[:alt] / pr[:alt].sum())
    ex = _parity.Excused()
    _parity.topk_compare(z, params, idx, Ua, lse, idx, U, lse, mg, ex)
    assert ex.excused == 1
    # a cut two tokens away from the oracle's is not
    far = kept - 2 if kept >= 3 else kept + 2
    Ub = np.full((1, 16), -np.inf, np.float32)
    Ub[0, :far] = np.log(pr[:far] / pr[:far].sum())
    with pytest.raises(AssertionError):
        _parity.topk_compare(z, params, idx, Ub, lse, idx, U, lse, mg, _parity.Excused())
