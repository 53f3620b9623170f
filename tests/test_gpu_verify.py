"""dflash2_verify against the oracle: bit-exact statuses, accept counts and
tokens, except at a decision whose oracle margin is below 1e-5, which must be a
valid outcome of a near-tie and after which the oracle goes on with the GPU's
decision forced (tests/_parity.py; at most 1% of the decisions excused); plus
a Monte Carlo of the committed-token marginals on the GPU."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests import _parity
from tests._util import MARGIN, cuda_or_skip, padded, params_np

pytestmark = pytest.mark.gpu


def oracle_walk_inputs(ref, inp, B, K):
    """Candidates, path and q from the oracle's topk/walk (selector term zero)."""
    idx, U, lse, _ = ref.topk16(inp.draft_logits, params=inp.params, rows_per_param=K)
    S = np.broadcast_to(U.reshape(B, K, 1, 16), (B, K, 16, 16)).copy()
    pt, ps, q, _ = ref.walk(idx, S, inp.params["temperature"], inp.u_walk, B, K)
    return idx.reshape(B, K, 16), pt, ps, q


def run_gpu_verify(inp, cand, pt, ps, q, params, B, K, trusted=False, V=None):
    dev = cuda_or_skip()
    pg = None if params is None else d2.sampling_params(params["temperature"], params["top_k"], params["top_p"],
                                                        device=dev)
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dt).to(dev)
    acc, out, st = d2.verify(padded(inp.target_logits.to(dev)), t(pt, torch.int32), t(cand, torch.int32),
                             t(q, torch.float32), t(ps, torch.int32), params=pg, u_acc=inp.u_acc.to(dev),
                             u_res=inp.u_res.to(dev), trusted=trusted, V=V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), st.cpu().numpy()


def check(ref, inp, cand, pt, ps, q, params, B, K, trusted=False):
    acc, out, st = run_gpu_verify(inp, cand, pt, ps, q, params, B, K, trusted)
    # the oracle sees the same f32 q the GPU sees
    ex = _parity.Excused()
    _parity.verify_compare(ref, inp.target_logits, pt, cand, q.astype(np.float32), ps, params, inp.u_acc.numpy(),
                           inp.u_res.numpy(), acc, out, st, ex, trusted=trusted)
    ex.check_bound(what="verify")
    return acc, ex


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [64, 4096 + 5, 20000])
def test_greedy_prefix(ref, dtype, V):
    B, K = 9, 7
    shp = synth.small_shape("27b_greedy", B=B, K=K, V=V, hidden=64, seed=V, dtype=dtype)
    inp = synth.make_inputs(shp, with_conv=False)
    zz = inp.target_logits.float().numpy()
    am = np.argmax(zz, axis=1).reshape(B, K + 1)
    pt = am[:, :K].copy().astype(np.int32)
    for b in range(B):
        if b < K:
            pt[b, b] = (pt[b, b] + 1) % V
    cand = np.zeros((B, K, 16), np.int32)
    cand[..., 0] = pt
    ps = np.zeros((B, K), np.int32)
    q = np.zeros((B, K, 16))
    q[..., 0] = 1.0
    acc, ex = check(ref, inp, cand, pt, ps, q, None, B, K)
    assert ex.excused == 0
    assert acc.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 7]


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("T,k,p", [(1.0, 20, 0.95), (0.7, 8, 1.0), (1.0, 64, 0.9), (1.5, 3, 0.6)])
def test_sampled_parity(ref, seed, T, k, p):
    B, K, V = 16, 7, 9000
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=seed, temperature=T, top_k=k, top_p=p,
                            target_noise=1.0)
    inp = synth.make_inputs(shp, with_conv=False)
    cand, pt, ps, q = oracle_walk_inputs(ref, inp, B, K)
    check(ref, inp, cand, pt, ps, q, inp.params, B, K)


def test_mixed_greedy_and_sampled(ref):
    B, K, V = 6, 4, 3000
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=9, target_noise=0.5)
    inp = synth.make_inputs(shp, with_conv=False)
    inp.params["temperature"][[1, 4]] = 0.0
    cand, pt, ps, q = oracle_walk_inputs(ref, inp, B, K)
    check(ref, inp, cand, pt, ps, q, inp.params, B, K)


def test_status_rows(ref):
    B, K, V = 6, 3, 500
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=11)
    inp = synth.make_inputs(shp, with_conv=False)
    cand, pt, ps, q = oracle_walk_inputs(ref, inp, B, K)
    inp.target_logits[0 * (K + 1) + 2, 7] = float("nan")
    q = q.copy()
    q[1] *= 1.01                                  # wrong total
    q[2, 1, 3] = np.nan
    ps = ps.copy()
    ps[3, 0] = (ps[3, 0] + 1) % 16                # drafted token not at its slot
    inp.params["top_p"][4] = 0.0                  # invalid
    acc, out, st = run_gpu_verify(inp, cand, pt, ps, q, inp.params, B, K)
    r_acc, r_out, r_st, _ = ref.verify(inp.target_logits, pt, cand, q, ps, inp.params, inp.u_acc, inp.u_res, B, K)
    np.testing.assert_array_equal(st, r_st)
    assert st.tolist()[:5] == [d2.binding.ST_NAN, d2.binding.ST_BAD_Q, d2.binding.ST_NAN, d2.binding.ST_BAD_Q,
                               d2.binding.ST_BAD_PARAMS]
    for b in range(5):
        assert acc[b] == 0 and np.all(out[b] == -1)
    # trusted: the wrong-total request is accepted as given
    acc2, out2, st2 = run_gpu_verify(inp, cand, pt, ps, q, inp.params, B, K, trusted=True)
    assert st2[1] == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("seed", [1, 2])
def test_wide_target_rows(ref, seed, dtype):
    """Sampled requests whose target distribution reaches past its 64 best tokens: no filter at all,
    top_p with top_k off, top_k above 64 with and without top_p.  p, the accept tests, the residual
    draw over the whole vocabulary in token-id order and the bonus draw against the oracle."""
    B, K, V = 12, 5, 20000
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=seed, target_noise=1.0, dtype=dtype)
    inp = synth.make_inputs(shp, with_conv=False)
    inp.params["temperature"] = np.resize(np.float32([1.0, 0.8, 1.2, 1.0]), B)
    inp.params["top_k"] = np.resize(np.int32([0, 0, 100, 500]), B)
    inp.params["top_p"] = np.resize(np.float32([1.0, 0.9, 1.0, 0.7]), B)
    cand, pt, ps, q = oracle_walk_inputs(ref, inp, B, K)
    acc, ex = check(ref, inp, cand, pt, ps, q, inp.params, B, K)
    assert 0 < int(np.sum(acc)) < B * K      # both accepts and rejects were exercised


def test_wide_and_narrow_requests_in_one_call(ref):
    """One batch mixing greedy requests, top_k 20 with top_p 0.95 (p within the 64 best), and
    wide targets (top_p 0.9 with top_k off, top_k 100): wide rows finished in their CTAs'
    epilogues next to rows finished at completion, against the oracle."""
    B, K, V = 16, 5, 20000
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=9, target_noise=1.0)
    inp = synth.make_inputs(shp, with_conv=False)
    inp.params["temperature"] = np.resize(np.float32([0.0, 1.0, 1.0, 0.9]), B)
    inp.params["top_k"] = np.resize(np.int32([0, 20, 0, 100]), B)
    inp.params["top_p"] = np.resize(np.float32([1.0, 0.95, 0.9, 1.0]), B)
    cand, pt, ps, q = oracle_walk_inputs(ref, inp, B, K)
    check(ref, inp, cand, pt, ps, q, inp.params, B, K)


@pytest.mark.parametrize("k,p", [(20, 0.95), (0, 0.9), (0, 1.0), (100, 1.0)])
def test_gpu_monte_carlo_marginals(ref, k, p):
    """6M verify rows on the GPU: committed-token marginals within 5e-3 of p_t (top_k 20 with top_p
    0.95, the pages' setting; then three targets whose p reaches past the 64 best, so that the
    residual and bonus draws walk the whole row: top_p 0.9 with top_k off, no filter at all, and
    top_k 100)."""
    dev = cuda_or_skip()
    B0, K, V = 4, 3, 2048
    shp = synth.small_shape("27b_sampled", B=B0, K=K, V=V, hidden=64, seed=31, target_noise=1.0)
    inp = synth.make_inputs(shp, with_conv=False)
    cand, _, _, _ = oracle_walk_inputs(ref, inp, B0, K)
    idx, U, _, _ = ref.topk16(inp.draft_logits, params=inp.params, rows_per_param=K)
    qrow = np.exp(U.reshape(B0, K, 16))
    qrow = qrow / qrow.sum(-1, keepdims=True)     # the walk's q with a zero selector term
    REP = 3000                                    # requests per call = B0 * REP
    B = B0 * REP
    tl = inp.target_logits.view(B0, K + 1, V).repeat(REP, 1, 1).view(B * (K + 1), V).to(dev)
    cand_g = torch.as_tensor(np.tile(cand, (REP, 1, 1))).to(dev)
    q_g = torch.as_tensor(np.tile(qrow, (REP, 1, 1))).float().to(dev)
    pg = d2.sampling_params([1.0] * B, [k] * B, [p] * B, device=dev)
    ws = d2.Workspace.for_verify(B, K, dev)
    gen = torch.Generator(device=dev).manual_seed(5)
    counts = [np.zeros((B0, V)) for _ in range(K + 1)]
    calls = 500                                   # 500 * 12000 = 6M rows
    for _ in range(calls):
        # draw the drafted slots from q, then verify
        u = torch.rand(B, K, generator=gen, device=dev)
        cdf = torch.cumsum(q_g, dim=-1)
        slot = torch.searchsorted(cdf, u.unsqueeze(-1) * cdf[..., -1:]).squeeze(-1).clamp_(max=15).to(torch.int32)
        pt = torch.gather(cand_g, 2, slot.long().unsqueeze(-1)).squeeze(-1).contiguous()
        acc, out, st = d2.verify(tl, pt, cand_g, q_g, slot.contiguous(), params=pg,
                                 u_acc=torch.rand(B, K, generator=gen, device=dev),
                                 u_res=torch.rand(B, K + 1, generator=gen, device=dev), ws=ws)
        assert int(st.abs().sum()) == 0
        for t in range(K + 1):
            reached = acc >= t
            tok = out[:, t]
            b_of = torch.arange(B, device=dev) % B0
            sel = reached.nonzero().flatten()
            flat = b_of[sel] * V + tok[sel].long()
            counts[t] += torch.bincount(flat, minlength=B0 * V).view(B0, V).cpu().numpy()
    for t in range(K + 1):
        for b in range(B0):
            n, ids, pr, _ = ref.target_dist(inp.target_logits[b * (K + 1) + t], 1.0, k, p)
            expect = np.zeros(V)
            expect[ids] = pr
            emp = counts[t][b] / counts[t][b].sum()
            assert np.max(np.abs(emp - expect)) < 5e-3, (t, b)


@pytest.mark.parametrize("name", ["27b_greedy", "27b_sampled"])
def test_full_size_sampled_requests(ref, name):
    dev = cuda_or_skip()
    shp = synth.WORKLOADS[name]
    inp = synth.make_inputs(shp, device=dev, with_conv=False)
    B, K, V = shp.B, shp.K, shp.V
    params = inp.params if shp.temperature > 0 else None
    pg = None if params is None else d2.sampling_params(params["temperature"], params["top_k"], params["top_p"],
                                                        device=dev)
    cand, U, lse = d2.topk16(inp.draft_logits, params=pg, rows_per_param=K)
    # a path with a zero selector term: walk over U
    S = U.view(B, K, 1, 16).expand(B, K, 16, 16)
    g = torch.zeros(B * K, 256, device=dev)
    Az = torch.zeros(V, 256, dtype=shp.dtype, device=dev)
    pt, ps, q, _ = d2.pair_score_walk(cand.view(B, K, 16), U.view(B, K, 16), inp.last_tok, Az, Az, g.view(B, K, 256),
                                      params=pg, u_walk=inp.u_walk if pg is not None else None)
    acc, out, st = d2.verify(inp.target_logits, pt, cand.view(B, K, 16), q, ps, params=pg,
                             u_acc=inp.u_acc if pg is not None else None, u_res=inp.u_res if pg is not None else None)
    torch.cuda.synchronize()
    ex = _parity.Excused()   # every request
    _parity.verify_compare(ref, inp.target_logits.cpu(), pt.cpu().numpy(), cand.view(B, K, 16).cpu().numpy(),
                           q.cpu().numpy(), ps.cpu().numpy(), params, inp.u_acc.cpu().numpy(), inp.u_res.cpu().numpy(),
                           acc.cpu().numpy(), out.cpu().numpy(), st.cpu().numpy(), ex, what=name)
    ex.check_bound(what=name)
    assert d2.device_error() == 0
