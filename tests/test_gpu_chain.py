"""The whole path (topk16 -> ctx_gate -> pair_score_walk -> verify) on the named
workloads, against the oracle run on the same inputs: every row and every
request of the full-size workloads, in the bench's launch configuration.
Near-tie decisions are excused only as tests/_parity.py allows (at most 1%
of the decisions, each checked to be a valid outcome)."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests import _parity
from tests._util import MARGIN, assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu


def gpu_chain(inp, dev):
    shp = inp.shape
    B, K = shp.B, shp.K
    sampled = shp.temperature > 0
    pg = d2.sampling_params(inp.params["temperature"], inp.params["top_k"], inp.params["top_p"], device=dev) \
        if sampled else None
    cand, U, lse = d2.topk16(inp.draft_logits, params=pg, rows_per_param=K)
    gate = d2.ctx_gate(inp.h, inp.Wg)
    pt, ps, q, S = d2.pair_score_walk(cand.view(B, K, 16), U.view(B, K, 16), inp.last_tok, inp.A, inp.Bt,
                                      gate.view(B, K, -1), params=pg, u_walk=inp.u_walk if sampled else None)
    acc, out, st = d2.verify(inp.target_logits, pt, cand.view(B, K, 16), q, ps, params=pg,
                             u_acc=inp.u_acc if sampled else None, u_res=inp.u_res if sampled else None)
    torch.cuda.synchronize()
    return dict(cand=cand, U=U, lse=lse, gate=gate, pt=pt, ps=ps, q=q, S=S, acc=acc, out=out, st=st)


def check_chain(ref, inp, res, reqs):
    """Each stage against the oracle fed the GPU's previous stage, for the requests `reqs`."""
    shp = inp.shape
    B, K, V = shp.B, shp.K, shp.V
    params = inp.params if shp.temperature > 0 else None
    rows = np.concatenate([np.arange(b * K, (b + 1) * K) for b in reqs])
    trows = np.concatenate([np.arange(b * (K + 1), (b + 1) * (K + 1)) for b in reqs])
    n = len(reqs)
    pr = None if params is None else params[reqs]
    prow = synth.make_params(len(rows), 0.0, 0, 1.0) if pr is None else np.repeat(pr, K)
    zd = inp.draft_logits[torch.as_tensor(rows).to(inp.draft_logits.device)].cpu()
    r_idx, r_U, r_lse, r_mg = ref.topk16(zd, params=pr, rows_per_param=K)
    ex_t = _parity.Excused()
    _parity.topk_compare(zd, prow, res["cand"].cpu().numpy()[rows], res["U"].cpu().numpy()[rows],
                         res["lse"].cpu().numpy()[rows], r_idx, r_U, r_lse, r_mg, ex_t, what=shp.name + " topk16")
    ex_t.check_bound(what="topk16")
    hd = inp.h[torch.as_tensor(rows).to(inp.h.device)].cpu()
    assert_close(res["gate"].cpu().numpy()[rows], ref.ctx_gate(hd, inp.Wg.cpu()), what="gate")
    cand = res["cand"].cpu().view(B, K, 16)[reqs]
    U = res["U"].cpu().view(B, K, 16)[reqs].double()
    gate = res["gate"].cpu().view(B, K, -1)[reqs].double()
    r_S = ref.pair_scores(cand, U, inp.last_tok.cpu()[reqs], inp.A.cpu(), inp.Bt.cpu(), gate, n, K)
    S = res["S"].cpu().double().numpy()[reqs]
    assert_close(S, r_S, what="scores")
    T = np.zeros(n, np.float32) if params is None else pr["temperature"]
    ex_w = _parity.Excused()
    _parity.walk_compare(ref, cand.numpy(), S, T, inp.u_walk.cpu().numpy()[reqs], res["pt"].cpu().numpy()[reqs],
                         res["ps"].cpu().numpy()[reqs], res["q"].cpu().numpy()[reqs], ex_w, what=shp.name + " walk")
    ex_w.check_bound(what="walk")
    tl = inp.target_logits[torch.as_tensor(trows).to(inp.target_logits.device)].cpu()
    ex_v = _parity.Excused()
    _parity.verify_compare(ref, tl, res["pt"].cpu().numpy()[reqs], cand.numpy(), res["q"].cpu().numpy()[reqs],
                           res["ps"].cpu().numpy()[reqs], pr, inp.u_acc.cpu().numpy()[reqs],
                           inp.u_res.cpu().numpy()[reqs], res["acc"].cpu().numpy()[reqs],
                           res["out"].cpu().numpy()[reqs], res["st"].cpu().numpy()[reqs], ex_v,
                           what=shp.name + " verify")
    ex_v.check_bound(what="verify")


def test_tiny_f32_whole_chain_matches_oracle_chain(ref):
    """The tiny fp32 workload: the GPU chain equals the oracle's own chain end to end."""
    dev = cuda_or_skip()
    inp = synth.make_inputs(synth.WORKLOADS["tiny_f32"], device="cpu", with_conv=False)
    ig = synth.Inputs(**{k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.__dict__.items()})
    res = gpu_chain(ig, dev)
    check_chain(ref, ig, res, np.arange(1))
    B, K = 1, 7
    idx, U, lse, _ = ref.topk16(inp.draft_logits)
    gate = ref.ctx_gate(inp.h, inp.Wg)
    S = ref.pair_scores(idx, U, inp.last_tok, inp.A, inp.Bt, gate, B, K)
    pt, ps, q, wm = ref.walk(idx, S, np.zeros(1, np.float32), inp.u_walk, B, K)
    acc, out, st, vm = ref.verify(inp.target_logits, pt, idx.reshape(B, K, 16), q, ps, None, inp.u_acc, inp.u_res,
                                  B, K)
    assert wm.min() >= MARGIN
    np.testing.assert_array_equal(res["pt"].cpu().numpy(), pt)
    np.testing.assert_array_equal(res["acc"].cpu().numpy(), acc)
    np.testing.assert_array_equal(res["out"].cpu().numpy(), out)


@pytest.mark.parametrize("name", ["4b_greedy", "27b_greedy", "27b_sampled", "27b_nucleus", "stress"])
def test_workload_chain(ref, name):
    dev = cuda_or_skip()
    inp = synth.make_inputs(synth.WORKLOADS[name], device=dev, with_conv=False)
    res = gpu_chain(inp, dev)
    B = inp.shape.B
    check_chain(ref, inp, res, np.arange(B))   # every request
    acc = res["acc"].cpu().numpy()
    assert np.all(res["st"].cpu().numpy() == 0)
    assert np.all((acc >= 0) & (acc <= inp.shape.K))
    assert d2.device_error() == 0


def test_stress_conv(ref):
    dev = cuda_or_skip()
    shp = synth.WORKLOADS["stress"]
    g = torch.Generator(device=dev).manual_seed(shp.seed)
    c = synth.make_conv(shp.B, shp.K + 1, shp.hidden, shp.dtype, g, dev)
    y = d2.conv2tap(c["x"], c["k0"], c["k1"], c["x_prev"])
    torch.cuda.synchronize()
    r = ref.conv2tap(c["x"].cpu(), c["k0"].cpu(), c["k1"].cpu(), c["x_prev"].cpu())   # all 256 requests
    assert torch.equal(y.cpu().view(torch.int16), r.view(torch.int16))
