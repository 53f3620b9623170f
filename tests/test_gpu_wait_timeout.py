"""A bounded device wait that runs out, made on the host without a fault.

The test hook makes every streaming warp of the row scan wait, for at most
2e6 SM cycles (about 1 ms), on a device word that nothing sets.  Each warp
gives up before its first copy.  The kernel must then return, set the device
error word, write -1 / NaN for every row (verify: status ST_NAN and nothing
committed) and leave the context usable: with the hook off and the workspace
zero-filled again, the next call agrees with the oracle."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests import _parity
from tests._util import cuda_or_skip, padded

pytestmark = pytest.mark.gpu

LIMIT = 2_000_000   # SM cycles, about 1 ms


def held(fn):
    """Run fn() with the hook waiting on a zero word; return fn's result and the error word."""
    dev = torch.device("cuda:0")
    flag = torch.zeros(1, dtype=torch.int32, device=dev)   # nothing ever sets it
    assert d2.device_error(clear=True) == 0
    d2.test_hold(flag, LIMIT)
    try:
        out = fn()
        code = d2.device_error(clear=True)
    finally:
        d2.test_hold(None)
    return out, code


@pytest.mark.parametrize("rows,V", [(24, 50000), (3, 262144)])   # whole rows per CTA; rows split over CTAs
def test_topk16_wait_runs_out_then_recovers(ref, rows, V):
    dev = cuda_or_skip()
    g = torch.Generator(device=dev).manual_seed(rows)
    z = synth.spike_logits(rows, V, g, dev).bfloat16()
    ws = d2.Workspace.for_topk16(rows, dev)
    (idx, U, lse), code = held(lambda: d2.topk16(z, ws=ws))
    assert code == 1   # DFLASH2_DEVERR_WAIT_TIMEOUT
    assert torch.all(idx == -1) and torch.all(torch.isnan(U)) and torch.all(torch.isnan(lse))
    ws.buf.zero_()
    idx, U, lse = d2.topk16(z, ws=ws)
    torch.cuda.synchronize()
    zc = z.cpu()
    r_idx, r_U, r_lse, r_mg = ref.topk16(zc)
    ex = _parity.Excused()
    _parity.topk_compare(zc, synth.make_params(rows, 0.0, 0, 1.0), idx.cpu().numpy(), U.cpu().numpy(),
                         lse.cpu().numpy(), r_idx, r_U, r_lse, r_mg, ex, what="after the time-out")
    ex.check_bound(what="after the time-out")
    assert d2.device_error() == 0


def test_noalloc_topk16_recovers_without_help():
    """The no-alloc call clears its own tickets, so the call after a time-out needs nothing from the caller."""
    dev = cuda_or_skip()
    g = torch.Generator(device=dev).manual_seed(7)
    z = synth.spike_logits(4, 200000, g, dev).bfloat16()
    (idx, _, _), code = held(lambda: d2.topk16_noalloc(z))
    assert code == 1 and torch.all(idx == -1)
    got = d2.topk16_noalloc(z)
    want = d2.topk16(z)
    torch.cuda.synchronize()
    for x, y in zip(got, want):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())
    assert d2.device_error() == 0


def test_verify_wait_runs_out_then_recovers(ref):
    dev = cuda_or_skip()
    B, K, V = 6, 7, 30000
    shp = synth.small_shape("27b_sampled", B=B, K=K, V=V, hidden=64, seed=11, dtype=torch.bfloat16)
    inp = synth.make_inputs(shp, with_conv=False)
    p = inp.params
    idx, U, _, _ = ref.topk16(inp.draft_logits, params=p, rows_per_param=K)
    S = np.broadcast_to(U.reshape(B, K, 1, 16), (B, K, 16, 16)).copy()
    pt, ps, q, _ = ref.walk(idx, S, p["temperature"], inp.u_walk, B, K)
    cand = idx.reshape(B, K, 16)
    pg = d2.sampling_params(p["temperature"], p["top_k"], p["top_p"], device=dev)
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dt).to(dev)
    tl = padded(inp.target_logits.to(dev))
    args = (tl, t(pt, torch.int32), t(cand, torch.int32), t(q, torch.float32), t(ps, torch.int32))
    ws = d2.Workspace.for_verify(B, K, dev)
    kw = dict(params=pg, u_acc=inp.u_acc.to(dev), u_res=inp.u_res.to(dev), ws=ws)
    (acc, out, st), code = held(lambda: d2.verify(*args, **kw))
    assert code == 1
    assert torch.all(st == d2.binding.ST_NAN) and torch.all(acc == 0) and torch.all(out == -1)
    ws.buf.zero_()
    acc, out, st = d2.verify(*args, **kw)
    torch.cuda.synchronize()
    ex = _parity.Excused()
    _parity.verify_compare(ref, inp.target_logits, pt, cand, q.astype(np.float32), ps, p, inp.u_acc.numpy(),
                           inp.u_res.numpy(), acc.cpu().numpy(), out.cpu().numpy(), st.cpu().numpy(), ex)
    ex.check_bound(what="verify after the time-out")
    assert d2.device_error() == 0
