"""dflash2_pair_score_walk_noalloc: the selector walk for callers that cannot
give this library any device memory (a plugin or engine whose memory pool
hands out no scratch).  Called through the C ABI, it must produce the same
scores, path, slots and q as dflash2_pair_score_walk with a workspace, on two
calls in a row (the second call must not see the first call's tickets).
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from tests._util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu


def noalloc_fn():
    L = d2.load_library()
    f = L.dflash2_pair_score_walk_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f.argtypes = [i64, i32, vp, vp, vp, vp, vp, i32, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    f.restype = i32
    return f


def make_inputs(seed, B, K, V, D, dev, sampled):
    g = torch.Generator(device=dev).manual_seed(seed)
    cand = torch.randint(0, V, (B, K, 16), generator=g, device=dev, dtype=torch.int32)
    U = (-torch.rand(B, K, 16, generator=g, device=dev) * 5).sort(dim=-1, descending=True).values
    last = torch.randint(0, V, (B,), generator=g, device=dev, dtype=torch.int32)
    A = (torch.randn(V, D, generator=g, device=dev) * 0.25).bfloat16()
    Bt = (torch.randn(V, D, generator=g, device=dev) * 0.25).bfloat16()
    gate = torch.rand(B, K, D, generator=g, device=dev)
    params = d2.sampling_params([1.0] * B, [0] * B, [1.0] * B, device=dev) if sampled else None
    u = torch.rand(B, K, generator=g, device=dev)
    return cand, U, last, A, Bt, gate, params, u


def call_noalloc(f, cand, U, last, A, Bt, gate, params, u):
    B, K, D = gate.shape
    V = A.shape[0]
    dev = cand.device
    pt = torch.empty(B, K, dtype=torch.int32, device=dev)
    ps = torch.empty(B, K, dtype=torch.int32, device=dev)
    q = torch.empty(B, K, 16, device=dev)
    S = torch.empty(B, K, 16, 16, device=dev)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = f(B, K, p(cand), p(U), p(last), p(A), p(Bt), 1, V, D, p(gate), p(params),
           p(u if params is not None else None), p(pt), p(ps), p(q), p(S),
           ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == 0, f"status {st}"
    return pt, ps, q, S


def test_noalloc_walk_matches_the_workspace_walk_twice():
    dev = cuda_or_skip()
    f = noalloc_fn()
    for seed, B, K, sampled in [(1, 64, 7, True), (2, 40, 5, False)]:
        ins = make_inputs(seed, B, K, 5000, 256, dev, sampled)
        cand, U, last, A, Bt, gate, params, u = ins
        ref = d2.pair_score_walk(cand, U, last, A, Bt, gate, params=params, u_walk=u if sampled else None)
        got = call_noalloc(f, *ins)
        torch.cuda.synchronize()
        for name, r, g in zip(("path_tok", "path_slot"), ref[:2], got[:2]):
            np.testing.assert_array_equal(g.cpu().numpy(), r.cpu().numpy(), err_msg=name)
        assert_close(got[2].cpu().numpy(), ref[2].cpu().numpy(), what="q_sel")
        assert_close(got[3].cpu().numpy(), ref[3].cpu().numpy(), what="scores")


def test_noalloc_rejects_batches_beyond_its_array():
    dev = cuda_or_skip()
    f = noalloc_fn()
    B = 16385
    p = ctypes.c_void_p(16)
    st = f(B, 2, p, p, p, p, p, 1, 5000, 256, p, None, None, p, p, p, p, None)
    assert st == 4  # DFLASH2_ERR_WORKSPACE: nothing launched
