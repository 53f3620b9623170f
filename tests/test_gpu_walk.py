"""dflash2_pair_score_walk against the oracle: scores within 1e-4 rel; paths and
slots bit-exact, except at a sampled step whose oracle margin is below 1e-5,
where the GPU's draw must be a neighbour of the CDF step and the comparison
goes on from it (at most 1% of the steps excused)."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from tests import _parity
from tests._util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu


def make(B, K, V, D, seed, dtype=torch.bfloat16, scale=0.25, filtered=False):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(B * K, V, generator=g) * 2
    A = (torch.randn(V, D, generator=g) * scale).to(dtype)
    Bt = (torch.randn(V, D, generator=g) * scale).to(dtype)
    gate = torch.rand(B * K, D, generator=g)
    last = torch.randint(0, V, (B,), generator=g, dtype=torch.int32)
    u = torch.rand(B, K, generator=g)
    return z, A, Bt, gate, last, u


def run(ref, B, K, V, D, seed, T=0.0, dtype=torch.bfloat16, scale=0.25, mutate=None):
    dev = cuda_or_skip()
    z, A, Bt, gate, last, u = make(B, K, V, D, seed, dtype, scale)
    idx, U, _, _ = ref.topk16(z)
    idx = idx.reshape(B, K, 16)
    U = U.astype(np.float32).reshape(B, K, 16)
    if mutate:
        idx, U = mutate(idx, U)
    params = None if T == 0.0 else d2.sampling_params([T] * B, [0] * B, [1.0] * B, device=dev)
    pt, ps, q, S = d2.pair_score_walk(torch.as_tensor(idx).to(dev), torch.as_tensor(U).to(dev), last.to(dev),
                                      A.to(dev), Bt.to(dev), gate.to(dev).view(B, K, D), params=params,
                                      u_walk=u.to(dev) if params is not None else None)
    torch.cuda.synchronize()
    r_S = ref.pair_scores(idx, U.astype(np.float64), last, A, Bt, gate.double().numpy(), B, K)
    assert_close(S.cpu().numpy(), r_S, what="scores")
    Tn = np.full(B, T, np.float32)
    # the walk: the oracle over the GPU's own scores, so only the walk is compared
    pt, ps, q = pt.cpu().numpy(), ps.cpu().numpy(), q.cpu().numpy()
    ex = _parity.Excused()
    _parity.walk_compare(ref, idx, S.cpu().double().numpy(), Tn, u.numpy(), pt, ps, q, ex)
    ex.check_bound(what="walk")
    r_mg = ref.walk(idx, S.cpu().double().numpy(), Tn, u.numpy(), B, K)[3]
    return pt, ps, q, r_mg


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [1, 2, 7, 15])
def test_greedy(ref, dtype, K):
    run(ref, 5, K, 3000, 256, seed=K, dtype=dtype)


@pytest.mark.parametrize("D", [16, 64, 256, 1024])
def test_embed_dims(ref, D):
    run(ref, 3, 4, 2000, D, seed=D, T=1.0)


@pytest.mark.parametrize("T", [0.5, 1.0])
def test_sampled(ref, T):
    run(ref, 16, 7, 5000, 256, seed=3, T=T, scale=1.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_largest_cluster_at_the_largest_D(ref, dtype):
    """K = 15 (a 15-CTA cluster, above the portable 8) at D = 1024 (the most
    shared memory a CTA of the walk takes): either the cluster can be resident
    and the result matches the oracle, or the call returns UNSUPPORTED and
    launches nothing."""
    try:
        run(ref, 3, 15, 3000, 1024, seed=15, T=1.0, dtype=dtype)
    except d2.DFlash2Error as e:
        assert e.code == 2, e  # DFLASH2_ERR_UNSUPPORTED
        assert d2.device_error() == 0


def test_zero_A_is_top1_chain(ref):
    dev = cuda_or_skip()
    B, K, V, D = 4, 7, 1000, 256
    z, A, Bt, gate, last, u = make(B, K, V, D, seed=4)
    idx, U, _, _ = ref.topk16(z)
    pt, ps, q, S = d2.pair_score_walk(torch.as_tensor(idx).view(B, K, 16).to(dev),
                                      torch.as_tensor(U).float().view(B, K, 16).to(dev), last.to(dev),
                                      torch.zeros_like(A).to(dev), Bt.to(dev), gate.to(dev).view(B, K, D))
    top1 = np.argmax(z.numpy(), axis=1).reshape(B, K)
    np.testing.assert_array_equal(pt.cpu().numpy(), top1)
    assert torch.all(ps == 0)


def test_filtered_candidates_never_drawn(ref):
    """Over 1M sampled walks the selector never draws a q = 0 candidate."""
    dev = cuda_or_skip()
    B, K, V, D = 25000, 2, 500, 64
    z, A, Bt, gate, last, _ = make(1, K, V, D, seed=5, scale=1.0)
    idx, U, _, _ = ref.topk16(z)
    U = U.astype(np.float32).reshape(1, K, 16)
    U[0, 0, [3, 9, 15]] = -np.inf
    U[0, 1, [0, 5]] = -np.inf
    idx_g = torch.as_tensor(idx).view(1, K, 16).repeat(B, 1, 1).to(dev)
    U_g = torch.as_tensor(U).repeat(B, 1, 1).to(dev)
    last_g = last.repeat(B).to(dev)
    gate_g = gate.view(1, K, D).repeat(B, 1, 1).to(dev)
    params = d2.sampling_params([1.0] * B, [0] * B, [1.0] * B, device=dev)
    gen = torch.Generator(device=dev).manual_seed(6)
    hist0 = torch.zeros(16, dtype=torch.int64, device=dev)
    for _ in range(40):  # 40 * 25000 = 1M walks
        pt, ps, q, S = d2.pair_score_walk(idx_g, U_g, last_g, A.to(dev), Bt.to(dev), gate_g, params=params,
                                          u_walk=torch.rand(B, K, generator=gen, device=dev))
        assert not torch.isin(ps[:, 0], torch.tensor([3, 9, 15], device=dev)).any()
        assert not torch.isin(ps[:, 1], torch.tensor([0, 5], device=dev)).any()
        hist0 += torch.bincount(ps[:, 0].long(), minlength=16)
    q0 = q[0, 0].double().cpu().numpy()
    emp = hist0.cpu().numpy() / hist0.sum().item()
    sd = np.sqrt(q0 * (1 - q0) / hist0.sum().item())
    assert np.all(np.abs(emp - q0) <= 5 * sd + 1e-9)


def test_nan_and_out_of_range(ref):
    def mutate(idx, U):
        idx = idx.copy()
        U = U.copy()
        U[1, 2, 4] = np.nan          # request 1 dies at step 2
        idx[2, 0, :] = 99999         # request 2: ids out of range -> NaN scores at t = 0 and 1
        return idx, U
    pt, ps, q, _ = run(ref, 3, 4, 3000, 64, seed=7, mutate=mutate)
    assert np.all(pt[2] == -1) and np.all(ps[2] == -1) and np.all(np.isnan(q[2]))
    assert np.all(pt[1, 2:] == -1) and pt[1, 1] >= 0
