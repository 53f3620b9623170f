"""dflash2_topk16_shard and dflash2_topk16_merge against the oracle: each
slice's partial (ids and logits bit for bit, the largest logit exactly, its
sum within 1e-4 rel), and the merge of the slices of whole rows against the
oracle's whole-row top-16 (ids bit for bit; U and lse within 1e-4 rel, near-tie
top_p cuts as tests/_parity.py allows), at the size of the 27B workloads."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests import _parity
from tests._util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu


def slices(z, cuts):
    b = [0] + list(cuts) + [z.shape[1]]
    return [(lo, z[:, lo:hi].contiguous()) for lo, hi in zip(b[:-1], b[1:])]


def gpu_sharded(z, cuts, params=None, rpp=1):
    dev = z.device
    V = z.shape[1]
    pg = None if params is None else d2.sampling_params(params["temperature"], params["top_k"], params["top_p"],
                                                        device=dev)
    parts = [d2.topk16_shard(zs, lo, V, params=pg, rows_per_param=rpp) for lo, zs in slices(z, cuts)]
    st = [torch.stack([p[i] for p in parts]).contiguous() for i in range(4)]
    return parts, d2.topk16_merge(*st, V, params=pg, rows_per_param=rpp)


def check_whole(ref, z, merged, params, rpp, what):
    zc = z.cpu()
    r = ref.topk16(zc, params=params, rows_per_param=rpp)
    rows = z.shape[0]
    prow = synth.make_params(rows, 0.0, 0, 1.0) if params is None else np.repeat(params, rpp)[:rows]
    ex = _parity.Excused()
    _parity.topk_compare(zc, prow, merged[0].cpu().numpy(), merged[1].cpu().numpy(), merged[2].cpu().numpy(),
                         *r, ex, what=what)
    ex.check_bound(what=what)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_partials_match_the_oracle(ref, dtype):
    dev = cuda_or_skip()
    g = torch.Generator(device=dev).manual_seed(1)
    z = (torch.randn(12, 40000, generator=g, device=dev) * 2).to(dtype)
    z[3, 30000:31000] = z[3].max()          # ties at the maximum inside one slice
    params = synth.make_params(6, [0.0, 1.0, 0.7, 1.0, 1.3, 0.0], [0, 20, 0, 64, 5, 0], [1.0, 0.95, 1.0, 1.0, 0.5, 1.0])
    pg = d2.sampling_params(params["temperature"], params["top_k"], params["top_p"], device=dev)
    for lo, zs in slices(z, [8000, 8016, 29992]):
        pi, pz, pm, ps = d2.topk16_shard(zs, lo, 40000, params=pg, rows_per_param=2)
        torch.cuda.synchronize()
        ri, rz, rm, rs = ref.topk16_shard(zs.cpu(), lo, 40000, params=params, rows_per_param=2)
        np.testing.assert_array_equal(pi.cpu().numpy(), ri, err_msg=f"ids of slice at {lo}")
        np.testing.assert_array_equal(pz.cpu().numpy(), rz.astype(np.float32), err_msg=f"logits of slice at {lo}")
        np.testing.assert_array_equal(pm.cpu().numpy(), rm.astype(np.float32))
        assert_close(ps.cpu().numpy(), rs, what=f"sums of slice at {lo}")
    assert d2.device_error() == 0


@pytest.mark.parametrize("name,cuts", [("27b_greedy", [40000, 40016, 100000]),
                                       ("27b_sampled", [37984, 75968, 113952]),
                                       ("27b_greedy", [])])
def test_merge_of_slices_is_the_whole_row_at_full_size(ref, name, cuts):
    dev = cuda_or_skip()
    shp = synth.WORKLOADS[name]
    g = torch.Generator(device=dev).manual_seed(shp.seed)
    z = synth.spike_logits(shp.B * shp.K, shp.V, g, dev).to(shp.dtype)
    params = None if shp.temperature == 0 else synth.make_params(shp.B, shp.temperature, shp.top_k, shp.top_p)
    _, merged = gpu_sharded(z, cuts, params, shp.K)
    torch.cuda.synchronize()
    check_whole(ref, z, merged, params, shp.K, f"{name} in {len(cuts) + 1} slices")
    assert d2.device_error() == 0


def test_masked_slice_bad_rows_and_refused_rows(ref):
    dev = cuda_or_skip()
    g = torch.Generator(device=dev).manual_seed(2)
    z = torch.randn(8, 6000, generator=g, device=dev) * 2
    z[:, 2000:4000] = -float("inf")        # a slice of masked tokens
    z[5, 4500] = float("nan")
    z[6, 100] = float("inf")
    params = synth.make_params(4, [0.0, 1.0, 1.0, 1.0], [0, 0, 65, 20], [1.0, 0.9, 1.0, 0.9])
    parts, merged = gpu_sharded(z, [2000, 4000], params, 2)
    torch.cuda.synchronize()
    pm = parts[1][2].cpu().numpy()
    assert np.all(np.isneginf(pm[[0, 1, 6, 7]])) and np.all(parts[1][3].cpu().numpy()[[0, 1]] == 0)
    idx, U, lse = (t.cpu().numpy() for t in merged)
    for r in (2, 3, 4, 5, 6):                # top_p with top_k off, top_k > 64, NaN, +Inf
        assert np.all(idx[r] == -1) and np.all(np.isnan(U[r])) and np.isnan(lse[r]), r
    ok = [0, 1, 7]
    zc = z.cpu()
    r_all = ref.topk16(zc, params=params, rows_per_param=2)
    ex = _parity.Excused()
    _parity.topk_compare(zc[ok], np.repeat(params, 2)[ok], idx[ok], U[ok], lse[ok], *(a[ok] for a in r_all), ex,
                         what="masked slice")
    assert d2.device_error() == 0
