"""Pins of the oracle's vocabulary-sharded top-16 (partials and merge) on the
CPU.  The merge of the slices' partials must give what the oracle's whole-row
top-16 gives (its own pins: library sorts, closed forms), for any split of
the vocabulary: ids bit for bit, U and lse within 1e-12; each partial must be
the slice's own ranking (a library sort with the slice's offset) and its sum
the closed form."""
import numpy as np
import pytest
import torch

from dflash_draft_selection_gb300 import synth

P = 64


def split(z, cuts, off=0, V_total=None, params=None, rpp=1, ref=None):
    V = z.shape[1]
    V_total = V if V_total is None else V_total
    bounds = [0] + list(cuts) + [V]
    parts = [ref.topk16_shard(z[:, a:b].contiguous(), off + a, V_total, params=params, rows_per_param=rpp)
             for a, b in zip(bounds[:-1], bounds[1:])]
    return [np.stack([p[i] for p in parts]) for i in range(4)]


def whole_and_merged(ref, z, cuts, params=None, rpp=1):
    w = ref.topk16(z, params=params, rows_per_param=rpp)
    m = ref.topk16_merge(*split(z, cuts, params=params, rpp=rpp, ref=ref), z.shape[1], params=params,
                         rows_per_param=rpp)
    return w, m


def assert_same(w, m, rows=None):
    rows = slice(None) if rows is None else rows
    np.testing.assert_array_equal(m[0][rows], w[0][rows])
    np.testing.assert_allclose(m[1][rows], w[1][rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(m[2][rows], w[2][rows], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cuts", [[], [1], [999], [17, 500], [100, 101, 102, 600, 900]])
def test_merge_of_any_split_is_the_whole_row(ref, dtype, cuts):
    g = torch.Generator().manual_seed(len(cuts))
    z = (torch.randn(6, 1000, generator=g) * 3).to(dtype)
    w, m = whole_and_merged(ref, z, cuts)
    assert_same(w, m)


def test_sampled_rows_filtered_and_not(ref):
    g = torch.Generator().manual_seed(3)
    z = torch.randn(8, 3000, generator=g) * 2
    params = synth.make_params(4, [0.7, 1.0, 1.3, 0.0], [0, 20, 64, 0], [1.0, 0.95, 0.8, 1.0])
    w, m = whole_and_merged(ref, z, [700, 1500, 2999], params=params, rpp=2)
    assert_same(w, m)


def test_ties_across_slices_keep_the_lower_id(ref):
    """The row maximum appears in three slices: the lowest global id ranks first, whatever slice holds it."""
    z = torch.randn(3, 512, generator=torch.Generator().manual_seed(4))
    for r, ids in enumerate([(400, 10, 250), (100, 300, 511), (0, 256, 257)]):
        for i in ids:
            z[r, i] = 9.0
    w, m = whole_and_merged(ref, z, [128, 256, 384])
    assert_same(w, m)
    for r, ids in enumerate([(400, 10, 250), (100, 300, 511), (0, 256, 257)]):
        assert list(m[0][r, :3]) == sorted(ids)


def test_masked_slice_and_bad_rows(ref):
    z = torch.randn(4, 600, generator=torch.Generator().manual_seed(5))
    z[:, 200:400] = -float("inf")      # a whole slice of masked tokens: not an error
    z[2, 450] = float("nan")           # a NaN in one slice: the row is bad
    z[3, 10] = float("inf")            # +Inf: bad
    w, m = whole_and_merged(ref, z, [200, 400])
    assert_same(w, m, rows=slice(0, 2))
    idx, z2, mm, ss = ref.topk16_shard(z[:, 200:400].contiguous(), 200, 600)
    assert np.all(np.isneginf(mm[:2])) and np.all(ss[:2] == 0) and np.all(idx[:2, :16] >= 200)
    for r in (2, 3):
        assert np.all(m[0][r] == -1) and np.all(np.isnan(m[1][r])) and np.isnan(m[2][r])


def test_rows_that_need_the_whole_row_are_refused(ref):
    """top_p with top_k off, and top_k above the list, cannot be merged from partials: -1 / NaN."""
    z = torch.randn(4, 900, generator=torch.Generator().manual_seed(6))
    params = synth.make_params(2, [1.0, 1.0], [0, 65], [0.9, 1.0])
    _, m = whole_and_merged(ref, z, [450], params=params, rpp=2)
    assert np.all(m[0] == -1) and np.all(np.isnan(m[2]))


def test_partial_is_the_slice_ranking_and_its_sum(ref):
    g = torch.Generator().manual_seed(7)
    z = torch.randn(5, 800, generator=g) * 2
    z[:, 37] = z[:, 5]   # a tie inside the slice
    off, V_total = 1000, 5000
    params = synth.make_params(5, [0.0, 0.8, 1.0, 1.0, 2.0], [0, 0, 30, 10, 0], [1.0, 1.0, 1.0, 0.9, 1.0])
    idx, pz, pm, ps = ref.topk16_shard(z, off, V_total, params=params)
    zz = z.double().numpy()
    for r in range(5):
        order = np.lexsort((np.arange(800), -zz[r]))     # value descending, then the lower id
        n = [16, 16, 30, 16, 16][r]
        np.testing.assert_array_equal(idx[r, :n], order[:n] + off)
        assert np.all(idx[r, n:] == -1) and np.all(np.isneginf(pz[r, n:]))
        np.testing.assert_array_equal(pz[r, :n], zz[r, order[:n]])
        assert pm[r] == zz[r].max()
        T = float(np.float32([1.0, 0.8, 1.0, 1.0, 2.0][r]))   # the parameters are f32
        filtered = r in (2, 3)
        want = 0.0 if filtered else np.exp((zz[r] - zz[r].max()) / T).sum()
        np.testing.assert_allclose(ps[r], want, rtol=1e-13)
