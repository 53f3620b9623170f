"""dflash2_topk16 against the oracle: bit-exact ids; U and lse within 1e-4 rel,
except on a row whose top_p cut is within 1e-5 of a cumulative mass, where
the GPU's cut may move by one token and its U must be that cut's filtered
distribution (tests/_parity.py; at most 1% of the rows)."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests import _parity
from tests._util import MARGIN, assert_close, cuda_or_skip, padded, params_np

pytestmark = pytest.mark.gpu


def run_both(ref, z, params=None, rpp=1, V=None):
    dev = cuda_or_skip()
    zg = padded(z.to(dev))
    pg = None if params is None else d2.sampling_params(params["temperature"], params["top_k"], params["top_p"],
                                                        device=dev)
    Vv = z.shape[1] if V is None else V
    idx, U, lse = d2.topk16(zg, params=pg, rows_per_param=rpp, V=Vv)
    torch.cuda.synchronize()
    r_idx, r_U, r_lse, r_mg = ref.topk16(z, params=params, rows_per_param=rpp, V=Vv, ld=z.shape[1])
    prow = synth.make_params(z.shape[0], 0.0, 0, 1.0) if params is None else np.repeat(params, rpp)[:z.shape[0]]
    return z, prow, idx.cpu().numpy(), U.cpu().numpy(), lse.cpu().numpy(), r_idx, r_U, r_lse, r_mg


def compare(res, what):
    ex = _parity.Excused()
    _parity.topk_compare(*res, ex, what=what)
    ex.check_bound(what=what)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [16, 17, 100, 4096, 8192 + 13, 40000])
def test_greedy_random(ref, dtype, V):
    g = torch.Generator().manual_seed(V)
    z = (torch.randn(11, V, generator=g) * 3).to(dtype)
    compare(run_both(ref, z), f"greedy V={V} {dtype}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ties_zero_signs_and_duplicates(ref, dtype):
    V = 9000
    g = torch.Generator().manual_seed(1)
    z = (torch.randint(-4, 4, (8, V), generator=g).float() * 0.25).to(dtype)
    z[1] = 2.0                           # all equal
    z[2, ::2] = -0.0
    z[2, 1::2] = 0.0
    z[3, [5, 8000, 20]] = 7.0            # triple maximum
    compare(run_both(ref, z), "ties")


@pytest.mark.parametrize("sampled", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tie_blocks_and_ramps_mid_row(ref, dtype, sampled):
    """Rows whose candidates pile up after the first chunk: a block of tied
    maxima, many spread-out ties, a dense tie cluster in one chunk, ascending
    and descending ramps.  Some overflow a warp's candidate buffer after the
    floor has risen and are ranked by the rescan; the rest are ranked from
    the streamed lists alone.  Either way the result must be exact."""
    V = 50000
    g = torch.Generator().manual_seed(7)
    z = torch.randn(8, V, generator=g) * 2
    z[0, 20000:20000 + 4096] = 9.0      # a whole chunk of tied maxima
    z[1, ::997] = 8.0                   # ~50 ties spread over the row
    z[2, 30000:30070] = 8.0             # 70 ties inside one chunk
    z[3] = torch.linspace(-5.0, 5.0, V)  # ascending: every chunk beats the last
    z[4] = torch.linspace(5.0, -5.0, V)  # descending: the first chunk holds the best
    z[5, 40000:40040] = z[5].max() + 1.0  # 40 ties near the row's end
    z = z.to(dtype)
    params = params_np(8, 1.0, 64, 1.0) if sampled else None
    compare(run_both(ref, z, params=params), f"tie blocks sampled={sampled}")


def test_padded_rows_ld_greater_than_V(ref):
    V, ld = 5000, 5008
    z = torch.randn(6, ld).bfloat16()
    z[:, V:] = 100.0                     # padding must not be read
    dev = cuda_or_skip()
    idx, U, lse = d2.topk16(z.to(dev), V=V)
    r_idx, r_U, r_lse, _ = ref.topk16(z, V=V, ld=ld)
    np.testing.assert_array_equal(idx.cpu().numpy(), r_idx)
    assert_close(U.cpu().numpy(), r_U)


@pytest.mark.parametrize("T,k,p", [(0.0, 0, 1.0), (0.7, 0, 1.0), (1.0, 20, 0.95), (1.0, 64, 1.0),
                                   (0.5, 5, 0.5), (2.0, 1, 1.0), (1.0, 16, 0.3), (1.3, 40, 0.99)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_sampled_filters(ref, T, k, p, dtype):
    g = torch.Generator().manual_seed(int(T * 10) + k)
    z = (torch.randn(12, 6000, generator=g) * 2.5).to(dtype)
    compare(run_both(ref, z, params=params_np(12, T, k, p)), f"T={T} k={k} p={p}")


def test_mixed_params_per_request(ref):
    B, K, V = 4, 3, 3000
    z = (torch.randn(B * K, V) * 2).bfloat16()
    p = params_np(B, 1.0, 20, 0.95)
    p["temperature"][1] = 0.0
    p["top_k"][2] = 0
    p["top_p"][2] = 1.0
    p["temperature"][3] = 0.5
    compare(run_both(ref, z, params=p, rpp=K), "mixed")


def test_bad_rows_and_params(ref):
    V = 700
    z = torch.randn(6, V)
    z[0, 5] = float("nan")
    z[1, 9] = float("inf")
    z[2, :] = float("-inf")
    z[3, :690] = float("-inf")
    _, _, idx, U, lse, r_idx, r_U, r_lse, _ = run_both(ref, z)
    np.testing.assert_array_equal(idx, r_idx)
    assert_close(U, r_U)
    p = params_np(6, 1.0, 10, 1.0)
    p["top_p"][4] = 0.0                  # invalid
    p["temperature"][5] = -1.0           # invalid
    _, _, idx, U, lse, r_idx, r_U, r_lse, _ = run_both(ref, z, params=p)
    np.testing.assert_array_equal(idx, r_idx)
    assert np.all(idx[4:] == -1) and np.all(np.isnan(U[4:]))


def wide_compare(ref, z, params, rpp, what):
    """Rows whose filter reaches past their 64 best (top_k > 64, or top_p with top_k off).  Ids are
    bit for bit.  A row whose kept prefix covers all 16 candidates has U and lse within 1e-4 rel
    whatever its exact cut: moving a deep cut by a few tokens of mass ~1e-5 changes U by less.  A
    row cut within its 16 candidates follows the near-tie rules of tests/_parity.py, bounded."""
    dev = cuda_or_skip()
    pg = d2.sampling_params(params["temperature"], params["top_k"], params["top_p"], device=dev)
    idx, U, lse = (t.cpu().numpy() for t in d2.topk16(padded(z.to(dev)), params=pg, rows_per_param=rpp))
    zc = z.cpu()
    r_idx, r_U, r_lse, r_mg = ref.topk16(zc, params=params, rows_per_param=rpp)
    np.testing.assert_array_equal(idx, r_idx, err_msg=what + " ids")
    deep = np.all(np.isfinite(r_U), axis=1)
    assert_close(U[deep], r_U[deep], what=what + " U (deep cuts)")
    assert_close(lse[deep], r_lse[deep], what=what + " lse (deep cuts)")
    sh = ~deep
    if sh.any():
        ex = _parity.Excused()
        prow = np.repeat(params, rpp)[: z.shape[0]]
        _parity.topk_compare(zc[sh], prow[sh], idx[sh], U[sh], lse[sh], r_idx[sh], r_U[sh], r_lse[sh], r_mg[sh], ex,
                             what=what + " (cuts within the candidates)")
        ex.check_bound(what=what)
    return deep


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_wide_filters(ref, dtype):
    """top_p with top_k off, top_k above 64 with and without top_p, on flat rows (deep cuts, found by
    passes over the row) and peaked rows (cuts within the 64 best, no pass), V = 40000."""
    g = torch.Generator().manual_seed(21)
    rows_per = 3
    flat = torch.randn(8 * rows_per, 40000, generator=g) * 1.5
    peaked = synth.spike_logits(8 * rows_per, 40000, torch.Generator().manual_seed(22), "cpu")
    z = torch.cat([flat, peaked]).to(dtype)
    T = [1.0, 0.7, 1.2, 1.0, 0.9, 1.0, 2.0, 1.0] * 2
    k = [0, 200, 1000, 0, 65, 30000, 0, 100] * 2
    p = [0.9, 1.0, 0.8, 0.5, 0.95, 0.99, 0.3, 1.0] * 2
    deep = wide_compare(ref, z, synth.make_params(16, T, k, p), rows_per, f"wide {dtype}")
    assert deep.any() and (~deep).any()


def test_exactly_64_with_ties_at_f(ref):
    """Lists exactly 64 long (top_k = 64, and top_p with top_k off) on rows whose best value is
    shared by 70 or by 300 tokens: the 64th slice maximum F is tied, so the extraction gathers
    every element that reaches F (70: within its buffer; 300: more than it holds, so every slice
    is ranked); the kept ties are the lowest ids.  bf16, V = 50000."""
    g = torch.Generator().manual_seed(64)
    rows_per, V = 3, 50000
    z = torch.randn(4 * rows_per, V, generator=g) * 2
    for r in range(z.shape[0]):
        n_tie = 300 if (r // rows_per) % 2 == 0 else 70
        pos = torch.randperm(V, generator=g)[:n_tie]
        z[r, pos] = z[r].max() + 1.0
    z = z.bfloat16()
    p = synth.make_params(4, [1.0, 1.0, 1.0, 1.0], [64, 64, 0, 0], [1.0, 1.0, 0.9, 0.5])
    wide_compare(ref, z, p, rows_per, "ties at F")


def test_many_wide_rows_per_cta(ref):
    """16384 flat rows of V = 4096 with top_p 0.9 and top_k off: about 36 wide rows per CTA, every
    one finished in its CTA's epilogue after the stream; 256 sampled rows against the oracle."""
    dev = cuda_or_skip()
    rows, V = 16384, 4096
    g = torch.Generator(device=dev).manual_seed(36)
    z = (torch.randn(rows, V, generator=g, device=dev) * 1.5).bfloat16()
    p = synth.make_params(rows, 1.0, 0, 0.9)
    pg = d2.sampling_params(p["temperature"], p["top_k"], p["top_p"], device=dev)
    idx, U, lse = (t.cpu().numpy() for t in d2.topk16(z, params=pg))
    assert d2.device_error() == 0
    pick = np.random.default_rng(5).choice(rows, 256, replace=False)
    zc = z[torch.as_tensor(pick, device=dev)].cpu()
    r_idx, r_U, r_lse, _ = ref.topk16(zc, params=p[pick])
    np.testing.assert_array_equal(idx[pick], r_idx)
    assert np.all(np.isfinite(r_U))          # every cut is deeper than the 16 candidates
    assert_close(U[pick], r_U, what="many wide rows U")
    assert_close(lse[pick], r_lse, what="many wide rows lse")


def test_wide_full_size(ref):
    """The 27B drafter's rows (448 x 151936 bf16) with top_p 0.95 and top_k off: every row."""
    dev = cuda_or_skip()
    shp = synth.WORKLOADS["27b_sampled"]
    g = torch.Generator(device=dev).manual_seed(shp.seed)
    z = synth.spike_logits(shp.B * shp.K, shp.V, g, dev).to(shp.dtype)
    wide_compare(ref, z.cpu(), synth.make_params(shp.B, 1.0, 0, 0.95), shp.K, "27b top_p 0.95")
    assert d2.device_error() == 0


def test_empty_and_invalid(ref):
    dev = cuda_or_skip()
    z = torch.randn(0, 100, device=dev)
    idx, U, lse = d2.topk16(z)
    assert idx.shape == (0, 16)
    with pytest.raises(d2.DFlash2Error):
        d2.topk16(torch.randn(2, 8, device=dev))          # V < 16
    with pytest.raises(d2.DFlash2Error):
        d2.topk16(torch.randn(2, 100, device=dev).bfloat16()[:, :99], V=99)  # ld*2 not 16-aligned? (ld=100 ok)


@pytest.mark.parametrize("name", ["27b_greedy", "27b_sampled", "stress"])
def test_full_size_all_rows(ref, name):
    """The full workload in the bench's launch configuration, every row checked against the oracle."""
    dev = cuda_or_skip()
    shp = synth.WORKLOADS[name]
    g = torch.Generator(device=dev).manual_seed(shp.seed)
    rows = shp.B * shp.K
    z = synth.spike_logits(rows, shp.V, g, dev).to(shp.dtype)
    if shp.dup_frac:
        synth.duplicate_max(z, shp.dup_frac, g)
    p = synth.make_params(shp.B, shp.temperature, shp.top_k, shp.top_p)
    pg = d2.sampling_params(p["temperature"], p["top_k"], p["top_p"], device=dev)
    idx, U, lse = d2.topk16(z, params=pg if shp.temperature > 0 else None, rows_per_param=shp.K)
    torch.cuda.synchronize()
    if shp.dup_frac:  # the rows with a duplicated maximum are among them
        zz = z.float()
        mx = zz.max(dim=1, keepdim=True).values
        assert ((zz == mx).sum(dim=1) > 1).any()
    zc = z.cpu()   # every row, checked one by one against the oracle
    pr = None if shp.temperature == 0 else p
    r_idx, r_U, r_lse, r_mg = ref.topk16(zc, params=pr, rows_per_param=shp.K)
    prow = synth.make_params(rows, 0.0, 0, 1.0) if pr is None else np.repeat(p, shp.K)
    ex = _parity.Excused()
    _parity.topk_compare(zc, prow, idx.cpu().numpy(), U.cpu().numpy(), lse.cpu().numpy(), r_idx, r_U, r_lse, r_mg,
                         ex, what=name)
    ex.check_bound(what=name)
    assert d2.device_error() == 0
