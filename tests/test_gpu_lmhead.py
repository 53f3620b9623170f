"""dflash2_lmhead_topk16 (the LM head and the top-16 fused, logits never in
memory) against the oracle (fp64 logits, then the top-16 definition).  With
logits exact in fp32 the candidates are bit for bit and U, lse within 1e-4
rel; with random bf16 inputs the fp32 accumulation may swap two candidates
whose fp64 logits are closer than 1e-4 (excused, at most 1% of the rows), and
U, lse are within 1e-4 (abs floor 1e-4).  Full size: the 27B drafter's LM head
(448 rows, hidden 5120, V 151936) on a sample of rows."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests._util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu

GAP = 1e-4


def exact_inputs(rows, hidden, V, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(-2, 3, (rows, hidden), generator=g).float().bfloat16()
    W = (torch.randint(-8, 9, (V, hidden), generator=g).float() / 8).bfloat16()
    return h, W


def run(h, W, params=None, rpp=1):
    dev = cuda_or_skip()
    pg = None if params is None else d2.sampling_params(params["temperature"], params["top_k"], params["top_p"],
                                                        device=dev)
    out = d2.lmhead_topk16(h.to(dev), W.to(dev), params=pg, rows_per_param=rpp)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


@pytest.mark.parametrize("rows,hidden,V", [(1, 64, 16), (130, 128, 3000), (257, 320, 4099)])
def test_exact_logits(ref, rows, hidden, V):
    h, W = exact_inputs(rows, hidden, V, rows)
    n = (rows + 1) // 2
    params = synth.make_params(n, np.resize([0.0, 1.0, 0.7, 1.0, 1.0], n), np.resize([0, 0, 16, 5, 20], n),
                               np.resize([1.0, 1.0, 0.9, 1.0, 1.0], n))
    idx, U, lse = run(h, W, params, 2)
    r_idx, r_U, r_lse, r_mg, _ = ref.lmhead_topk16(h, W, params=params, rows_per_param=2)
    np.testing.assert_array_equal(idx, r_idx)
    ok = r_mg >= 1e-5                       # top_p cuts at a near-tie are left to the U check below
    assert_close(U[ok], r_U[ok], what="U")
    assert_close(lse[ok], r_lse[ok], what="lse")
    assert d2.device_error() == 0


def check_random(ref, h, W, idx, U, lse, rows_checked):
    r_idx, r_U, r_lse, _, gap = ref.lmhead_topk16(h[rows_checked], W)
    excused = 0
    for k, r in enumerate(rows_checked):
        if gap[k] < GAP and not np.array_equal(idx[r], r_idx[k]):
            assert sorted(idx[r]) == sorted(r_idx[k]) or gap[k] < GAP, r
            excused += 1
            continue
        np.testing.assert_array_equal(idx[r], r_idx[k], err_msg=f"row {r}")
        assert_close(U[r], r_U[k], atol=1e-4, what=f"U row {r}")
        assert_close(lse[r], r_lse[k], atol=1e-4, what=f"lse row {r}")
    assert excused <= max(1, len(rows_checked) // 100), excused


def test_random_logits(ref):
    g = torch.Generator().manual_seed(5)
    h = torch.randn(130, 512, generator=g).bfloat16()
    W = (torch.randn(5000, 512, generator=g) / 512 ** 0.5).bfloat16()
    idx, U, lse = run(h, W)
    check_random(ref, h, W, idx, U, lse, np.arange(130))
    assert d2.device_error() == 0


def test_full_size_sampled_rows(ref):
    """The 27B drafter's LM head at full size; 8 rows (spread over the M tiles) checked one by one."""
    dev = cuda_or_skip()
    g = torch.Generator(device=dev).manual_seed(7)
    h = torch.randn(448, 5120, generator=g, device=dev).bfloat16()
    W = (torch.randn(151936, 5120, generator=g, device=dev) / 5120 ** 0.5).bfloat16()
    idx, U, lse = (t.cpu().numpy() for t in d2.lmhead_topk16(h, W))
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 255, 300, 383, 447])
    check_random(ref, h.cpu(), W.cpu(), idx, U, lse, rows)
    assert d2.device_error() == 0
