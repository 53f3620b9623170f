"""dflash2_topk16_noalloc: the drafter-row reduction for callers that cannot
give this library any device memory (a plugin, or an engine whose memory pool
hands out no scratch).  Called through the C ABI it must give the same
candidates, U and lse as dflash2_topk16 with a workspace, on two calls in a
row whose rows are split over several CTAs (the split rows use the tickets and
partial records of the fixed scratch, so the second call would go wrong if the
first left its tickets behind), and at its largest batch.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from dflash_draft_selection_gb300 import synth
from tests._util import cuda_or_skip

pytestmark = pytest.mark.gpu

MAX_ROWS = 16384   # DFLASH2_TOPK16_NOALLOC_MAX_ROWS


def _same(a, b, what):
    for name, x, y in zip(("cand_idx", "cand_U", "lse"), a, b):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy(), err_msg=f"{what} {name}")


def _logits(seed, rows, V, dev, dtype=torch.bfloat16):
    g = torch.Generator(device=dev).manual_seed(seed)
    return synth.spike_logits(rows, V, g, dev).to(dtype)


def test_noalloc_topk16_matches_the_workspace_call_twice():
    """Few long rows (each split over many CTAs), then a sampled batch: each
    call's outputs equal the workspace call's bit for bit."""
    dev = cuda_or_skip()
    z1 = _logits(1, 6, 262144, dev)                      # 6 rows x 64 chunks: every row is split
    z2 = _logits(2, 7 * 9, 151936, dev, torch.float32)   # 63 rows, sampled, rows_per_param 7
    p2 = d2.sampling_params([1.0, 0.7, 1.3] * 3, [20, 0, 5] * 3, [0.95, 0.8, 1.0] * 3, device=dev)
    got1 = d2.topk16_noalloc(z1)
    got2 = d2.topk16_noalloc(z2, params=p2, rows_per_param=7)
    ref1 = d2.topk16(z1)
    ref2 = d2.topk16(z2, params=p2, rows_per_param=7)
    torch.cuda.synchronize()
    _same(got1, ref1, "first call")
    _same(got2, ref2, "second call")
    assert d2.device_error() == 0


def test_noalloc_topk16_at_its_largest_batch():
    dev = cuda_or_skip()
    z = _logits(3, MAX_ROWS, 4096, dev)
    got = d2.topk16_noalloc(z)
    ref = d2.topk16(z)
    torch.cuda.synchronize()
    _same(got, ref, f"rows={MAX_ROWS}")


def test_noalloc_topk16_wide_rows_at_its_largest_batch():
    """top_p with top_k off on every row of the largest batch: each CTA marks and finishes about 36
    wide rows in the fixed scratch; equal to the workspace call, twice in a row (the marks must
    be cleared between calls)."""
    dev = cuda_or_skip()
    z = _logits(4, MAX_ROWS, 4096, dev)
    p = d2.sampling_params([1.0], [0], [0.9], device=dev)
    for _ in range(2):
        got = d2.topk16_noalloc(z, params=p, rows_per_param=MAX_ROWS)
        ref = d2.topk16(z, params=p, rows_per_param=MAX_ROWS)
        torch.cuda.synchronize()
        _same(got, ref, "wide rows")
    assert d2.device_error() == 0


def test_noalloc_topk16_rejects_batches_beyond_its_array():
    cuda_or_skip()
    L = d2.load_library()
    p = ctypes.c_void_p(256)
    st = L.dflash2_topk16_noalloc(p, 1, MAX_ROWS + 1, 4096, 4096, None, 1, p, p, p, None)
    assert st == 4  # DFLASH2_ERR_WORKSPACE: nothing launched
    assert L.dflash2_topk16_noalloc(p, 1, 0, 4096, 4096, None, 1, p, p, p, None) == 0
    assert L.dflash2_topk16_noalloc(p, 1, -1, 4096, 4096, None, 1, p, p, p, None) == 1
