"""Pins of the oracle's fused LM head + top-16 on the CPU.  With inputs whose
logits are exact in f32 (small multiples of 1/8), the fused oracle must give
what the oracle's top-16 gives on those logits computed by a numpy matmul
(ids bit for bit, U and lse within 1e-12), for every sampling mode it takes;
rows that need more than 16 candidates or the whole row come out -1 / NaN;
and its gap is the smallest difference between consecutive best logits."""
import numpy as np
import torch

from dflash_draft_selection_gb300 import synth


def exact_inputs(rows, hidden, V, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(-2, 3, (rows, hidden), generator=g).float().bfloat16()
    W = (torch.randint(-8, 9, (V, hidden), generator=g).float() / 8).bfloat16()
    z = (h.double() @ W.double().T).float()   # exact: small multiples of 1/8
    assert torch.equal(z.double(), h.double() @ W.double().T)
    return h, W, z


def test_fused_equals_top16_of_the_logits(ref):
    h, W, z = exact_inputs(12, 128, 3000, 1)
    params = synth.make_params(6, [0.0, 1.0, 0.7, 1.0, 1.2, 0.0], [0, 0, 16, 10, 0, 0], [1.0, 1.0, 0.9, 1.0, 1.0, 1.0])
    f = ref.lmhead_topk16(h, W, params=params, rows_per_param=2)
    w = ref.topk16(z, params=params, rows_per_param=2)
    np.testing.assert_array_equal(f[0], w[0])
    np.testing.assert_allclose(f[1], w[1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(f[2], w[2], rtol=0, atol=1e-12)


def test_rows_needing_more_than_16_are_refused(ref):
    h, W, _ = exact_inputs(4, 64, 500, 2)
    params = synth.make_params(2, [1.0, 1.0], [20, 0], [1.0, 0.9])
    idx, U, lse, _, _ = ref.lmhead_topk16(h, W, params=params, rows_per_param=2)
    assert np.all(idx == -1) and np.all(np.isnan(U)) and np.all(np.isnan(lse))


def test_gap_is_the_closest_pair_among_the_best(ref):
    h, W, z = exact_inputs(3, 64, 800, 3)
    gap = ref.lmhead_topk16(h, W)[4]
    for r in range(3):
        s = np.sort(z[r].double().numpy())[::-1][:17]
        assert gap[r] == np.min(s[:-1] - s[1:])
