"""Shared helpers of the parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

RTOL = 1e-4   # relative tolerance on fp scores / probabilities / log-probabilities
ATOL = 1e-5   # absolute floor
MARGIN = 1e-5  # oracle decision margin below which either outcome is accepted


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dflash_draft_selection_gb300 as d2
    d2.load_library()
    return torch.device("cuda:0")


def assert_close(gpu, ref, rtol=RTOL, atol=ATOL, what=""):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN pattern differs"
    inf_g, inf_r = np.isinf(g), np.isinf(r)
    assert np.array_equal(inf_g, inf_r) and np.array_equal(g[inf_g], r[inf_r]), f"{what}: inf pattern differs"
    fin = np.isfinite(r)
    err = np.abs(g[fin] - r[fin])
    lim = atol + rtol * np.abs(r[fin])
    if err.size:
        worst = int(np.argmax(err - lim))
        assert np.all(err <= lim), f"{what}: |gpu-ref| {err[worst]:.3g} > {lim[worst]:.3g} (ref {r[fin][worst]:.6g})"


def params_np(B, T, k, p):
    from dflash_draft_selection_gb300 import synth
    return synth.make_params(B, T, k, p)


def padded(z):
    """z [rows, V] copied into rows whose stride is a multiple of 16 bytes (the ABI's row alignment)."""
    rows, V = z.shape
    per = 16 // z.element_size()
    ld = (V + per - 1) // per * per
    buf = torch.zeros(rows, ld, dtype=z.dtype, device=z.device)
    buf[:, :V] = z
    return buf[:, :V]
