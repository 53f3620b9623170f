"""dflash2_dynconv2tap against the oracle: the taps (sigmoid of the tensor-core projection, fp32
accumulation) within 2e-5 of the fp64 taps.  y = x_{t-1} + k0 (x_t - x_{t-1}), so a tap off by d
moves y by d |x_t - x_{t-1}|: bf16 outputs are within one bf16 ulp of the exactly rounded fp64
value plus 2e-5 |x_t - x_{t-1}|, and equal to it almost everywhere; f32 outputs within 1e-5
relative plus the same tap term."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from tests._util import cuda_or_skip

pytestmark = pytest.mark.gpu


def _inputs(seed, B, T, H, G, dtype):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, T, H, generator=g).to(dtype)
    xp = torch.randn(B, H, generator=g).to(dtype)
    W = (torch.randn(H // G, H, generator=g) * (2.0 / H ** 0.5)).to(dtype)
    return x, xp, W


def _ulp_bf16(v):
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _compare(ref, x, xp, W, G):
    dev = cuda_or_skip()
    taps, y = d2.dynconv2tap(x.to(dev), xp.to(dev), W.to(dev), G)
    torch.cuda.synchronize()
    r_taps, r_y = ref.dynconv2tap(x, xp, W, G)
    np.testing.assert_allclose(taps.cpu().numpy().astype(np.float64), r_taps, rtol=0, atol=2e-5)
    yg = y.float().cpu().numpy().astype(np.float64)
    yr = (r_y.float().numpy() if isinstance(r_y, torch.Tensor) else r_y).astype(np.float64)
    _check_y(yg, yr, _step(x, xp), x.dtype)
    assert d2.device_error() == 0


def _step(x, xp):
    """|x_t - x_{t-1}| (x_prev at t = 0) in fp64."""
    xd = x.double()
    prev = torch.cat([xp.double()[:, None, :], xd[:, :-1, :]], dim=1)
    return (xd - prev).abs().numpy()


def _check_y(yg, yr, step, dtype):
    tap = 2e-5 * step
    diff = np.abs(yg - yr)
    if dtype == torch.bfloat16:
        assert np.all(diff <= _ulp_bf16(yr) * 1.0000001 + tap), float(np.max(diff - _ulp_bf16(yr) - tap))
        assert np.mean(diff == 0) > 0.99
    else:
        assert np.all(diff <= 1e-5 * np.abs(yr) + 1e-6 + tap)


@pytest.mark.parametrize("B,T,H,G", [(3, 5, 256, 16), (2, 4, 512, 8), (4, 3, 1024, 64)])
def test_bf16_vector_path(ref, B, T, H, G):
    """Group sizes that are multiples of 8: 16-byte vectors sharing one tap."""
    _compare(ref, *_inputs(B * 100 + G, B, T, H, G, torch.bfloat16), G)


def test_bf16_scalar_path(ref):
    """group_size 12 (not a multiple of 8): one element per step."""
    _compare(ref, *_inputs(7, 2, 6, 192, 12, torch.bfloat16), 12)


@pytest.mark.parametrize("H,G", [(256, 16), (100, 4)])
def test_f32(ref, H, G):
    """f32 on the CUDA cores, including a group count (25) the tensor-core path does not take."""
    _compare(ref, *_inputs(H + G, 3, 4, H, G, torch.float32), G)


def test_stress_shape_sampled_rows(ref):
    """B = 256, T = 16, H = 5120, group_size 80 (64 groups): the GPU runs the whole batch; 200
    sampled positions are compared element by element."""
    B, T, H, G = 256, 16, 5120, 80
    x, xp, W = _inputs(11, B, T, H, G, torch.bfloat16)
    rows = np.random.default_rng(3).choice(B * T, 200, replace=False)
    # the oracle on the sampled positions (and their predecessors) only
    dev = cuda_or_skip()
    taps, y = d2.dynconv2tap(x.to(dev), xp.to(dev), W.to(dev), G)
    torch.cuda.synchronize()
    b, t = rows // T, rows % T
    bt_, tt_, tp_ = torch.as_tensor(b), torch.as_tensor(t), torch.as_tensor(np.maximum(t - 1, 0))
    xs = torch.stack([x[bt_, tt_], torch.where(tt_[:, None] == 0, xp[bt_], x[bt_, tp_])], 1)
    # two-position sequences (predecessor, position) reproduce each sampled position's inputs
    x2 = torch.stack([xs[:, 1], xs[:, 0]], 1)
    r_taps, r_y = ref.dynconv2tap(x2, xs[:, 1], W, G)
    np.testing.assert_allclose(taps.cpu().numpy()[b, t].astype(np.float64), r_taps[:, 1], rtol=0, atol=2e-5)
    yg = y.float().cpu().numpy()[b, t].astype(np.float64)
    yr = r_y.float().numpy()[:, 1].astype(np.float64)
    _check_y(yg, yr, (xs[:, 0].double() - xs[:, 1].double()).abs().numpy(), torch.bfloat16)
    assert d2.device_error() == 0


def test_argument_errors():
    dev = cuda_or_skip()
    x = torch.randn(2, 3, 192, device=dev).bfloat16()
    xp = torch.randn(2, 192, device=dev).bfloat16()
    with pytest.raises(d2.DFlash2Error):
        d2.dynconv2tap(x, xp, torch.randn(5, 192, device=dev).bfloat16(), 40)    # 40 does not divide 192
    with pytest.raises(d2.DFlash2Error):
        d2.dynconv2tap(x, xp, torch.randn(24, 192, device=dev).bfloat16(), 8)    # 24 groups: not a power of two
