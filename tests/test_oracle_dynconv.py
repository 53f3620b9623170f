"""Pins of the oracle's grouped dynamic two-tap convolution (taps k0 = sigmoid(Wd . x_t) per group
of channels, k1 = 1 - k0; y_t = k0 x_t + k1 x_{t-1}, x_prev at t = 0) to things other than
itself: scipy's expit for the taps, closed forms for Wd = 0 (the mean of the two positions) and
for saturated taps (y = x_t, or the shift y = x_{t-1}).  No GPU needed."""
import numpy as np
import torch
from scipy.special import expit


def _inputs(seed, B, T, H, G, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, T, H, generator=g).to(dtype)
    xp = torch.randn(B, H, generator=g).to(dtype)
    W = (torch.randn(H // G, H, generator=g) / H ** 0.5).to(dtype)
    return x, xp, W


def _prev(x, xp):
    """x_{t-1} for every position, x_prev at t = 0."""
    return torch.cat([xp[:, None, :], x[:, :-1, :]], dim=1)


def test_taps_are_expit_of_the_projection(ref):
    x, xp, W = _inputs(1, 3, 5, 64, 8)
    taps, _ = ref.dynconv2tap(x, xp, W, 8)
    want = expit(np.einsum("bth,gh->btg", x.double().numpy(), W.double().numpy()))
    np.testing.assert_allclose(taps, want, rtol=1e-12, atol=0)


def test_zero_projection_averages_the_two_positions(ref):
    x, xp, W = _inputs(2, 2, 6, 48, 16)
    taps, y = ref.dynconv2tap(x, xp, torch.zeros_like(W), 16)
    assert np.all(taps == 0.5)
    # (x_t + x_{t-1}) / 2 is exact in fp64 for bf16 operands; torch rounds it to bf16 (nearest even)
    want = ((x.double() + _prev(x, xp).double()) / 2).to(torch.bfloat16)
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_saturated_taps_select_one_position(ref):
    """A projection of +-60 on one channel held at 1 drives every tap to 1 or 0 (within e^-60):
    y is x_t itself, or the sequence shifted by one (x_prev first)."""
    B, T, H, G = 2, 4, 32, 8
    x, xp, _ = _inputs(3, B, T, H, G)
    x[:, :, 5] = 1.0
    W = torch.zeros(H // G, H, dtype=torch.bfloat16)
    W[:, 5] = 60.0
    _, y = ref.dynconv2tap(x, xp, W, G)
    keep = torch.ones(H, dtype=torch.bool)
    keep[5] = False
    assert torch.equal(y[..., keep].view(torch.int16), x[..., keep].view(torch.int16))
    W[:, 5] = -60.0
    _, y = ref.dynconv2tap(x, xp, W, G)
    assert torch.equal(y[..., keep].view(torch.int16), _prev(x, xp)[..., keep].view(torch.int16))


def test_f32_saturated_and_zero_cases(ref):
    x, xp, W = _inputs(4, 2, 3, 40, 10, torch.float32)
    _, y = ref.dynconv2tap(x, xp, torch.zeros_like(W), 10)
    np.testing.assert_array_equal(y, ((x.double() + _prev(x, xp).double()) / 2).float().numpy())
