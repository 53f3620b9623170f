"""dflash2_ctx_gate (tensor cores for bf16) and dflash2_conv2tap against the oracle."""
import numpy as np
import pytest
import torch

import dflash_draft_selection_gb300 as d2
from tests._util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,hidden,D", [(1, 64, 16), (7, 256, 256), (128, 512, 64), (200, 2560, 256),
                                        (448, 5120, 256), (3840, 5120, 256), (130, 128, 32), (33, 1024, 512)])
def test_gate_bf16_tensor_cores(ref, n, hidden, D):
    dev = cuda_or_skip()
    g = torch.Generator().manual_seed(n + hidden)
    h = torch.randn(n, hidden, generator=g).bfloat16()
    W = (torch.randn(D, hidden, generator=g) / 16).bfloat16()
    out = d2.ctx_gate(h.to(dev), W.to(dev))
    torch.cuda.synchronize()
    rows = np.arange(n) if n <= 512 else np.r_[0:64, n - 64:n, 1000:1064]
    r = ref.ctx_gate(h[rows], W)
    assert_close(out.cpu().numpy()[rows], r, what=f"gate n={n} hidden={hidden} D={D}")
    assert d2.device_error() == 0


def test_gate_special_cases(ref):
    dev = cuda_or_skip()
    h = torch.randn(300, 256).bfloat16().to(dev)
    W = torch.zeros(256, 256).bfloat16().to(dev)
    assert torch.all(d2.ctx_gate(h, W) == 0.5)
    assert torch.all(d2.ctx_gate(torch.zeros_like(h), torch.randn_like(W)) == 0.5)


@pytest.mark.parametrize("n,hidden,D", [(7, 256, 256), (5, 100, 16)])
def test_gate_f32(ref, n, hidden, D):
    dev = cuda_or_skip()
    h = torch.randn(n, hidden)
    W = torch.randn(D, hidden) / 16
    out = d2.ctx_gate(h.to(dev), W.to(dev))
    assert_close(out.cpu().numpy(), ref.ctx_gate(h, W), what="gate f32")


def test_gate_invalid():
    dev = cuda_or_skip()
    with pytest.raises(d2.DFlash2Error):
        d2.ctx_gate(torch.randn(4, 100, device=dev).bfloat16(), torch.randn(256, 100, device=dev).bfloat16())
    with pytest.raises(d2.DFlash2Error):
        d2.ctx_gate(torch.randn(4, 128, device=dev).bfloat16(), torch.randn(48, 128, device=dev).bfloat16())


@pytest.mark.parametrize("B,T,H,G", [(2, 8, 2560, 1), (3, 5, 24, 1), (2, 4, 17, 1), (2, 8, 64, 4),
                                     (1, 1, 16, 16), (4, 16, 5120, 1)])
def test_conv_bf16_bit_exact(ref, B, T, H, G):
    dev = cuda_or_skip()
    g = torch.Generator().manual_seed(B * T + H)
    x = torch.randn(B, T, H, generator=g).bfloat16()
    k0 = (torch.rand(B, T, H // G, generator=g) * 2 - 1).bfloat16()
    k1 = (torch.rand(B, T, H // G, generator=g) * 2 - 1).bfloat16()
    xp = torch.randn(B, H, generator=g).bfloat16()
    y = d2.conv2tap(x.to(dev), k0.to(dev), k1.to(dev), xp.to(dev), group=G)
    r = ref.conv2tap(x, k0, k1, xp, group=G)
    assert torch.equal(y.cpu().view(torch.int16), r.view(torch.int16))


def test_conv_bf16_midpoints(ref):
    dev = cuda_or_skip()
    # exact midpoints decided by a tiny second product (see the oracle pins)
    vals = [(37 / 32, 7 / 8, -(2 ** -30), 2 ** -30), (37 / 32, 7 / 8, 2 ** -30, 2 ** -30),
            (1.0, 1.0, 2 ** -8, 1.0), (1.0, 1.0, 2 ** -8, 1 + 2 ** -7), (1.0, 1 + 2 ** -7, 2 ** -8, 1.0)]
    x = torch.tensor([[[v[0] for v in vals]]]).bfloat16()
    k0 = torch.tensor([[[v[1] for v in vals]]]).bfloat16()
    k1 = torch.tensor([[[v[2] for v in vals]]]).bfloat16()
    xp = torch.tensor([[v[3] for v in vals]]).bfloat16()
    y = d2.conv2tap(x.to(dev), k0.to(dev), k1.to(dev), xp.to(dev))
    r = ref.conv2tap(x, k0, k1, xp)
    assert torch.equal(y.cpu().view(torch.int16), r.view(torch.int16))


def test_conv_f32(ref):
    dev = cuda_or_skip()
    x = torch.randn(2, 6, 40)
    k0 = torch.rand(2, 6, 40) * 2 - 1
    k1 = torch.rand(2, 6, 40) * 2 - 1
    xp = torch.randn(2, 40)
    y = d2.conv2tap(x.to(dev), k0.to(dev), k1.to(dev), xp.to(dev)).cpu().numpy()
    r = ref.conv2tap(x, k0, k1, xp)
    prev = torch.cat([xp[:, None], x[:, :-1]], dim=1)
    scale = (k0.abs() * x.abs() + k1.abs() * prev.abs()).numpy()
    assert np.all(np.abs(y - r) <= 2 ** -22 * scale + 1e-30)
