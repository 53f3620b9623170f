"""Seeded synthetic inputs for the DFlash 2 draft-selection + verify path.

This module only draws random numbers in the shapes and value distributions
of the workloads the DFlash 2 pages describe; it holds none of the method's
arithmetic.  Both the CUDA path and the CPU oracle are fed from here, and
nothing else is shared between them.

Recipes (one per named workload; sigma is always a standard deviation):

* ``tiny_f32``    B=1, K=7, V=4096, hidden=256, D=256, fp32.  Draft and target
  logits iid N(0, 2).  A, B, W_g ~ N(0, 1/16); h ~ N(0, 1).  Greedy.
* ``4b_greedy``   B=16, K=7, V=151936, hidden=2560, bf16.  Draft logits are
  Gumbel(0,1) per element plus one spike per row at a uniform token whose
  softmax mass is 0.85 (the 85.4% per-position Recall@1 of the DFlash 2
  proposer issue, "What upstream shipped").  Target = draft + N(0, 0.5).
  Conv inputs [16, 8, 2560]: x ~ N(0,1), taps ~ U(-1, 1).
* ``27b_greedy``  B=64, K=7, V=151936, hidden=5120, bf16; logits as above.
* ``27b_sampled`` as 27b_greedy with temperature 1, top_k 20, top_p 0.95 on
  both sides (the recommended sampling of the FreeToken DFlash 2 PR, "Speed")
  and U(0,1) uniforms for the walk, the accept test and the resample.
* ``27b_nucleus`` as 27b_sampled with top_k off (top_p 0.95 alone): the kept
  prefix reaches past the 64 best tokens of the rows.
* ``stress``      B=256, K=15, V=262144, hidden=5120, bf16; logits as above,
  and in 5% of draft and target rows one extra uniform token is set equal to
  the row maximum.  Conv inputs [256, 16, 5120] with a per-request x_prev.

The sampling parameters of a request are packed as 12-byte records
(float temperature, int32 top_k, float top_p).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SPIKE_MASS = 0.85

SAMPLING_DTYPE = np.dtype([("temperature", "<f4"), ("top_k", "<i4"), ("top_p", "<f4")])


@dataclass
class Shape:
    name: str
    B: int
    K: int
    V: int
    hidden: int
    D: int = 256
    dtype: torch.dtype = torch.bfloat16
    logits: str = "spike"          # "normal2" (N(0,2) iid) or "spike" (Gumbel + spike)
    target_noise: float = 0.5      # sigma of target - draft (spike recipe)
    temperature: float = 0.0
    top_k: int = 0
    top_p: float = 1.0
    dup_frac: float = 0.0          # fraction of rows with a duplicated maximum
    table_sigma: float = 1.0 / 16.0
    conv: bool = True
    seed: int = 0


WORKLOADS = {
    "tiny_f32": Shape("tiny_f32", 1, 7, 4096, 256, dtype=torch.float32, logits="normal2",
                      conv=False, seed=0),
    "4b_greedy": Shape("4b_greedy", 16, 7, 151936, 2560, seed=2),
    "27b_greedy": Shape("27b_greedy", 64, 7, 151936, 5120, seed=3),
    "27b_sampled": Shape("27b_sampled", 64, 7, 151936, 5120, temperature=1.0, top_k=20,
                         top_p=0.95, seed=4),
    "27b_nucleus": Shape("27b_nucleus", 64, 7, 151936, 5120, temperature=1.0, top_k=0,
                         top_p=0.95, seed=6),
    "stress": Shape("stress", 256, 15, 262144, 5120, dup_frac=0.05, seed=5),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def spike_logits(rows: int, V: int, g: torch.Generator, device, mass: float = SPIKE_MASS) -> torch.Tensor:
    """fp32 [rows, V]: Gumbel(0,1) noise plus one spike per row holding `mass` of the softmax."""
    u = torch.rand(rows, V, generator=g, device=device, dtype=torch.float32)
    u.clamp_(min=1e-12, max=1.0 - 1e-7)
    z = -torch.log(-torch.log(u))
    s = torch.randint(0, V, (rows,), generator=g, device=device)
    lse_all = torch.logsumexp(z.double(), dim=1)
    zs = z.gather(1, s[:, None]).squeeze(1).double()
    lse_rest = lse_all + torch.log1p(-torch.exp(zs - lse_all))
    spike = math.log(mass / (1.0 - mass)) + lse_rest
    z.scatter_(1, s[:, None], spike.float()[:, None])
    return z


def duplicate_max(x: torch.Tensor, frac: float, g: torch.Generator) -> torch.Tensor:
    """In a seeded `frac` of the rows of x, copy the row maximum to one more uniform token."""
    rows, V = x.shape
    n = int(round(frac * rows))
    if n == 0:
        return x
    dev = x.device
    pick = torch.randperm(rows, generator=g, device=dev)[:n]
    tok = torch.randint(0, V, (n,), generator=g, device=dev)
    amax = x[pick].float().argmax(dim=1)
    tok = torch.where(tok == amax, (tok + 1) % V, tok)
    mx = x[pick].max(dim=1).values
    x[pick, tok] = mx
    return x


@dataclass
class Inputs:
    shape: Shape
    draft_logits: torch.Tensor       # [B*K, V]
    target_logits: torch.Tensor      # [B*(K+1), V]
    A: torch.Tensor                  # [V, D]
    Bt: torch.Tensor                 # [V, D]
    Wg: torch.Tensor                 # [D, hidden]
    h: torch.Tensor                  # [B*K, hidden]
    last_tok: torch.Tensor           # [B] int32
    params: np.ndarray               # [B] SAMPLING_DTYPE
    u_walk: torch.Tensor             # [B, K] f32
    u_acc: torch.Tensor              # [B, K] f32
    u_res: torch.Tensor              # [B, K+1] f32
    conv: dict = field(default_factory=dict)


def make_logits(shp: Shape, g: torch.Generator, device):
    B, K, V = shp.B, shp.K, shp.V
    if shp.logits == "normal2":
        d = torch.randn(B * K, V, generator=g, device=device) * 2.0
        t = torch.randn(B * (K + 1), V, generator=g, device=device) * 2.0
    else:
        d = spike_logits(B * K, V, g, device)
        # target rows: t < K follow the draft rows plus noise; the bonus row is a fresh block row
        bonus = spike_logits(B, V, g, device)
        t = torch.empty(B, K + 1, V, device=device)
        t[:, :K] = d.to(shp.dtype).float().view(B, K, V)
        t[:, K] = bonus
        t += torch.randn(B, K + 1, V, generator=g, device=device) * shp.target_noise
        t = t.view(B * (K + 1), V)
    d = d.to(shp.dtype)
    t = t.to(shp.dtype)
    if shp.dup_frac > 0:
        duplicate_max(d, shp.dup_frac, g)
        duplicate_max(t, shp.dup_frac, g)
    return d, t


def make_params(B: int, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    p = np.zeros(B, dtype=SAMPLING_DTYPE)
    p["temperature"] = temperature
    p["top_k"] = top_k
    p["top_p"] = top_p
    return p


def make_inputs(shp: Shape, device="cpu", with_conv: bool | None = None) -> Inputs:
    g = _gen(shp.seed, device)
    B, K, V, D, Hd = shp.B, shp.K, shp.V, shp.D, shp.hidden
    d, t = make_logits(shp, g, device)
    sig = shp.table_sigma
    A = (torch.randn(V, D, generator=g, device=device) * sig).to(shp.dtype)
    Bt = (torch.randn(V, D, generator=g, device=device) * sig).to(shp.dtype)
    Wg = (torch.randn(D, Hd, generator=g, device=device) * (1.0 / 16.0)).to(shp.dtype)
    h = torch.randn(B * K, Hd, generator=g, device=device).to(shp.dtype)
    last_tok = torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int32)
    u_walk = torch.rand(B, K, generator=g, device=device)
    u_acc = torch.rand(B, K, generator=g, device=device)
    u_res = torch.rand(B, K + 1, generator=g, device=device)
    params = make_params(B, shp.temperature, shp.top_k, shp.top_p)
    inp = Inputs(shp, d, t, A, Bt, Wg, h, last_tok, params, u_walk, u_acc, u_res)
    if (shp.conv if with_conv is None else with_conv):
        inp.conv = make_conv(B, K + 1, Hd, shp.dtype, g, device)
    return inp


def make_conv(B: int, T: int, H: int, dtype, g: torch.Generator, device, group: int = 1) -> dict:
    """Two-tap conv inputs: x ~ N(0,1) [B,T,H], taps ~ U(-1,1) [B,T,H/group], x_prev ~ N(0,1) [B,H]."""
    Hk = H // group
    x = torch.randn(B, T, H, generator=g, device=device).to(dtype)
    k0 = (torch.rand(B, T, Hk, generator=g, device=device) * 2 - 1).to(dtype)
    k1 = (torch.rand(B, T, Hk, generator=g, device=device) * 2 - 1).to(dtype)
    x_prev = torch.randn(B, H, generator=g, device=device).to(dtype)
    return {"x": x, "k0": k0, "k1": k1, "x_prev": x_prev, "group": group}


def small_shape(name: str, **kw) -> Shape:
    """A workload with the recipe of `name` and some sizes overridden (for parity tests)."""
    base = WORKLOADS[name]
    d = dict(base.__dict__)
    d.update(kw)
    return Shape(**d)
