"""CPU oracle for the DFlash 2 draft-selection + verify path (TEST INFRASTRUCTURE).

A plain fp64 C restatement of each step (``dflash2_ref.c``) behind numpy
wrappers.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the CUDA library never does, and
the two share no code.  Inputs are torch CPU tensors or numpy arrays; bf16
tensors are passed as their raw 16-bit words and widened inside the C code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash2_ref.c")
_LIB = os.path.join(_HERE, "libdflash2_ref.so")
_lock = threading.Lock()
_lib = None

NC = 16
ST_OK, ST_NAN, ST_BAD_Q, ST_BAD_PARAMS = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no machine-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            L.dflash2_ref_topk16.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, i64, vp, vp, vp, vp]
            L.dflash2_ref_topk16_shard.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, vp, vp, i64, i32, vp, vp,
                                                   vp, vp]
            L.dflash2_ref_topk16_merge.argtypes = [i32, i64, i32, vp, vp, vp, vp, i64, vp, vp, vp, i64, vp, vp, vp,
                                                   vp]
            L.dflash2_ref_lmhead_topk16.argtypes = [vp, vp, i32, i64, i64, i64, vp, vp, vp, i64, vp, vp, vp, vp,
                                                    vp]
            L.dflash2_ref_ctx_gate.argtypes = [vp, i32, i64, i64, vp, i64, vp]
            L.dflash2_ref_pair_scores.argtypes = [i64, i32, vp, vp, vp, vp, vp, i32, i64, i32, vp, vp]
            L.dflash2_ref_walk.argtypes = [i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.dflash2_ref_target_dist.argtypes = [vp, i32, i64, f32, ctypes.c_int32, f32, vp, vp, i64, vp]
            L.dflash2_ref_target_dist.restype = i64
            L.dflash2_ref_verify.argtypes = [vp, i32, i64, i32, i64, i64, vp, vp, vp, vp, vp, vp, vp,
                                             vp, vp, i32, vp, vp, vp, vp]
            L.dflash2_ref_accept_sparse.argtypes = [i64, i64, i32, vp, vp, vp, i64, vp, vp, vp, vp, vp,
                                                    vp, vp, i32, vp, vp, vp]
            L.dflash2_ref_walk_accept_mc.argtypes = [i64, i64, i32, vp, vp, vp, vp, vp, vp, i64, vp, vp,
                                                     vp, vp, vp]
            L.dflash2_ref_conv2tap.argtypes = [vp, vp, vp, vp, i32, i64, i32, i64, i32, vp]
            L.dflash2_ref_dynconv2tap.argtypes = [vp, vp, vp, i32, i64, i32, i64, i32, vp, vp]
            L.dflash2_ref_num_threads.restype = i32
            L.dflash2_ref_set_num_threads.argtypes = [i32]
            _lib = L
    return _lib


def num_threads() -> int:
    return lib().dflash2_ref_num_threads()


def set_num_threads(n: int) -> None:
    lib().dflash2_ref_set_num_threads(int(n))


# ---------------------------------------------------------------- marshalling
def _raw(x):
    """(contiguous numpy array, dtype code) for a float tensor/array: 0 = f32, 1 = bf16 words."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), 1
            return x.to(torch.float32).numpy(), 0
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 1
    return np.ascontiguousarray(x, dtype=np.float32), 0


def _arr(x, dtype):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _params(params, n):
    """Split a SAMPLING_DTYPE record array (or None = greedy) into three arrays."""
    if params is None:
        return None, None, None
    p = np.asarray(params)
    return (np.ascontiguousarray(p["temperature"], dtype=np.float32),
            np.ascontiguousarray(p["top_k"], dtype=np.int32),
            np.ascontiguousarray(p["top_p"], dtype=np.float32))


# ------------------------------------------------------------------ functions
def topk16(logits, params=None, rows_per_param=1, V=None, ld=None):
    """Returns (cand_idx [rows,16] i32, cand_U [rows,16] f64, lse [rows] f64, margin [rows])."""
    raw, dt = _raw(logits)
    rows = raw.shape[0]
    ld = raw.shape[1] if ld is None else ld
    V = raw.shape[1] if V is None else V
    T, tk, tp = _params(params, rows)
    idx = np.empty((rows, NC), np.int32)
    U = np.empty((rows, NC), np.float64)
    lse = np.empty(rows, np.float64)
    mg = np.empty(rows, np.float64)
    lib().dflash2_ref_topk16(_p(raw), dt, rows, V, ld, _p(T), _p(tk), _p(tp), rows_per_param,
                             _p(idx), _p(U), _p(lse), _p(mg))
    return idx, U, lse, mg


SHARD_P = 64  # list entries per row of a shard partial


def topk16_shard(logits, off, V_total, params=None, rows_per_param=1, P=SHARD_P):
    """One vocabulary shard's partial.  logits [rows, Vs] hold tokens off..off+Vs-1.
    Returns (part_idx [rows,P] i32, part_z [rows,P] f64, part_m [rows], part_s [rows])."""
    raw, dt = _raw(logits)
    rows, Vs = raw.shape
    T, tk, tp = _params(params, rows)
    idx = np.empty((rows, P), np.int32)
    z = np.empty((rows, P), np.float64)
    m = np.empty(rows, np.float64)
    sm = np.empty(rows, np.float64)
    lib().dflash2_ref_topk16_shard(_p(raw), dt, rows, Vs, Vs, off, V_total, _p(T), _p(tk), _p(tp),
                                   rows_per_param, P, _p(idx), _p(z), _p(m), _p(sm))
    return idx, z, m, sm


def topk16_merge(part_idx, part_z, part_m, part_s, V_total, params=None, rows_per_param=1):
    """Merge partials stacked [S, rows, P] / [S, rows].  Returns (cand_idx, cand_U, lse, margin)."""
    pi = _arr(part_idx, np.int32)
    pz = _arr(part_z, np.float64)
    pm = _arr(part_m, np.float64)
    ps = _arr(part_s, np.float64)
    S, rows, P = pi.shape
    T, tk, tp = _params(params, rows)
    idx = np.empty((rows, NC), np.int32)
    U = np.empty((rows, NC), np.float64)
    lse = np.empty(rows, np.float64)
    mg = np.empty(rows, np.float64)
    lib().dflash2_ref_topk16_merge(S, rows, P, _p(pi), _p(pz), _p(pm), _p(ps), V_total, _p(T), _p(tk), _p(tp),
                                   rows_per_param, _p(idx), _p(U), _p(lse), _p(mg))
    return idx, U, lse, mg


def lmhead_topk16(h, W, params=None, rows_per_param=1):
    """h [rows, hidden], W [V, hidden] (bf16 or f32).  Returns (cand_idx, cand_U, lse, margin, gap)."""
    hr, dt = _raw(h)
    wr, dt2 = _raw(W)
    assert dt == dt2
    rows, hidden = hr.shape
    V = wr.shape[0]
    T, tk, tp = _params(params, rows)
    idx = np.empty((rows, NC), np.int32)
    U = np.empty((rows, NC), np.float64)
    lse = np.empty(rows, np.float64)
    mg = np.empty(rows, np.float64)
    gap = np.empty(rows, np.float64)
    lib().dflash2_ref_lmhead_topk16(_p(hr), _p(wr), dt, rows, hidden, V, _p(T), _p(tk), _p(tp), rows_per_param,
                                    _p(idx), _p(U), _p(lse), _p(mg), _p(gap))
    return idx, U, lse, mg, gap


def ctx_gate(h, Wg):
    hr, dt = _raw(h)
    wr, dt2 = _raw(Wg)
    assert dt == dt2
    n, hidden = hr.shape
    D = wr.shape[0]
    out = np.empty((n, D), np.float64)
    lib().dflash2_ref_ctx_gate(_p(hr), dt, n, hidden, _p(wr), D, _p(out))
    return out


def pair_scores(cand_idx, cand_U, last_tok, A, Bt, gate, B, K):
    ar, dt = _raw(A)
    br, dt2 = _raw(Bt)
    assert dt == dt2
    V, D = ar.shape
    ci = _arr(cand_idx, np.int32)
    cu = _arr(cand_U, np.float64)
    lt = _arr(last_tok, np.int32)
    g = _arr(gate, np.float64)
    S = np.empty((B, K, NC, NC), np.float64)
    lib().dflash2_ref_pair_scores(B, K, _p(ci), _p(cu), _p(lt), _p(ar), _p(br), dt, V, D, _p(g), _p(S))
    return S


def walk(cand_idx, scores, temperature, u_walk, B, K, R=1):
    """u_walk [R,B,K] (or [B,K] with R=1).  Returns path_tok, path_slot, q_sel, margin."""
    ci = _arr(cand_idx, np.int32)
    S = _arr(scores, np.float64)
    T = _arr(temperature, np.float32)
    u = _arr(u_walk, np.float32)
    shp = (R, B, K) if R > 1 else (B, K)
    pt = np.empty(shp, np.int32)
    ps = np.empty(shp, np.int32)
    q = np.empty(shp + (NC,), np.float64)
    mg = np.empty(shp, np.float64)
    lib().dflash2_ref_walk(R, B, K, _p(ci), _p(S), _p(T), _p(u), _p(pt), _p(ps), _p(q), _p(mg))
    return pt, ps, q, mg


def target_dist(row, temperature=0.0, top_k=0, top_p=1.0, cap=None):
    raw, dt = _raw(row)
    raw = raw.reshape(-1)
    V = raw.shape[0]
    cap = V if cap is None else cap
    ids = np.empty(cap, np.int32)
    pr = np.empty(cap, np.float64)
    mg = np.empty(1, np.float64)
    n = lib().dflash2_ref_target_dist(_p(raw), dt, V, float(temperature), int(top_k), float(top_p),
                                      _p(ids), _p(pr), cap, _p(mg))
    if n < 0:
        return n, None, None, float(mg[0])
    return int(n), ids[:n].copy(), pr[:n].copy(), float(mg[0])


def verify(tlogits, path_tok, cand_idx, q_sel, path_slot, params, u_acc, u_res, B, K,
           trusted=False, V=None, ld=None):
    raw, dt = _raw(tlogits)
    ld = raw.shape[-1] if ld is None else ld
    V = raw.shape[-1] if V is None else V
    T, tk, tp = _params(params, B)
    pt = _arr(path_tok, np.int32)
    ci = _arr(cand_idx, np.int32)
    q = _arr(q_sel, np.float64)
    ps = _arr(path_slot, np.int32)
    ua = _arr(u_acc, np.float32)
    ur = _arr(u_res, np.float32)
    acc = np.empty(B, np.int32)
    out = np.empty((B, K + 1), np.int32)
    st = np.empty(B, np.int32)
    mg = np.empty(B, np.float64)
    lib().dflash2_ref_verify(_p(raw), dt, B, K, V, ld, _p(pt), _p(ci), _p(q), _p(ps), _p(T), _p(tk),
                             _p(tp), _p(ua), _p(ur), int(trusted), _p(acc), _p(out), _p(st), _p(mg))
    return acc, out, st, mg


def accept_sparse(dist_ids, dist_p, dist_n, temperature, path_tok, cand_idx, q_sel, path_slot,
                  u_acc, u_res, B, K, R, trusted=False):
    di = _arr(dist_ids, np.int32)
    dp = _arr(dist_p, np.float64)
    dn = _arr(dist_n, np.int64)
    cap = di.shape[-1]
    T = _arr(temperature, np.float32)
    pt = _arr(path_tok, np.int32)
    ci = _arr(cand_idx, np.int32)
    q = _arr(q_sel, np.float64)
    ps = _arr(path_slot, np.int32)
    ua = _arr(u_acc, np.float32)
    ur = _arr(u_res, np.float32)
    acc = np.empty((R, B), np.int32)
    out = np.empty((R, B, K + 1), np.int32)
    st = np.empty((R, B), np.int32)
    lib().dflash2_ref_accept_sparse(R, B, K, _p(di), _p(dp), _p(dn), cap, _p(T), _p(pt), _p(ci), _p(q),
                                    _p(ps), _p(ua), _p(ur), int(trusted), _p(acc), _p(out), _p(st))
    return acc, out, st


def walk_accept_mc(cand_idx, scores, temperature, dist_ids, dist_p, dist_n, u_walk, u_acc, u_res,
                   B, K, R):
    """R repetitions of (sampled walk, accept) over fixed scores and target distributions."""
    ci = _arr(cand_idx, np.int32)
    S = _arr(scores, np.float64)
    T = _arr(temperature, np.float32)
    di = _arr(dist_ids, np.int32)
    dp = _arr(dist_p, np.float64)
    dn = _arr(dist_n, np.int64)
    cap = di.shape[-1]
    uw = _arr(u_walk, np.float32)
    ua = _arr(u_acc, np.float32)
    ur = _arr(u_res, np.float32)
    acc = np.empty((R, B), np.int32)
    out = np.empty((R, B, K + 1), np.int32)
    lib().dflash2_ref_walk_accept_mc(R, B, K, _p(ci), _p(S), _p(T), _p(di), _p(dp), _p(dn), cap, _p(uw),
                                     _p(ua), _p(ur), _p(acc), _p(out))
    return acc, out


def conv2tap(x, k0, k1, x_prev, group=1):
    """Returns y with x's dtype (bf16 as torch tensor when x is a bf16 torch tensor)."""
    xr, dt = _raw(x)
    k0r, _ = _raw(k0)
    k1r, _ = _raw(k1)
    xpr, _ = _raw(x_prev)
    B, T, H = xr.shape
    y = np.empty_like(xr)
    lib().dflash2_ref_conv2tap(_p(xr), _p(k0r), _p(k1r), _p(xpr), dt, B, T, H, group, _p(y))
    if dt == 1:
        import torch
        return torch.from_numpy(y.view(np.int16)).view(torch.bfloat16)
    return y


def dynconv2tap(x, x_prev, Wd, group=1):
    """Grouped dynamic taps k0 = sigmoid(Wd . x_t) per group (k1 = 1 - k0) and the two-tap conv.
    Returns (taps [B, T, H/group] float64, y with x's dtype)."""
    xr, dt = _raw(x)
    xpr, _ = _raw(x_prev)
    wr, _ = _raw(Wd)
    B, T, H = xr.shape
    taps = np.empty((B, T, H // group), np.float64)
    y = np.empty_like(xr)
    lib().dflash2_ref_dynconv2tap(_p(xr), _p(xpr), _p(wr), dt, B, T, H, group, _p(taps), _p(y))
    if dt == 1:
        import torch
        return taps, torch.from_numpy(y.view(np.int16)).view(torch.bfloat16)
    return taps, y
