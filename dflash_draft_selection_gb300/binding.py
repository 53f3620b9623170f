"""ctypes binding of libdflash2.so: torch CUDA tensors in, pointers out.

Every function here has the name of the C entry point it calls (without the
``dflash2_`` prefix) and does argument marshalling only: shapes are read from
the tensors, outputs are allocated when not passed in, and the call is made on
the current CUDA stream.  Nothing is computed in Python; if the library cannot
be loaded the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash2.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 0, 1, 2, 3, 4
F32, BF16 = 0, 1
ST_OK, ST_NAN, ST_BAD_Q, ST_BAD_PARAMS, ST_UNSUPPORTED = 0, 1, 2, 3, 4
VERIFY_TRUST_Q = 1
NC = 16
SHARD_LIST = 64

SAMPLING_DTYPE = np.dtype([("temperature", "<f4"), ("top_k", "<i4"), ("top_p", "<f4")])

_lib = None
_lock = threading.Lock()


class DFlash2Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {_status_string(code)} (status {code})")


def load_library():
    """Load libdflash2.so (built in-tree by the package's build step)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with `python -m dflash_draft_selection_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
        L.dflash2_topk16_workspace_bytes.argtypes = [i64]
        L.dflash2_topk16_workspace_bytes.restype = sz
        L.dflash2_topk16.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, vp, vp, vp, sz, vp]
        L.dflash2_topk16_noalloc.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, vp, vp, vp]
        L.dflash2_topk16_shard.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, i64, vp, vp, vp, vp, vp, sz, vp]
        L.dflash2_topk16_merge.argtypes = [i32, i64, vp, vp, vp, vp, i64, vp, i64, vp, vp, vp, vp]
        L.dflash2_lmhead_topk16_workspace_bytes.argtypes = [i64, i64]
        L.dflash2_lmhead_topk16_workspace_bytes.restype = sz
        L.dflash2_lmhead_topk16.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, vp, vp, vp, sz, vp]
        L.dflash2_ctx_gate.argtypes = [vp, i32, i64, i64, vp, i32, vp, vp]
        L.dflash2_pair_score_walk.argtypes = [i64, i32, vp, vp, vp, vp, vp, i32, i64, i32, vp, vp, vp, vp, vp,
                                              vp, vp, vp]
        L.dflash2_verify_workspace_bytes.argtypes = [i64, i32]
        L.dflash2_verify_workspace_bytes.restype = sz
        L.dflash2_verify.argtypes = [vp, i32, i64, i32, i64, i64, vp, vp, vp, vp, vp, vp, vp, u32, vp, vp, vp,
                                     vp, sz, vp]
        L.dflash2_conv2tap.argtypes = [vp, vp, vp, vp, i32, i64, i32, i64, i32, vp, vp]
        L.dflash2_dynconv2tap.argtypes = [vp, vp, vp, i32, i64, i32, i64, i32, vp, vp, vp]
        L.dflash2_status_string.argtypes = [i32]
        L.dflash2_status_string.restype = ctypes.c_char_p
        L.dflash2_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        L.dflash2_test_hold.argtypes = [vp, i64]
        for fn in ("dflash2_topk16", "dflash2_topk16_noalloc", "dflash2_topk16_shard", "dflash2_topk16_merge",
                   "dflash2_lmhead_topk16",
                   "dflash2_ctx_gate", "dflash2_pair_score_walk",
                   "dflash2_verify", "dflash2_conv2tap", "dflash2_dynconv2tap", "dflash2_device_error",
                   "dflash2_test_hold"):
            getattr(L, fn).restype = i32
        _lib = L
        return _lib


def _status_string(code: int) -> str:
    try:
        return load_library().dflash2_status_string(code).decode()
    except OSError:
        return "library not loaded"


def _check(fn: str, code: int):
    if code != OK:
        raise DFlash2Error(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("dflash2 tensors must be CUDA tensors")


def sampling_params(temperature, top_k, top_p, n: int | None = None, device="cuda") -> torch.Tensor:
    """Pack per-request sampling parameters into the C record layout (12 bytes each) on `device`."""
    if n is None:
        n = np.broadcast(np.asarray(temperature), np.asarray(top_k), np.asarray(top_p)).size
    rec = np.zeros(n, dtype=SAMPLING_DTYPE)
    rec["temperature"] = temperature
    rec["top_k"] = top_k
    rec["top_p"] = top_p
    return torch.from_numpy(rec.view(np.uint8).copy()).to(device)


def _params_from(params, device):
    if params is None or isinstance(params, torch.Tensor):
        return params
    rec = np.ascontiguousarray(np.asarray(params, dtype=SAMPLING_DTYPE))
    return torch.from_numpy(rec.view(np.uint8).copy()).to(device)


class Workspace:
    """A zero-filled device workspace, reusable across calls (kept zeroed by them)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.buf = torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    @staticmethod
    def for_topk16(rows: int, device="cuda") -> "Workspace":
        return Workspace(load_library().dflash2_topk16_workspace_bytes(rows), device)

    @staticmethod
    def for_lmhead(rows: int, V: int, device="cuda") -> "Workspace":
        return Workspace(load_library().dflash2_lmhead_topk16_workspace_bytes(rows, V), device)

    @staticmethod
    def for_verify(B: int, K: int, device="cuda") -> "Workspace":
        return Workspace(load_library().dflash2_verify_workspace_bytes(B, K), device)


# ------------------------------------------------------------------ calls ----
def topk16(logits: torch.Tensor, params=None, rows_per_param: int = 1, V: int | None = None, ws=None, out=None):
    """dflash2_topk16.  logits [rows, ld] (bf16/f32).  Returns (cand_idx, cand_U, lse)."""
    L = load_library()
    _need_cuda(logits)
    assert logits.dim() == 2 and logits.stride(1) == 1
    rows, ld = logits.shape[0], logits.stride(0)
    V = logits.shape[1] if V is None else V
    dev = logits.device
    if out is None:
        out = (torch.empty(rows, NC, dtype=torch.int32, device=dev),
               torch.empty(rows, NC, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    cand_idx, cand_U, lse = out
    if ws is None:
        ws = Workspace.for_topk16(rows, dev)
    p = _params_from(params, dev)
    _check("dflash2_topk16", L.dflash2_topk16(_ptr(logits), _dtype(logits), rows, V, ld, _ptr(p), rows_per_param,
                                              _ptr(cand_idx), _ptr(cand_U), _ptr(lse), ws.ptr(), ws.nbytes,
                                              _stream(dev)))
    return cand_idx, cand_U, lse


def topk16_noalloc(logits: torch.Tensor, params=None, rows_per_param: int = 1, V: int | None = None, out=None):
    """dflash2_topk16_noalloc: topk16 with the library's own fixed scratch.  Returns (cand_idx, cand_U, lse)."""
    L = load_library()
    _need_cuda(logits)
    assert logits.dim() == 2 and logits.stride(1) == 1
    rows, ld = logits.shape[0], logits.stride(0)
    V = logits.shape[1] if V is None else V
    dev = logits.device
    if out is None:
        out = (torch.empty(rows, NC, dtype=torch.int32, device=dev),
               torch.empty(rows, NC, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    cand_idx, cand_U, lse = out
    p = _params_from(params, dev)
    _check("dflash2_topk16_noalloc",
           L.dflash2_topk16_noalloc(_ptr(logits), _dtype(logits), rows, V, ld, _ptr(p), rows_per_param,
                                    _ptr(cand_idx), _ptr(cand_U), _ptr(lse), _stream(dev)))
    return cand_idx, cand_U, lse


def topk16_shard(logits: torch.Tensor, id_offset: int, V_total: int, params=None, rows_per_param: int = 1,
                 V: int | None = None, ws=None, out=None):
    """dflash2_topk16_shard: one vocabulary slice's partial.  logits [rows, ld] hold tokens id_offset.. .
    Returns (part_idx [rows, 64] i32, part_z [rows, 64] f32, part_m [rows] f32, part_s [rows] f32)."""
    L = load_library()
    _need_cuda(logits)
    assert logits.dim() == 2 and logits.stride(1) == 1
    rows, ld = logits.shape[0], logits.stride(0)
    V = logits.shape[1] if V is None else V
    dev = logits.device
    if out is None:
        out = (torch.empty(rows, SHARD_LIST, dtype=torch.int32, device=dev),
               torch.empty(rows, SHARD_LIST, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev), torch.empty(rows, dtype=torch.float32, device=dev))
    pi, pz, pm, ps = out
    if ws is None:
        ws = Workspace.for_topk16(rows, dev)
    p = _params_from(params, dev)
    _check("dflash2_topk16_shard",
           L.dflash2_topk16_shard(_ptr(logits), _dtype(logits), rows, V, ld, id_offset, V_total, _ptr(p),
                                  rows_per_param, _ptr(pi), _ptr(pz), _ptr(pm), _ptr(ps), ws.ptr(), ws.nbytes,
                                  _stream(dev)))
    return pi, pz, pm, ps


def topk16_merge(part_idx, part_z, part_m, part_s, V_total: int, params=None, rows_per_param: int = 1, out=None):
    """dflash2_topk16_merge: partials stacked [S, rows, 64] / [S, rows].  Returns (cand_idx, cand_U, lse)."""
    L = load_library()
    _need_cuda(part_idx, part_z, part_m, part_s)
    for t in (part_idx, part_z, part_m, part_s):
        assert t.is_contiguous()
    S, rows = part_idx.shape[0], part_idx.shape[1]
    dev = part_idx.device
    if out is None:
        out = (torch.empty(rows, NC, dtype=torch.int32, device=dev),
               torch.empty(rows, NC, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    cand_idx, cand_U, lse = out
    p = _params_from(params, dev)
    _check("dflash2_topk16_merge",
           L.dflash2_topk16_merge(S, rows, _ptr(part_idx), _ptr(part_z), _ptr(part_m), _ptr(part_s), V_total,
                                  _ptr(p), rows_per_param, _ptr(cand_idx), _ptr(cand_U), _ptr(lse), _stream(dev)))
    return cand_idx, cand_U, lse


def lmhead_topk16(h: torch.Tensor, W: torch.Tensor, params=None, rows_per_param: int = 1, ws=None, out=None):
    """dflash2_lmhead_topk16: h [rows, hidden] bf16, W [V, hidden] bf16.  Returns (cand_idx, cand_U, lse)."""
    L = load_library()
    _need_cuda(h, W)
    assert h.dtype == torch.bfloat16 and W.dtype == torch.bfloat16 and h.is_contiguous() and W.is_contiguous()
    rows, hidden = h.shape
    V = W.shape[0]
    dev = h.device
    if out is None:
        out = (torch.empty(rows, NC, dtype=torch.int32, device=dev),
               torch.empty(rows, NC, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    cand_idx, cand_U, lse = out
    if ws is None:
        ws = Workspace.for_lmhead(rows, V, dev)
    p = _params_from(params, dev)
    _check("dflash2_lmhead_topk16",
           L.dflash2_lmhead_topk16(_ptr(h), _ptr(W), rows, hidden, V, _ptr(p), rows_per_param, _ptr(cand_idx),
                                   _ptr(cand_U), _ptr(lse), ws.ptr(), ws.nbytes, _stream(dev)))
    return cand_idx, cand_U, lse


def ctx_gate(h: torch.Tensor, Wg: torch.Tensor, out=None):
    """dflash2_ctx_gate.  h [n, hidden], Wg [D, hidden] (same dtype).  Returns gate [n, D] f32."""
    L = load_library()
    _need_cuda(h, Wg)
    assert h.is_contiguous() and Wg.is_contiguous() and h.dtype == Wg.dtype
    n, hidden = h.shape
    D = Wg.shape[0]
    gate = torch.empty(n, D, dtype=torch.float32, device=h.device) if out is None else out
    _check("dflash2_ctx_gate", L.dflash2_ctx_gate(_ptr(h), _dtype(h), n, hidden, _ptr(Wg), D, _ptr(gate),
                                                  _stream(h.device)))
    return gate


def pair_score_walk(cand_idx, cand_U, last_tok, A, Bt, gate, params=None, u_walk=None, out=None):
    """dflash2_pair_score_walk.  cand_idx/cand_U [B, K, 16], gate [B, K, D], A/Bt [V, D].

    Returns (path_tok [B,K], path_slot [B,K], q_sel [B,K,16], scores [B,K,16,16]).
    """
    L = load_library()
    _need_cuda(cand_idx, cand_U, last_tok, A, Bt, gate)
    B, K = cand_idx.shape[0], cand_idx.shape[1]
    V, D = A.shape
    dev = cand_idx.device
    if out is None:
        out = (torch.empty(B, K, dtype=torch.int32, device=dev), torch.empty(B, K, dtype=torch.int32, device=dev),
               torch.empty(B, K, NC, dtype=torch.float32, device=dev),
               torch.empty(B, K, NC, NC, dtype=torch.float32, device=dev))
    path_tok, path_slot, q_sel, scores = out
    p = _params_from(params, dev)
    _check("dflash2_pair_score_walk",
           L.dflash2_pair_score_walk(B, K, _ptr(cand_idx), _ptr(cand_U), _ptr(last_tok), _ptr(A), _ptr(Bt),
                                     _dtype(A), V, D, _ptr(gate), _ptr(p), _ptr(u_walk), _ptr(path_tok),
                                     _ptr(path_slot), _ptr(q_sel), _ptr(scores), _stream(dev)))
    return path_tok, path_slot, q_sel, scores


def verify(tlogits, path_tok, cand_idx, q_sel, path_slot, params=None, u_acc=None, u_res=None, ws=None,
           trusted: bool = False, V: int | None = None, out=None):
    """dflash2_verify.  tlogits [B*(K+1), ld].  Returns (accept_len [B], out_tok [B, K+1], status [B])."""
    L = load_library()
    _need_cuda(tlogits, path_tok, cand_idx, q_sel, path_slot)
    B, K = path_tok.shape
    assert tlogits.dim() == 2 and tlogits.stride(1) == 1 and tlogits.shape[0] == B * (K + 1)
    ld = tlogits.stride(0)
    V = tlogits.shape[1] if V is None else V
    dev = tlogits.device
    if ws is None:
        ws = Workspace.for_verify(B, K, dev)
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, K + 1, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    accept_len, out_tok, status = out
    p = _params_from(params, dev)
    _check("dflash2_verify",
           L.dflash2_verify(_ptr(tlogits), _dtype(tlogits), B, K, V, ld, _ptr(path_tok), _ptr(cand_idx),
                            _ptr(q_sel), _ptr(path_slot), _ptr(p), _ptr(u_acc), _ptr(u_res),
                            VERIFY_TRUST_Q if trusted else 0, _ptr(accept_len), _ptr(out_tok), _ptr(status),
                            ws.ptr(), ws.nbytes, _stream(dev)))
    return accept_len, out_tok, status


def conv2tap(x, k0, k1, x_prev, group: int = 1, out=None):
    """dflash2_conv2tap.  x [B, T, H], k0/k1 [B, T, H/group], x_prev [B, H].  Returns y [B, T, H]."""
    L = load_library()
    _need_cuda(x, k0, k1, x_prev)
    B, T, H = x.shape
    y = torch.empty_like(x) if out is None else out
    _check("dflash2_conv2tap", L.dflash2_conv2tap(_ptr(x), _ptr(k0), _ptr(k1), _ptr(x_prev), _dtype(x), B, T, H,
                                                  group, _ptr(y), _stream(x.device)))
    return y


def dynconv2tap(x, x_prev, Wd, group: int = 1, out=None):
    """dflash2_dynconv2tap.  x [B, T, H], x_prev [B, H], Wd [H/group, H].  Returns (taps [B, T, H/group]
    f32, y [B, T, H])."""
    L = load_library()
    _need_cuda(x, x_prev, Wd)
    B, T, H = x.shape
    if out is None:
        out = (torch.empty(B, T, H // group, dtype=torch.float32, device=x.device), torch.empty_like(x))
    taps, y = out
    _check("dflash2_dynconv2tap", L.dflash2_dynconv2tap(_ptr(x), _ptr(x_prev), _ptr(Wd), _dtype(x), B, T, H, group,
                                                        _ptr(taps), _ptr(y), _stream(x.device)))
    return taps, y


def device_error(clear: bool = False) -> int:
    """The library's device error word (synchronises the device)."""
    L = load_library()
    code = ctypes.c_uint32(0)
    _check("dflash2_device_error", L.dflash2_device_error(ctypes.byref(code), int(clear)))
    return code.value


def test_hold(flag=None, max_cycles: int = 0):
    """dflash2_test_hold: with `flag` (a CUDA int32 tensor of one element) set, later scan
    kernels wait on it for at most `max_cycles` before their first copy; None switches it off."""
    L = load_library()
    _need_cuda(flag)
    _check("dflash2_test_hold", L.dflash2_test_hold(_ptr(flag), int(max_cycles) if flag is not None else 0))
