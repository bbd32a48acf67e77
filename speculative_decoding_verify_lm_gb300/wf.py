"""Python binding of ``libwf.so`` (the C ABI declared in include/wf.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtype / device / contiguity, and passes raw device pointers and the current
(or given) CUDA stream to the library; all arithmetic runs in the library's
kernels.  The functions carry the C names.  If the shared library is missing
it is built with nvcc; if that fails, loading raises - there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

WF_MAX_SEQ_NODES = 256
WF_MAX_TOPK = 16
STATUS = {0: "WF_OK", 1: "WF_ERR_INVALID_ARG", 2: "WF_ERR_WORKSPACE", 3: "WF_ERR_CUDA", 4: "WF_ERR_UNSUPPORTED",
          5: "WF_ERR_BAD_DATA", 6: "WF_ERR_TIMEOUT"}


class WfError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib().wf_status_string(status).decode()} (status {status})")


_c_void_p = ctypes.c_void_p
_i32 = ctypes.c_int
_f32 = ctypes.c_float
_u64 = ctypes.c_uint64
_sz = ctypes.c_size_t


class RoundArgs(ctypes.Structure):
    """Mirror of ``wf_round_args``."""
    _fields_ = [
        ("hidden", _c_void_p), ("W", _c_void_p), ("P", _i32), ("d", _i32), ("V", _i32),
        ("B", _i32), ("pos_off", _c_void_p), ("node_off", _c_void_p), ("kind", _c_void_p), ("tok", _c_void_p),
        ("parent", _c_void_p), ("path_stride", _i32),
        ("m", _i32), ("W1", _c_void_p), ("b1", _c_void_p), ("w2", _c_void_p), ("b2", _f32), ("tau", _f32),
        ("x", _c_void_p), ("Wd", _c_void_p), ("d2t", _c_void_p), ("Vd", _i32), ("k", _i32),
        ("ids", _c_void_p), ("maxlogit", _c_void_p), ("n_accept", _c_void_p), ("bonus", _c_void_p),
        ("last_pos", _c_void_p), ("path", _c_void_p), ("delta_al", _c_void_p), ("route", _c_void_p),
        ("draft_ids", _c_void_p), ("tids", _c_void_p), ("vals", _c_void_p), ("router_kind", _i32),
        ("lse", _c_void_p),
    ]


WF_ROUTER_NEURAL = 0
WF_ROUTER_ENTROPY = 1


class CatchupArgs(ctypes.Structure):
    """Mirror of ``wf_catchup_args``."""
    _fields_ = [
        ("u", _c_void_p), ("bl_off", _c_void_p), ("cache_len", _c_void_p), ("B", _i32), ("N", _i32), ("din", _i32),
        ("H", _i32), ("G", _i32), ("D", _i32), ("gamma", _c_void_p), ("eps", _f32), ("theta", _f32),
        ("Wq", _c_void_p), ("Wk", _c_void_p), ("Wv", _c_void_p), ("Wo", _c_void_p), ("Kc", _c_void_p),
        ("Vc", _c_void_p), ("cap", _i32), ("out", _c_void_p), ("attn", _c_void_p),
    ]


_SIGS = {
    "wf_status_string": (ctypes.c_char_p, [_i32]),
    "wf_version": (_i32, []),
    "wf_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "wf_lmhead_entropy": (_i32, [_c_void_p, _i32, _i32, _c_void_p, _i32, _c_void_p, _i32, _f32, _c_void_p, _c_void_p,
                                 _c_void_p, _sz, _c_void_p]),
    "wf_workspace_init": (_i32, [_c_void_p, _sz, _c_void_p]),
    "wf_read_device_error": (_i32, [_c_void_p, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _i32, _c_void_p]),
    "wf_set_wait_timeout_ns": (None, [_u64]),
    "wf_probe_bounded_wait": (_i32, [_u64, _c_void_p, _sz, _c_void_p]),
    "wf_lmhead_argmax": (_i32, [_c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _sz,
                                _c_void_p]),
    "wf_lmhead_argmax_noalloc": (_i32, [_c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p]),
    "wf_noalloc_read_device_error": (_i32, [ctypes.POINTER(_i32), ctypes.POINTER(_i32), _i32, _c_void_p]),
    "wf_build_tree": (_i32, [_c_void_p, _c_void_p, _i32, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                             _c_void_p, _sz, _c_void_p]),
    "wf_accepted_rows": (_i32, [_c_void_p, _c_void_p, _i32, _c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p, _i32,
                                _c_void_p, _c_void_p]),
    "wf_verify_chain": (_i32, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p,
                               _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "wf_verify_tree": (_i32, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p,
                              _c_void_p, _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "wf_router_mlp": (_i32, [_c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _f32, _f32,
                             _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "wf_draft_topk": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i32, _c_void_p, _c_void_p,
                             _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "wf_lmhead_draft_topk": (_i32, [_c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                                    _c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                                    _c_void_p, _c_void_p, _sz, _c_void_p]),
    "wf_round": (_i32, [ctypes.POINTER(RoundArgs), _c_void_p, _sz, _c_void_p]),
    "wf_catchup_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "wf_catchup_kv": (_i32, [ctypes.POINTER(CatchupArgs), _c_void_p, _sz, _c_void_p]),
    "wf_catchup": (_i32, [ctypes.POINTER(CatchupArgs), _c_void_p, _sz, _c_void_p]),
}


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load (building first if missing or stale) the native library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def exported_symbols() -> list:
    return list(_SIGS)


# ------------------------------------------------------------------ marshalling
def _check(t: Optional[torch.Tensor], name: str, dtypes, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if t.numel() == 0:   # an empty array still needs a valid (never read) device address
        return _placeholder(t.device)
    return t.data_ptr()


_placeholders = {}


def _placeholder(device) -> int:
    if device not in _placeholders:
        _placeholders[device] = torch.zeros(16, dtype=torch.int32, device=device)
    return _placeholders[device].data_ptr()


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _raise(st: int, where: str):
    if st != 0:
        raise WfError(st, where)


class Workspace:
    """Caller-owned device workspace sized by wf_workspace_bytes and zeroed once."""

    def __init__(self, P: int, B: int = 1, m: int = 1, Vd: int = 0, k: int = 0, device=None, stream=None,
                 d: int = 0):
        self.nbytes = int(lib().wf_workspace_bytes(P, B, d, m, Vd, k))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _raise(lib().wf_workspace_init(self.buf.data_ptr(), self.nbytes, _stream(stream)), "wf_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def device_error(self, clear: bool = True, stream=None):
        code, info = _i32(0), _i32(0)
        _raise(lib().wf_read_device_error(self.ptr, ctypes.byref(code), ctypes.byref(info), int(clear),
                                          _stream(stream)), "wf_read_device_error")
        return code.value, info.value


def wf_workspace_bytes(P: int, B: int = 1, m: int = 1, Vd: int = 0, k: int = 0, d: int = 0) -> int:
    return int(lib().wf_workspace_bytes(P, B, d, m, Vd, k))


def wf_lmhead_entropy(hidden, W, tau: float, ws: Workspace, rows=None, B=None, H=None, route=None, stream=None):
    """Entropy of the target's next-token distribution at the given rows (all rows if None) and the
    WhiFlash-Entropy route (H > tau)."""
    P, d = hidden.shape
    V = W.shape[0]
    B = (rows.numel() if rows is not None else P) if B is None else B
    H = torch.empty(B, dtype=torch.float32, device=hidden.device) if H is None else H
    route = torch.empty(B, dtype=torch.int32, device=hidden.device) if route is None else route
    st = lib().wf_lmhead_entropy(_check(hidden, "hidden", _BF16), P, d, _check(rows, "rows", _I32, True), B,
                                 _check(W, "W", _BF16), V, float(tau), _check(H, "H", _F32),
                                 _check(route, "route", _I32, True), ws.ptr, ws.nbytes, _stream(stream))
    _raise(st, "wf_lmhead_entropy")
    return H, route


def wf_set_wait_timeout_ns(ns: int) -> None:
    lib().wf_set_wait_timeout_ns(int(ns))


def wf_probe_bounded_wait(timeout_ns: int, ws: Workspace, stream=None) -> None:
    _raise(lib().wf_probe_bounded_wait(int(timeout_ns), ws.ptr, ws.nbytes, _stream(stream)), "wf_probe_bounded_wait")


def wf_lmhead_argmax(hidden, W, ws: Workspace, ids=None, maxlogit=None, stream=None):
    P, d = hidden.shape
    V = W.shape[0]
    if ids is None:
        ids = torch.empty(P, dtype=torch.int32, device=hidden.device)
    st = lib().wf_lmhead_argmax(_check(hidden, "hidden", _BF16), _check(W, "W", _BF16), P, d, V,
                                _check(ids, "ids", _I32), _check(maxlogit, "maxlogit", _F32, True), ws.ptr, ws.nbytes,
                                _stream(stream))
    _raise(st, "wf_lmhead_argmax")
    return ids


def wf_lmhead_argmax_noalloc(hidden, W, ids=None, maxlogit=None, stream=None):
    """The LM-head argmax without a workspace (scratch in a fixed array inside the
    library), for callers that cannot allocate device memory.  Calls on one device
    share that array: do not let them overlap on the GPU."""
    P, d = hidden.shape
    V = W.shape[0]
    if ids is None:
        ids = torch.empty(P, dtype=torch.int32, device=hidden.device)
    st = lib().wf_lmhead_argmax_noalloc(_check(hidden, "hidden", _BF16), _check(W, "W", _BF16), P, d, V,
                                        _check(ids, "ids", _I32), _check(maxlogit, "maxlogit", _F32, True),
                                        _stream(stream))
    _raise(st, "wf_lmhead_argmax_noalloc")
    return ids


def wf_noalloc_read_device_error(clear: bool = True, stream=None):
    """(code, info) left on the device by the last wf_lmhead_argmax_noalloc call."""
    code, info = _i32(0), _i32(0)
    _raise(lib().wf_noalloc_read_device_error(ctypes.byref(code), ctypes.byref(info), int(clear), _stream(stream)),
           "wf_noalloc_read_device_error")
    return code.value, info.value


def wf_build_tree(tid, lp, N: int, ws: Workspace, parent=None, token=None, score=None, depth=None, stream=None):
    """EAGLE-3 draft tree from per-step, per-slot top-k children -> (parent, token, score, depth) [B, N].
    Outputs not given are allocated."""
    B, D, k, _ = tid.shape
    dev = tid.device
    parent = torch.empty((B, N), dtype=torch.int32, device=dev) if parent is None else parent
    token = torch.empty((B, N), dtype=torch.int32, device=dev) if token is None else token
    score = torch.empty((B, N), dtype=torch.float32, device=dev) if score is None else score
    depth = torch.empty((B, N), dtype=torch.int32, device=dev) if depth is None else depth
    for name, t_, dt in (("parent", parent, _I32), ("token", token, _I32), ("score", score, _F32),
                         ("depth", depth, _I32)):
        if t_.numel() < B * N:
            raise ValueError(f"{name}: needs {B * N} elements")
        _check(t_, name, dt)
    st = lib().wf_build_tree(_check(tid, "tid", _I32), _check(lp, "lp", _F32), B, D, k, N, parent.data_ptr(),
                             token.data_ptr(), score.data_ptr(), depth.data_ptr(), ws.ptr, ws.nbytes, _stream(stream))
    _raise(st, "wf_build_tree")
    return parent, token, score, depth


def wf_accepted_rows(n_accept, path, pos_off, hidden=None, acc_rows=None, acc_off=None, hidden_out=None,
                     stream=None):
    """Kept rows of each sequence (root + accepted path), their packed offsets and,
    if ``hidden`` is given, the packed hidden states of those rows.  Outputs not
    given are allocated; a ``hidden_out`` not given is sized by a host read of
    n_accept (pass one with room for B * (path stride + 1) rows to stay on the
    stream, e.g. inside a CUDA graph)."""
    B, ps = path.shape
    dev = n_accept.device
    acc_rows = torch.empty((B, ps + 1), dtype=torch.int32, device=dev) if acc_rows is None else acc_rows
    acc_off = torch.empty(B + 1, dtype=torch.int32, device=dev) if acc_off is None else acc_off
    if acc_rows.numel() < B * (ps + 1) or acc_off.numel() < B + 1:
        raise ValueError("acc_rows needs B * (path stride + 1) elements and acc_off B + 1")
    out = hidden_out
    d = 0
    if hidden is not None:
        d = hidden.shape[1]
        if out is not None and (out.dim() != 2 or out.shape[1] != d or out.shape[0] < B * (ps + 1)):
            raise ValueError("hidden_out needs room for B * (path stride + 1) rows of d columns")
        if out is None:
            total = int(n_accept.clamp(min=-1).add(1).sum().item())   # host read of the packed size
            out = torch.empty((max(total, 1), d), dtype=hidden.dtype, device=dev)
    st = lib().wf_accepted_rows(_check(n_accept, "n_accept", _I32), _check(path, "path", _I32), ps,
                                _check(pos_off, "pos_off", _I32), B, _check(acc_rows, "acc_rows", _I32),
                                _check(acc_off, "acc_off", _I32), _check(hidden, "hidden", _BF16, True), d,
                                _check(out, "hidden_out", _BF16, True), _stream(stream))
    _raise(st, "wf_accepted_rows")
    return acc_rows, acc_off, out


def _verify_outputs(B, path_stride, device, n_accept, bonus, last_pos, path):
    mk = lambda: torch.empty(B, dtype=torch.int32, device=device)  # noqa: E731
    n_accept = mk() if n_accept is None else n_accept
    bonus = mk() if bonus is None else bonus
    last_pos = mk() if last_pos is None else last_pos
    if path is None and path_stride > 0:
        path = torch.empty((B, path_stride), dtype=torch.int32, device=device)
    return n_accept, bonus, last_pos, path


def wf_verify_chain(g, draft, pos_off, node_off, ws: Workspace, path_stride: int = 0, n_accept=None, bonus=None,
                    last_pos=None, path=None, stream=None):
    B = pos_off.numel() - 1
    n_accept, bonus, last_pos, path = _verify_outputs(B, path_stride, g.device, n_accept, bonus, last_pos, path)
    st = lib().wf_verify_chain(_check(g, "g", _I32), _check(draft, "draft", _I32), _check(pos_off, "pos_off", _I32),
                               _check(node_off, "node_off", _I32), B, path_stride, _check(n_accept, "n_accept", _I32),
                               _check(bonus, "bonus", _I32), _check(last_pos, "last_pos", _I32),
                               _check(path, "path", _I32, True), ws.ptr, ws.nbytes, _stream(stream))
    _raise(st, "wf_verify_chain")
    return n_accept, bonus, last_pos, path


def wf_verify_tree(g, tok, parent, node_off, pos_off, ws: Workspace, path_stride: int = 0, n_accept=None,
                   bonus=None, last_pos=None, path=None, stream=None):
    B = pos_off.numel() - 1
    n_accept, bonus, last_pos, path = _verify_outputs(B, path_stride, g.device, n_accept, bonus, last_pos, path)
    st = lib().wf_verify_tree(_check(g, "g", _I32), _check(tok, "tok", _I32), _check(parent, "parent", _I32),
                              _check(node_off, "node_off", _I32), _check(pos_off, "pos_off", _I32), B, path_stride,
                              _check(n_accept, "n_accept", _I32), _check(bonus, "bonus", _I32),
                              _check(last_pos, "last_pos", _I32), _check(path, "path", _I32, True), ws.ptr,
                              ws.nbytes, _stream(stream))
    _raise(st, "wf_verify_tree")
    return n_accept, bonus, last_pos, path


def wf_router_mlp(hidden, rows, W1, b1, w2, b2: float, tau: float, ws: Workspace, delta_al=None, route=None,
                  stream=None):
    B = rows.numel()
    m, d = W1.shape
    if delta_al is None:
        delta_al = torch.empty(B, dtype=torch.float32, device=hidden.device)
    if route is None:
        route = torch.empty(B, dtype=torch.int32, device=hidden.device)
    st = lib().wf_router_mlp(_check(hidden, "hidden", _BF16), _check(rows, "rows", _I32), B, d, m,
                             _check(W1, "W1", _F32), _check(b1, "b1", _F32), _check(w2, "w2", _F32), float(b2),
                             float(tau), _check(delta_al, "delta_al", _F32), _check(route, "route", _I32), ws.ptr,
                             ws.nbytes, _stream(stream))
    _raise(st, "wf_router_mlp")
    return delta_al, route


def wf_draft_topk(x, Wd, d2t, k: int, ws: Workspace, draft_ids=None, tids=None, vals=None, lse=None,
                  stream=None):
    """-> (draft_ids, tids, vals); pass ``lse`` (a [B] fp32 tensor) to also receive
    each row's log-sum-exp over the draft vocabulary."""
    B, d = x.shape
    Vd = Wd.shape[0]
    dev = x.device
    draft_ids = torch.empty((B, k), dtype=torch.int32, device=dev) if draft_ids is None else draft_ids
    tids = torch.empty((B, k), dtype=torch.int32, device=dev) if tids is None else tids
    vals = torch.empty((B, k), dtype=torch.float32, device=dev) if vals is None else vals
    st = lib().wf_draft_topk(_check(x, "x", _BF16), _check(Wd, "Wd", _BF16), _check(d2t, "d2t", _I32), B, d, Vd, k,
                             _check(draft_ids, "draft_ids", _I32), _check(tids, "tids", _I32),
                             _check(vals, "vals", _F32), _check(lse, "lse", _F32, True), ws.ptr, ws.nbytes,
                             _stream(stream))
    _raise(st, "wf_draft_topk")
    return draft_ids, tids, vals


def wf_lmhead_draft_topk(hidden, W, x, Wd, d2t, k: int, ws: Workspace, ids=None, maxlogit=None, draft_ids=None,
                         tids=None, vals=None, lse=None, stream=None):
    """Target argmax over the rows of hidden and draft top-k over the rows of x
    in one weight sweep (P, B <= 128, or P > 128 and B <= 256)."""
    P, d = hidden.shape
    V = W.shape[0]
    B = x.shape[0]
    Vd = Wd.shape[0]
    if x.shape[1] != d or W.shape[1] != d or Wd.shape[1] != d:
        raise ValueError("hidden, W, x and Wd must share the hidden size d")
    dev = hidden.device
    ids = torch.empty(P, dtype=torch.int32, device=dev) if ids is None else ids
    draft_ids = torch.empty((B, k), dtype=torch.int32, device=dev) if draft_ids is None else draft_ids
    tids = torch.empty((B, k), dtype=torch.int32, device=dev) if tids is None else tids
    vals = torch.empty((B, k), dtype=torch.float32, device=dev) if vals is None else vals
    st = lib().wf_lmhead_draft_topk(_check(hidden, "hidden", _BF16), _check(W, "W", _BF16), P, d, V,
                                    _check(ids, "ids", _I32), _check(maxlogit, "maxlogit", _F32, True),
                                    _check(x, "x", _BF16), _check(Wd, "Wd", _BF16), _check(d2t, "d2t", _I32), B, Vd,
                                    k, _check(draft_ids, "draft_ids", _I32), _check(tids, "tids", _I32),
                                    _check(vals, "vals", _F32), _check(lse, "lse", _F32, True), ws.ptr, ws.nbytes,
                                    _stream(stream))
    _raise(st, "wf_lmhead_draft_topk")
    return ids, draft_ids, tids, vals


class CatchupWorkspace(Workspace):
    """Workspace of wf_catchup / wf_catchup_kv for B sequences, N backlog rows and the drafter's shapes."""

    def __init__(self, B: int, N: int, din: int, H: int, G: int, D: int, device=None, stream=None):
        self.nbytes = int(lib().wf_catchup_workspace_bytes(B, N, din, H, G, D))
        if self.nbytes == 0:
            raise ValueError("catch-up shapes outside the library's range")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _raise(lib().wf_workspace_init(self.buf.data_ptr(), self.nbytes, _stream(stream)), "wf_workspace_init")


class Catchup:
    """One KV-only catch-up call (wf_catchup, or wf_catchup_kv with kv_only) over
    device tensors, repeatable and capturable in a CUDA graph.  u [N, din],
    bl_off [B+1], cache_len [B] int32; gamma [din], Wq [H*D, din], Wk / Wv
    [G*D, din], Wo [din, H*D] bf16; caches Kc / Vc [B, cap, G*D] bf16 (updated
    in place); outputs out [B, din] and attn [B, H*D] fp32."""

    def __init__(self, u, bl_off, cache_len, gamma, Wk, Wv, Kc, Vc, G: int, Wq=None, Wo=None, eps: float = 1e-6,
                 theta: float = 1e4, kv_only: bool = False, with_attn: bool = True):
        N, din = u.shape
        B = bl_off.numel() - 1
        D = Wk.shape[0] // G
        H = Wq.shape[0] // D if Wq is not None else G
        if Kc.shape != Vc.shape or Kc.dim() != 3 or Kc.shape[0] != B or Kc.shape[2] != G * D:
            raise ValueError("caches must be [B, cap, G*D]")
        if Wk.shape != (G * D, din) or Wv.shape != Wk.shape or gamma.numel() != din:
            raise ValueError("Wk / Wv must be [G*D, din] and gamma [din]")
        if not kv_only and (Wq is None or Wo is None or Wq.shape != (H * D, din) or Wo.shape != (din, H * D)):
            raise ValueError("wf_catchup needs Wq [H*D, din] and Wo [din, H*D]")
        dev = u.device
        self.kv_only = kv_only
        self.out = None if kv_only else torch.empty((B, din), dtype=torch.float32, device=dev)
        self.attn = None if kv_only or not with_attn else torch.empty((B, H * D), dtype=torch.float32, device=dev)
        self.ws = CatchupWorkspace(B, N, din, H, G, D, device=dev)
        self.tensors = (u, bl_off, cache_len, gamma, Wq, Wk, Wv, Wo, Kc, Vc)   # kept alive
        a = CatchupArgs()
        a.u = _check(u, "u", _BF16)
        a.bl_off = _check(bl_off, "bl_off", _I32)
        a.cache_len = _check(cache_len, "cache_len", _I32)
        a.B, a.N, a.din, a.H, a.G, a.D = B, N, din, H, G, D
        a.gamma = _check(gamma, "gamma", _BF16)
        a.eps, a.theta = float(eps), float(theta)
        a.Wq = _check(Wq, "Wq", _BF16, True)
        a.Wk = _check(Wk, "Wk", _BF16)
        a.Wv = _check(Wv, "Wv", _BF16)
        a.Wo = _check(Wo, "Wo", _BF16, True)
        a.Kc = _check(Kc, "Kc", _BF16)
        a.Vc = _check(Vc, "Vc", _BF16)
        a.cap = Kc.shape[1]
        a.out = _check(self.out, "out", _F32, True)
        a.attn = _check(self.attn, "attn", _F32, True)
        self.args = a

    def __call__(self, stream=None):
        fn = lib().wf_catchup_kv if self.kv_only else lib().wf_catchup
        st = fn(ctypes.byref(self.args), self.ws.ptr, self.ws.nbytes, _stream(stream))
        _raise(st, "wf_catchup_kv" if self.kv_only else "wf_catchup")
        return self.out, self.attn


def _packed(spec, device):
    """One uint8 device buffer holding every (name, dtype, shape) of ``spec`` at
    256-byte aligned offsets; returns (buffer, {name: typed view})."""
    offs, total = {}, 0
    for name, dt, shape in spec:
        n = 1
        for s in shape:
            n *= s
        offs[name] = total
        total += (n * torch.empty((), dtype=dt).element_size() + 255) // 256 * 256
    buf = torch.zeros(max(total, 256), dtype=torch.uint8, device=device)
    views = {}
    for name, dt, shape in spec:
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        views[name] = buf[offs[name]:offs[name] + nbytes].view(dt).view(*shape)
    return buf, views


class Round:
    """Inputs and output buffers of wf_round, held as device tensors so the
    call can be repeated (and captured in a CUDA graph) without re-marshalling.

    The per-round inputs (hidden states, drafted tokens, tree parents, offsets,
    kinds, drafter hidden states) live in one packed device buffer and all
    outputs in another, so a host program moves a round in and out with one
    copy each (pinned_inputs / upload, pinned_outputs / download).  Weights
    (W, W1, b1, w2, Wd, d2t) stay where the caller keeps them."""

    def __init__(self, hidden, W, pos_off, node_off, tok, W1, b1, w2, b2: float, tau: float, kind=None, parent=None,
                 path_stride: int = 0, x=None, Wd=None, d2t=None, k: int = 0, with_maxlogit: bool = False,
                 router_kind: int = WF_ROUTER_NEURAL):
        dev = hidden.device
        P, d = hidden.shape
        B = pos_off.numel() - 1
        m = W1.shape[0]
        N = tok.numel()
        draft = Wd is not None
        in_spec = [("hidden", hidden.dtype, (P, d)), ("tok", torch.int32, (N,)), ("pos_off", torch.int32, (B + 1,)),
                   ("node_off", torch.int32, (B + 1,))]
        if kind is not None:
            in_spec.append(("kind", torch.int32, (B,)))
        if parent is not None:
            in_spec.append(("parent", torch.int32, (N,)))
        if draft:
            in_spec.append(("x", x.dtype, (B, d)))
        self.in_buf, views = _packed(in_spec, dev)
        for name, src in (("hidden", hidden), ("tok", tok), ("pos_off", pos_off), ("node_off", node_off),
                          ("kind", kind), ("parent", parent), ("x", x)):
            if name in views:
                views[name].copy_(src.reshape(views[name].shape))
        self.inputs = dict(W=W, W1=W1, b1=b1, w2=w2, Wd=Wd, d2t=d2t, kind=None, parent=None, x=None)
        self.inputs.update(views)
        hidden, tok, pos_off, node_off = views["hidden"], views["tok"], views["pos_off"], views["node_off"]
        kind, parent, x = views.get("kind"), views.get("parent"), views.get("x")
        out_spec = [("ids", torch.int32, (P,)), ("n_accept", torch.int32, (B,)), ("bonus", torch.int32, (B,)),
                    ("last_pos", torch.int32, (B,)), ("delta_al", torch.float32, (B,)), ("route", torch.int32, (B,))]
        if path_stride:
            out_spec.append(("path", torch.int32, (B, path_stride)))
        if with_maxlogit:
            out_spec.append(("maxlogit", torch.float32, (P,)))
        if draft:
            out_spec += [("draft_ids", torch.int32, (B, k)), ("tids", torch.int32, (B, k)),
                         ("vals", torch.float32, (B, k)), ("lse", torch.float32, (B,))]
        self.out_buf, outs = _packed(out_spec, dev)
        self.out = {name: outs.get(name) for name in ("ids", "n_accept", "bonus", "last_pos", "path", "delta_al",
                                                      "route", "maxlogit", "draft_ids", "tids", "vals", "lse")}
        self._in_spec, self._out_spec = in_spec, out_spec
        a = RoundArgs()
        a.hidden = _check(hidden, "hidden", _BF16)
        a.W = _check(W, "W", _BF16)
        a.P, a.d, a.V = P, d, W.shape[0]
        a.B = B
        a.pos_off = _check(pos_off, "pos_off", _I32)
        a.node_off = _check(node_off, "node_off", _I32)
        a.kind = _check(kind, "kind", _I32, True)
        a.tok = _check(tok, "tok", _I32)
        a.parent = _check(parent, "parent", _I32, True)
        a.path_stride = path_stride
        a.m = m
        a.W1 = _check(W1, "W1", _F32)
        a.b1 = _check(b1, "b1", _F32)
        a.w2 = _check(w2, "w2", _F32)
        a.b2, a.tau = float(b2), float(tau)
        a.x = _check(x, "x", _BF16, True)
        a.Wd = _check(Wd, "Wd", _BF16, True)
        a.d2t = _check(d2t, "d2t", _I32, True)
        a.Vd = Wd.shape[0] if Wd is not None else 0
        a.k = k if Wd is not None else 0
        a.router_kind = int(router_kind)
        for name in ("ids", "maxlogit", "n_accept", "bonus", "last_pos", "path", "delta_al", "route", "draft_ids",
                     "tids", "vals", "lse"):
            t = self.out[name]
            setattr(a, name, t.data_ptr() if t is not None else None)
        self.args = a
        self.ws = Workspace(P, B, m, a.Vd, a.k, device=dev, d=d)

    def __call__(self, stream=None):
        _raise(lib().wf_round(ctypes.byref(self.args), self.ws.ptr, self.ws.nbytes, _stream(stream)), "wf_round")
        return self.out

    # ---- host staging: one pinned buffer in, one out
    def pinned_inputs(self):
        """A pinned host copy of the packed inputs (same layout as the device buffer)."""
        return self.in_buf.cpu().pin_memory()

    def pinned_outputs(self):
        return torch.empty(self.out_buf.numel(), dtype=torch.uint8).pin_memory()

    def upload(self, host_inputs, stream=None):
        with torch.cuda.stream(stream) if stream is not None else _nullctx():
            self.in_buf.copy_(host_inputs, non_blocking=True)

    def download(self, host_outputs, stream=None):
        with torch.cuda.stream(stream) if stream is not None else _nullctx():
            host_outputs.copy_(self.out_buf, non_blocking=True)

    def capture_host_step(self, host_inputs, host_outputs):
        """Capture one host-to-host step - copy the packed inputs in from pinned
        memory, run the round, copy every output back - as a CUDA graph;
        ``replay_host_step()`` then runs it with one launch.  Call once the round
        has run eagerly at least once (its kernels are configured on first use)."""
        self._host_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self._host_graph):
            self.in_buf.copy_(host_inputs, non_blocking=True)
            self()
            host_outputs.copy_(self.out_buf, non_blocking=True)
        return self._host_graph

    def replay_host_step(self):
        self._host_graph.replay()

    def host_views(self, host_outputs):
        """Typed views of the outputs inside a downloaded pinned buffer."""
        _, views = _packed_views(host_outputs, self._out_spec)
        return views


class _nullctx:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False


def _packed_views(buf, spec):
    off, views = 0, {}
    for name, dt, shape in spec:
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        views[name] = buf[off:off + nbytes].view(dt).view(*shape)
        off += (nbytes + 255) // 256 * 256
    return buf, views


def wf_round(hidden, W, pos_off, node_off, tok, W1, b1, w2, b2, tau, kind=None, parent=None, path_stride=0, x=None,
             Wd=None, d2t=None, k=0, stream=None):
    """One-shot round (allocates outputs and a workspace)."""
    r = Round(hidden, W, pos_off, node_off, tok, W1, b1, w2, b2, tau, kind=kind, parent=parent,
              path_stride=path_stride, x=x, Wd=Wd, d2t=d2t, k=k)
    return r(stream)
