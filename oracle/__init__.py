"""CPU oracle for the WhiFlash verify-and-route round (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package; the library never does.  The
arithmetic lives in ``wf_oracle.c`` (plain fp64 loops, OpenMP across
positions); this module compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wf_oracle.c")
_LIB = os.path.join(_HERE, "libwf_oracle.so")
_lock = threading.Lock()
_default = None


def compile_c(src: str, out: str) -> str:
    """gcc -O2 with OpenMP and strict IEEE evaluation (no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_c(_SRC, _LIB)
    return _LIB


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class Oracle:
    """numpy front end of one compiled copy of the oracle."""

    def __init__(self, path: str):
        self.lib = ctypes.CDLL(path)
        self.lib.oracle_gelu.restype = ctypes.c_double
        self.lib.oracle_gelu.argtypes = [ctypes.c_double]

    def threads(self) -> int:
        return int(self.lib.oracle_threads())

    def gelu(self, x: float) -> float:
        return float(self.lib.oracle_gelu(float(x)))

    def lmhead_argmax(self, h: np.ndarray, W: np.ndarray):
        """h [P, d] bf16 bits, W [V, d] bf16 bits -> (ids int32 [P], maxlogit f64 [P], gap f64 [P])."""
        h = np.ascontiguousarray(h, np.uint16)
        W = np.ascontiguousarray(W, np.uint16)
        P, d = h.shape
        V = W.shape[0]
        assert W.shape[1] == d
        ids = np.empty(P, np.int32)
        mx = np.empty(P, np.float64)
        gap = np.empty(P, np.float64)
        rc = self.lib.oracle_lmhead_argmax(_p(h), _p(W), ctypes.c_int64(P), ctypes.c_int64(d), ctypes.c_int64(V),
                                        _p(ids), _p(mx), _p(gap))
        assert rc == 0, rc
        return ids, mx, gap

    def verify_chain(self, g, draft, pos_off, node_off, path_stride: int = 0):
        g = np.ascontiguousarray(g, np.int32)
        draft = np.ascontiguousarray(draft, np.int32)
        pos_off = np.ascontiguousarray(pos_off, np.int32)
        node_off = np.ascontiguousarray(node_off, np.int32)
        B = len(pos_off) - 1
        n = np.empty(B, np.int32)
        bonus = np.empty(B, np.int32)
        last = np.empty(B, np.int32)
        path = np.empty((B, path_stride), np.int32) if path_stride else None
        rc = self.lib.oracle_verify_chain(_p(g), _p(draft), _p(pos_off), _p(node_off), ctypes.c_int(B), _p(n),
                                       _p(bonus), _p(last), _p(path), ctypes.c_int(path_stride))
        assert rc == 0, rc
        return n, bonus, last, path

    def verify_tree(self, g, tok, parent, node_off, pos_off, path_stride: int = 0):
        """Returns (n_accept, bonus, last_pos, path, rc); rc 2 flags a bad parent index."""
        g = np.ascontiguousarray(g, np.int32)
        tok = np.ascontiguousarray(tok, np.int32)
        parent = np.ascontiguousarray(parent, np.int32)
        node_off = np.ascontiguousarray(node_off, np.int32)
        pos_off = np.ascontiguousarray(pos_off, np.int32)
        B = len(pos_off) - 1
        n = np.empty(B, np.int32)
        bonus = np.empty(B, np.int32)
        last = np.empty(B, np.int32)
        path = np.empty((B, path_stride), np.int32) if path_stride else None
        rc = self.lib.oracle_verify_tree(_p(g), _p(tok), _p(parent), _p(node_off), _p(pos_off), ctypes.c_int(B),
                                      _p(n), _p(bonus), _p(last), _p(path), ctypes.c_int(path_stride))
        return n, bonus, last, path, rc

    def router(self, hidden, rows, W1, b1, w2, b2: float, tau: float):
        """-> (delta f64 [B], route int32 [B])."""
        hidden = np.ascontiguousarray(hidden, np.uint16)
        rows = np.ascontiguousarray(rows, np.int32)
        W1 = np.ascontiguousarray(W1, np.float32)
        b1 = np.ascontiguousarray(b1, np.float32)
        w2 = np.ascontiguousarray(w2, np.float32)
        B = len(rows)
        m, d = W1.shape
        assert hidden.shape[1] == d
        delta = np.empty(B, np.float64)
        route = np.empty(B, np.int32)
        rc = self.lib.oracle_router(_p(hidden), _p(rows), ctypes.c_int(B), ctypes.c_int64(d), ctypes.c_int64(m),
                                 _p(W1), _p(b1), _p(w2), ctypes.c_double(b2), ctypes.c_double(tau),
                                 _p(delta), _p(route))
        assert rc == 0, rc
        return delta, route

    def build_tree(self, tid, lp, N):
        """tid int32 [B, D, k, k], lp f32 [B, D, k, k] -> (parent, token, score f32, depth) each [B, N], rc."""
        tid = np.ascontiguousarray(tid, np.int32)
        lp = np.ascontiguousarray(lp, np.float32)
        B, D, k, _ = tid.shape
        parent = np.empty((B, N), np.int32)
        token = np.empty((B, N), np.int32)
        score = np.empty((B, N), np.float32)
        depth = np.empty((B, N), np.int32)
        rc = self.lib.oracle_build_tree(_p(tid), _p(lp), ctypes.c_int(B), ctypes.c_int(D), ctypes.c_int(k),
                                        ctypes.c_int(N), _p(parent), _p(token), _p(score), _p(depth))
        return parent, token, score, depth, rc

    def accepted_rows(self, n_accept, path, pos_off):
        """-> (acc_rows int32 [B, path_stride + 1], acc_off int32 [B + 1])."""
        n_accept = np.ascontiguousarray(n_accept, np.int32)
        path = np.ascontiguousarray(path, np.int32)
        pos_off = np.ascontiguousarray(pos_off, np.int32)
        B, ps = path.shape
        acc_rows = np.empty((B, ps + 1), np.int32)
        acc_off = np.empty(B + 1, np.int32)
        rc = self.lib.oracle_accepted_rows(_p(n_accept), _p(path), ctypes.c_int(ps), _p(pos_off), ctypes.c_int(B),
                                           _p(acc_rows), _p(acc_off))
        assert rc == 0, rc
        return acc_rows, acc_off

    def entropy(self, hidden, rows, W, tau: float = 0.0):
        """Entropy of softmax(<h, W_v>) at each row -> (H f64 [B], route int32 [B])."""
        hidden = np.ascontiguousarray(hidden, np.uint16)
        rows = np.ascontiguousarray(rows, np.int32)
        W = np.ascontiguousarray(W, np.uint16)
        B = len(rows)
        d = hidden.shape[1]
        V = W.shape[0]
        H = np.empty(B, np.float64)
        route = np.empty(B, np.int32)
        rc = self.lib.oracle_entropy(_p(hidden), _p(rows), ctypes.c_int(B), _p(W), ctypes.c_int64(d),
                                     ctypes.c_int64(V), ctypes.c_double(tau), _p(H), _p(route))
        assert rc == 0, rc
        return H, route

    def draft_topk(self, x, Wd, d2t, k: int):
        """-> (draft_ids [B,k], target_ids [B,k], logits f64 [B,k], lse f64 [B], min_gap f64 [B])."""
        x = np.ascontiguousarray(x, np.uint16)
        Wd = np.ascontiguousarray(Wd, np.uint16)
        d2t = np.ascontiguousarray(d2t, np.int32)
        B, d = x.shape
        Vd = Wd.shape[0]
        dids = np.empty((B, k), np.int32)
        tids = np.empty((B, k), np.int32)
        vals = np.empty((B, k), np.float64)
        lse = np.empty(B, np.float64)
        mg = np.empty(B, np.float64)
        rc = self.lib.oracle_draft_topk(_p(x), _p(Wd), _p(d2t), ctypes.c_int(B), ctypes.c_int64(d), ctypes.c_int64(Vd),
                                     ctypes.c_int(k), _p(dids), _p(tids), _p(vals), _p(lse), _p(mg))
        assert rc == 0, rc
        return dids, tids, vals, lse, mg

    def round_(self, hidden, W, pos_off, node_off, kind, tok, parent, W1, b1, w2, b2, tau, path_stride):
        """Full round -> dict(ids, n_accept, bonus, last_pos, path, delta, route)."""
        hidden = np.ascontiguousarray(hidden, np.uint16)
        W = np.ascontiguousarray(W, np.uint16)
        pos_off = np.ascontiguousarray(pos_off, np.int32)
        node_off = np.ascontiguousarray(node_off, np.int32)
        kind = np.ascontiguousarray(kind, np.int32)
        tok = np.ascontiguousarray(tok, np.int32)
        parent = np.ascontiguousarray(parent, np.int32)
        W1 = np.ascontiguousarray(W1, np.float32)
        b1 = np.ascontiguousarray(b1, np.float32)
        w2 = np.ascontiguousarray(w2, np.float32)
        B = len(pos_off) - 1
        P = int(pos_off[-1])
        d = hidden.shape[1]
        V = W.shape[0]
        m = W1.shape[0]
        out = dict(ids=np.empty(P, np.int32), n_accept=np.empty(B, np.int32), bonus=np.empty(B, np.int32),
                   last_pos=np.empty(B, np.int32), path=np.empty((B, path_stride), np.int32),
                   delta=np.empty(B, np.float64), route=np.empty(B, np.int32))
        rc = self.lib.oracle_round(_p(hidden), _p(W), ctypes.c_int64(d), ctypes.c_int64(V), _p(pos_off), _p(node_off),
                                _p(kind), _p(tok), _p(parent), ctypes.c_int(B), ctypes.c_int64(m), _p(W1), _p(b1),
                                _p(w2), ctypes.c_double(b2), ctypes.c_double(tau), _p(out["ids"]),
                                _p(out["n_accept"]), _p(out["bonus"]), _p(out["last_pos"]), _p(out["path"]),
                                ctypes.c_int(path_stride), _p(out["delta"]), _p(out["route"]))
        assert rc == 0, rc
        return out

    def rmsnorm(self, u, gamma, eps: float):
        """u [din] bf16 bits, gamma [din] bf16 bits -> a f64 [din]."""
        u = np.ascontiguousarray(u, np.uint16)
        gamma = np.ascontiguousarray(gamma, np.uint16)
        a = np.empty(u.shape[0], np.float64)
        self.lib.oracle_rmsnorm(_p(u), ctypes.c_int64(u.shape[0]), _p(gamma), ctypes.c_double(eps), _p(a))
        return a

    def rope(self, x, pos: float, theta: float):
        """x f64 [D] -> the rotated vector f64 [D]."""
        x = np.ascontiguousarray(x, np.float64)
        y = np.empty_like(x)
        self.lib.oracle_rope(_p(x), ctypes.c_int(x.shape[0]), ctypes.c_double(pos), ctypes.c_double(theta), _p(y))
        return y

    def catchup(self, u, bl_off, cache_len, gamma, eps, theta, Wq, Wk, Wv, Wo, Kc, Vc, H: int, G: int):
        """KV-only catch-up.  u [N, din], Wq [H*D, din], Wk / Wv [G*D, din], Wo [din, H*D], gamma [din],
        caches Kc / Vc [B, cap, G*D] (all bf16 bits; the caches are copied, not modified) ->
        dict(Kc, Vc, q [B, H*D], attn [B, H*D], out [B, din]) and rc (2: a sequence without backlog or
        beyond its cache)."""
        u = np.ascontiguousarray(u, np.uint16)
        bl_off = np.ascontiguousarray(bl_off, np.int32)
        cache_len = np.ascontiguousarray(cache_len, np.int32)
        gamma = np.ascontiguousarray(gamma, np.uint16)
        Wq, Wk, Wv, Wo = (np.ascontiguousarray(w, np.uint16) for w in (Wq, Wk, Wv, Wo))
        Kc = np.array(Kc, np.uint16, copy=True, order="C")
        Vc = np.array(Vc, np.uint16, copy=True, order="C")
        B = len(bl_off) - 1
        din = u.shape[1]
        D = Wk.shape[0] // G
        cap = Kc.shape[1]
        assert Wq.shape == (H * D, din) and Wk.shape == (G * D, din) and Wv.shape == Wk.shape
        assert Wo.shape == (din, H * D) and Kc.shape == (B, cap, G * D) and Vc.shape == Kc.shape
        out = dict(Kc=Kc, Vc=Vc, q=np.empty((B, H * D)), attn=np.empty((B, H * D)), out=np.empty((B, din)))
        rc = self.lib.oracle_catchup(_p(u), _p(bl_off), _p(cache_len), ctypes.c_int(B), ctypes.c_int64(din),
                                     ctypes.c_int(H), ctypes.c_int(G), ctypes.c_int(D), _p(gamma),
                                     ctypes.c_double(eps), ctypes.c_double(theta), _p(Wq), _p(Wk), _p(Wv), _p(Wo),
                                     _p(Kc), _p(Vc), ctypes.c_int64(cap), _p(out["q"]), _p(out["attn"]),
                                     _p(out["out"]))
        return out, rc


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads():
    return default().threads()


def gelu(x):
    return default().gelu(x)


def lmhead_argmax(h, W):
    return default().lmhead_argmax(h, W)


def verify_chain(*a, **k):
    return default().verify_chain(*a, **k)


def verify_tree(*a, **k):
    return default().verify_tree(*a, **k)


def router(*a, **k):
    return default().router(*a, **k)


def draft_topk(*a, **k):
    return default().draft_topk(*a, **k)


def entropy(*a, **k):
    return default().entropy(*a, **k)


def round_(*a, **k):
    return default().round_(*a, **k)


def catchup(*a, **k):
    return default().catchup(*a, **k)


# ---- adapters in the shape the input generator asks for --------------------------------
def argmax_fn(W, rows):
    ids, _, gap = lmhead_argmax(rows, W)
    return ids, gap


def router_fn(W1, b1, w2, b2, rows):
    delta, _ = router(rows, np.arange(len(rows), dtype=np.int32), W1, b1, w2, b2, 0.0)
    return delta


def topk_gap_fn(Wd, k, rows):
    d2t = np.arange(Wd.shape[0], dtype=np.int32)
    return draft_topk(rows, Wd, d2t, k)[4]
