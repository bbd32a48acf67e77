"""Helpers for the GPU parity tests: host <-> device marshalling and the
properties a verify-and-route result must satisfy at any size."""
from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_verify_lm_gb300 import wf
from speculative_decoding_verify_lm_gb300.synth import bf16_bits_to_f32

DEV = "cuda:0"


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def host(t):
    return None if t is None else t.cpu().numpy()


def round_on_gpu(wl, path_stride=None, with_draft=True, maxlogit=False):
    ps = wl.max_depth if path_stride is None else path_stride
    draft = with_draft and wl.Wd is not None
    r = wf.Round(dev(wl.hidden), dev(wl.W), dev(wl.pos_off), dev(wl.node_off), dev(wl.tok), dev(wl.W1), dev(wl.b1),
                 dev(wl.w2), wl.b2, wl.tau, kind=dev(wl.kind), parent=dev(wl.parent), path_stride=ps,
                 x=dev(wl.x) if draft else None, Wd=dev(wl.Wd) if draft else None,
                 d2t=dev(wl.d2t) if draft else None, k=wl.topk if draft else 0, with_maxlogit=maxlogit)
    out = {k: host(v) for k, v in r().items()}
    torch.cuda.synchronize()
    return r, out


def logit_error_bound(h_bits, W_bits, ids):
    """Worst-case |fp32 accumulation - exact| for logit <h_p, W_id>: 2 d u sum|h||W|."""
    h = bf16_bits_to_f32(h_bits).astype(np.float64)
    W = bf16_bits_to_f32(W_bits[ids]).astype(np.float64)
    d = h.shape[1]
    return 2.0 * d * 2.0 ** -24 * np.abs(h * W).sum(axis=1)


def check_round_properties(wl, out):
    """Holds at any size for every sequence, planted or not: the accepted path is
    a valid matched root path, nothing deeper is accepted, and bonus / last row agree."""
    ids = out["ids"]
    for b in range(wl.B):
        r0, r1 = int(wl.pos_off[b]), int(wl.pos_off[b + 1])
        n0, n1 = int(wl.node_off[b]), int(wl.node_off[b + 1])
        tok = wl.tok[n0:n1]
        n = int(out["n_accept"][b])
        last = int(out["last_pos"][b])
        assert r0 <= last < r1 and out["bonus"][b] == ids[last]
        if wl.kind[b] == 0:
            assert 0 <= n <= n1 - n0 and last == r0 + n
            assert all(tok[j] == ids[r0 + j] for j in range(n))
            assert n == n1 - n0 or tok[n] != ids[r0 + n]
            continue
        par = wl.parent[n0:n1]
        depth = np.zeros(len(tok), np.int64)
        acc = np.zeros(len(tok), bool)
        for i in range(len(tok)):
            prow = r0 if par[i] < 0 else r0 + 1 + par[i]
            depth[i] = 1 + (0 if par[i] < 0 else depth[par[i]])
            acc[i] = tok[i] == ids[prow] and (par[i] < 0 or acc[par[i]])
        assert n == (depth[acc].max() if acc.any() else 0)
        if n:
            node = last - r0 - 1
            assert acc[node] and depth[node] == n
        if out.get("path") is not None:
            path = [int(x) for x in out["path"][b] if x >= 0]
            assert len(path) == min(n, out["path"].shape[1])
            for j, node in enumerate(path):
                assert depth[node] == j + 1 and acc[node]
                assert (par[node] == -1) if j == 0 else (par[node] == path[j - 1])
