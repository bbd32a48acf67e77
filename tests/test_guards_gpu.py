"""Operands the kernels read with the tensor-memory accelerator must be memory
of the current GPU: every entry point that builds a tensor map refuses a host
pointer (pageable or pinned) with WF_ERR_INVALID_ARG before it enqueues
anything, so such a pointer never reaches a copy engine."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import DEV
from speculative_decoding_verify_lm_gb300 import wf

pytestmark = pytest.mark.gpu

INVALID = 1


def _host_buffers(nbytes):
    pageable = np.zeros(nbytes // 2 + 64, np.uint16)
    off = (-pageable.ctypes.data) % 16 // 2          # 16-byte aligned like a device buffer
    pinned = torch.zeros(nbytes + 64, dtype=torch.uint8).pin_memory()
    return [("pageable", pageable.ctypes.data + 2 * off, pageable), ("pinned", pinned.data_ptr(), pinned)]


def test_lmhead_and_draft_refuse_host_operands():
    P, d, V, Vd, k = 4, 64, 300, 200, 4
    h = torch.zeros((P, d), dtype=torch.int16, device=DEV)
    W = torch.zeros((V, d), dtype=torch.int16, device=DEV)
    x = torch.zeros((1, d), dtype=torch.int16, device=DEV)
    Wd = torch.zeros((Vd, d), dtype=torch.int16, device=DEV)
    d2t = torch.arange(Vd, dtype=torch.int32, device=DEV)
    ids = torch.full((P,), -7, dtype=torch.int32, device=DEV)
    tids = torch.full((1, k), -7, dtype=torch.int32, device=DEV)
    ws = wf.Workspace(P, 1, 1, Vd, k, d=d)
    L = wf.lib()
    s = torch.cuda.current_stream().cuda_stream
    for name, hp, keep in _host_buffers(V * d * 2):
        assert L.wf_lmhead_argmax(hp, W.data_ptr(), P, d, V, ids.data_ptr(), None, ws.ptr, ws.nbytes, s) == INVALID
        assert L.wf_lmhead_argmax(h.data_ptr(), hp, P, d, V, ids.data_ptr(), None, ws.ptr, ws.nbytes, s) == INVALID
        assert L.wf_lmhead_argmax_noalloc(h.data_ptr(), hp, P, d, V, ids.data_ptr(), None, s) == INVALID
        assert L.wf_draft_topk(hp, Wd.data_ptr(), d2t.data_ptr(), 1, d, Vd, k, None, tids.data_ptr(), None, None,
                               ws.ptr, ws.nbytes, s) == INVALID
        assert L.wf_draft_topk(x.data_ptr(), hp, d2t.data_ptr(), 1, d, Vd, k, None, tids.data_ptr(), None, None,
                               ws.ptr, ws.nbytes, s) == INVALID
        assert L.wf_lmhead_draft_topk(h.data_ptr(), W.data_ptr(), P, d, V, ids.data_ptr(), None, x.data_ptr(), hp,
                                      d2t.data_ptr(), 1, Vd, k, None, tids.data_ptr(), None, None, ws.ptr, ws.nbytes,
                                      s) == INVALID
        assert L.wf_lmhead_entropy(hp, P, d, None, P, W.data_ptr(), V, 1.0, torch.empty(P, device=DEV).data_ptr(),
                                   None, ws.ptr, ws.nbytes, s) == INVALID
    torch.cuda.synchronize()
    # nothing was enqueued: the outputs keep their fill, the workspace is clean
    assert (ids == -7).all().item() and (tids == -7).all().item()
    assert ws.device_error() == (0, 0) and not ws.buf.any().item()


def test_round_refuses_host_weights():
    P, d, V, m = 17, 64, 300, 8
    hidden = torch.zeros((P, d), dtype=torch.int16, device=DEV)
    W = torch.zeros((V, d), dtype=torch.int16, device=DEV)
    pos_off = torch.tensor([0, P], dtype=torch.int32, device=DEV)
    node_off = torch.tensor([0, P - 1], dtype=torch.int32, device=DEV)
    tok = torch.zeros(P - 1, dtype=torch.int32, device=DEV)
    W1 = torch.zeros((m, d), dtype=torch.float32, device=DEV)
    b1 = torch.zeros(m, dtype=torch.float32, device=DEV)
    r = wf.Round(hidden, W, pos_off, node_off, tok, W1, b1, b1, 0.0, 1.0, kind=torch.zeros(1, dtype=torch.int32,
                 device=DEV), path_stride=16)
    r.out["n_accept"].fill_(-7)
    for name, hp, keep in _host_buffers(V * d * 2):
        a = wf.RoundArgs.from_buffer_copy(r.args)
        a.W = hp
        st = wf.lib().wf_round(ctypes.byref(a), r.ws.ptr, r.ws.nbytes, torch.cuda.current_stream().cuda_stream)
        assert st == INVALID, name
    torch.cuda.synchronize()
    assert (r.out["n_accept"] == -7).all().item()
    r()   # the same round with device weights runs
    torch.cuda.synchronize()
    assert r.ws.device_error() == (0, 0)


def test_catchup_refuses_host_weights():
    B, N, din, H, G, D = 1, 2, 64, 4, 2, 16
    dev = lambda *shape: torch.zeros(shape, dtype=torch.int16, device=DEV)  # noqa: E731
    u, gamma = dev(N, din), dev(din)
    Wq, Wk, Wv, Wo = dev(H * D, din), dev(G * D, din), dev(G * D, din), dev(din, H * D)
    Kc, Vc = dev(B, 8, G * D), dev(B, 8, G * D)
    bl_off = torch.tensor([0, N], dtype=torch.int32, device=DEV)
    cache_len = torch.tensor([3], dtype=torch.int32, device=DEV)
    cu = wf.Catchup(u, bl_off, cache_len, gamma, Wk, Wv, Kc, Vc, G, Wq=Wq, Wo=Wo)
    for name, hp, keep in _host_buffers(H * D * din * 2):
        for field in ("Wk", "Wv", "Wq", "Wo", "u", "Kc", "Vc"):
            a = wf.CatchupArgs.from_buffer_copy(cu.args)
            setattr(a, field, hp)
            st = wf.lib().wf_catchup(ctypes.byref(a), cu.ws.ptr, cu.ws.nbytes, torch.cuda.current_stream().cuda_stream)
            assert st == INVALID, (name, field)
    torch.cuda.synchronize()
    assert cu.ws.device_error() == (0, 0)
