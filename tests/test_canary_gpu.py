"""Writes past an output buffer.  Every entry point writes its outputs into
buffers that sit between canary bytes; a kernel that writes past either end
of an output changes them.  Sizes are odd on purpose (rows, k and strides that
are no multiple of a tile or a vector width).  The GPUs here offer no memory
checker, so this stands in for one on every output; the workspace side is
covered by the zero-at-rest checks of the parity tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import DEV, dev, host
from speculative_decoding_verify_lm_gb300 import synth, wf
from test_parity_gpu import _draft_case, _gapped_hidden, _random_trees

pytestmark = pytest.mark.gpu

CANARY = 0xA5
GUARD = 256   # bytes on each side; a multiple of 16 keeps the buffer 16-byte aligned


class Guarded:
    """A device tensor of `shape` inside GUARD canary bytes on each side."""

    def __init__(self, shape, dtype):
        shape = tuple(shape)
        n = int(np.prod(shape)) if shape else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        r = self.raw.cpu().numpy()
        return bool((r[:GUARD] == CANARY).all() and (r[GUARD + self.nbytes:] == CANARY).all())


def o():
    return oracle.default()


def all_intact(*gs):
    return all(g.intact() for g in gs)


@pytest.mark.parametrize("P,d,V", [(37, 128, 4999), (3, 2560, 151936)])
def test_lmhead_argmax_outputs(P, d, V):
    W = synth.normal_bf16(5 + P, 0, V, d, 0.02 if d >= 256 else 0.1)
    h = _gapped_hidden(13 + V, P, d, W)
    ids_ref, _, _ = o().lmhead_argmax(h, W)
    ids, mx = Guarded((P,), torch.int32), Guarded((P,), torch.float32)
    wf.wf_lmhead_argmax(dev(h), dev(W), wf.Workspace(P), ids=ids.t, maxlogit=mx.t)
    assert np.array_equal(host(ids.t), ids_ref) and all_intact(ids, mx)
    ids2, mx2 = Guarded((P,), torch.int32), Guarded((P,), torch.float32)
    wf.wf_lmhead_argmax_noalloc(dev(h), dev(W), ids=ids2.t, maxlogit=mx2.t)
    assert np.array_equal(host(ids2.t), ids_ref) and all_intact(ids2, mx2)


def test_verify_outputs():
    g, tok, par, pos_off, node_off, kinds = _random_trees(9, 13, 40)
    B, ps = 13, 5   # a path stride shorter than the deepest accepted path
    ws = wf.Workspace(int(pos_off[-1]), B)
    for which in ("tree", "chain"):
        outs = [Guarded((B,), torch.int32) for _ in range(3)] + [Guarded((B, ps), torch.int32)]
        n, bo, la, pa = (x.t for x in outs)
        if which == "tree":
            wf.wf_verify_tree(dev(g), dev(tok), dev(par), dev(node_off), dev(pos_off), ws, path_stride=ps,
                              n_accept=n, bonus=bo, last_pos=la, path=pa)
            rn, rb, rl, rp, _ = o().verify_tree(g, tok, par, node_off, pos_off, ps)
        else:
            wf.wf_verify_chain(dev(g), dev(tok), dev(pos_off), dev(node_off), ws, path_stride=ps, n_accept=n,
                               bonus=bo, last_pos=la, path=pa)
            rn, rb, rl, rp = o().verify_chain(g, tok, pos_off, node_off, ps)
        assert np.array_equal(host(n), rn) and np.array_equal(host(bo), rb) and np.array_equal(host(la), rl)
        assert np.array_equal(host(pa), rp) and all_intact(*outs)


@pytest.mark.parametrize("B,d,m", [(5, 2560, 1024), (13, 2560, 1024), (37, 72, 40)])
def test_router_outputs(B, d, m):
    rng = np.random.default_rng(B + m)
    P = B + 4
    h = synth.normal_bf16(B + d, 1, P, d, 1.0)
    rows = rng.permutation(P)[:B].astype(np.int32)
    W1 = (rng.standard_normal((m, d)) * 0.05).astype(np.float32)
    b1 = (rng.standard_normal(m) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal(m) * 0.05).astype(np.float32)
    ref, _ = o().router(h, rows, W1, b1, w2, 0.1, 0.3)
    delta, route = Guarded((B,), torch.float32), Guarded((B,), torch.int32)
    wf.wf_router_mlp(dev(h), dev(rows), dev(W1), dev(b1), dev(w2), 0.1, 0.3, wf.Workspace(P, B, m),
                     delta_al=delta.t, route=route.t)
    assert np.max(np.abs(host(delta.t) - ref)) <= 1e-3 and all_intact(delta, route)


def test_draft_topk_outputs():
    B, d, Vd, k = 3, 128, 3001, 7
    Wd, d2t, x, dids, tids, _ = _draft_case(B, d, Vd, k)
    outs = [Guarded((B, k), torch.int32), Guarded((B, k), torch.int32), Guarded((B, k), torch.float32),
            Guarded((B,), torch.float32)]
    wf.wf_draft_topk(dev(x), dev(Wd), dev(d2t), k, wf.Workspace(1, B, 1, Vd, k), draft_ids=outs[0].t,
                     tids=outs[1].t, vals=outs[2].t, lse=outs[3].t)
    assert np.array_equal(host(outs[0].t), dids) and np.array_equal(host(outs[1].t), tids) and all_intact(*outs)
    assert np.isfinite(host(outs[3].t)).all()


@pytest.mark.parametrize("P,B,d,V,Vd,k", [(17, 1, 256, 8192, 4000, 10), (61, 3, 2560, 151936, 32000, 10)])
def test_shared_sweep_outputs(P, B, d, V, Vd, k):
    W = synth.normal_bf16(3 + P, 0, V, d, 0.02 if d >= 2560 else 0.1)
    h = _gapped_hidden(17 + V, P, d, W)
    ids_ref, _, _ = o().lmhead_argmax(h, W)
    Wd, d2t, x, dids, tids, _ = _draft_case(B, d, Vd, k)
    outs = [Guarded((P,), torch.int32), Guarded((P,), torch.float32), Guarded((B, k), torch.int32),
            Guarded((B, k), torch.int32), Guarded((B, k), torch.float32), Guarded((B,), torch.float32)]
    wf.wf_lmhead_draft_topk(dev(h), dev(W), dev(x), dev(Wd), dev(d2t), k, wf.Workspace(P, B, 1, Vd, k),
                            ids=outs[0].t, maxlogit=outs[1].t, draft_ids=outs[2].t, tids=outs[3].t, vals=outs[4].t,
                            lse=outs[5].t)
    assert np.array_equal(host(outs[0].t), ids_ref)
    assert np.array_equal(host(outs[2].t), dids) and np.array_equal(host(outs[3].t), tids) and all_intact(*outs)


def test_entropy_outputs():
    P, d, V = 20, 64, 999
    W = synth.normal_bf16(V + d, 0, V, d, d ** -0.5 * 2.0)
    h = synth.normal_bf16(P + d, 1, P, d, 1.0)
    rows = np.array([19, 0, 7, 7, 3], np.int32)
    H_ref, _ = o().entropy(h, rows, W)
    H, route = Guarded((5,), torch.float32), Guarded((5,), torch.int32)
    wf.wf_lmhead_entropy(dev(h), dev(W), 1.0, wf.Workspace(P, 5, d=d), rows=dev(rows), H=H.t, route=route.t)
    assert np.max(np.abs(host(H.t) - H_ref)) <= 1e-3 and all_intact(H, route)


def test_build_tree_outputs():
    B, D, k, N = 2, 4, 5, 13
    rng = np.random.default_rng(31)
    tid = rng.integers(0, 151936, (B, D, k, k)).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(k) * 0.7, (B, D, k))).astype(np.float32)
    lp[lp < -60] = -60.0
    ref = o().build_tree(tid, lp, N)
    outs = [Guarded((B, N), torch.int32), Guarded((B, N), torch.int32), Guarded((B, N), torch.float32),
            Guarded((B, N), torch.int32)]
    ws = wf.Workspace(1)
    t_tid, t_lp = dev(tid), dev(lp)
    wf.wf_build_tree(t_tid, t_lp, N, ws, parent=outs[0].t, token=outs[1].t, score=outs[2].t, depth=outs[3].t)
    for g, e in zip(outs, ref[:4]):
        assert np.array_equal(host(g.t), e)
    assert all_intact(*outs)


def test_accepted_rows_outputs():
    g, tok, par, pos_off, node_off, _ = _random_trees(12, 7, 30)
    ps = 30
    n, _, _, path, _ = o().verify_tree(g, tok, par, node_off, pos_off, ps)
    acc_rows, acc_off = o().accepted_rows(n, path, pos_off)
    d = 72
    h = synth.normal_bf16(12, 1, int(pos_off[-1]), d, 1.0)
    total = int(np.sum(n + 1))
    rows_g, off_g = Guarded((7, ps + 1), torch.int32), Guarded((8,), torch.int32)
    hid_g = Guarded((7 * (ps + 1), d), torch.int16)   # the bound the binding asks for
    wf.wf_accepted_rows(dev(n), dev(path), dev(pos_off), hidden=dev(h), acc_rows=rows_g.t, acc_off=off_g.t,
                        hidden_out=hid_g.t)
    assert np.array_equal(host(rows_g.t), acc_rows) and np.array_equal(host(off_g.t), acc_off)
    kept = np.concatenate([acc_rows[b][:n[b] + 1] for b in range(7)])
    assert len(kept) == total
    assert np.array_equal(host(hid_g.t)[:total].view(np.uint16), h[kept]) and all_intact(rows_g, off_g, hid_g)


@pytest.mark.parametrize("n,L,cap", [((3, 1, 5), (2, 0, 9), 16), ((50,), (4000,), 4096)])
def test_catchup_outputs(n, L, cap):
    c = pins.catchup_case(41, din=96, H=6, G=3, D=16, n=n, L=L, cap=cap)
    ref, rc = oracle.catchup(**c)
    assert rc == 0
    B, HD = len(n), 6 * 16
    Kc, Vc = dev(c["Kc"]), dev(c["Vc"])
    cu = wf.Catchup(dev(c["u"]), dev(c["bl_off"]), dev(c["cache_len"]), dev(c["gamma"]), dev(c["Wk"]), dev(c["Wv"]),
                    Kc, Vc, c["G"], Wq=dev(c["Wq"]), Wo=dev(c["Wo"]), eps=c["eps"], theta=c["theta"])
    out, attn = Guarded((B, 96), torch.float32), Guarded((B, HD), torch.float32)
    cu.args.out = ctypes.c_void_p(out.t.data_ptr())
    cu.args.attn = ctypes.c_void_p(attn.t.data_ptr())
    cu()
    assert cu.ws.device_error() == (0, 0)
    assert np.allclose(host(out.t), ref["out"], rtol=0, atol=5e-2) and np.allclose(host(attn.t), ref["attn"], rtol=0,
                                                                                     atol=5e-2)
    assert all_intact(out, attn)


def test_accepted_rows_counts_past_the_stride():
    """Accepted counts beyond the path's columns (outside the documented input
    range) are taken as the columns and -1 keeps no row: the result equals the
    oracle's on the clamped counts, and nothing is written past the buffers
    sized for path_stride + 1 rows a sequence."""
    g, tok, par, pos_off, node_off, _ = _random_trees(14, 4, 30)
    ps = 5
    n_ref, _, _, path_ref, _ = o().verify_tree(g, tok, par, node_off, pos_off, ps)
    n = np.array([3, 12, -1, 9], np.int32)   # 12 and 9 exceed the 5 path columns
    path = path_ref.copy()
    clamped = np.clip(n, -1, ps)
    acc_rows, acc_off = o().accepted_rows(clamped, path, pos_off)
    d = 16
    h = synth.normal_bf16(14, 1, int(pos_off[-1]), d, 1.0)
    rows_g, off_g = Guarded((4, ps + 1), torch.int32), Guarded((5,), torch.int32)
    hid_g = Guarded((4 * (ps + 1), d), torch.int16)
    wf.wf_accepted_rows(dev(n), dev(path), dev(pos_off), hidden=dev(h), acc_rows=rows_g.t, acc_off=off_g.t,
                        hidden_out=hid_g.t)
    torch.cuda.synchronize()
    assert np.array_equal(host(rows_g.t), acc_rows) and np.array_equal(host(off_g.t), acc_off)
    kept = np.concatenate([acc_rows[b][:clamped[b] + 1] for b in range(4)])
    assert np.array_equal(host(hid_g.t)[:len(kept)].view(np.uint16), h[kept])
    assert all_intact(rows_g, off_g, hid_g)
