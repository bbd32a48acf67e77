"""GPU library vs CPU oracle, through the C ABI.

Integer results (target argmax ids, acceptance lengths, bonus tokens, last
rows, accepted paths, routes, draft top-k ids) must match bit-exactly; the
router output within 1e-3 absolute; logits within the worst-case fp32
accumulation bound 2*d*u*sum|h*w| (u = 2^-24).  Inputs obey the rejection
rules (top-2 logit gap, router margin and adjacent draft top-k gaps all
>= 1e-2), so the fp64 oracle and the fp32 kernels take the same decisions.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, dev, host, logit_error_bound, round_on_gpu
from speculative_decoding_verify_lm_gb300 import synth, wf

pytestmark = pytest.mark.gpu

ORACLE = None


def o():
    global ORACLE
    if ORACLE is None:
        ORACLE = oracle.default()
    return ORACLE


def _gapped_hidden(seed, P, d, W, reject=True):
    h = synth.normal_bf16(seed, 1, P, d, 1.0)
    if not reject:
        return h
    for a in range(1, 400):
        _, _, gap = o().lmhead_argmax(h, W)
        bad = np.nonzero(gap < synth.GAP_MIN)[0]
        if not len(bad):
            return h
        for r in bad:
            h[r] = synth.hidden_row(seed, int(r), a, d)
    raise RuntimeError("gap rule not met")


# ------------------------------------------------------------------ LM head
@pytest.mark.parametrize("P,d,V", [(1, 64, 300), (17, 256, 8192), (61, 128, 1000), (200, 64, 513), (130, 72, 777),
                                   (5, 8, 40), (256, 192, 2048), (129, 256, 257),
                                   # evened-out tiles of two heights; the last one past the matrix
                                   (40, 256, 76000), (97, 128, 76003),
                                   (9, 16384, 1000),    # the largest hidden size
                                   # paired CTAs with an odd count of activation tiles: the last
                                   # pair's second CTA loads rows past the matrix (zero fill)
                                   (300, 128, 3001), (1100, 64, 2049), (383, 2560, 5000)])
def test_lmhead_argmax(P, d, V):
    W = synth.normal_bf16(7 + P, 0, V, d, 0.02 if d >= 256 else 0.1)
    h = _gapped_hidden(11 + V, P, d, W)
    ids_ref, mx_ref, gap = o().lmhead_argmax(h, W)
    ws = wf.Workspace(P)
    ids = torch.empty(P, dtype=torch.int32, device=DEV)
    mx = torch.empty(P, dtype=torch.float32, device=DEV)
    for _ in range(2):   # the workspace is reused: the second call must see it clean
        wf.wf_lmhead_argmax(dev(h), dev(W), ws, ids=ids, maxlogit=mx)
        torch.cuda.synchronize()
        assert np.array_equal(host(ids), ids_ref)
        assert np.all(np.abs(host(mx) - mx_ref) <= logit_error_bound(h, W, ids_ref))
    assert ws.device_error() == (0, 0)
    assert not ws.buf.any().item(), "workspace must be left zeroed"


def test_lmhead_argmax_ties_lowest_id():
    d, V, P = 64, 600, 3
    W = synth.normal_bf16(3, 0, V, d, 0.05)
    W[[17, 333, 599]] = synth.to_bf16_bits(np.full((3, d), 0.5, np.float32))   # identical, dominant rows
    h = synth.to_bf16_bits(np.abs(np.random.default_rng(0).standard_normal((P, d))).astype(np.float32))
    ws = wf.Workspace(P)
    ids = wf.wf_lmhead_argmax(dev(h), dev(W), ws)
    assert host(ids).tolist() == [17, 17, 17]


# ------------------------------------------------------------------ verify
def _random_trees(seed, B, max_nodes):
    rng = np.random.default_rng(seed)
    pos_off, node_off, par, tok, kinds = [0], [0], [], [], []
    for b in range(B):
        N = int(rng.integers(0, max_nodes + 1))
        kinds.append(int(rng.integers(0, 2)))
        p = [int(rng.integers(-1, i)) if i else -1 for i in range(N)] if kinds[-1] else list(range(-1, N - 1))
        par += p
        tok += rng.integers(0, 3, N).tolist()
        pos_off.append(pos_off[-1] + N + 1)
        node_off.append(node_off[-1] + N)
    P = pos_off[-1]
    g = rng.integers(0, 3, P).astype(np.int32)
    return (g, np.array(tok, np.int32), np.array(par, np.int32), np.array(pos_off, np.int32),
            np.array(node_off, np.int32), np.array(kinds, np.int32))


@pytest.mark.parametrize("seed,B,max_nodes", [(1, 1, 60), (2, 37, 8), (3, 300, 70), (4, 5, 256), (5, 64, 0)])
def test_verify_tree_and_chain(seed, B, max_nodes):
    g, tok, par, pos_off, node_off, kinds = _random_trees(seed, B, max_nodes)
    ws = wf.Workspace(int(pos_off[-1]), B)
    ps = 12
    n, bo, la, pa = wf.wf_verify_tree(dev(g), dev(tok), dev(par), dev(node_off), dev(pos_off), ws, path_stride=ps)
    rn, rb, rl, rp, rc = o().verify_tree(g, tok, par, node_off, pos_off, ps)
    assert rc == 0
    assert np.array_equal(host(n), rn) and np.array_equal(host(bo), rb) and np.array_equal(host(la), rl)
    assert np.array_equal(host(pa), rp)
    # chains on their own (every sequence read as a DFlash block)
    cn, cb, cl, cp = wf.wf_verify_chain(dev(g), dev(tok), dev(pos_off), dev(node_off), ws, path_stride=ps)
    rn, rb, rl, rp = o().verify_chain(g, tok, pos_off, node_off, ps)
    assert np.array_equal(host(cn), rn) and np.array_equal(host(cb), rb) and np.array_equal(host(cl), rl)
    assert np.array_equal(host(cp), rp)
    assert ws.device_error() == (0, 0)


def test_verify_golden_cases():
    import pins
    for fname, tree in (("trees.txt", True), ("chains.txt", False)):
        cases = pins.read_cases(fname)
        seqs = [(c["g"], c.get("tok", c.get("draft")), c.get("parent", list(range(-1, len(c.get("draft", [])) - 1))))
                for c in cases]
        g, tok, par, pos_off, node_off = pins._pack(seqs)
        ws = wf.Workspace(len(g), len(cases))
        if tree:
            n, bo, la, _ = wf.wf_verify_tree(dev(g), dev(tok), dev(par), dev(node_off), dev(pos_off), ws)
        else:
            n, bo, la, _ = wf.wf_verify_chain(dev(g), dev(tok), dev(pos_off), dev(node_off), ws)
        for b, c in enumerate(cases):
            e = c["expect"]
            assert host(n)[b] == e["n"] and host(bo)[b] == e["bonus"], c["name"]
            assert host(la)[b] - pos_off[b] == e["last"], c["name"]


def test_verify_bad_parent_sets_error():
    g = np.array([1, 2, 3, 5, 6, 1, 2], np.int32)
    tok = np.array([1, 2, 5, 1], np.int32)
    par = np.array([-1, 1, -1, 3], np.int32)       # seq 0: parent[1] = 1 (not < 1); seq 1 fine
    pos_off = np.array([0, 3, 5, 7], np.int32)
    node_off = np.array([0, 2, 3, 4], np.int32)    # seq 2: node 0 has parent 3 (out of range)
    par = np.array([-1, 1, -1, 3], np.int32)
    ws = wf.Workspace(7, 3)
    n, bo, la, _ = wf.wf_verify_tree(dev(g), dev(tok), dev(par), dev(node_off), dev(pos_off), ws)
    assert host(n)[0] == -1 and host(n)[2] == -1 and host(n)[1] == 1 and host(bo)[1] == 6
    code, info = ws.device_error()
    assert code == 5 and info in (0, 2)


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("B,d,m", [(1, 2560, 1024), (1, 2560, 320), (7, 256, 128), (8, 72, 40), (9, 72, 40),
                                   (12, 2560, 1024), (33, 64, 5), (256, 512, 64),
                                   # the GEMM's row groups at their edges: lower groups only, the
                                   # first upper group, a second row tile of one row
                                   (64, 256, 200), (65, 256, 200), (129, 128, 300),
                                   (3, 4096, 256), (20, 4096, 256)])   # rows too wide for W1 in registers
def test_router(B, d, m):
    rng = np.random.default_rng(B * 7 + m)
    P = B + 3
    h = synth.normal_bf16(B + d, 1, P, d, 1.0)
    rows = rng.permutation(P)[:B].astype(np.int32)
    W1 = (rng.standard_normal((m, d)) * 0.05).astype(np.float32)
    b1 = (rng.standard_normal(m) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal(m) * 0.05).astype(np.float32)
    b2, tau = 0.1, 0.3
    ref, rroute = o().router(h, rows, W1, b1, w2, b2, tau)
    ws = wf.Workspace(P, B, m)
    for _ in range(2):
        delta, route = wf.wf_router_mlp(dev(h), dev(rows), dev(W1), dev(b1), dev(w2), b2, tau, ws)
        torch.cuda.synchronize()
        assert np.max(np.abs(host(delta) - ref)) <= 1e-3
        clear = np.abs(ref - tau) >= synth.GAP_MIN
        assert np.array_equal(host(route)[clear], rroute[clear])
    assert not ws.buf.any().item()


# ------------------------------------------------------------------ draft head
def _draft_case(B, d, Vd, k):
    """Draft weights, id map and inputs whose adjacent top-(k+1) logits are
    >= 1e-2 apart, with the oracle's answer.  Logit scale ~1 at d = 2560 (std
    0.02), larger for the small shapes so that the rule holds in a few draws."""
    Wd = synth.normal_bf16(Vd + d, 0, Vd, d, 0.02 if d >= 2560 else 4.0 / d ** 0.5)
    d2t = np.random.default_rng(Vd).permutation(151936)[:Vd].astype(np.int32)
    x = synth.normal_bf16(B + 1, 1, B, d, 1.0)
    dids, tids, vals, lse, mg = o().draft_topk(x, Wd, d2t, k)
    for a in range(1, 400):   # resample the offending rows only
        bad = np.nonzero(mg < synth.GAP_MIN)[0]
        if not len(bad):
            break
        for r in bad:
            x[r] = synth.hidden_row(B + 1, int(r), a, d)
        got = o().draft_topk(x[bad], Wd, d2t, k)
        for full, part in zip((dids, tids, vals, lse, mg), got):
            full[bad] = part
    assert (mg >= synth.GAP_MIN).all(), "gap rule not met: expected ids would be stale"
    _lse_ref[id(x)] = lse
    return Wd, d2t, x, dids, tids, vals


_lse_ref = {}   # the oracle's log-sum-exp of each _draft_case's rows, by the x array


def _check_lse(got, x):
    """Log-sum-exp over the draft vocabulary: fp32 partial sums of e^(L - max)
    per tile, merged in fp32; well within 1e-3 of the fp64 value at these sizes."""
    assert np.max(np.abs(got - _lse_ref[id(x)])) <= 1e-3


@pytest.mark.parametrize("B,d,Vd,k", [(1, 256, 1000, 10), (3, 128, 32000, 10), (130, 64, 700, 16), (2, 72, 300, 1),
                                      (1, 2560, 32000, 10), (2, 16384, 500, 16),
                                      (300, 128, 4000, 10),    # paired CTAs, odd count of activation tiles
                                      (5, 96, 3000, 12)])      # the 16-wide candidate lists, 12 kept
def test_draft_topk(B, d, Vd, k):
    Wd, d2t, x, dids, tids, vals = _draft_case(B, d, Vd, k)
    ws = wf.Workspace(1, B, 1, Vd, k)
    lse = torch.empty(B, dtype=torch.float32, device=DEV)
    for it in range(3):   # with the log-sum-exp, without it, with it again (the workspace stays clean)
        gi, gt, gv = wf.wf_draft_topk(dev(x), dev(Wd), dev(d2t), k, ws, lse=lse if it != 1 else None)
        torch.cuda.synchronize()
        assert np.array_equal(host(gi), dids) and np.array_equal(host(gt), tids)
        bound = np.stack([logit_error_bound(x[b:b + 1].repeat(k, 0), Wd, dids[b]) for b in range(B)])
        assert np.all(np.abs(host(gv) - vals) <= bound)
        if it != 1:
            _check_lse(host(lse), x)
    assert ws.device_error() == (0, 0)
    assert not ws.buf.any().item()


@pytest.mark.parametrize("P,B,d,V,Vd,k", [(17, 1, 256, 8192, 4000, 10), (128, 128, 64, 777, 300, 16),
                                          (61, 2, 72, 1000, 129, 1), (1, 1, 2560, 151936, 32000, 10),
                                          (40, 2, 256, 76000, 19456, 10),
                                          # several activation tiles: the paired sweep carries the draft head
                                          (300, 200, 128, 5000, 3000, 10), (257, 64, 96, 2000, 1000, 16),
                                          (600, 256, 64, 4096, 2050, 4), (129, 129, 2560, 33000, 7000, 10)])
def test_lmhead_draft_topk_shared_sweep(P, B, d, V, Vd, k):
    """Both heads in one sweep give the oracle's argmax and top-k (and leave the
    workspace zeroed), here and on a reused workspace."""
    W = synth.normal_bf16(7 + P, 0, V, d, 0.02 if d >= 256 else 0.1)
    h = _gapped_hidden(11 + V, P, d, W)
    ids_ref, mx_ref, _ = o().lmhead_argmax(h, W)
    Wd, d2t, x, dids, tids, vals = _draft_case(B, d, Vd, k)
    ws = wf.Workspace(P, B, 1, Vd, k, d=d)
    mx = torch.empty(P, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, dtype=torch.float32, device=DEV)
    for it in range(2):
        ids, gi, gt, gv = wf.wf_lmhead_draft_topk(dev(h), dev(W), dev(x), dev(Wd), dev(d2t), k, ws, maxlogit=mx,
                                                  lse=lse if it == 0 else None)
        torch.cuda.synchronize()
        if it == 0:
            _check_lse(host(lse), x)
        assert np.array_equal(host(ids), ids_ref)
        assert np.all(np.abs(host(mx) - mx_ref) <= logit_error_bound(h, W, ids_ref))
        assert np.array_equal(host(gi), dids) and np.array_equal(host(gt), tids)
        bound = np.stack([logit_error_bound(x[b:b + 1].repeat(k, 0), Wd, dids[b]) for b in range(B)])
        assert np.all(np.abs(host(gv) - vals) <= bound)
    assert ws.device_error() == (0, 0)
    assert not ws.buf.any().item(), "workspace must be left zeroed"


def test_draft_topk_bad_map():
    Wd = synth.normal_bf16(5, 0, 300, 64, 0.1)
    x = synth.normal_bf16(6, 1, 2, 64, 1.0)
    d2t = np.full(300, -1, np.int32)
    ws = wf.Workspace(1, 2, 1, 300, 4)
    _, gt, _ = wf.wf_draft_topk(dev(x), dev(Wd), dev(d2t), 4, ws)
    assert (host(gt) == -1).all()
    assert ws.device_error()[0] == 5


# ------------------------------------------------------------------ whole rounds
def _compare_round(wl, out, seqs=None):
    ref = o().round_(wl.hidden, wl.W, wl.pos_off, wl.node_off, wl.kind, wl.tok, wl.parent, wl.W1, wl.b1, wl.w2,
                     wl.b2, wl.tau, out["path"].shape[1]) if seqs is None else None
    if ref is not None:
        for key in ("ids", "n_accept", "bonus", "last_pos", "path", "route"):
            assert np.array_equal(out[key], ref[key]), key
        assert np.max(np.abs(out["delta_al"] - ref["delta"])) <= 1e-3
    assert np.array_equal(out["n_accept"][wl.planted], wl.cut[wl.planted])


# The five round workloads at full size are compared with the oracle's stored
# answers in test_full_size_gpu.py.


@pytest.mark.parametrize("kinds,K,d,V,Vd,k", [([1], 16, 128, 3000, 1000, 10), ([0, 1], 16, 64, 777, 301, 16),
                                               ([0] * 8, 15, 72, 2049, 129, 1), ([0] * 7 + [1], 3, 256, 8192, 4000, 10)])
def test_round_shared_sweep_with_draft(kinds, K, d, V, Vd, k):
    """At most 128 verified rows and 128 sequences: the draft head shares the
    LM head's weight sweep (W, then Wd) and its candidate lists are merged
    after acceptance.  Ragged vocabularies; 128 rows exactly in one case."""
    wl = synth.small_workload(500 + d + k, d=d, V=V, kinds=kinds, argmax_fn=oracle.argmax_fn, m=16, K=K,
                              Vd=Vd, topk=k, router_fn=oracle.router_fn, topk_gap_fn=oracle.topk_gap_fn)
    assert wl.P <= 128
    r, out = round_on_gpu(wl)
    assert r.ws.device_error() == (0, 0)
    _compare_round(wl, out)
    dids, tids, vals, _, _ = o().draft_topk(wl.x, wl.Wd, wl.d2t, wl.topk)
    assert np.array_equal(out["draft_ids"], dids) and np.array_equal(out["tids"], tids)
    assert np.max(np.abs(out["vals"] - vals)) <= 1e-3
    out2 = {key: host(v) for key, v in r().items()}
    for key in ("ids", "n_accept", "route", "draft_ids", "tids"):
        assert np.array_equal(out2[key], out[key]), key


def test_round_edge_shapes():
    """One-row sequences (no drafts), tiny vocabulary, d = 8, a lone chain."""
    for kinds, d, V in (([0], 8, 40), ([1, 0, 1], 64, 257), ([0, 0], 16, 2)):
        wl = synth.small_workload(31 + d, d=d, V=V, kinds=kinds, argmax_fn=oracle.argmax_fn, m=8, K=3,
                                  n_nodes=4, depth=2, branch=2, router_fn=oracle.router_fn, reject=V > 2)
        r, out = round_on_gpu(wl)
        assert r.ws.device_error() == (0, 0)
        _compare_round(wl, out)


# ------------------------------------------------------------------ entropy router
@pytest.mark.parametrize("P,d,V,rows", [(17, 256, 8192, None), (5, 64, 300, None), (61, 128, 5000, [60, 0, 7]),
                                        (300, 64, 1000, list(range(299, 43, -1))), (40, 2560, 151936, [3, 39]),
                                        (200, 256, 20000, None),    # two row tiles (paired CTAs), ragged second
                                        (129, 128, 3000, None)])    # the second tile holds one row
def test_entropy(P, d, V, rows):
    W = synth.normal_bf16(V + d, 0, V, d, d ** -0.5 * 2.0)
    h = synth.normal_bf16(P + d, 1, P, d, 1.0)
    r = np.arange(P, dtype=np.int32) if rows is None else np.array(rows, np.int32)
    H_ref, _ = o().entropy(h, r, W)
    tau = float(np.median(H_ref)) + 0.0037
    ws = wf.Workspace(P, len(r), d=d)
    for _ in range(2):
        H, route = wf.wf_lmhead_entropy(dev(h), dev(W), tau, ws, rows=None if rows is None else dev(r))
        torch.cuda.synchronize()
        assert np.max(np.abs(host(H) - H_ref)) <= 1e-3
        clear = np.abs(H_ref - tau) >= synth.GAP_MIN
        assert np.array_equal(host(route)[clear], (H_ref > tau).astype(np.int32)[clear])
    assert ws.device_error() == (0, 0)
    if rows is None:   # gathered rows stay in their staging area; everything else is left zeroed
        assert not ws.buf.any().item()


def test_entropy_bad_row():
    W = synth.normal_bf16(3, 0, 500, 64, 0.2)
    h = synth.normal_bf16(4, 1, 10, 64, 1.0)
    ws = wf.Workspace(10, 3, d=64)
    H, route = wf.wf_lmhead_entropy(dev(h), dev(W), 1.0, ws, rows=dev(np.array([2, 10, -1], np.int32)))
    assert np.isnan(host(H)[1:]).all() and list(host(route)[1:]) == [-1, -1] and not np.isnan(host(H)[0])
    assert ws.device_error()[0] == 5


@pytest.mark.parametrize("kinds", [[0, 1], [1, 1, 1, 0]])
def test_round_entropy_router(kinds):
    """WhiFlash-Entropy routing inside a round: fused into the LM-head sweep for
    <= 128 rows, a second sweep over the accepted rows otherwise."""
    wl = synth.small_workload(77 + len(kinds), d=128, V=3000, kinds=kinds, argmax_fn=oracle.argmax_fn, m=8,
                              n_nodes=60, depth=8, branch=10)
    assert (wl.P <= 128) == (len(kinds) == 2)   # both paths: the fused sweep and the second sweep
    _check_entropy_round(wl)


def test_round_entropy_router_with_draft_head():
    """The same with a draft head: its top-k shares the LM head's sweep (which
    also gathers the entropy statistics) and is merged in the verification
    launch."""
    wl = synth.small_workload(91, d=128, V=3000, kinds=[1, 0], argmax_fn=oracle.argmax_fn, m=8, n_nodes=60,
                              depth=8, branch=10, Vd=700, topk=10, topk_gap_fn=oracle.topk_gap_fn)
    out = _check_entropy_round(wl)
    dids, tids, _, _, _ = o().draft_topk(wl.x, wl.Wd, wl.d2t, wl.topk)
    assert np.array_equal(out["draft_ids"], dids) and np.array_equal(out["tids"], tids)


def _check_entropy_round(wl):
    rr = wl.pos_off[1:]
    ref = o().round_(wl.hidden, wl.W, wl.pos_off, wl.node_off, wl.kind, wl.tok, wl.parent, wl.W1, wl.b1, wl.w2,
                     wl.b2, wl.tau, wl.max_depth)
    H_ref, _ = o().entropy(wl.hidden, ref["last_pos"], wl.W)
    tau = float(np.median(H_ref)) + 0.0041
    draft = wl.Wd is not None
    r = wf.Round(dev(wl.hidden), dev(wl.W), dev(wl.pos_off), dev(wl.node_off), dev(wl.tok), dev(wl.W1),
                 dev(wl.b1), dev(wl.w2), wl.b2, tau, kind=dev(wl.kind), parent=dev(wl.parent),
                 path_stride=wl.max_depth, router_kind=wf.WF_ROUTER_ENTROPY, x=dev(wl.x) if draft else None,
                 Wd=dev(wl.Wd) if draft else None, d2t=dev(wl.d2t) if draft else None,
                 k=wl.topk if draft else 0)
    assert rr[-1] == wl.P
    for _ in range(2):
        out = {k: host(v) for k, v in r().items()}
        torch.cuda.synchronize()
        for key in ("ids", "n_accept", "bonus", "last_pos", "path"):
            assert np.array_equal(out[key], ref[key]), key
        assert np.max(np.abs(out["delta_al"] - H_ref)) <= 1e-3
        clear = np.abs(H_ref - tau) >= synth.GAP_MIN
        assert np.array_equal(out["route"][clear], (H_ref > tau).astype(np.int32)[clear])
    assert r.ws.device_error() == (0, 0)
    return out


# ------------------------------------------------------------------ kept rows
@pytest.mark.parametrize("seed,B,max_nodes", [(11, 3, 60), (12, 1500, 12), (13, 7, 0)])
def test_accepted_rows(seed, B, max_nodes):
    g, tok, par, pos_off, node_off, kinds = _random_trees(seed, B, max_nodes)
    ps = max(max_nodes, 1)
    n, _, _, path, _ = o().verify_tree(g, tok, par, node_off, pos_off, ps)
    acc_rows, acc_off = o().accepted_rows(n, path, pos_off)
    d = 64
    h = synth.normal_bf16(seed, 1, int(pos_off[-1]), d, 1.0)
    gr, go, gh = wf.wf_accepted_rows(dev(n), dev(path), dev(pos_off), hidden=dev(h))
    torch.cuda.synchronize()
    assert np.array_equal(host(gr), acc_rows) and np.array_equal(host(go), acc_off)
    kept = np.concatenate([acc_rows[b][:n[b] + 1] for b in range(B)])
    assert np.array_equal(host(gh).view(np.uint16), h[kept])


# ------------------------------------------------------------------ draft-tree construction
@pytest.mark.parametrize("B,D,k,N", [(1, 8, 10, 60), (64, 8, 10, 60), (5, 3, 4, 20), (3, 16, 16, 200), (2, 1, 6, 6)])
def test_build_tree(B, D, k, N):
    rng = np.random.default_rng(B * 100 + D)
    tid = rng.integers(0, 151936, (B, D, k, k)).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(k) * 0.7, (B, D, k))).astype(np.float32)
    lp[lp < -60] = -60.0
    ref = o().build_tree(tid, lp, N)
    assert ref[4] == 0
    ws = wf.Workspace(1)
    got = wf.wf_build_tree(dev(tid), dev(lp), N, ws)
    torch.cuda.synchronize()
    for a, e in zip(got, ref[:4]):
        assert np.array_equal(host(a), e)
    assert ws.device_error() == (0, 0)


def test_verify_right_after_tree_construction():
    """A verify call enqueued straight after the call that builds its tree (same
    stream, no synchronisation in between) sees the built parents and tokens:
    a call on its own reads its inputs only after the work before it."""
    B, D, k, N = 6, 6, 4, 40
    rng = np.random.default_rng(5)
    tid = rng.integers(0, 4, (B, D, k, k)).astype(np.int32)    # a tiny alphabet: many matches
    lp = np.log(rng.dirichlet(np.ones(k) * 0.7, (B, D, k))).astype(np.float32)
    lp[lp < -60] = -60.0
    rpar, rtok, _, _, rc = o().build_tree(tid, lp, N)
    assert rc == 0
    node_off = (np.arange(B + 1) * N).astype(np.int32)
    pos_off = (np.arange(B + 1) * (N + 1)).astype(np.int32)
    g = rng.integers(0, 4, B * (N + 1)).astype(np.int32)
    ref = o().verify_tree(g, rtok.ravel(), rpar.ravel(), node_off, pos_off, 8)
    assert ref[4] == 0 and ref[0].max() >= 2
    ws = wf.Workspace(B * (N + 1), B)
    g_d, no_d, po_d = dev(g), dev(node_off), dev(pos_off)
    for _ in range(3):
        parent, token, _, _ = wf.wf_build_tree(dev(tid), dev(lp), N, ws)
        n, bo, la, pa = wf.wf_verify_tree(g_d, token.view(-1), parent.view(-1), no_d, po_d, ws, path_stride=8)
        torch.cuda.synchronize()
        assert np.array_equal(host(n), ref[0]) and np.array_equal(host(bo), ref[1])
        assert np.array_equal(host(la), ref[2]) and np.array_equal(host(pa), ref[3])
    assert ws.device_error() == (0, 0)


def test_draft_head_to_tree_construction_chain():
    """The draft head feeds tree construction on one stream: top-10 target ids
    and logits over the 32,000-id draft vocabulary with the log-sum-exp
    (wf_draft_topk), log-probabilities = logits - lse, then the depth-8,
    60-node tree (wf_build_tree) - the EAGLE-3 settings (WhiFlash paper App. A
    Table 7; Qwen3-4B-EAGLE3 card, "Factors").  Each (step, slot) has its own
    drafter state.  The oracle runs the same chain in fp64.  Tree construction
    ranks sums of log-probabilities, which have no gap rule; so the oracle's
    tree is first checked to stay the same when every log-probability moves by
    up to 1e-4, and the GPU's log-probabilities are checked to lie within 1e-4
    of the oracle's, before the trees are compared."""
    D, k, N, d, Vd, seed = 8, 10, 60, 2560, 32000, 81
    Wd = synth.normal_bf16(Vd + d, 0, Vd, d, 0.02)
    d2t = np.random.default_rng(Vd).permutation(151936)[:Vd].astype(np.int32)
    x = synth.normal_bf16(seed, 1, D * k, d, 1.0)
    dids, tids, vals, lse_ref, mg = o().draft_topk(x, Wd, d2t, k)
    for a in range(1, 400):   # adjacent top-11 gaps >= 1e-2: the GPU picks the same children in the same order
        bad = np.nonzero(mg < synth.GAP_MIN)[0]
        if not len(bad):
            break
        for r in bad:
            x[r] = synth.hidden_row(seed, int(r), a, d)
        got = o().draft_topk(x[bad], Wd, d2t, k)
        for full, part in zip((dids, tids, vals, lse_ref, mg), got):
            full[bad] = part
    assert (mg >= synth.GAP_MIN).all()
    lp_ref = (vals - lse_ref[:, None]).astype(np.float32).reshape(1, D, k, k)
    tid_ref = tids.reshape(1, D, k, k)
    tree_ref = o().build_tree(tid_ref, lp_ref, N)
    assert tree_ref[4] == 0
    rng = np.random.default_rng(7)
    for _ in range(16):
        jitter = rng.uniform(-1e-4, 1e-4, lp_ref.shape).astype(np.float32)
        alt = o().build_tree(tid_ref, np.minimum(lp_ref + jitter, 0).astype(np.float32), N)
        assert all(np.array_equal(a_, e) for a_, e in zip(alt[:2], tree_ref[:2])), "oracle tree hinges on rounding"
    ws = wf.Workspace(1, D * k, 1, Vd, k, d=d)
    lse = torch.empty(D * k, dtype=torch.float32, device=DEV)
    _, gt, gv = wf.wf_draft_topk(dev(x), dev(Wd), dev(d2t), k, ws, lse=lse)
    lp = (gv - lse[:, None]).view(1, D, k, k)   # same stream, no synchronisation
    parent, token, score, depth = wf.wf_build_tree(gt.view(1, D, k, k), lp, N, ws)
    torch.cuda.synchronize()
    assert np.max(np.abs(host(lse) - lse_ref)) <= 1e-3
    assert np.array_equal(host(gt).reshape(tid_ref.shape), tid_ref)
    assert np.max(np.abs(host(lp) - lp_ref)) <= 1e-4
    assert np.array_equal(host(parent), tree_ref[0]) and np.array_equal(host(token), tree_ref[1])
    assert np.array_equal(host(depth), tree_ref[3])
    assert np.max(np.abs(host(score) - tree_ref[2])) <= 8e-4   # sums of 8 log-probabilities
    assert ws.device_error() == (0, 0)


def test_build_tree_bad_logprob():
    tid = np.zeros((2, 2, 2, 2), np.int32)
    lp = np.full((2, 2, 2, 2), -0.5, np.float32)
    lp[1, 1, 1, 0] = 0.25
    ws = wf.Workspace(1)
    parent, token, _, _ = wf.wf_build_tree(dev(tid), dev(lp), 3, ws)
    assert (host(parent)[1] == -1).all() and (host(token)[1] == -1).all() and host(parent)[0][0] == -1
    assert ws.device_error()[0] == 5


# ------------------------------------------------------------------ failure path
def test_bounded_wait_gives_up_and_context_survives():
    ws = wf.Workspace(8)
    wf.wf_probe_bounded_wait(20_000_000, ws)          # 20 ms on a barrier nothing arrives on
    assert ws.device_error(clear=True) == (6, 0xFFFF)
    # the context is still usable: a normal call afterwards succeeds
    W = synth.normal_bf16(1, 0, 300, 64, 0.1)
    h = _gapped_hidden(2, 4, 64, W)
    ids = wf.wf_lmhead_argmax(dev(h), dev(W), ws)
    assert np.array_equal(host(ids), o().lmhead_argmax(h, W)[0])
    assert ws.device_error() == (0, 0)
