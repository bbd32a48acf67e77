"""Checks that pin the CPU oracle to facts outside itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  Expected values come from brute force written differently from
the oracle (walk-to-root for trees, numpy/scipy library routines for dot
products, sorting, erf and log-sum-exp), closed forms, textbook constants,
and the hand-worked fixtures under tests/golden/.  tests/test_oracle_mutants.py
compiles deliberately broken copies of the oracle and asserts that these
checks catch each one.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
from scipy.special import erf, logsumexp

from speculative_decoding_verify_lm_gb300.synth import bf16_bits_to_f32, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_bf16(rng, shape, std):
    return to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def read_cases(name):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            if ln.startswith("case "):
                cur = {"name": ln[5:]}
                cases.append(cur)
                continue
            key, _, val = ln.partition(":")
            val = val.strip()
            if key == "expect":
                exp = {}
                for item in val.split():
                    k, _, v = item.partition("=")
                    exp[k] = [int(t) for t in v.split(",") if t] if k == "path" else int(v)
                cur["expect"] = exp
            else:
                cur[key] = [int(t) if t.lstrip("-").isdigit() else float(t) for t in val.split()]
    return cases


# ---------------------------------------------------------------- LM head argmax
def check_argmax_bruteforce(o):
    """ids / max logit / top-2 gap against numpy float64 matmul + a full sort.

    Shapes are pairwise distinct so a transposed operand cannot pass."""
    rng = np.random.default_rng(1)
    for P, d, V in [(1, 8, 5), (5, 24, 37), (7, 40, 301), (3, 16, 1)]:
        h = _rand_bf16(rng, (P, d), 1.0)
        W = _rand_bf16(rng, (V, d), 0.2)
        L = _f64(h) @ _f64(W).T
        ids, mx, gap = o.lmhead_argmax(h, W)
        for p in range(P):
            order = sorted(range(V), key=lambda v: (-L[p, v], v))
            assert ids[p] == order[0], (P, d, V, p)
            assert abs(mx[p] - L[p, order[0]]) <= 1e-12 * max(1.0, abs(L[p, order[0]]))
            if V > 1:
                want = L[p, order[0]] - L[p, order[1]]
                assert abs(gap[p] - want) <= 1e-12 * max(1.0, abs(L[p]).max()), (gap[p], want)
            else:
                assert gap[p] == math.inf


def check_argmax_ties(o):
    """Equal maximal logits: the lowest id wins and the gap is exactly 0."""
    rng = np.random.default_rng(2)
    d, V = 16, 12
    h = to_bf16_bits(np.abs(rng.standard_normal((2, d))).astype(np.float32) + np.float32(0.1))
    W = _rand_bf16(rng, (V, d), 0.05)
    W[3] = to_bf16_bits(np.full(d, 4.0, np.float32))     # identical rows, far above the rest
    W[7] = W[3]
    ids, mx, gap = o.lmhead_argmax(h, W)
    L = _f64(h) @ _f64(W).T
    assert list(ids) == [3, 3] and list(gap) == [0.0, 0.0] and np.allclose(mx, L[:, 3], rtol=1e-12)


def check_argmax_closed_form(o):
    """One-hot weight rows: logit(p, v) = c_v * h[p, v mod d], exact in binary."""
    d, V, P = 8, 20, 3
    hv = np.array([[1, -2, 3, 0.5, -1, 2, 0.25, 1.5],
                   [-1, -1, -1, -1, -1, -1, -1, -4],
                   [2, 2, 2, 2, 2, 2, 2, 2]], np.float32)
    c = np.array([(v % 7) - 3 for v in range(V)], np.float32)
    Wv = np.zeros((V, d), np.float32)
    for v in range(V):
        Wv[v, v % d] = c[v]
    ids, mx, gap = o.lmhead_argmax(to_bf16_bits(hv), to_bf16_bits(Wv))
    for p in range(P):
        L = [float(c[v]) * float(hv[p, v % d]) for v in range(V)]
        best = max(L)
        first = L.index(best)
        second = max(L[:first] + L[first + 1:])
        assert ids[p] == first and mx[p] == best and gap[p] == best - second, (p, ids[p], first)


# ---------------------------------------------------------------- verification
def _pack(seqs):
    """seqs: list of (g_rows, tok, parent) -> packed arrays + offsets."""
    pos_off, node_off = [0], [0]
    for g, tok, _ in seqs:
        pos_off.append(pos_off[-1] + len(g))
        node_off.append(node_off[-1] + len(tok))
    g = np.concatenate([np.asarray(s[0], np.int32) for s in seqs])
    tok = np.concatenate([np.asarray(s[1], np.int32) for s in seqs]) if node_off[-1] else np.zeros(0, np.int32)
    par = np.concatenate([np.asarray(s[2], np.int32) for s in seqs]) if node_off[-1] else np.zeros(0, np.int32)
    return g, tok, par, np.array(pos_off, np.int32), np.array(node_off, np.int32)


def check_chain_golden(o):
    cases = read_cases("chains.txt")
    seqs = [(c["g"], c["draft"], list(range(-1, len(c["draft"]) - 1))) for c in cases]
    g, tok, _, pos_off, node_off = _pack(seqs)
    n, bonus, last, path = o.verify_chain(g, tok, pos_off, node_off, path_stride=16)
    for b, c in enumerate(cases):
        e = c["expect"]
        assert n[b] == e["n"] and bonus[b] == e["bonus"] and last[b] - pos_off[b] == e["last"], c["name"]
        assert list(path[b][: e["n"]]) == list(range(e["n"])) and all(path[b][e["n"]:] == -1), c["name"]


def check_tree_golden(o):
    cases = read_cases("trees.txt")
    seqs = [(c["g"], c["tok"], c["parent"]) for c in cases]
    g, tok, par, pos_off, node_off = _pack(seqs)
    n, bonus, last, path, rc = o.verify_tree(g, tok, par, node_off, pos_off, path_stride=8)
    assert rc == 0
    for b, c in enumerate(cases):
        e = c["expect"]
        assert n[b] == e["n"], (c["name"], n[b])
        assert bonus[b] == e["bonus"] and last[b] - pos_off[b] == e["last"], c["name"]
        assert [x for x in path[b] if x >= 0] == e["path"], (c["name"], path[b])


def _brute_tree(g, tok, parent):
    """Walk every node up to the root and require every hop to match."""
    N = len(tok)

    def depth(i):
        return 0 if i < 0 else 1 + depth(parent[i])

    def row(i):
        return 0 if i < 0 else i + 1

    acc_nodes = []
    for i in range(N):
        ok, j = True, i
        while j >= 0:
            if tok[j] != g[row(parent[j])]:
                ok = False
                break
            j = parent[j]
        if ok:
            acc_nodes.append(i)
    if not acc_nodes:
        return 0, 0, []
    best = min(acc_nodes, key=lambda i: (-depth(i), i))
    path, j = [], best
    while j >= 0:
        path.append(j)
        j = parent[j]
    return depth(best), best + 1, path[::-1]


def check_tree_bruteforce(o, max_nodes=6):
    """Every parent array with parent[i] in [-1, i) up to ``max_nodes`` nodes,
    tokens and target choices over a 2-letter alphabet."""
    rng = np.random.default_rng(3)
    seqs, expect = [], []
    for N in range(0, max_nodes + 1):
        for parent in itertools.product(*[range(-1, i) for i in range(N)]):
            for _ in range(2):
                tok = rng.integers(0, 2, N).tolist()
                g = rng.integers(0, 2, N + 1).tolist()
                seqs.append((g, tok, list(parent)))
                expect.append(_brute_tree(g, tok, list(parent)))
    g, tok, par, pos_off, node_off = _pack(seqs)
    n, bonus, last, path, rc = o.verify_tree(g, tok, par, node_off, pos_off, path_stride=max_nodes)
    assert rc == 0
    for b, (en, elast, epath) in enumerate(expect):
        assert n[b] == en and last[b] - pos_off[b] == elast, (b, seqs[b], n[b], en)
        assert bonus[b] == seqs[b][0][elast]
        assert [x for x in path[b] if x >= 0] == epath


def check_chain_is_linear_tree(o):
    rng = np.random.default_rng(4)
    seqs = []
    for _ in range(200):
        K = int(rng.integers(0, 17))
        g = rng.integers(0, 3, K + 1).tolist()
        draft = rng.integers(0, 3, K).tolist()
        seqs.append((g, draft, list(range(-1, K - 1))))
    g, tok, par, pos_off, node_off = _pack(seqs)
    c = o.verify_chain(g, tok, pos_off, node_off, path_stride=16)
    t = o.verify_tree(g, tok, par, node_off, pos_off, path_stride=16)
    for a, b in zip(c[:4], t[:4]):
        assert np.array_equal(a, b)


def check_tree_bad_parent(o):
    seqs = [([1, 2, 3], [1, 2], [-1, 1]), ([5, 6], [5], [-1]), ([1, 2], [1], [-2])]
    g, tok, par, pos_off, node_off = _pack(seqs)
    n, bonus, last, path, rc = o.verify_tree(g, tok, par, node_off, pos_off, path_stride=2)
    assert rc == 2
    assert n[0] == bonus[0] == last[0] == -1 and n[2] == -1
    assert n[1] == 1 and bonus[1] == 6


# ---------------------------------------------------------------- router
PHI_1 = 0.8413447460685429     # standard normal CDF at 1 (textbook table value)
PHI_3 = 0.9986501019683699     # ... at 3


def check_gelu_values(o):
    assert o.gelu(0.0) == 0.0
    assert abs(o.gelu(1.0) - PHI_1) < 1e-15
    assert abs(o.gelu(-1.0) - (-(1.0 - PHI_1))) < 1e-15
    assert abs(o.gelu(3.0) - 3.0 * PHI_3) < 1e-14
    assert o.gelu(10.0) == 10.0
    assert -1e-20 < o.gelu(-10.0) <= 0.0


def _router_numpy(h_bits, W1, b1, w2, b2):
    z = W1.astype(np.float64) @ _f64(h_bits).T + b1.astype(np.float64)[:, None]
    a = 0.5 * z * (1.0 + erf(z / np.sqrt(2.0)))
    return b2 + w2.astype(np.float64) @ a


def check_router_closed_forms(o):
    rng = np.random.default_rng(5)
    d, m, B = 24, 10, 4
    h = _rand_bf16(rng, (B, d), 1.0)
    rows = np.arange(B, dtype=np.int32)
    b1 = rng.standard_normal(m).astype(np.float32)
    w2 = rng.standard_normal(m).astype(np.float32)
    b2 = 0.375
    # W1 = 0: delta = b2 + sum_j w2_j * GELU(b1_j), independent of h
    delta, _ = o.router(h, rows, np.zeros((m, d), np.float32), b1, w2, b2, 0.0)
    want = b2 + sum(float(w2[j]) * 0.5 * float(b1[j]) * (1.0 + math.erf(float(b1[j]) / math.sqrt(2.0)))
                    for j in range(m))
    assert np.allclose(delta, want, rtol=0, atol=1e-13)
    # one unit far on the linear side of GELU: delta = b2 + w2 * (b1 + c * h[k])
    k, c = 5, 0.75
    W1 = np.zeros((1, d), np.float32)
    W1[0, k] = c
    delta, _ = o.router(h, rows, W1, np.array([20.0], np.float32), np.array([-0.5], np.float32), b2, 0.0)
    want = b2 - 0.5 * (20.0 + c * _f64(h)[:, k])
    assert np.allclose(delta, want, rtol=0, atol=1e-12)
    # random weights against numpy / scipy
    W1 = (rng.standard_normal((m, d)) * 0.3).astype(np.float32)
    delta, _ = o.router(h, rows[::-1].copy(), W1, b1, w2, b2, 0.0)
    want = _router_numpy(h[::-1], W1, b1, w2, b2)
    assert np.allclose(delta, want, rtol=1e-12, atol=1e-12)


def check_route_strict(o):
    """route = 1 only when the prediction strictly exceeds tau; tau -> -inf / +inf
    gives all-EAGLE-3 / all-DFlash (the standalone drafters)."""
    d, m = 8, 3
    h = np.zeros((2, d), np.uint16)
    rows = np.array([0, 1], np.int32)
    W1 = np.zeros((m, d), np.float32)
    z = np.zeros(m, np.float32)
    b2 = 1.25
    _, r = o.router(h, rows, W1, z, z, b2, 1.25)
    assert list(r) == [0, 0]
    _, r = o.router(h, rows, W1, z, z, b2, 1.2499999)
    assert list(r) == [1, 1]
    rng = np.random.default_rng(6)
    hh = _rand_bf16(rng, (2, d), 1.0)
    W1 = rng.standard_normal((m, d)).astype(np.float32)
    w2 = rng.standard_normal(m).astype(np.float32)
    assert list(o.router(hh, rows, W1, z, w2, 0.0, -math.inf)[1]) == [1, 1]
    assert list(o.router(hh, rows, W1, z, w2, 0.0, math.inf)[1]) == [0, 0]


def router_param_count(d, m):
    return d * m + m + m + 1


def check_router_param_table():
    """m = d/8 with both biases reproduces the sizes printed in Table 6."""
    with open(os.path.join(GOLDEN, "router_param_counts.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for name, d, printed in rows:
        n = router_param_count(int(d), int(d) // 8)
        assert round(n / 1e6, 2) == float(printed), (name, n)


# ---------------------------------------------------------------- draft head
def check_topk_bruteforce(o):
    rng = np.random.default_rng(7)
    for B, d, Vd, k in [(1, 16, 40, 10), (3, 24, 100, 5), (2, 8, 10, 10), (2, 32, 257, 1)]:
        x = _rand_bf16(rng, (B, d), 1.0)
        Wd = _rand_bf16(rng, (Vd, d), 0.3)
        d2t = rng.permutation(10 * Vd)[:Vd].astype(np.int32)
        L = _f64(x) @ _f64(Wd).T
        dids, tids, vals, lse, mg = o.draft_topk(x, Wd, d2t, k)
        for b in range(B):
            order = np.lexsort((np.arange(Vd), -L[b]))
            assert list(dids[b]) == list(order[:k])
            assert list(tids[b]) == list(d2t[order[:k]])
            assert np.allclose(vals[b], L[b, order[:k]], rtol=1e-12, atol=1e-12)
            assert abs(lse[b] - logsumexp(L[b])) < 1e-10
            srt = L[b, order]
            want = min(srt[j] - srt[j + 1] for j in range(min(k, Vd - 1))) if Vd > 1 else math.inf
            assert abs(mg[b] - want) < 1e-10


def check_topk_ties(o):
    """Equal logits keep the lower draft id first."""
    rng = np.random.default_rng(8)
    d, Vd = 8, 12
    x = _rand_bf16(rng, (1, d), 1.0)
    Wd = _rand_bf16(rng, (Vd, d), 0.01)
    Wd[9] = to_bf16_bits(np.sign(bf16_bits_to_f32(x[0]) + 1e-3) * np.float32(2.0))
    Wd[2] = Wd[9]
    d2t = np.arange(Vd, dtype=np.int32)
    dids, _, vals, _, mg = o.draft_topk(x, Wd, d2t, 3)
    assert list(dids[0][:2]) == [2, 9] and vals[0][0] == vals[0][1] and mg[0] == 0.0


# ---------------------------------------------------------------- entropy router
def check_entropy(o):
    """H = -sum p log p of softmax(<h, W_v>): closed forms and scipy."""
    from scipy.stats import entropy as sp_entropy
    from scipy.special import softmax
    rng = np.random.default_rng(9)
    d, V = 16, 50
    h = _rand_bf16(rng, (3, d), 1.0)
    rows = np.array([0, 1, 2], np.int32)
    # all logits equal: the uniform distribution, H = log V exactly (up to rounding)
    H, _ = o.entropy(h, rows, np.zeros((V, d), np.uint16))
    assert np.allclose(H, math.log(V), rtol=0, atol=1e-12)
    # two identical rows far above the rest: H -> log 2
    hp = to_bf16_bits(np.abs(rng.standard_normal((2, d))).astype(np.float32) + np.float32(0.5))
    W = _rand_bf16(rng, (V, d), 0.01)
    W[4] = to_bf16_bits(np.full(d, 8.0, np.float32))
    W[30] = W[4]
    H, _ = o.entropy(hp, np.array([0, 1], np.int32), W)
    assert np.allclose(H, math.log(2.0), atol=1e-9)
    # random weights against scipy
    W = _rand_bf16(rng, (V, d), 0.5)
    L = _f64(h) @ _f64(W).T
    H, _ = o.entropy(h, rows[::-1].copy(), W)
    want = [sp_entropy(softmax(L[r])) for r in rows[::-1]]
    assert np.allclose(H, want, rtol=1e-12, atol=1e-12)
    # softmax is shift invariant: adding 800 to every logit (exp(800) overflows
    # a double) must leave H unchanged
    hs, Ws = h.copy(), W.copy()
    hs[:, -1] = to_bf16_bits(np.array([1.0], np.float32))[0]
    Ws[:, -1] = to_bf16_bits(np.array([800.0], np.float32))[0]
    Ls = _f64(hs) @ _f64(Ws).T
    assert Ls.min() > 700
    H, _ = o.entropy(hs, rows, Ws)
    assert np.all(np.isfinite(H))
    assert np.allclose(H, [sp_entropy(softmax(Ls[r] - 800.0)) for r in rows], rtol=1e-9, atol=1e-9)


def check_entropy_route_strict(o):
    d, V = 8, 16
    h = np.zeros((1, d), np.uint16)
    W = np.zeros((V, d), np.uint16)
    logV = math.log(V)
    _, r = o.entropy(h, np.array([0], np.int32), W, tau=logV)
    assert list(r) == [0]
    _, r = o.entropy(h, np.array([0], np.int32), W, tau=logV - 1e-6)
    assert list(r) == [1]


# ---------------------------------------------------------------- kept rows
def check_accepted_rows(o):
    """Hand-worked: the golden trees' accepted paths map to their rows, in order,
    root first; offsets count n_accept + 1 per sequence."""
    cases = read_cases("trees.txt")
    seqs = [(c["g"], c["tok"], c["parent"]) for c in cases]
    g, tok, par, pos_off, node_off = _pack(seqs)
    n, _, last, path, _ = o.verify_tree(g, tok, par, node_off, pos_off, path_stride=4)
    acc_rows, acc_off = o.accepted_rows(n, path, pos_off)
    for b, c in enumerate(cases):
        e = c["expect"]
        want = [int(pos_off[b])] + [int(pos_off[b]) + 1 + x for x in e["path"]]
        got = [int(x) for x in acc_rows[b] if x >= 0]
        assert got == want, (c["name"], got, want)
        assert acc_rows[b][-1 if len(want) <= 4 else 0] == (-1 if len(want) <= 4 else want[0])
        assert acc_off[b + 1] - acc_off[b] == e["n"] + 1
        assert got[-1] == last[b]        # the last kept row is the last accepted row
    assert acc_off[0] == 0


# ---------------------------------------------------------------- draft-tree construction
def _tree_by_beam(tid, lp, N):
    """The same construction written as an explicit beam search over Python
    lists (scores in numpy float32, added in the same order)."""
    D, k = tid.shape[0], tid.shape[1]
    pool = []                                   # (score, creation index, parent, token, depth)
    frontier = [None]                           # the root
    for t in range(D):
        created = []
        for j, par in enumerate(frontier if t else [None]):
            for c in range(k):
                base = np.float32(0.0) if par is None else pool[par][0]
                created.append((np.float32(base + np.float32(lp[t, j, c])), len(pool) + len(created), par,
                                int(tid[t, j, c]), t + 1))
        pool += created
        frontier = [e[1] for e in sorted(created, key=lambda e: (-float(e[0]), e[1]))[:k]]
    best = sorted(pool, key=lambda e: (-float(e[0]), e[1]))[:N]
    order = sorted(best, key=lambda e: e[4])    # stable: keeps score order within a depth
    new_of = {e[1]: i for i, e in enumerate(order)}
    return ([-1 if e[2] is None else new_of[e[2]] for e in order], [e[3] for e in order],
            [float(e[0]) for e in order], [e[4] for e in order])


def check_build_tree(o):
    c = read_cases("tree_build.txt")[0]
    D, k, N = c["D"][0], c["k"][0], c["N"][0]
    tid = np.array(c["tid"], np.int32).reshape(1, D, k, k)
    lp = np.array(c["lp"], np.float32).reshape(1, D, k, k)
    parent, token, score, depth, rc = o.build_tree(tid, lp, N)
    assert rc == 0
    assert list(parent[0]) == c["expect_parent"] and list(token[0]) == c["expect_token"]
    assert list(depth[0]) == c["expect_depth"]
    rng = np.random.default_rng(10)
    for D, k, N in [(8, 10, 60), (3, 4, 20), (5, 2, 9), (1, 6, 6)]:
        B = 3
        tid = rng.integers(0, 1000, (B, D, k, k)).astype(np.int32)
        lp = np.log(rng.dirichlet(np.ones(k) * 0.7, (B, D, k))).astype(np.float32)
        parent, token, score, depth, rc = o.build_tree(tid, lp, N)
        assert rc == 0
        for b in range(B):
            wp, wt, ws, wd = _tree_by_beam(tid[b], lp[b], N)
            assert list(parent[b]) == wp and list(token[b]) == wt and list(depth[b]) == wd
            assert np.array_equal(score[b], np.array(ws, np.float32))
            assert all(parent[b][i] < i for i in range(N))          # listed depth by depth
    # equal scores everywhere: the earlier-created node wins every tie
    tid = np.arange(3 * 2 * 2, dtype=np.int32).reshape(1, 3, 2, 2)
    lp = np.full((1, 3, 2, 2), -0.5, np.float32)
    parent, token, _, depth, rc = o.build_tree(tid, lp, 5)
    wp, wt, _, wd = _tree_by_beam(tid[0], lp[0], 5)
    assert rc == 0 and list(parent[0]) == wp and list(token[0]) == wt and list(depth[0]) == wd
    assert list(token[0]) == [0, 1, 4, 5, 6]
    bad = np.zeros((1, 2, 2, 2), np.float32)
    bad[0, 1, 0, 1] = 0.5                                           # a log-probability above 0
    assert o.build_tree(np.zeros((1, 2, 2, 2), np.int32), bad, 3)[4] == 2


# ---------------------------------------------------------------- KV-only catch-up
def check_rmsnorm(o):
    """Hand-worked: u = (3, 4, 0, 0), unit gain, eps = 0 -> rms 2.5 -> (1.2, 1.6, 0, 0).
    Constant input c: every element is gamma_i * c / sqrt(c^2 + eps) (eps inside the root);
    with eps = 0 the result does not change when u doubles."""
    one = to_bf16_bits(np.ones(4, np.float32))
    a = o.rmsnorm(to_bf16_bits(np.array([3, 4, 0, 0], np.float32)), one, 0.0)
    assert np.allclose(a, [1.2, 1.6, 0.0, 0.0], rtol=1e-15, atol=0)
    rng = np.random.default_rng(40)
    gamma = _rand_bf16(rng, 16, 1.0)
    for c, eps in ((1.5, 0.0), (-0.375, 1e-6), (0.0078125, 0.25)):
        a = o.rmsnorm(to_bf16_bits(np.full(16, c, np.float32)), gamma, eps)
        assert np.allclose(a, _f64(gamma) * c / math.sqrt(c * c + eps), rtol=1e-14, atol=0)
    u = _rand_bf16(rng, 16, 1.0)
    assert np.allclose(o.rmsnorm(u, gamma, 0.0), o.rmsnorm(to_bf16_bits(_f64(u) * 2), gamma, 0.0), rtol=1e-14)


def check_rope(o):
    """Basis vectors: with theta = 10^4 and D = 8 the pair frequencies are 1, 10^-1,
    10^-2, 10^-3, so e_0 at position p turns to (cos p) e_0 + (sin p) e_4 and e_2 at
    p = 100 to (cos 1) e_2 + (sin 1) e_6.  Position 0 is the identity; turning by a
    then b is turning by a + b; scores depend only on the distance of the positions."""
    th, D = 1e4, 8
    for p in (0.0, 1.0, 2.5, 1000.0):
        y = o.rope(np.eye(D)[0], p, th)
        assert np.allclose(y, np.cos(p) * np.eye(D)[0] + np.sin(p) * np.eye(D)[4], atol=1e-13)
    y = o.rope(np.eye(D)[2], 100.0, th)
    assert np.allclose(y, np.cos(1.0) * np.eye(D)[2] + np.sin(1.0) * np.eye(D)[6], atol=1e-12)
    y = o.rope(np.eye(D)[7], 5000.0, th)       # frequency 10^-3: angle 5, second member of the pair
    assert np.allclose(y, np.cos(5.0) * np.eye(D)[7] - np.sin(5.0) * np.eye(D)[3], atol=1e-12)
    rng = np.random.default_rng(41)
    x, k = rng.standard_normal(D), rng.standard_normal(D)
    assert np.allclose(o.rope(x, 0.0, th), x, atol=0)
    assert np.allclose(o.rope(o.rope(x, 3.0, th), 11.0, th), o.rope(x, 14.0, th), atol=1e-12)
    for m, n in ((5, 2), (40, 33), (7, 7)):
        assert np.isclose(o.rope(x, m, th) @ o.rope(k, n, th), o.rope(x, m - n, th) @ k, atol=1e-12)


def catchup_case(seed, din=16, H=4, G=2, D=4, n=(3, 1), L=(2, 0), cap=8, theta=1e4, eps=1e-6):
    """A small random catch-up problem (weights ~N(0, 1/din), inputs ~N(0, 1))."""
    rng = np.random.default_rng(seed)
    B = len(n)
    bl_off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    c = dict(u=_rand_bf16(rng, (int(bl_off[-1]), din), 1.0), bl_off=bl_off, cache_len=np.array(L, np.int32),
             gamma=to_bf16_bits((1.0 + 0.1 * rng.standard_normal(din)).astype(np.float32)), eps=eps, theta=theta,
             Wq=_rand_bf16(rng, (H * D, din), din ** -0.5), Wk=_rand_bf16(rng, (G * D, din), din ** -0.5),
             Wv=_rand_bf16(rng, (G * D, din), din ** -0.5), Wo=_rand_bf16(rng, (din, H * D), (H * D) ** -0.5),
             Kc=_rand_bf16(rng, (B, cap, G * D), 1.0), Vc=_rand_bf16(rng, (B, cap, G * D), 1.0), H=H, G=G)
    return c


def check_catchup_single_entry(o):
    """An empty cache and one backlog token: every head attends to that token alone,
    so its output is the token's own cached value; with Wo = 0 the output is the input."""
    c = catchup_case(42, n=(1,), L=(0,))
    c["Wo"] = np.zeros_like(c["Wo"])
    r, rc = o.catchup(**c)
    assert rc == 0
    D = c["Wk"].shape[0] // c["G"]
    for h in range(c["H"]):
        g = h // (c["H"] // c["G"])
        assert np.allclose(r["attn"][0, h * D:(h + 1) * D], _f64(r["Vc"][0, 0, g * D:(g + 1) * D]), atol=1e-15)
    assert np.array_equal(r["out"][0], _f64(c["u"][0]))


def check_catchup_two_entries(o):
    """Two cache rows (one cached, one new): each head's output is the logistic mix
    s(x) v0 + s(-x) v1 with x = (<q, k0> - <q, k1>) / 2 (D = 4, so sqrt D = 2);
    identical keys give the mean of the two values."""
    c = catchup_case(43, n=(1,), L=(1,), H=2, G=1)
    r, rc = o.catchup(**c)
    assert rc == 0
    D = 4
    k = _f64(r["Kc"][0, :2]).reshape(2, 1, D)
    v = _f64(r["Vc"][0, :2]).reshape(2, 1, D)
    for h in range(2):
        q = r["q"][0, h * D:(h + 1) * D]
        x = (q @ k[0, 0] - q @ k[1, 0]) / 2.0
        w0 = 1.0 / (1.0 + math.exp(-x))
        assert np.allclose(r["attn"][0, h * D:(h + 1) * D], w0 * v[0, 0] + (1 - w0) * v[1, 0], atol=1e-12)
    c2 = catchup_case(44, n=(1,), L=(1,), H=2, G=1)
    # a zero key projection and a zero cached key: every score is 0, equal weights
    c2["Wk"] = np.zeros_like(c2["Wk"])
    c2["Kc"] = np.zeros_like(c2["Kc"])
    r, rc = o.catchup(**c2)
    mean = (_f64(r["Vc"][0, 0]) + _f64(r["Vc"][0, 1])) / 2
    assert np.allclose(r["attn"][0, :D], mean, atol=1e-14) and np.allclose(r["attn"][0, D:], mean, atol=1e-14)


def check_catchup_head_groups(o):
    """8 query heads over 2 KV heads: heads 0-3 read KV head 0, heads 4-7 KV head 1.
    A KV head whose values are all zero silences exactly its own group."""
    c = catchup_case(45, H=8, G=2, D=4, n=(2,), L=(3,))
    D = 4
    c["Vc"][:, :, D:] = 0
    c["Wv"][D:] = 0
    r, rc = o.catchup(**c)
    assert rc == 0
    assert np.all(r["attn"][0, 4 * D:] == 0) and np.all(np.abs(r["attn"][0, :4 * D]).max() > 0)


def check_catchup_lazy_equals_eager(o):
    """Lazy catch-up leaves the result unchanged (paper Sec. 4, Table 3: the accepted
    tokens are identical): entering the backlog in one batch gives the same caches and
    final output as entering it one token at a time.  Rows outside the backlog are
    untouched."""
    c = catchup_case(46, n=(3, 1, 4), L=(2, 0, 1), cap=6)
    batch, rc = o.catchup(**c)
    assert rc == 0
    Kc, Vc = c["Kc"].copy(), c["Vc"].copy()
    L = c["cache_len"].copy()
    out_last = {}
    for b in range(3):
        for j in range(int(c["bl_off"][b]), int(c["bl_off"][b + 1])):
            one = dict(c, u=c["u"][j:j + 1], bl_off=np.array([0, 1], np.int32), cache_len=L[b:b + 1],
                       Kc=Kc[b:b + 1], Vc=Vc[b:b + 1])
            r, rc = o.catchup(**one)
            assert rc == 0
            Kc[b], Vc[b] = r["Kc"][0], r["Vc"][0]
            L[b] += 1
            out_last[b] = r["out"][0]
    assert np.array_equal(Kc, batch["Kc"]) and np.array_equal(Vc, batch["Vc"])
    for b in range(3):
        assert np.allclose(out_last[b], batch["out"][b], rtol=0, atol=1e-13)
        end = int(c["cache_len"][b] + c["bl_off"][b + 1] - c["bl_off"][b])
        assert np.array_equal(batch["Kc"][b, :c["cache_len"][b]], c["Kc"][b, :c["cache_len"][b]])
        assert np.array_equal(batch["Kc"][b, end:], c["Kc"][b, end:])


def check_catchup_final_query(o):
    """With Wq = Wk and one query head per KV head, the final token's rotated query,
    rounded to bf16, is the key it wrote at its own position L + n - 1.  Identity
    value weights (G D = din) cache the normalised input itself."""
    c = catchup_case(47, din=8, H=2, G=2, D=4, n=(3, 2), L=(1, 4), cap=8)
    c["Wq"] = c["Wk"].copy()
    c["Wv"] = to_bf16_bits(np.eye(8, dtype=np.float32))
    r, rc = o.catchup(**c)
    assert rc == 0
    for b, (L, n) in enumerate(((1, 3), (4, 2))):
        assert np.array_equal(to_bf16_bits(r["q"][b].astype(np.float32)), r["Kc"][b, L + n - 1])
        f = int(c["bl_off"][b + 1]) - 1
        a = o.rmsnorm(c["u"][f], c["gamma"], c["eps"])
        assert np.array_equal(r["Vc"][b, L + n - 1], to_bf16_bits(a.astype(np.float32)))


def check_catchup_output_projection(o):
    """Wo maps the attention output (H D wide) to the layer width din, out x in: with a
    single unit weight at (row 0, column 5) the output is the input plus attn[5] in
    element 0, and the input unchanged everywhere else."""
    c = catchup_case(49, din=16, H=4, G=2, D=4, n=(2,), L=(1,))
    Wo = np.zeros((16, 16), np.float32)
    Wo[0, 5] = 1.0
    c["Wo"] = to_bf16_bits(Wo)
    r, rc = o.catchup(**c)
    assert rc == 0
    u = _f64(c["u"][1])
    assert r["out"][0, 0] == u[0] + r["attn"][0, 5]
    assert np.array_equal(r["out"][0, 1:], u[1:])


def check_catchup_rejects_overflow(o):
    """A backlog that does not fit the cache, or an empty one, is refused."""
    c = catchup_case(48, n=(3,), L=(6,), cap=8)
    assert o.catchup(**c)[1] == 2
    c = catchup_case(48, n=(0, 2), L=(0, 0), cap=8)
    assert o.catchup(**c)[1] == 2


ALL_CHECKS = [check_argmax_bruteforce, check_argmax_ties, check_argmax_closed_form, check_chain_golden,
              check_tree_golden, check_tree_bruteforce, check_chain_is_linear_tree, check_tree_bad_parent,
              check_gelu_values, check_router_closed_forms, check_route_strict, check_topk_bruteforce,
              check_topk_ties, check_entropy, check_entropy_route_strict, check_accepted_rows,
              check_build_tree, check_rmsnorm, check_rope, check_catchup_single_entry, check_catchup_two_entries,
              check_catchup_head_groups, check_catchup_lazy_equals_eager, check_catchup_final_query,
              check_catchup_output_projection, check_catchup_rejects_overflow]
