"""Seeded synthetic workloads for the WhiFlash verify-and-route round.

This module draws random inputs and builds their structure (draft trees,
DFlash blocks, matched-prefix cuts, the draft-to-target id map).  It holds
none of the round's arithmetic: wherever a drafted token has to agree with
the target's greedy choice, the caller hands in a function that returns the
target argmax (and, for the input-rejection rules, the top-2 logit gap, the
router output and the draft-head top-k gaps).  The tests pass the CPU oracle
there; the benchmark passes the library's own LM-head kernel, whose output
only shapes the benchmark input and is never used as an expected value.

Shapes and distributions follow the WhiFlash paper (arXiv 2606.07710):
hidden size 2560 and target vocabulary 151,936 for Qwen3-4B, a 32,000-id
EAGLE-3 draft vocabulary (Qwen3-4B-EAGLE3 model card, "Technical
Specifications"), EAGLE-3 trees of depth 8 / top-k 10 / 60 draft tokens and
DFlash blocks of 16 (paper App. A, "Drafter Hyperparameters", Table 7).

Every random stream is derived from ``numpy.random.SeedSequence`` keyed by the
workload seed plus a fixed tag, so each tensor is reproducible on its own and
independent of how many threads draw it.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Optional

import numpy as np

BASE_SEED = 20261202

# Stream tags (second word of every SeedSequence entropy tuple).
_T_W, _T_HID, _T_HID_RS, _T_STRUCT, _T_TOK, _T_ROUTER, _T_WD, _T_X, _T_X_RS, _T_D2T = range(10)

GAP_MIN = 1e-2        # minimum top-2 logit gap, adjacent top-(k+1) gap and router margin


# --------------------------------------------------------------------------- bf16
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 bits to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, *words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *words])))


def normal_bf16(seed: int, tag: int, rows: int, cols: int, std: float,
                chunk_rows: int = 1024, threads: int = 8) -> np.ndarray:
    """[rows, cols] bf16 bits drawn ~N(0, std^2) in fp32 then rounded to bf16.

    Row block i (of ``chunk_rows`` rows) comes from its own stream, so the
    result does not depend on the thread count."""
    out = np.empty((rows, cols), dtype=np.uint16)

    def fill(i: int) -> None:
        r0, r1 = i * chunk_rows, min(rows, (i + 1) * chunk_rows)
        x = _rng(seed, tag, i).standard_normal((r1 - r0, cols), dtype=np.float32)
        x *= np.float32(std)
        out[r0:r1] = to_bf16_bits(x)

    nblk = (rows + chunk_rows - 1) // chunk_rows
    if nblk <= 1:
        for i in range(nblk):
            fill(i)
    else:
        with ThreadPoolExecutor(min(threads, nblk)) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def hidden_row(seed: int, row: int, attempt: int, d: int, tag: int = _T_HID_RS) -> np.ndarray:
    """One resampled hidden row (bf16 bits), ~N(0, 1), for the rejection rules."""
    x = _rng(seed, tag, row, attempt).standard_normal(d, dtype=np.float32)
    return to_bf16_bits(x)


# --------------------------------------------------------------------------- configs
@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    d: int
    V: int
    B: int
    kind: str            # "chain", "tree" or "mixed"
    m: int               # router width
    cut: str             # "uniform16" (U{0..16}), "geom" (min(Geom0(0.25),16)) ; trees use U{0..8}
    draft_head: bool
    K: int = 16          # DFlash block size
    n_nodes: int = 60    # EAGLE-3 draft tokens
    depth: int = 8       # EAGLE-3 tree depth
    branch: int = 10     # EAGLE-3 top-k (max children per node)
    Vd: int = 32000
    topk: int = 10
    w_std: float = 0.02
    r_std: float = 0.05
    tau: float = 1.0


CONFIGS = [
    Config("tiny_chain_b1", d=256, V=8192, B=1, kind="chain", m=128, cut="uniform16", draft_head=False),
    Config("qwen3_4b_dflash_chain_b1", d=2560, V=151936, B=1, kind="chain", m=1024, cut="geom", draft_head=False),
    Config("qwen3_4b_eagle3_tree_b1", d=2560, V=151936, B=1, kind="tree", m=1024, cut="tree", draft_head=True),
    Config("qwen3_4b_mixed_b32", d=2560, V=151936, B=32, kind="mixed", m=1024, cut="geom", draft_head=False),
    Config("qwen3_4b_tree_b256", d=2560, V=151936, B=256, kind="tree", m=1024, cut="tree", draft_head=True),
]


def seed_of(index: int) -> int:
    return BASE_SEED + index


# --------------------------------------------------------------------------- structure
def random_tree(rng: np.random.Generator, n_nodes: int, depth: int, branch: int):
    """A random draft tree of exactly ``depth`` levels, <= ``branch`` children per node.

    Returns (parent, node_depth) with nodes relabelled breadth-first so that
    parent[i] < i; parent -1 means the root (the last committed token)."""
    assert n_nodes >= depth
    par = [-1]                       # creation order; the spine first
    dep = [1]
    for j in range(1, depth):
        par.append(j - 1)
        dep.append(j + 1)
    nchild = {-1: 1}
    for j in range(depth - 1):
        nchild[j] = 1
    while len(par) < n_nodes:
        cands = [-1] + [i for i in range(len(par)) if dep[i] < depth]
        cands = [c for c in cands if nchild.get(c, 0) < branch]
        p = int(cands[rng.integers(len(cands))])
        nchild[p] = nchild.get(p, 0) + 1
        par.append(p)
        dep.append(1 if p < 0 else dep[p] + 1)
    # breadth-first relabel: sort by (depth, random key)
    key = rng.random(n_nodes)
    order = sorted(range(n_nodes), key=lambda i: (dep[i], key[i]))
    new_of = {old: new for new, old in enumerate(order)}
    parent = np.array([-1 if par[o] < 0 else new_of[par[o]] for o in order], dtype=np.int32)
    node_depth = np.array([dep[o] for o in order], dtype=np.int32)
    assert all(parent[i] < i for i in range(n_nodes))
    return parent, node_depth


def _draw_token_not(rng: np.random.Generator, V: int, banned: set) -> int:
    while True:
        t = int(rng.integers(V))
        if t not in banned:
            return t


# --------------------------------------------------------------------------- workload
@dataclasses.dataclass
class Workload:
    cfg: Config
    seed: int
    hidden: np.ndarray     # [P, d] bf16 bits
    W: np.ndarray          # [V, d] bf16 bits
    pos_off: np.ndarray    # [B+1] int32
    node_off: np.ndarray   # [B+1] int32
    kind: np.ndarray       # [B] int32, 0 DFlash chain, 1 EAGLE-3 tree
    tok: np.ndarray        # [N] int32 drafted target-vocabulary ids
    parent: np.ndarray     # [N] int32 sequence-local parent (-1 = root)
    W1: np.ndarray         # [m, d] f32
    b1: np.ndarray         # [m] f32
    w2: np.ndarray         # [m] f32
    b2: float
    tau: float
    cut: np.ndarray        # [B] planted matched depth (the expected n_accept where planted)
    planted: np.ndarray    # [B] bool: sequence planted from the supplied target argmax
    max_depth: int
    Wd: Optional[np.ndarray] = None   # [Vd, d] bf16 bits
    x: Optional[np.ndarray] = None    # [B, d] bf16 bits (drafter hidden state)
    d2t: Optional[np.ndarray] = None  # [Vd] int32
    topk: int = 0
    path_nodes: list = dataclasses.field(default_factory=list)  # per sequence: planted root path (tree)
    # rejection record: final resample attempt of each resampled hidden row / drafter row
    hidden_attempts: dict = dataclasses.field(default_factory=dict)
    x_attempts: dict = dataclasses.field(default_factory=dict)

    @property
    def P(self) -> int:
        return int(self.pos_off[-1])

    @property
    def B(self) -> int:
        return len(self.kind)

    def expected_last_pos(self, b: int) -> int:
        """Global row of the deepest planted match (valid where planted)."""
        root = int(self.pos_off[b])
        c = int(self.cut[b])
        if c == 0:
            return root
        if self.kind[b] == 0:
            return root + c
        return root + 1 + int(self.path_nodes[b][c - 1])


def _structure(cfg: Config, seed: int, B: int):
    rng = _rng(seed, _T_STRUCT)
    if cfg.kind == "chain":
        kinds = np.zeros(B, np.int32)
    elif cfg.kind == "tree":
        kinds = np.ones(B, np.int32)
    else:   # mixed: exactly half of each drafter, in random order
        kinds = np.array([0] * (B // 2) + [1] * (B - B // 2), np.int32)
        rng.shuffle(kinds)
    parents, paths, cuts = [], [], []
    for b in range(B):
        if kinds[b] == 0:
            parents.append(np.arange(-1, cfg.K - 1, dtype=np.int32))
            paths.append(list(range(cfg.K)))
            if cfg.cut == "uniform16":
                cuts.append(int(rng.integers(0, cfg.K + 1)))
            else:
                cuts.append(min(int(rng.geometric(0.25)) - 1, cfg.K))
        else:
            parent, ndep = random_tree(rng, cfg.n_nodes, cfg.depth, cfg.branch)
            leaves = np.nonzero(ndep == cfg.depth)[0]
            leaf = int(leaves[rng.integers(len(leaves))])
            path = []
            i = leaf
            while i >= 0:
                path.append(i)
                i = int(parent[i])
            path.reverse()
            parents.append(parent)
            paths.append(path)
            cuts.append(int(rng.integers(0, cfg.depth + 1)))
    rows = np.array([len(p) + 1 for p in parents], np.int64)
    pos_off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    node_off = np.concatenate([[0], np.cumsum(rows - 1)]).astype(np.int32)
    return kinds, parents, paths, np.array(cuts, np.int32), pos_off, node_off


def _plant(cfg: Config, V: int, rng: np.random.Generator, kind: int, parent: np.ndarray,
           path: list, cut: int, g_rows: Optional[np.ndarray]) -> np.ndarray:
    """Draft tokens of one sequence.  ``g_rows[r]`` is the target argmax at the
    sequence's row r (row 0 = root).  Nodes on the planted path up to ``cut``
    agree with the target; every other node disagrees with the target's choice
    at its parent's row, and siblings carry distinct tokens.  With ``g_rows``
    None the tokens are drawn uniformly (an unplanted sequence)."""
    n = len(parent)
    if g_rows is None:
        return rng.integers(0, V, size=n).astype(np.int32)
    tok = np.empty(n, np.int32)
    on_path = {node: depth for depth, node in enumerate(path, start=1)}
    used = {}
    for i in range(n):
        prow = 0 if parent[i] < 0 else int(parent[i]) + 1
        target = int(g_rows[prow])
        sib = used.setdefault(int(parent[i]), set())
        if kind == 0 and i > cut:
            t = int(rng.integers(V))          # past the first mismatch: unconstrained
        elif on_path.get(i, 10 ** 9) <= cut:
            t = target
        else:
            t = _draw_token_not(rng, V, sib | {target})
        sib.add(t)
        tok[i] = t
    return tok


# argmax_fn(W [V, d], h rows [n, d]) -> (ids [n], top-2 gap [n] or None)
ArgmaxFn = Callable[[np.ndarray, np.ndarray], tuple]
# router_fn(W1, b1, w2, b2, h rows [n, d]) -> delta_al [n]
RouterFn = Callable[..., np.ndarray]
# topk_gap_fn(Wd, k, x rows [n, d]) -> smallest adjacent gap among the top k+1 logits [n]
TopkGapFn = Callable[[np.ndarray, int, np.ndarray], np.ndarray]


def make_workload(index: int, argmax_fn: ArgmaxFn, router_fn: Optional[RouterFn] = None,
                  topk_gap_fn: Optional[TopkGapFn] = None, reject: bool = True,
                  plant_seqs: Optional[list] = None, B: Optional[int] = None,
                  m: Optional[int] = None, max_rounds: int = 64) -> Workload:
    """Build workload ``index`` (0-based position in ``CONFIGS``).

    argmax_fn: target argmax over rows of ``hidden`` (and the top-2 gap when
      ``reject``).  Only rows of planted sequences are passed to it.
    plant_seqs: sequences whose draft tokens are planted from the target
      argmax (default all); the rest carry uniform random tokens.
    reject: apply the rejection rules (top-2 gap, router margin, draft top-k
      gaps, all >= 1e-2) by resampling the offending hidden / drafter rows.
    B, m: override the batch size / router width (same distributions)."""
    cfg = CONFIGS[index]
    seed = seed_of(index)
    B = cfg.B if B is None else B
    m = cfg.m if m is None else m
    d, V = cfg.d, cfg.V
    kinds, parents, paths, cuts, pos_off, node_off = _structure(cfg, seed, B)
    P = int(pos_off[-1])
    W = normal_bf16(seed, _T_W, V, d, cfg.w_std)
    hidden = normal_bf16(seed, _T_HID, P, d, 1.0)
    rr = _rng(seed, _T_ROUTER)
    W1 = (rr.standard_normal((m, d), dtype=np.float32) * np.float32(cfg.r_std))
    b1 = (rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std))
    w2 = (rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std))
    b2 = float(np.float32(rr.standard_normal() * cfg.r_std))
    planted = np.zeros(B, bool)
    planted[list(range(B)) if plant_seqs is None else list(plant_seqs)] = True

    attempts = {}

    def resample(row: int) -> None:
        a = attempts.get(row, 0) + 1
        attempts[row] = a
        if a > max_rounds:
            raise RuntimeError(f"row {row}: rejection rule not met after {max_rounds} resamples")
        hidden[row] = hidden_row(seed, row, a, d)

    # target argmax at every row of the planted sequences, with the top-2 gap rule
    prow = np.concatenate([np.arange(pos_off[b], pos_off[b + 1]) for b in range(B) if planted[b]]) \
        if planted.any() else np.zeros(0, np.int64)
    g = np.full(P, -1, np.int64)

    def refresh(rows: np.ndarray) -> None:
        todo = np.asarray(rows, np.int64)
        while len(todo):
            ids, gap = argmax_fn(W, hidden[todo])
            g[todo] = ids
            if not reject or gap is None:
                return
            bad = todo[np.asarray(gap) < GAP_MIN]
            for r in bad:
                resample(int(r))
            todo = bad

    refresh(prow)
    tok_rng = _rng(seed, _T_TOK)
    toks = []
    for b in range(B):
        gr = g[pos_off[b]:pos_off[b + 1]] if planted[b] else None
        toks.append(_plant(cfg, V, tok_rng, int(kinds[b]), parents[b], paths[b], int(cuts[b]), gr))

    wl = Workload(cfg=cfg, seed=seed, hidden=hidden, W=W, pos_off=pos_off, node_off=node_off,
                  kind=kinds, tok=np.concatenate(toks).astype(np.int32),
                  parent=np.concatenate(parents).astype(np.int32), W1=W1, b1=b1, w2=w2, b2=b2,
                  tau=cfg.tau, cut=cuts, planted=planted,
                  max_depth=cfg.K if cfg.kind == "chain" else (cfg.depth if cfg.kind == "tree" else max(cfg.K, cfg.depth)),
                  path_nodes=paths)

    # router margin: resample the hidden row the router reads, then re-plant the sequence
    if reject and router_fn is not None:
        for _ in range(max_rounds):
            seqs = [b for b in range(B) if planted[b]]
            rows = np.array([wl.expected_last_pos(b) for b in seqs], np.int64)
            if not len(rows):
                break
            delta = np.asarray(router_fn(W1, b1, w2, b2, hidden[rows]))
            bad = [(b, int(r)) for b, r, dl in zip(seqs, rows, delta) if abs(float(dl) - wl.tau) < GAP_MIN]
            if not bad:
                break
            for b, r in bad:
                resample(r)
                refresh(np.array([r]))
                gr = g[pos_off[b]:pos_off[b + 1]]
                t = _plant(cfg, V, _rng(seed, _T_TOK, b, attempts[r]), int(kinds[b]), parents[b],
                           paths[b], int(cuts[b]), gr)
                wl.tok[node_off[b]:node_off[b + 1]] = t
        else:
            raise RuntimeError("router margin rule not met")

    if cfg.draft_head:
        wl.Wd = normal_bf16(seed, _T_WD, cfg.Vd, d, cfg.w_std)
        wl.x = normal_bf16(seed, _T_X, B, d, 1.0)
        wl.d2t = _rng(seed, _T_D2T).choice(V, size=cfg.Vd, replace=False).astype(np.int32)
        wl.topk = cfg.topk
        if reject and topk_gap_fn is not None:
            # only the planted sequences are compared against the oracle; with
            # ~N(0,1) logits over 32,000 ids a draw meets the rule ~8% of the time
            xa = {}
            todo = np.nonzero(planted)[0]
            for _ in range(max(max_rounds, 1000)):
                gaps = np.asarray(topk_gap_fn(wl.Wd, wl.topk, wl.x[todo]))
                bad = todo[gaps < GAP_MIN]
                if not len(bad):
                    break
                for b in bad:
                    xa[int(b)] = xa.get(int(b), 0) + 1
                    wl.x[b] = hidden_row(seed, int(b), xa[int(b)], d, tag=_T_X_RS)
                todo = bad
            else:
                raise RuntimeError("draft top-k gap rule not met")
            wl.x_attempts = dict(xa)
    wl.hidden_attempts = dict(attempts)
    return wl


def replay_workload(index: int, hidden_attempts: dict, x_attempts: dict, tok: np.ndarray,
                    m: Optional[int] = None) -> Workload:
    """Rebuild workload ``index`` as ``make_workload`` left it, from its record:
    the final resample attempt of each rejected hidden row and drafter row and
    the drafted tokens (which ``make_workload`` planted from the target argmax).
    Everything else is redrawn from the seed, so no argmax is needed here."""
    cfg = CONFIGS[index]
    seed = seed_of(index)
    B = cfg.B
    m = cfg.m if m is None else m
    d, V = cfg.d, cfg.V
    kinds, parents, paths, cuts, pos_off, node_off = _structure(cfg, seed, B)
    P = int(pos_off[-1])
    W = normal_bf16(seed, _T_W, V, d, cfg.w_std)
    hidden = normal_bf16(seed, _T_HID, P, d, 1.0)
    for row, a in hidden_attempts.items():
        hidden[int(row)] = hidden_row(seed, int(row), int(a), d)
    rr = _rng(seed, _T_ROUTER)
    W1 = (rr.standard_normal((m, d), dtype=np.float32) * np.float32(cfg.r_std))
    b1 = (rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std))
    w2 = (rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std))
    b2 = float(np.float32(rr.standard_normal() * cfg.r_std))
    tok = np.asarray(tok, np.int32)
    if len(tok) != int(node_off[-1]):
        raise ValueError(f"record holds {len(tok)} drafted tokens, the workload has {int(node_off[-1])}")
    wl = Workload(cfg=cfg, seed=seed, hidden=hidden, W=W, pos_off=pos_off, node_off=node_off,
                  kind=kinds, tok=tok.copy(), parent=np.concatenate(parents).astype(np.int32), W1=W1, b1=b1,
                  w2=w2, b2=b2, tau=cfg.tau, cut=cuts, planted=np.ones(B, bool),
                  max_depth=cfg.K if cfg.kind == "chain" else (cfg.depth if cfg.kind == "tree" else max(cfg.K, cfg.depth)),
                  path_nodes=paths, hidden_attempts={int(k): int(v) for k, v in hidden_attempts.items()},
                  x_attempts={int(k): int(v) for k, v in x_attempts.items()})
    if cfg.draft_head:
        wl.Wd = normal_bf16(seed, _T_WD, cfg.Vd, d, cfg.w_std)
        wl.x = normal_bf16(seed, _T_X, B, d, 1.0)
        for b, a in x_attempts.items():
            wl.x[int(b)] = hidden_row(seed, int(b), int(a), d, tag=_T_X_RS)
        wl.d2t = _rng(seed, _T_D2T).choice(V, size=cfg.Vd, replace=False).astype(np.int32)
        wl.topk = cfg.topk
    return wl


def workload_from_record(rec: dict, m: Optional[int] = None) -> Workload:
    """``replay_workload`` from a stored record: a dict with the workload index
    and an ``inputs`` entry holding ``hidden_attempts`` and ``x_attempts`` as
    [row, attempt] pairs and the drafted tokens ``tok``."""
    inp = rec["inputs"]
    return replay_workload(int(rec["index"]), {r: a for r, a in inp["hidden_attempts"]},
                           {b: a for b, a in inp["x_attempts"]}, np.array(inp["tok"], np.int32), m=m)


def small_workload(seed: int, d: int, V: int, kinds: list, argmax_fn: ArgmaxFn,
                   m: int = 32, K: int = 16, n_nodes: int = 60, depth: int = 8, branch: int = 10,
                   Vd: int = 0, topk: int = 0, router_fn: Optional[RouterFn] = None,
                   topk_gap_fn: Optional[TopkGapFn] = None, reject: bool = True) -> Workload:
    """A free-shaped workload for parity sweeps (same distributions as the configs).

    kinds: per sequence 0 (chain of K) or 1 (tree of n_nodes, depth ``depth``)."""
    # weights ~N(0, 1/d): logits of unit scale at any d, as at d = 2560 with std 0.02
    cfg = Config(f"custom_{seed}", d=d, V=V, B=len(kinds), kind="mixed", m=m, cut="uniform16",
                 draft_head=Vd > 0, K=K, n_nodes=n_nodes, depth=depth, branch=branch, Vd=max(Vd, 1),
                 topk=topk, w_std=float(d) ** -0.5)
    rng = _rng(seed, _T_STRUCT)
    parents, paths, cuts = [], [], []
    for k in kinds:
        if k == 0:
            parents.append(np.arange(-1, K - 1, dtype=np.int32))
            paths.append(list(range(K)))
            cuts.append(int(rng.integers(0, K + 1)))
        else:
            parent, ndep = random_tree(rng, n_nodes, depth, branch)
            leaves = np.nonzero(ndep == depth)[0]
            i = int(leaves[rng.integers(len(leaves))])
            path = []
            while i >= 0:
                path.append(i)
                i = int(parent[i])
            path.reverse()
            parents.append(parent)
            paths.append(path)
            cuts.append(int(rng.integers(0, depth + 1)))
    B = len(kinds)
    rows = np.array([len(p) + 1 for p in parents], np.int64)
    pos_off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    node_off = np.concatenate([[0], np.cumsum(rows - 1)]).astype(np.int32)
    P = int(pos_off[-1])
    W = normal_bf16(seed, _T_W, V, d, cfg.w_std)
    hidden = normal_bf16(seed, _T_HID, P, d, 1.0)
    attempts = {}
    todo = np.arange(P)
    g = np.full(P, -1, np.int64)
    for _ in range(256):
        ids, gap = argmax_fn(W, hidden[todo])
        g[todo] = ids
        if not reject or gap is None:
            break
        bad = todo[np.asarray(gap) < GAP_MIN]
        if not len(bad):
            break
        for r in bad:
            attempts[int(r)] = attempts.get(int(r), 0) + 1
            hidden[r] = hidden_row(seed, int(r), attempts[int(r)], d)
        todo = bad
    else:
        raise RuntimeError("top-2 gap rule not met")
    tok_rng = _rng(seed, _T_TOK)
    toks = [_plant(cfg, V, tok_rng, int(kinds[b]), parents[b], paths[b], cuts[b],
                   g[pos_off[b]:pos_off[b + 1]]) for b in range(B)]
    rr = _rng(seed, _T_ROUTER)
    W1 = rr.standard_normal((m, d), dtype=np.float32) * np.float32(cfg.r_std)
    b1 = rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std)
    w2 = rr.standard_normal(m, dtype=np.float32) * np.float32(cfg.r_std)
    b2 = float(np.float32(rr.standard_normal() * cfg.r_std))
    wl = Workload(cfg=cfg, seed=seed, hidden=hidden, W=W, pos_off=pos_off, node_off=node_off,
                  kind=np.array(kinds, np.int32), tok=np.concatenate(toks).astype(np.int32),
                  parent=np.concatenate(parents).astype(np.int32), W1=W1, b1=b1, w2=w2, b2=b2,
                  tau=cfg.tau, cut=np.array(cuts, np.int32), planted=np.ones(B, bool),
                  max_depth=max(K if 0 in kinds else 0, depth if 1 in kinds else 0), path_nodes=paths)
    if reject and router_fn is not None:
        for _ in range(256):
            rows = np.array([wl.expected_last_pos(b) for b in range(B)], np.int64)
            delta = np.asarray(router_fn(W1, b1, w2, b2, hidden[rows]))
            bad = [b for b in range(B) if abs(float(delta[b]) - wl.tau) < GAP_MIN]
            if not bad:
                break
            # shift the decision threshold away from the offending values instead of
            # resampling hidden rows (keeps the planted argmax intact)
            wl.tau = float(wl.tau + 0.0371)
        else:
            raise RuntimeError("router margin rule not met")
    if Vd > 0:
        wl.Wd = normal_bf16(seed, _T_WD, Vd, d, cfg.w_std)
        wl.x = normal_bf16(seed, _T_X, B, d, 1.0)
        wl.d2t = _rng(seed, _T_D2T).choice(V, size=Vd, replace=False).astype(np.int32)
        wl.topk = topk
        if reject and topk_gap_fn is not None:
            xa = {}
            todo = np.arange(B)
            for _ in range(256):
                gaps = np.asarray(topk_gap_fn(wl.Wd, wl.topk, wl.x[todo]))
                bad = todo[gaps < GAP_MIN]
                if not len(bad):
                    break
                for b in bad:
                    xa[int(b)] = xa.get(int(b), 0) + 1
                    wl.x[b] = hidden_row(seed, int(b), xa[int(b)], d, tag=_T_X_RS)
                todo = bad
            else:
                raise RuntimeError("draft top-k gap rule not met")
    return wl


# --------------------------------------------------------------------------- KV-only catch-up
# The EAGLE-3 drafter of the Qwen3-4B-EAGLE3 card ("Technical Specifications":
# one decoder layer, hidden 2560, 32 attention heads, 8 KV heads; head size
# 2560 / 32 = 80) catching up its backlog after a switch.  Cache lengths and
# backlogs span the switching-cost tables of the paper (Sec. 4, Table 4 and
# App. Table 12: base KV lengths 512 .. 16384, backlogs 1 .. 1024, typically
# 80-90 tokens).  Layer inputs ~N(0, 1) like hidden states, weights ~N(0, 0.02^2)
# like the other weights here, RMSNorm gains 1 + N(0, 0.1^2), cached keys and
# values ~N(0, 1); all bf16.
_T_CU = 100   # first stream tag of the catch-up tensors


@dataclasses.dataclass(frozen=True)
class CatchupConfig:
    name: str
    n: tuple             # backlog tokens per sequence
    L: tuple             # entries already cached per sequence
    din: int = 2560
    H: int = 32
    G: int = 8
    D: int = 80
    eps: float = 1e-6
    theta: float = 10000.0
    w_std: float = 0.02


CATCHUP_CONFIGS = [
    CatchupConfig("eagle3_catchup_b1_L2048_n85", n=(85,), L=(2048,)),
    CatchupConfig("eagle3_catchup_b1_L16384_n1024", n=(1024,), L=(16384,)),
    CatchupConfig("eagle3_catchup_b4_mixed", n=(1, 64, 128, 7), L=(0, 511, 1024, 4000)),
    CatchupConfig("eagle3_catchup_b8_L8192_n128", n=(128,) * 8, L=(8192,) * 8),
]


def catchup_workload(index: int, cap_extra: int = 0) -> dict:
    """Inputs of one catch-up call (bf16 bits / int32), keyed like the oracle's arguments.
    Each cache holds cache_len + backlog (+ cap_extra) rows."""
    cfg = CATCHUP_CONFIGS[index]
    seed = BASE_SEED + 1000 + index
    B = len(cfg.n)
    GD, HD = cfg.G * cfg.D, cfg.H * cfg.D
    cap = max(L + n for L, n in zip(cfg.L, cfg.n)) + cap_extra
    bl_off = np.concatenate([[0], np.cumsum(cfg.n)]).astype(np.int32)
    N = int(bl_off[-1])
    g = _rng(seed, _T_CU + 1).standard_normal(cfg.din, dtype=np.float32)
    return dict(
        u=normal_bf16(seed, _T_CU + 0, N, cfg.din, 1.0),
        bl_off=bl_off, cache_len=np.array(cfg.L, np.int32),
        gamma=to_bf16_bits(np.float32(1.0) + np.float32(0.1) * g),
        eps=cfg.eps, theta=cfg.theta,
        Wq=normal_bf16(seed, _T_CU + 2, HD, cfg.din, cfg.w_std),
        Wk=normal_bf16(seed, _T_CU + 3, GD, cfg.din, cfg.w_std),
        Wv=normal_bf16(seed, _T_CU + 4, GD, cfg.din, cfg.w_std),
        Wo=normal_bf16(seed, _T_CU + 5, cfg.din, HD, cfg.w_std),
        Kc=normal_bf16(seed, _T_CU + 6, B * cap, GD, 1.0).reshape(B, cap, GD),
        Vc=normal_bf16(seed, _T_CU + 7, B * cap, GD, 1.0).reshape(B, cap, GD),
        H=cfg.H, G=cfg.G)
