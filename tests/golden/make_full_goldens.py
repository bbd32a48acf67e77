#!/usr/bin/env python3
"""Write the CPU oracle's answers for the five round workloads at full size.

For workload i (``synth.CONFIGS[i]``) this builds the inputs exactly as the
tests do - ``synth.make_workload(i, oracle.argmax_fn, oracle.router_fn,
oracle.topk_gap_fn)``, every sequence planted from the oracle's target argmax
and every rejection rule applied - then runs the oracle over the whole
workload and stores, in ``round_<workload>.json`` next to this script:

  inputs    the generation record that ``synth.replay_workload`` rebuilds the
            inputs from without an argmax (the final resample attempt of each
            rejected hidden / drafter row and the drafted tokens), plus a
            SHA-256 of every input array to check the rebuild;
  expected  the oracle's round (target argmax of every verified row,
            acceptance, bonus, last row, accepted path, router output and
            route), its draft-head top-k with the log-sum-exp over the draft
            vocabulary (EAGLE-3 workloads), and the entropy of the target's
            distribution at each sequence's last accepted row (WhiFlash-Entropy).

Only ``oracle/`` and the seeded generator are called; no value comes from the
GPU library.  The largest workload (256 trees, 15,616 rows over 151,936 x
2,560 weights) takes roughly 40 minutes on 8 host cores.

    python tests/golden/make_full_goldens.py [index ...]
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from speculative_decoding_verify_lm_gb300 import synth  # noqa: E402


def sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def input_hashes(wl) -> dict:
    h = {"hidden": sha(wl.hidden), "W": sha(wl.W), "tok": sha(wl.tok), "parent": sha(wl.parent),
         "pos_off": sha(wl.pos_off), "W1": sha(wl.W1)}
    if wl.Wd is not None:
        h.update(Wd=sha(wl.Wd), x=sha(wl.x), d2t=sha(wl.d2t))
    return h


def oracle_sha() -> str:
    with open(os.path.join(ROOT, "oracle", "wf_oracle.c"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def golden_path(index: int) -> str:
    return os.path.join(HERE, f"round_{synth.CONFIGS[index].name}.json")


def floats(a) -> list:
    return [float(v) for v in np.asarray(a, np.float64).ravel()]


def ints(a) -> list:
    return [int(v) for v in np.asarray(a).ravel()]


def make(index: int) -> dict:
    o = oracle.default()
    t0 = time.time()
    wl = synth.make_workload(index, oracle.argmax_fn, oracle.router_fn, oracle.topk_gap_fn)
    t_gen = time.time() - t0
    ref = o.round_(wl.hidden, wl.W, wl.pos_off, wl.node_off, wl.kind, wl.tok, wl.parent, wl.W1, wl.b1, wl.w2,
                   wl.b2, wl.tau, wl.max_depth)
    H, _ = o.entropy(wl.hidden, ref["last_pos"], wl.W)
    exp = {"ids": ints(ref["ids"]), "n_accept": ints(ref["n_accept"]), "bonus": ints(ref["bonus"]),
           "last_pos": ints(ref["last_pos"]), "path": ints(ref["path"]), "delta": floats(ref["delta"]),
           "route": ints(ref["route"]), "entropy_at_last": floats(H)}
    if wl.Wd is not None:
        dids, tids, vals, lse, mg = o.draft_topk(wl.x, wl.Wd, wl.d2t, wl.topk)
        exp.update(draft_ids=ints(dids), tids=ints(tids), vals=floats(vals), lse=floats(lse),
                   topk_min_gap=floats(mg))
    cfg = wl.cfg
    return {
        "workload": cfg.name, "index": index, "seed": int(wl.seed),
        "generator": "synth.make_workload(index, oracle.argmax_fn, oracle.router_fn, oracle.topk_gap_fn)",
        "oracle_source_sha256": oracle_sha(), "oracle_threads": o.threads(),
        "seconds": {"generate": round(t_gen, 1), "total": round(time.time() - t0, 1)},
        "shape": {"B": int(wl.B), "P": int(wl.P), "N": int(len(wl.tok)), "d": cfg.d, "V": cfg.V,
                  "m": int(wl.W1.shape[0]), "path_stride": int(wl.max_depth),
                  "Vd": cfg.Vd if wl.Wd is not None else 0, "k": int(wl.topk)},
        "tau": float(wl.tau), "b2": float(wl.b2),
        "cut": ints(wl.cut),
        "inputs": {"hidden_attempts": sorted([int(r), int(a)] for r, a in wl.hidden_attempts.items()),
                   "x_attempts": sorted([int(b), int(a)] for b, a in wl.x_attempts.items()),
                   "tok": ints(wl.tok), "sha256": input_hashes(wl)},
        "expected": exp,
    }


def load(index: int) -> dict:
    with open(golden_path(index)) as f:
        return json.load(f)


def replay(index: int, rec: dict | None = None):
    """The workload rebuilt from its stored record (no argmax needed)."""
    return synth.workload_from_record(load(index) if rec is None else rec)


def main(argv):
    idx = [int(a) for a in argv] or list(range(len(synth.CONFIGS)))
    for i in idx:
        t0 = time.time()
        rec = make(i)
        wl = replay(i, rec)   # the record rebuilds the same inputs
        assert input_hashes(wl) == rec["inputs"]["sha256"], "replay does not rebuild the inputs"
        tmp = golden_path(i) + ".tmp"
        with open(tmp, "w") as f:
            json.dump(rec, f, separators=(",", ":"))
            f.write("\n")
        os.replace(tmp, golden_path(i))
        print(f"{rec['workload']}: {time.time() - t0:.0f} s -> {golden_path(i)}", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
