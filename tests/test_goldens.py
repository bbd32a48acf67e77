"""The stored full-size oracle answers (tests/golden/round_*.json) on the CPU:
they were written by the current oracle, the generation record rebuilds the
inputs they were computed on, they reproduce when written again (the three
batch-1 workloads), and they hold the properties every round result has
(planted acceptance depths, valid accepted paths, routes that agree with the
router output).  The GPU side compares with them in test_full_size_gpu.py."""
import os
import sys

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_lm_gb300 import synth

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_full_goldens as fg  # noqa: E402

SMALL = (0, 1, 2)


@pytest.mark.parametrize("index", range(len(synth.CONFIGS)))
def test_golden_written_by_current_oracle(index):
    rec = fg.load(index)
    assert rec["oracle_source_sha256"] == fg.oracle_sha(), "oracle changed: rerun make_full_goldens.py"
    assert rec["workload"] == synth.CONFIGS[index].name and rec["index"] == index


@pytest.mark.parametrize("index", SMALL)
def test_golden_reproduces(index):
    """Writing the record again gives the same inputs and the same answers."""
    rec = fg.load(index)
    again = fg.make(index)
    for key in ("inputs", "expected", "cut", "tau", "b2", "shape", "seed"):
        assert again[key] == rec[key], key


def _invariants(rec, wl):
    e = rec["expected"]
    out = {k: np.array(e[k]) for k in ("ids", "n_accept", "bonus", "last_pos", "route")}
    out["path"] = np.array(e["path"], np.int32).reshape(wl.B, -1)
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from gpu_util import check_round_properties   # numpy-only property check
    check_round_properties(wl, out)
    assert np.array_equal(out["n_accept"], np.array(rec["cut"]))
    delta = np.array(e["delta"])
    assert np.array_equal(out["route"], (delta > rec["tau"]).astype(int))
    assert np.all(np.abs(delta - rec["tau"]) >= synth.GAP_MIN)
    if wl.Wd is not None:
        assert np.all(np.array(e["topk_min_gap"]) >= synth.GAP_MIN)
        lse = np.array(e["lse"])
        top = np.array(e["vals"]).reshape(wl.B, -1)[:, 0]
        assert np.all(lse > top) and np.all(lse < top + np.log(synth.CONFIGS[rec["index"]].Vd))


@pytest.mark.parametrize("index", range(len(synth.CONFIGS)))
def test_golden_record_rebuilds_inputs_and_holds_invariants(index):
    rec = fg.load(index)
    wl = fg.replay(index, rec)
    assert fg.input_hashes(wl) == rec["inputs"]["sha256"]
    _invariants(rec, wl)


def test_large_golden_rows_are_the_oracles():
    """Rows spread over the 256-tree workload, recomputed by the oracle now."""
    rec = fg.load(4)
    wl = fg.replay(4, rec)
    rows = np.linspace(0, wl.P - 1, 9).astype(np.int64)
    ids, _, _ = oracle.lmhead_argmax(wl.hidden[rows], wl.W)
    assert np.array_equal(ids, np.array(rec["expected"]["ids"])[rows])
    seqs = [0, 128, 255]
    dids, tids, vals, lse, _ = oracle.draft_topk(wl.x[seqs], wl.Wd, wl.d2t, wl.topk)
    k = wl.topk
    assert np.array_equal(dids, np.array(rec["expected"]["draft_ids"]).reshape(-1, k)[seqs])
    assert np.array_equal(lse, np.array(rec["expected"]["lse"])[seqs])
