"""Every round workload at full size against the CPU oracle, element by element.

The oracle's answers for the five workloads (tiny chain; Qwen3-4B-shaped
DFlash chain and EAGLE-3 tree at batch 1; the mixed batch of 32; 256 trees,
15,616 verified rows) are stored under tests/golden/ by make_full_goldens.py,
which calls only the oracle.  Here the inputs are rebuilt from the stored
generation record (checked against the stored input hashes) and one round runs
through the C ABI: every target argmax id, acceptance length, bonus token, last
row, accepted path and route must equal the oracle's, the router output and
the entropy within 1e-3, the draft head's top-k ids and target ids exactly and
its logits within the fp32 accumulation bound.  The generation rules (top-2
logit gap, router margin, adjacent top-k gaps all >= 1e-2) keep every decision
clear of the fp32 / fp64 rounding difference.
"""
import os
import sys

import numpy as np
import pytest

from gpu_util import check_round_properties, dev, host, logit_error_bound, round_on_gpu
from speculative_decoding_verify_lm_gb300 import synth, wf

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_full_goldens as fg  # noqa: E402

pytestmark = pytest.mark.gpu

_cache = {}


def _workload(index):
    if index not in _cache:
        _cache.clear()   # the large workloads hold ~1 GB of host arrays each
        rec = fg.load(index)
        wl = fg.replay(index, rec)
        assert fg.input_hashes(wl) == rec["inputs"]["sha256"], "rebuilt inputs differ from the oracle's"
        _cache[index] = (rec, wl)
    return _cache[index]


def _compare(rec, wl, out, entropy=False):
    e = rec["expected"]
    B = wl.B
    assert np.array_equal(out["ids"], np.array(e["ids"], np.int32)), "target argmax"
    for key in ("n_accept", "bonus", "last_pos"):
        assert np.array_equal(out[key], np.array(e[key], np.int32)), key
    assert np.array_equal(out["path"], np.array(e["path"], np.int32).reshape(B, -1)), "path"
    if entropy:
        H = np.array(e["entropy_at_last"])
        assert np.max(np.abs(out["delta_al"] - H)) <= 1e-3, "entropy"
    else:
        assert np.max(np.abs(out["delta_al"] - np.array(e["delta"]))) <= 1e-3, "router output"
        assert np.array_equal(out["route"], np.array(e["route"], np.int32)), "route"
    assert np.array_equal(out["n_accept"], np.array(rec["cut"], np.int32)), "planted depth"
    if wl.Wd is not None:
        k = wl.topk
        dids = np.array(e["draft_ids"], np.int32).reshape(B, k)
        assert np.array_equal(out["draft_ids"], dids), "draft ids"
        assert np.array_equal(out["tids"], np.array(e["tids"], np.int32).reshape(B, k)), "target ids"
        vals = np.array(e["vals"]).reshape(B, k)
        bound = np.stack([logit_error_bound(wl.x[b:b + 1].repeat(k, 0), wl.Wd, dids[b]) for b in range(B)])
        assert np.all(np.abs(out["vals"] - vals) <= bound), "draft logits"
        assert np.max(np.abs(out["lse"] - np.array(e["lse"]))) <= 1e-3, "draft log-sum-exp"


@pytest.mark.parametrize("index", range(len(synth.CONFIGS)))
def test_round_full_size(index):
    rec, wl = _workload(index)
    r, out = round_on_gpu(wl)
    assert r.ws.device_error() == (0, 0)
    _compare(rec, wl, out)
    check_round_properties(wl, out)
    # the same round again on the same workspace
    out2 = {k: host(v) for k, v in r().items()}
    _compare(rec, wl, out2)
    assert r.ws.device_error() == (0, 0)


@pytest.mark.parametrize("index", range(1, len(synth.CONFIGS)))
def test_round_full_size_entropy_routed(index):
    """WhiFlash-Entropy routing at full size: one sweep with the entropy
    statistics (<= 128 rows), else a second sweep over the accepted rows."""
    rec, wl = _workload(index)
    H = np.array(rec["expected"]["entropy_at_last"])
    tau = float(np.median(H)) + 0.0043
    draft = wl.Wd is not None
    r = wf.Round(dev(wl.hidden), dev(wl.W), dev(wl.pos_off), dev(wl.node_off), dev(wl.tok), dev(wl.W1),
                 dev(wl.b1), dev(wl.w2), wl.b2, tau, kind=dev(wl.kind), parent=dev(wl.parent),
                 path_stride=wl.max_depth, x=dev(wl.x) if draft else None, Wd=dev(wl.Wd) if draft else None,
                 d2t=dev(wl.d2t) if draft else None, k=wl.topk if draft else 0, router_kind=wf.WF_ROUTER_ENTROPY)
    for _ in range(2):
        out = {k: host(v) for k, v in r().items()}
        _compare(rec, wl, out, entropy=True)
        clear = np.abs(H - tau) >= synth.GAP_MIN
        assert np.array_equal(out["route"][clear], (H > tau).astype(np.int32)[clear])
    assert r.ws.device_error() == (0, 0)
