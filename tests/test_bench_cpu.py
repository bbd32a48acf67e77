"""bench.py on the CPU: the side-step inputs are well formed and the reference
arm of each side step prints one JSON line with the fields the benchmark
contract asks for."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_kept_rows_inputs_are_accepted_paths():
    x = bench.op_inputs("kept_rows", 9)
    n, path, pos_off = x["n"], x["path"], x["pos_off"]
    assert ((0 <= n) & (n <= 8)).all() and path.shape == (9, 8)
    for b in range(9):
        assert (path[b, :n[b]] >= 0).all() and (path[b, n[b]:] == -1).all()
        assert len(set(path[b, :n[b]].tolist())) == n[b]          # distinct nodes
    rows, off = oracle.default().accepted_rows(n, path, pos_off)
    assert off[-1] == int(np.sum(n + 1))
    for b in range(9):   # root row first, then rows of the path, all inside the sequence
        kept = rows[b, :n[b] + 1]
        assert kept[0] == pos_off[b] and (kept < pos_off[b + 1]).all()


def test_build_tree_inputs_shape():
    x = bench.op_inputs("build_tree", 3)
    assert x["tid"].shape == (3, 8, 10, 10) and x["lp"].shape == (3, 8, 10, 10) and x["N"] == 60
    assert (x["lp"] <= 0).all()


@pytest.mark.parametrize("op", ["build_tree", "kept_rows"])
def test_reference_arm_line(op):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op,
                          "--op-batch", "2", "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle"
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]


@pytest.mark.parametrize("mode,metric", [(["--config", "0"], "METRIC"), (["--config", "0", "--router", "entropy"], "METRIC"),
                                         (["--catchup", "0"], "CATCHUP_METRIC")])
def test_reference_arm_matches_own_arm(mode, metric):
    """The reference arm of a round or a catch-up prints the metric, unit and
    workload keys the GPU arm prints for the same mode (the driver compares
    the two lines)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *mode,
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == getattr(bench, metric) and j["higher_is_better"] is True
    assert j["value"] > 0 and j["e2e"]["value"] == j["value"] and j["cpu_baseline"]["kind"] == "oracle"
    from speculative_decoding_verify_lm_gb300 import synth
    if metric == "METRIC":
        cfg = synth.CONFIGS[0]
        wl = bench.load_workload(0)
        entropy = "entropy" in mode
        want = bench.round_config(cfg.name + ("_entropy" if entropy else ""), cfg, wl, entropy, 1)
        assert j["unit"] == bench.UNIT
        assert j["config"] == want   # exactly the keys the GPU arm prints
    else:
        want = bench.catchup_config(synth.CATCHUP_CONFIGS[0])
        assert j["unit"] == "backlog tokens/s"
    for k, v in want.items():
        assert j["config"][k] == v, k


def test_round_launch_count_follows_the_composition():
    """The launch count a round line claims, per wf_round's composition."""
    assert bench.round_launches(17, 1, False, False) == 3       # LM head, router beside it, acceptance
    assert bench.round_launches(61, 1, True, False) == 3        # both heads in one sweep, acceptance + merge, router
    assert bench.round_launches(1248, 32, False, False) == 4    # LM head, acceptance, router GEMM + finish
    assert bench.round_launches(15616, 256, True, False) == 4   # both heads in one paired sweep, acceptance + merge,
    #                                                              router GEMM + finish
    assert bench.round_launches(15616, 300, True, False) == 6   # draft rows past one tile pair: its own sweep + merge
    assert bench.round_launches(17, 1, False, True) == 2        # entropy sweep, acceptance
    assert bench.round_launches(15616, 256, True, True) == 4    # both heads, acceptance + merge, gather, entropy sweep


def test_bench_workload_is_the_stored_record():
    """Both arms rebuild the inputs the oracle's stored answers were computed on."""
    import sys as _s
    _s.path.insert(0, os.path.join(ROOT, "tests", "golden"))
    import make_full_goldens as fg
    rec = fg.load(1)
    wl = bench.load_workload(1)
    assert fg.input_hashes(wl) == rec["inputs"]["sha256"]
