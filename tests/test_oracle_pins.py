"""The CPU oracle pinned to brute force, closed forms and hand-worked cases."""
import numpy as np
import pytest

import pins
from speculative_decoding_verify_lm_gb300 import synth


@pytest.fixture(scope="module")
def o(oracle_mod):
    return oracle_mod.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(o, check):
    check(o)


def test_router_param_table():
    pins.check_router_param_table()


def test_round_is_composition(o, oracle_mod):
    """oracle_round = argmax, per-kind acceptance, router at the last accepted row."""
    wl = synth.small_workload(11, d=64, V=300, kinds=[0, 1, 1, 0, 1], argmax_fn=oracle_mod.argmax_fn,
                              m=16, K=16, n_nodes=20, depth=5, branch=4)
    out = o.round_(wl.hidden, wl.W, wl.pos_off, wl.node_off, wl.kind, wl.tok, wl.parent, wl.W1, wl.b1,
                   wl.w2, wl.b2, wl.tau, 16)
    ids, _, _ = o.lmhead_argmax(wl.hidden, wl.W)
    assert np.array_equal(ids, out["ids"])
    for b in range(wl.B):
        po = np.array([0, wl.pos_off[b + 1] - wl.pos_off[b]], np.int32)
        no = np.array([0, wl.node_off[b + 1] - wl.node_off[b]], np.int32)
        gb = ids[wl.pos_off[b]:wl.pos_off[b + 1]]
        tb = wl.tok[wl.node_off[b]:wl.node_off[b + 1]]
        if wl.kind[b] == 0:
            n, bo, la, pa = o.verify_chain(gb, tb, po, no, 16)
        else:
            n, bo, la, pa, _ = o.verify_tree(gb, tb, wl.parent[wl.node_off[b]:wl.node_off[b + 1]], no, po, 16)
        assert out["n_accept"][b] == n[0] and out["bonus"][b] == bo[0]
        assert out["last_pos"][b] == la[0] + wl.pos_off[b]
        assert np.array_equal(out["path"][b], pa[0])
        # constructive: the planted matched depth is what verification finds
        assert n[0] == wl.cut[b]
    delta, route = o.router(wl.hidden, out["last_pos"], wl.W1, wl.b1, wl.w2, wl.b2, wl.tau)
    assert np.array_equal(delta, out["delta"]) and np.array_equal(route, out["route"])


@pytest.mark.parametrize("index", [0, 1])
def test_config_planted_cut(o, oracle_mod, index):
    """Full-size chain configs: verification finds exactly the planted cut."""
    wl = synth.make_workload(index, oracle_mod.argmax_fn, oracle_mod.router_fn, oracle_mod.topk_gap_fn)
    out = o.round_(wl.hidden, wl.W, wl.pos_off, wl.node_off, wl.kind, wl.tok, wl.parent, wl.W1, wl.b1,
                   wl.w2, wl.b2, wl.tau, wl.max_depth)
    assert np.array_equal(out["n_accept"], wl.cut)
    assert all(abs(out["delta"] - wl.tau) >= synth.GAP_MIN)
    assert out["last_pos"][0] == wl.expected_last_pos(0)
