"""The C ABI library builds, loads without a GPU, exports what include/wf.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_verify_lm_gb300 import wf

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "wf.h")


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"WF_API\s+[\w\s\*]+?\b(wf_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("wf_lmhead_argmax", "wf_verify_chain", "wf_verify_tree", "wf_router_mlp", "wf_draft_topk",
                 "wf_round", "wf_workspace_bytes", "wf_status_string", "wf_catchup", "wf_catchup_kv"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = wf.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", wf.lib_path()], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared():
        assert name in exported, name
        assert getattr(L, name) is not None
    assert set(wf.exported_symbols()) == set(declared())
    # nothing but the declared API is exported
    assert {e for e in exported if not e.startswith("_")} == set(declared())


def test_status_strings_and_sizes():
    L = wf.lib()
    assert L.wf_version() >= 100
    for s in range(7):
        assert L.wf_status_string(s).decode().startswith(wf.STATUS[s])
    small = L.wf_workspace_bytes(17, 1, 2560, 1024, 0, 0)
    big = L.wf_workspace_bytes(15616, 256, 2560, 1024, 32000, 10)
    assert 0 < small < big and big % 256 == 0
    # keys for every row + draft candidates + router partials
    assert big >= 256 + 8 * 15616 + 125 * 2 * 128 * 10 * 8 + 4 * 256 * 128


NULL = None


@pytest.mark.parametrize("call,args", [
    ("wf_lmhead_argmax", (NULL, NULL, 1, 64, 10, NULL, NULL, NULL, 0, NULL)),
    ("wf_lmhead_argmax", (256, 256, 0, 64, 10, 256, NULL, 256, 1 << 20, NULL)),       # P = 0
    ("wf_lmhead_argmax", (256, 256, 4, 60, 10, 256, NULL, 256, 1 << 20, NULL)),       # d % 8 != 0
    ("wf_lmhead_argmax", (258, 256, 4, 64, 10, 256, NULL, 256, 1 << 20, NULL)),       # misaligned hidden
    ("wf_verify_tree", (256, 256, NULL, 256, 256, 1, 0, 256, 256, 256, NULL, 256, 1 << 20, NULL)),
    ("wf_verify_chain", (256, 256, 256, 256, -1, 0, 256, 256, 256, NULL, 256, 1 << 20, NULL)),
    ("wf_router_mlp", (256, 256, 1, 64, 0, 256, 256, 256, 0.0, 1.0, 256, 256, 256, 1 << 20, NULL)),  # m = 0
    ("wf_draft_topk", (256, 256, 256, 1, 64, 100, 17, 256, 256, 256, NULL, 256, 1 << 20, NULL)),    # k > 16
    ("wf_draft_topk", (256, 256, 256, 1, 64, 5, 6, 256, 256, 256, NULL, 256, 1 << 20, NULL)),       # k > Vd
    ("wf_draft_topk", (256, 256, 256, 1, 64, 100, 4, NULL, NULL, NULL, NULL, 256, 1 << 20, NULL)),  # no output
    ("wf_lmhead_draft_topk", (256, 256, 4, 64, 100, 256, NULL, 256, 256, 256, 1, 50, 0, NULL, 256, 256, NULL,
                              256, 1 << 20, NULL)),                                                # k = 0
    ("wf_lmhead_draft_topk", (256, 256, 4, 64, 100, 256, NULL, 264, 256, 256, 1, 50, 4, NULL, 256, 256, NULL,
                              256, 1 << 20, NULL)),                                                # misaligned x
])
def test_invalid_arguments_rejected_on_host(call, args):
    assert getattr(wf.lib(), call)(*args) == 1


@pytest.mark.parametrize("ws,nbytes", [(NULL, 1 << 20), (256 + 64, 1 << 20), (256, 16)])
def test_workspace_checked_on_host(ws, nbytes):
    st = wf.lib().wf_lmhead_argmax(256, 256, 4, 64, 10, 256, NULL, ws, nbytes, NULL)
    assert st == 2


def test_shared_sweep_limits():
    # draft rows past one activation tile (target rows in one tile) or past one
    # tile pair (target rows in several): unsupported, nothing enqueued (no
    # device needed)
    L = wf.lib()
    assert L.wf_lmhead_draft_topk(256, 256, 128, 64, 100, 256, NULL, 256, 256, 256, 129, 50, 4, NULL, 256, 256,
                                  NULL, 256, 1 << 20, NULL) == 4
    assert L.wf_lmhead_draft_topk(256, 256, 129, 64, 100, 256, NULL, 256, 256, 256, 257, 50, 4, NULL, 256, 256,
                                  NULL, 256, 1 << 20, NULL) == 4


def test_catchup_shapes_checked_on_host():
    L = wf.lib()
    assert L.wf_catchup_workspace_bytes(1, 85, 2560, 32, 8, 80) > 0
    assert L.wf_catchup_workspace_bytes(1, 85, 2560, 32, 8, 72) == 0     # head size not a multiple of 16
    assert L.wf_catchup_workspace_bytes(1, 85, 2560, 30, 8, 80) == 0     # query heads not a multiple of KV heads
    assert L.wf_catchup_workspace_bytes(2, 1, 2560, 32, 8, 80) == 0      # fewer backlog rows than sequences
    a = wf.CatchupArgs()
    a.u = a.bl_off = a.cache_len = a.gamma = a.Wq = a.Wk = a.Wv = a.Wo = a.Kc = a.Vc = a.out = 256
    a.B, a.N, a.din, a.H, a.G, a.D, a.cap, a.eps, a.theta = 1, 4, 64, 4, 2, 16, 8, 1e-6, 1e4
    ws = 256
    nbytes = L.wf_catchup_workspace_bytes(1, 4, 64, 4, 2, 16)
    a.Wq = None
    assert L.wf_catchup(ctypes.byref(a), ws, nbytes, None) == 1          # the full call needs Wq
    a.Wq, a.theta = 256, 0.0
    assert L.wf_catchup_kv(ctypes.byref(a), ws, nbytes, None) == 1       # rotary base must be positive
    a.theta, a.Kc = 1e4, 264
    assert L.wf_catchup_kv(ctypes.byref(a), ws, nbytes, None) == 1       # misaligned cache
    a.Kc = 256
    assert L.wf_catchup_kv(ctypes.byref(a), ws, nbytes - 256, None) == 2  # workspace too small


def test_round_rejects_missing_tree_description():
    a = wf.RoundArgs()
    a.hidden = a.W = 256
    a.P, a.d, a.V, a.B = 17, 64, 100, 1
    a.pos_off = a.node_off = a.tok = 256
    a.kind = a.parent = None         # neither a kind array nor parents
    a.m = 8
    a.W1 = a.b1 = a.w2 = 256
    a.ids = a.n_accept = a.bonus = a.last_pos = a.delta_al = a.route = 256
    assert wf.lib().wf_round(ctypes.byref(a), 256, 1 << 20, None) == 1
