"""KV-only catch-up on the GPU vs the CPU oracle, through the C ABI.

The oracle computes the exact definition in fp64 and rounds only what the
method stores in bf16 (the cache rows).  The GPU rounds at more points: the
normalised inputs a, the query and the attention probabilities (bf16
tensor-core operands), the fp32 accumulations, and the attention output
before Wo (bf16 operand).  Every comparison uses a
first-order bound built from those rounding points (unit roundoff u = 2^-8
for bf16, 2^-24 per fp32 addition) with a factor 2 of slack:
  k, v before storing   |dk| <= (u + din 2^-24) sum_i |W_i a_i|  (+ the rotation mixes a pair)
  cache entries         |dk| plus one bf16 rounding of either side
  scores                |ds_t| <= (|dq| |k_t| + |q| |dk_t|) / sqrt(D),  |dq| including u |q|
  attention output      |do| <= 2 max|ds| sum_t p_t |v_t| + sum_t p_t |dv_t| + u sum_t p_t |v_t|
  output                |dout| <= sum_c |Wo_c| (|do_c| + u |o_c|)
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import dev, host
from speculative_decoding_verify_lm_gb300 import wf
from speculative_decoding_verify_lm_gb300.synth import bf16_bits_to_f32, catchup_workload

pytestmark = pytest.mark.gpu

U = 2.0 ** -8
E32 = 2.0 ** -24


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def run_gpu(c, kv_only=False):
    Kc, Vc = dev(c["Kc"]), dev(c["Vc"])
    cu = wf.Catchup(dev(c["u"]), dev(c["bl_off"]), dev(c["cache_len"]), dev(c["gamma"]), dev(c["Wk"]),
                    dev(c["Wv"]), Kc, Vc, c["G"], Wq=dev(c["Wq"]), Wo=dev(c["Wo"]), eps=c["eps"], theta=c["theta"],
                    kv_only=kv_only)
    out, attn = cu()
    torch.cuda.synchronize()
    res = dict(Kc=host(Kc).view(np.uint16), Vc=host(Vc).view(np.uint16))
    if not kv_only:
        res.update(out=host(out), attn=host(attn))
    return res, cu


def bounds(c, ref):
    """Per-element tolerances (cache rows, attention output, output) from the rounding points above."""
    o = oracle.default()
    H, G = c["H"], c["G"]
    din = c["u"].shape[1]
    D = c["Wk"].shape[0] // G
    half = D // 2
    B = len(c["bl_off"]) - 1
    a = np.stack([o.rmsnorm(r, c["gamma"], c["eps"]) for r in c["u"]])
    g_acc = U + din * E32
    ek = g_acc * (np.abs(a) @ np.abs(_f64(c["Wk"])).T)          # [N, GD] before the rotation
    ev = g_acc * (np.abs(a) @ np.abs(_f64(c["Wv"])).T)
    ek = ek.reshape(len(a), G, 2, half)
    ek = (ek + ek[:, :, ::-1]).reshape(len(a), G * D)
    tolK = np.zeros(c["Kc"].shape)
    tolV = np.zeros(c["Vc"].shape)
    for b in range(B):
        L = int(c["cache_len"][b])
        for j, r in enumerate(range(int(c["bl_off"][b]), int(c["bl_off"][b + 1]))):
            kref = _f64(ref["Kc"][b, L + j])
            vref = _f64(ref["Vc"][b, L + j])
            tolK[b, L + j] = ek[r] * (1 + U) + 2 * U * np.abs(kref) + 1e-6 * np.abs(kref)
            tolV[b, L + j] = ev[r] * (1 + U) + 2 * U * np.abs(vref)
    if "attn" not in ref or ref["attn"] is None:
        return tolK, tolV, None, None
    tolA = np.zeros((B, H * D))
    tolO = np.zeros((B, din))
    hq = H // G
    for b in range(B):
        f = int(c["bl_off"][b + 1]) - 1
        T = int(c["cache_len"][b]) + int(c["bl_off"][b + 1] - c["bl_off"][b])
        eq = g_acc * (np.abs(_f64(c["Wq"])) @ np.abs(a[f]))     # [HD] before the rotation
        eq = eq.reshape(H, 2, half)
        eq = (eq + eq[:, ::-1]).reshape(H * D) + 1e-6 * np.abs(ref["q"][b])
        K = _f64(ref["Kc"][b, :T]).reshape(T, G, D)
        V = _f64(ref["Vc"][b, :T]).reshape(T, G, D)
        dK = tolK[b, :T].reshape(T, G, D)
        dV = tolV[b, :T].reshape(T, G, D)
        for h in range(H):
            g = h // hq
            q = ref["q"][b, h * D:(h + 1) * D]
            dq = eq[h * D:(h + 1) * D] + U * np.abs(q)        # + the bf16 query operand
            s = K[:, g] @ q / math.sqrt(D)
            p = np.exp(s - s.max())
            p /= p.sum()
            ds = (np.abs(K[:, g]) @ dq + (dK[:, g] @ (np.abs(q) + dq))) / math.sqrt(D)
            tolA[b, h * D:(h + 1) * D] = 2 * ((2 * ds.max() + U) * (p @ np.abs(V[:, g])) + p @ dV[:, g]) + \
                1e-5 * (p @ np.abs(V[:, g]))                    # U: the bf16 probabilities
        oabs = np.abs(ref["attn"][b])
        tolO[b] = 2 * (np.abs(_f64(c["Wo"])) @ (tolA[b] + U * oabs)) + 2 * (H * D) * E32 * \
            (np.abs(_f64(c["Wo"])) @ oabs) + 1e-6
    return tolK, tolV, tolA, tolO


def check_against_oracle(c, res, kv_only=False):
    ref, rc = oracle.catchup(**c)
    assert rc == 0
    tolK, tolV, tolA, tolO = bounds(c, ref if not kv_only else dict(ref, attn=None))
    dK = np.abs(_f64(res["Kc"]) - _f64(ref["Kc"]))
    dV = np.abs(_f64(res["Vc"]) - _f64(ref["Vc"]))
    assert np.all(dK <= tolK), f"key cache off by {np.max(dK - tolK)}"
    assert np.all(dV <= tolV), f"value cache off by {np.max(dV - tolV)}"
    # rows outside the backlog are exactly what they were
    for b in range(len(c["bl_off"]) - 1):
        L = int(c["cache_len"][b])
        end = L + int(c["bl_off"][b + 1] - c["bl_off"][b])
        for name in ("Kc", "Vc"):
            assert np.array_equal(res[name][b, :L], c[name][b, :L])
            assert np.array_equal(res[name][b, end:], c[name][b, end:])
    if not kv_only:
        assert np.all(np.abs(res["attn"] - ref["attn"]) <= tolA), np.max(np.abs(res["attn"] - ref["attn"]) - tolA)
        assert np.all(np.abs(res["out"] - ref["out"]) <= tolO), np.max(np.abs(res["out"] - ref["out"]) - tolO)
    return ref


@pytest.mark.parametrize("seed,din,H,G,D,n,L,cap", [
    (1, 64, 4, 2, 16, (3, 1), (2, 0), 8),                                 # tiny, two sequences
    (2, 256, 8, 2, 32, (5, 1, 17), (0, 10, 40), 64),                      # ragged backlogs
    (3, 512, 8, 8, 64, (1,), (300,), 301),                                # one token, cache filled exactly
    (4, 128, 4, 1, 128, (40, 200), (7, 0), 256),                          # one KV head, > 128 rows
    (5, 192, 6, 3, 48, tuple([1] * 130), tuple(range(130)), 131),         # 130 sequences: two row tiles
    (6, 64, 2, 1, 16, (50,), (4000,), 4096),                              # 16 splits: the largest cluster merge
    (7, 128, 4, 2, 32, (40,), (5000,), 5100),                             # 20 splits by rows, capped at 16 (on chip)
    (8, 160, 4, 2, 32, (2, 3, 1, 5, 2, 1, 4, 2), (5,) * 8, 16),           # 8 sequences: the few-row output projection
    (9, 160, 4, 2, 32, (2, 3, 1, 5, 2, 1, 4, 2, 3), (5,) * 9, 16),        # 9: the tensor-core output projection
    (10, 4096, 8, 2, 64, (6, 2), (20, 3), 32),                            # a wide input (64 K blocks)
    (11, 1024, 128, 8, 128, (3,), (10,), 16),                             # H x D = 16384, the largest
    (12, 2560, 32, 8, 80, (300,), (700,), 1000),                          # EAGLE-3 shape, 40 tiles: 6 K splits
    (13, 2560, 32, 8, 80, (450,), (50,), 500),                            # 48 tiles: 5 K splits
    # D = 128: one attention CTA an SM, 12 clusters of 16 splits cannot all be
    # resident, so the splits merge through global memory
    (14, 256, 16, 4, 128, (5, 3, 7), (4000, 4090, 3000), 4096),
    (15, 384, 8, 4, 96, (5, 2), (300, 7), 320),                           # D = 96 (12 dim tiles)
    (16, 448, 8, 4, 112, (3,), (700,), 720),                              # D = 112 (14 dim tiles, 112-wide tiles)
])
def test_catchup_small_shapes(seed, din, H, G, D, n, L, cap):
    c = pins.catchup_case(seed, din=din, H=H, G=G, D=D, n=n, L=L, cap=cap)
    res, cu = run_gpu(c)
    assert cu.ws.device_error() == (0, 0)
    check_against_oracle(c, res)


def test_catchup_eagle3_geometry_representative_backlog():
    """The drafter of the EAGLE3 card (hidden 2560, 32 heads, 8 KV heads, D = 80)
    catching up 85 backlog tokens onto a 2048-entry cache (the paper's representative
    80-90 token backlog)."""
    c = catchup_workload(0)
    res, cu = run_gpu(c)
    assert cu.ws.device_error() == (0, 0)
    check_against_oracle(c, res)


def test_catchup_eagle3_geometry_batch():
    c = catchup_workload(2)
    res, cu = run_gpu(c)
    assert cu.ws.device_error() == (0, 0)
    check_against_oracle(c, res)


@pytest.mark.parametrize("index", [1, 3])
def test_catchup_eagle3_geometry_long_backlogs(index):
    """The two long-backlog workloads the bench times: 1,024 tokens onto a
    16,384-entry cache (eight activation tiles, three K splits, 16 attention
    splits merged on chip) and 8 sequences of 128 onto 8,192 (three cache
    splits a sequence)."""
    c = catchup_workload(index)
    res, cu = run_gpu(c)
    assert cu.ws.device_error() == (0, 0)
    check_against_oracle(c, res)


def test_catchup_kv_only_and_repeat():
    """The KV-only call writes exactly the backlog rows (same values as the full
    call), and a repeated call on the same workspace gives identical bits."""
    c = pins.catchup_case(21, din=256, H=8, G=4, D=32, n=(9, 2, 30), L=(3, 0, 11), cap=48)
    kv, _ = run_gpu(c, kv_only=True)
    check_against_oracle(c, kv, kv_only=True)
    full, cu = run_gpu(c)
    assert np.array_equal(kv["Kc"], full["Kc"]) and np.array_equal(kv["Vc"], full["Vc"])
    out1, attn1 = (host(t) for t in cu())
    torch.cuda.synchronize()
    assert np.array_equal(out1, full["out"]) and np.array_equal(attn1, full["attn"])


def test_catchup_overflow_sets_error_and_spares_the_cache():
    c = pins.catchup_case(22, din=64, H=4, G=2, D=16, n=(3, 2), L=(6, 1), cap=8)   # sequence 0: 6 + 3 > 8
    res, cu = run_gpu(c)
    code, info = cu.ws.device_error()
    assert code == 5 and info == 0
    assert np.array_equal(res["Kc"][0, :6], c["Kc"][0, :6])   # nothing written before the overflow's rows
    ref, _ = oracle.catchup(**dict(c, bl_off=c["bl_off"][1:] - c["bl_off"][1], cache_len=c["cache_len"][1:],
                                   u=c["u"][3:], Kc=c["Kc"][1:], Vc=c["Vc"][1:]))
    tolK, _, _, _ = bounds(dict(c, bl_off=c["bl_off"][1:] - c["bl_off"][1], cache_len=c["cache_len"][1:],
                                u=c["u"][3:], Kc=c["Kc"][1:], Vc=c["Vc"][1:]), dict(ref, attn=None))
    assert np.all(np.abs(_f64(res["Kc"][1]) - _f64(ref["Kc"][0])) <= tolK[0])
