"""wf_lmhead_argmax_noalloc, the variant for callers that cannot allocate
device memory (its scratch is a fixed array inside the library), must give
exactly what the workspace-based wf_lmhead_argmax gives, call after call, and
the CPU oracle's argmax on inputs whose top-2 logit gap is at least 1e-2.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verify_lm_gb300 import synth, wf

pytestmark = pytest.mark.gpu


def _inputs(seed, P, d, V):
    W = synth.normal_bf16(seed, 0, V, d, d ** -0.5)
    h = synth.normal_bf16(seed, 1, P, d, 1.0)
    t = lambda a: torch.from_numpy(a.view(np.int16)).to("cuda:0")  # noqa: E731
    return t(h), t(W), h, W


@pytest.mark.parametrize("P,d,V", [(17, 2560, 151936), (300, 256, 5000), (1, 64, 300)])
def test_noalloc_matches_workspace_call(P, d, V):
    h, W, h_np, W_np = _inputs(100 + P, P, d, V)
    ws = wf.Workspace(P)
    ids_ref = torch.empty(P, dtype=torch.int32, device="cuda:0")
    mx_ref = torch.empty(P, dtype=torch.float32, device="cuda:0")
    wf.wf_lmhead_argmax(h, W, ws, ids=ids_ref, maxlogit=mx_ref)
    for _ in range(2):          # two calls in a row: the shared array must not carry state over
        ids = torch.full((P,), -7, dtype=torch.int32, device="cuda:0")
        mx = torch.full((P,), float("nan"), dtype=torch.float32, device="cuda:0")
        st = wf.lib().wf_lmhead_argmax_noalloc(ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()), P, d,
                                               V, ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(mx.data_ptr()),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, wf.lib().wf_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref)
        # same kernel, same operands: the logits agree to fp32 accumulation (bound 2 d u sum|h w|)
        hf = synth.bf16_bits_to_f32(h_np).astype(np.float64)
        wf_ = synth.bf16_bits_to_f32(W_np[ids_ref.cpu().numpy()]).astype(np.float64)
        bound = 2.0 * d * 2.0 ** -24 * np.abs(hf * wf_).sum(axis=1)
        assert np.all(np.abs(mx.cpu().numpy() - mx_ref.cpu().numpy()) <= bound)


@pytest.mark.parametrize("P,d,V", [(17, 2560, 151936), (300, 256, 5000)])
def test_noalloc_matches_oracle(P, d, V):
    """Against the oracle, on inputs resampled until every row's top-2 logit gap
    is >= 1e-2 (fp32 accumulation and fp64 then pick the same id)."""
    import oracle
    W = synth.normal_bf16(300 + P, 0, V, d, d ** -0.5)
    h = synth.normal_bf16(300 + P, 1, P, d, 1.0)
    ids_ref, mx_ref, gap = oracle.lmhead_argmax(h, W)
    for a in range(1, 100):
        bad = np.nonzero(gap < synth.GAP_MIN)[0]
        if not len(bad):
            break
        for r in bad:
            h[r] = synth.hidden_row(300 + P, int(r), a, d)
        i2, m2, g2 = oracle.lmhead_argmax(h[bad], W)
        ids_ref[bad], mx_ref[bad], gap[bad] = i2, m2, g2
    assert (gap >= synth.GAP_MIN).all()
    t = lambda a: torch.from_numpy(a.view(np.int16)).to("cuda:0")  # noqa: E731
    hd, Wdv = t(h), t(W)
    for _ in range(2):
        ids = torch.full((P,), -7, dtype=torch.int32, device="cuda:0")
        mx = torch.empty(P, dtype=torch.float32, device="cuda:0")
        wf.wf_lmhead_argmax_noalloc(hd, Wdv, ids=ids, maxlogit=mx)
        assert wf.wf_noalloc_read_device_error() == (0, 0)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        hf = synth.bf16_bits_to_f32(h).astype(np.float64)
        wr = synth.bf16_bits_to_f32(W[ids_ref]).astype(np.float64)
        assert np.all(np.abs(mx.cpu().numpy() - mx_ref) <= 2.0 * d * 2.0 ** -24 * np.abs(hf * wr).sum(axis=1))


def test_noalloc_rejects_rows_beyond_its_array():
    P = 16385                          # WF_NOALLOC_MAX_ROWS + 1
    h = torch.zeros((P, 64), dtype=torch.int16, device="cuda:0")
    W = torch.zeros((8, 64), dtype=torch.int16, device="cuda:0")
    ids = torch.empty(P, dtype=torch.int32, device="cuda:0")
    st = wf.lib().wf_lmhead_argmax_noalloc(ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()), P, 64, 8,
                                           ctypes.c_void_p(ids.data_ptr()), None, None)
    assert st == 1
