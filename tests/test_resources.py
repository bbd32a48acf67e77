"""Register and spill budgets of the kernels, read from ptxas's resource report
of the in-tree build (no GPU needed).

At batch 1 the neural router runs beside the LM-head argmax sweep on the same
SMs.  An SM sub-partition holds 16K registers, and it receives two warps of
each: two sweep warps at 96 registers and two router warps at 160 fill it
exactly (2 x 32 x 96 + 2 x 32 x 160 = 16,384).  One register more in either
kernel and the router's blocks wait until the sweep has finished (measured:
a DFlash round 15 us longer on a GB300)."""
import re

import pytest

from speculative_decoding_verify_lm_gb300 import build as B


def kernels(name):
    """{mangled kernel name: (registers, spill bytes)} of csrc/<name>."""
    rep = B.ptxas_report(name)
    if not rep:
        B.build(force=True)
        rep = B.ptxas_report(name)
    out, cur, spill = {}, None, 0
    for ln in rep.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", ln)
        if m:
            cur, spill = m.group(1), 0
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", ln)
        if m and cur:
            spill = int(m.group(1)) + int(m.group(2))
            continue
        m = re.search(r"Used (\d+) registers", ln)
        if m and cur:
            out[cur] = (int(m.group(1)), spill)
            cur = None
    return out


def one(ks, needle):
    hits = [v for k, v in ks.items() if needle in k]
    assert len(hits) == 1, (needle, sorted(ks))
    return hits[0]


def test_argmax_sweep_fits_beside_the_router():
    regs, _ = one(kernels("wf_gemm_select.cu"), "gemm_select_kernelILi1ELb0ELb0ELb0E")
    assert regs <= 96, f"the batch-1 argmax sweep uses {regs} registers; the router no longer fits beside it"


def test_router_fits_beside_the_argmax_sweep():
    regs, _ = one(kernels("wf_router.cu"), "13router_kernel")
    assert regs <= 160, f"the router uses {regs} registers; it no longer fits beside the argmax sweep"


@pytest.mark.parametrize("name", [s.rsplit("/", 1)[-1] for s in B.sources()])
def test_no_kernel_spills(name):
    spills = {k: s for k, (_, s) in kernels(name).items() if s}
    assert not spills, spills
