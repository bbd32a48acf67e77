#!/usr/bin/env python3
"""Benchmark of one WhiFlash verify-and-route round on GB300.

A step is one whole round through the library's C ABI (wf_round): target
LM-head argmax at every verified row, chain / tree acceptance with the bonus
token, the neural router on each sequence's last accepted row, and (for the
EAGLE-3 workloads) the draft head's top-10.  Inputs are the seeded synthetic
workloads of ``speculative_decoding_verify_lm_gb300.synth`` (default: the
largest one, 256 EAGLE-3 trees of 60 nodes plus a root each = 15,616 verified
rows over the Qwen3-4B-shaped LM head, hidden 2560, vocabulary 151,936, with
the draft head's top-10 over 32,000 ids), rebuilt from the record that the
oracle's full-size answers are stored with, so that every drafted token is
planted from the oracle's target argmax and both arms time the same inputs.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a deliberately slow baseline, not a GPU program).
Several GPUs run independent replicas (one process per GPU, weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified positions/s and accepted tokens/s per round; % of HBM/TC roofline"
CATCHUP_METRIC = "KV-only catch-up: backlog tokens entered per second; % of HBM roofline"
UNIT = "verified positions/s"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4,
                    help="workload index 0-4 (default 4: 256 EAGLE-3 trees, 15,616 verified rows)")
    ap.add_argument("--router-width", type=int, default=None, help="override m (the paper's m = d/8 = 320)")
    ap.add_argument("--router", choices=["neural", "entropy"], default="neural",
                    help="the round's routing policy: the neural router (default) or WhiFlash-Entropy")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct wf_round calls instead of a CUDA graph")
    ap.add_argument("--op", choices=["build_tree", "kept_rows"], default=None,
                    help="time one of the round's side steps instead of a round: the EAGLE-3 draft-tree "
                         "construction or the kept rows of the accepted paths")
    ap.add_argument("--op-batch", type=int, default=1, help="sequences per --op call")
    ap.add_argument("--catchup", type=int, default=None,
                    help="time the drafter's KV-only catch-up on this workload (index 0-3) instead of a round")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def allreduce_max(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, read while the timed
    region runs: NVML (read-only queries through ctypes) polled in a loop while the
    host waits for the region's last event, else nvidia-smi every 200 ms."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_uuid):
        import ctypes
        self.ct = ctypes
        self.sm, self.mx, self.reasons = [], [], set()
        self.nvml = self.handle = self.proc = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if lib.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(h)) == 0:
                    self.nvml, self.handle = lib, h
                    fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                    self.reason_fn = fn or lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is None:
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                              "-lms", "200", "-i", gpu_uuid], stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None

    def sample(self):
        if self.nvml is None:
            return
        ct = self.ct
        c, m, r = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(c)) == 0:          # NVML_CLOCK_SM
            self.sm.append(float(c.value))
        if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(m)) == 0:
            self.mx.append(float(m.value))
        if self.reason_fn(self.handle, ct.byref(r)) == 0:
            for bit, name in self.REASONS.items():
                if r.value & bit:
                    self.reasons.add(name)

    def wait(self, event):
        """Sample until `event` (the timed region's last event) has completed."""
        while not event.query():
            self.sample()
            time.sleep(0.0002)
        self.sample()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 7:
                    continue
                try:
                    self.sm.append(float(f[0]))
                    self.mx.append(float(f[1]))
                except ValueError:
                    continue
                for name, v in zip(self.NAMES, f[3:7]):
                    if v.lower().startswith("active"):
                        self.reasons.add(name)
        src = "nvml" if self.nvml is not None else ("nvidia-smi" if self.proc is not None else "unavailable")
        return {"sm_mhz": statistics.median(self.sm) if self.sm else None,
                "sm_max_mhz": max(self.mx) if self.mx else None, "reasons": sorted(self.reasons),
                "samples": len(self.sm), "source": src}


# kernel label -> the source files it is built from (template arguments: top-k
# width, entropy, both heads, paired CTAs)
KERNEL_SOURCES = {name: ("wf_gemm_select.cu", "wf_internal.cuh")
                  for name in ("gemm_select_kernel<1,0,0,0>", "gemm_select_kernel<1,0,0,1>",
                               "gemm_select_kernel<1,1,0,0>", "gemm_select_kernel<1,0,1,0>",
                               "gemm_select_kernel<1,0,1,1>")}


def source_sha(kernel: str) -> str:
    """Hash of the source files a kernel is built from (its ncu counters go stale when they change)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verify_lm_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j["hbm_gbs"], j["bf16_tflops"], j.get("bf16_tflops_sustained", j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def traffic_for(kernel: str, workload: str):
    """ncu DRAM bytes per launch recorded under profiles/ for this exact source, else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(f"{kernel}@{workload}")
    if not e or e.get("source_sha") != source_sha(kernel):
        return None
    return e.get("bytes_per_launch")


# ----------------------------------------------------------------------------- CPU oracle arm
def oracle_round(o, sub, entropy: bool):
    """One oracle round: LM-head argmax, acceptance and the neural router, or
    with entropy routing also the entropy of the target distribution at each
    sequence's accepted row."""
    out = o.round_(*sub)
    if entropy:
        o.entropy(sub[0], out["last_pos"], sub[1], sub[11])
    return out


def cpu_sample(wl, budget_s: float, entropy: bool = False):
    """Time the oracle round on a bounded sample of the workload; returns (positions/s, sample text, cores)."""
    import oracle
    o = oracle.default()
    B = wl.B
    # sequences in order until the sample is about budget-sized (one probe round first)
    seqs, rows = [], 0
    t_probe = None
    for b in range(B):
        seqs.append(b)
        rows += int(wl.pos_off[b + 1] - wl.pos_off[b])
        if rows >= 17:
            break
    sub = _subset(wl, seqs)
    t0 = time.perf_counter()
    oracle_round(o, sub, entropy)
    t_probe = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(t_probe, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_round(o, sub, entropy)
    dt = time.perf_counter() - t0
    P_sub = int(sub[2][-1])
    return P_sub * reps / dt, f"{reps} oracle rounds over {len(seqs)} of {B} sequences ({P_sub} verified rows each)", \
        o.threads(), dt / reps, P_sub


def _subset(wl, seqs):
    rows = np.concatenate([np.arange(wl.pos_off[b], wl.pos_off[b + 1]) for b in seqs])
    nodes = np.concatenate([np.arange(wl.node_off[b], wl.node_off[b + 1]) for b in seqs])
    lens = np.array([wl.pos_off[b + 1] - wl.pos_off[b] for b in seqs])
    pos_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    node_off = np.concatenate([[0], np.cumsum(lens - 1)]).astype(np.int32)
    return (wl.hidden[rows], wl.W, pos_off, node_off, wl.kind[seqs], wl.tok[nodes], wl.parent[nodes], wl.W1,
            wl.b1, wl.w2, wl.b2, wl.tau, wl.max_depth)


def round_config(cfg_name, cfg, wl, entropy, world=1):
    """The workload keys of a round's JSON line, the same for both arms."""
    draft = wl.Wd is not None
    weight_bytes = cfg.V * cfg.d * 2 + (wl.Wd.nbytes if draft else 0) + wl.W1.nbytes
    return {"workload": cfg_name, "P": int(wl.P), "B": int(wl.B), "d": cfg.d, "V": cfg.V,
            "router": "entropy" if entropy else f"neural, m = {int(wl.W1.shape[0])}",
            "draft_head": f"{cfg.Vd}x{cfg.d} top-{wl.topk}" if draft else None,
            "inputs": "rebuilt from the stored oracle record: every sequence planted from the oracle's target argmax",
            "l2": "flushed between steps (working set < 2x L2)" if flush_l2(weight_bytes)
            else f"inputs larger than L2 (weights {weight_bytes / 1e6:.0f} MB streamed per step)",
            "parallelism": f"replicas x{world}"}


def flush_l2(weight_bytes: int) -> bool:
    return weight_bytes < 2 * L2_BYTES


def golden_record(index: int) -> dict:
    """The oracle's stored full-size answers for workload ``index`` (written by
    tests/golden/make_full_goldens.py, which calls only the oracle); read here
    only for the generation record that rebuilds the inputs."""
    from speculative_decoding_verify_lm_gb300 import synth
    path = os.path.join(ROOT, "tests", "golden", f"round_{synth.CONFIGS[index].name}.json")
    with open(path) as f:
        return json.load(f)


def load_workload(index: int, m=None):
    from speculative_decoding_verify_lm_gb300 import synth
    return synth.workload_from_record(golden_record(index), m=m)


def round_launches(P: int, B: int, draft: bool, entropy: bool) -> int:
    """Kernel launches of one wf_round (the composition in wf_round: the LM
    head or both heads in one sweep, acceptance, the router, the draft head)."""
    shared = draft and (B <= 128 if P <= 128 else B <= 256)
    if entropy:
        if P <= 128:
            return 2 + (0 if shared else (2 if draft else 0))
        # the draft head in the first sweep (rows in one tile pair), else its own sweep and merge after the round
        return 4 + (0 if draft and B <= 256 else (2 if draft else 0))
    if P <= 32:   # router beside the LM head over every row
        return 3 + (0 if shared else (2 if draft else 0))
    router = 1 if B <= 8 else 2
    return 2 + router + (0 if shared else (2 if draft else 0))


def run_reference(args, cfg_name, cfg, wl, world):
    """--impl reference: the CPU oracle, as it stands, on the host cores.  Each
    step is one oracle round over a bounded sample of the workload (its first
    sequence; the whole workload would take minutes to hours per step)."""
    import oracle
    o = oracle.default()
    entropy = args.router == "entropy"
    sub = _subset(wl, [0])
    for _ in range(args.warmup):
        oracle_round(o, sub, entropy)
    t0 = time.perf_counter()
    acc = 0
    for _ in range(args.steps):
        out = oracle_round(o, sub, entropy)
        acc += int((out["n_accept"] + 1).sum())
    dt = time.perf_counter() - t0
    P1 = int(sub[2][-1])
    val = P1 * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": round_config(cfg_name, cfg, wl, entropy, world),
            "accepted_tokens_per_s": acc / dt,
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": o.threads(), "kind": "oracle",
                             "sample": f"each step: one oracle round over the workload's first sequence "
                                       f"({P1} of {wl.P} verified rows)"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- KV-only catch-up
def catchup_config(cfg):
    """The workload keys of a catch-up JSON line, the same for both arms."""
    return {"workload": cfg.name, "B": len(cfg.n), "backlog": list(cfg.n), "cache_len": list(cfg.L),
            "din": cfg.din, "H": cfg.H, "G": cfg.G, "D": cfg.D, "l2": "L2 flushed (256 MB write) before every call"}


def run_catchup_reference(args):
    """The oracle's catch-up, timed on the host cores (the reference arm of --catchup)."""
    import oracle
    from speculative_decoding_verify_lm_gb300 import synth
    cfg = synth.CATCHUP_CONFIGS[args.catchup]
    c = synth.catchup_workload(args.catchup)
    for _ in range(args.warmup):
        oracle.catchup(**c)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.catchup(**c)
    dt = time.perf_counter() - t0
    N = int(c["bl_off"][-1])
    val = N * args.steps / dt
    print(json.dumps({"impl": "reference", "metric": CATCHUP_METRIC,
                      "value": val, "unit": "backlog tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                      "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": catchup_config(cfg),
                      "cpu_baseline": {"value": val, "unit": "backlog tokens/s", "cores": oracle.threads(),
                                       "kind": "oracle", "sample": "whole oracle catch-up calls of this workload"},
                      "e2e": {"value": val, "unit": "backlog tokens/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}), flush=True)



def catchup_work(c):
    """Algorithmic bytes and flops of one catch-up call."""
    N, din = c["u"].shape
    B = len(c["bl_off"]) - 1
    GD, HD = c["Wk"].shape[0], c["Wq"].shape[0]
    T = int(sum(int(L) + int(c["bl_off"][b + 1] - c["bl_off"][b]) for b, L in enumerate(c["cache_len"])))
    weights = 2 * (2 * GD * din + 2 * HD * din + din)
    nbytes = weights + 2 * N * din + 2 * 2 * N * GD + 2 * 2 * T * GD + 4 * B * din + 4 * B * HD + 4 * (2 * B + 1)
    flops = 2.0 * N * din * 2 * GD + 2.0 * B * din * HD + 4.0 * T * HD + 2.0 * B * HD * din
    return nbytes, flops, T


def run_catchup(args, rank, local, pg):
    import torch
    from speculative_decoding_verify_lm_gb300 import synth, wf
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = synth.CATCHUP_CONFIGS[args.catchup]
    c = synth.catchup_workload(args.catchup)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16  # noqa: E731
                                   else np.ascontiguousarray(a)).to(device)
    Kc, Vc = t(c["Kc"]), t(c["Vc"])
    u = t(c["u"])
    cu = wf.Catchup(u, t(c["bl_off"]), t(c["cache_len"]), t(c["gamma"]), t(c["Wk"]), t(c["Wv"]), Kc, Vc, c["G"],
                    Wq=t(c["Wq"]), Wo=t(c["Wo"]), eps=c["eps"], theta=c["theta"])
    stream = torch.cuda.current_stream(device)
    l2buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    for _ in range(max(args.warmup, 3)):
        cu()
    torch.cuda.synchronize(device)
    code, info = cu.ws.device_error()
    if code:
        raise RuntimeError(f"device error {code} (info {info}) during warm-up")
    step = cu
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cu()
        step = g.replay
        step()
    torch.cuda.synchronize(device)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        l2buf.zero_()   # weights and caches come from HBM every call
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    sampler.wait(ev[-1][1])
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_mean = statistics.mean(ms)
    N = int(c["bl_off"][-1])
    B = len(cfg.n)
    nbytes, flops, T = catchup_work(c)
    hbm_peak, tc_peak, _, peak_src = measured_peaks()
    achieved = nbytes / (ms_mean / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": None, "kernel": "catch-up call (norm, projections, attention, output projection)",
            "algorithmic_per_launch": nbytes, "launch_ms": ms_mean,
            "flops_per_call": flops, "peak_source": f"{peak_src} (hbm_gbs, burst)"}
    # end to end: the backlog's layer inputs in from pinned host memory, the output back
    h_u = torch.empty(u.shape, dtype=u.dtype, pin_memory=True)
    h_u.copy_(u)
    h_out = torch.empty(cu.out.shape, dtype=cu.out.dtype, pin_memory=True)
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for _ in range(2):
        u.copy_(h_u, non_blocking=True)
        step()
        h_out.copy_(cu.out, non_blocking=True)
    torch.cuda.synchronize(device)
    e2e_ev[0].record(stream)
    for _ in range(args.steps):
        u.copy_(h_u, non_blocking=True)
        step()
        h_out.copy_(cu.out, non_blocking=True)
    e2e_ev[1].record(stream)
    torch.cuda.synchronize(device)
    e2e_s = e2e_ev[0].elapsed_time(e2e_ev[1]) / 1e3
    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        import oracle
        oracle.catchup(**c)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 30.0) or reps == 0:
            oracle.catchup(**c)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": N * reps / dt, "unit": "backlog tokens/s", "cores": oracle.threads(), "kind": "oracle",
               "sample": f"{reps} whole oracle catch-up call(s) of this workload"}
    line = {"metric": CATCHUP_METRIC,
            "value": N * args.steps / (sum(ms) / 1e3), "unit": "backlog tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_mean, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": catchup_config(cfg),
            "launch": "wf_catchup captured in a CUDA graph" if not args.no_graph else "direct calls",
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": N * args.steps / e2e_s, "unit": "backlog tokens/s",
                    "h2d_bytes_per_step": int(h_u.numel() * h_u.element_size()),
                    "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size())},
            "clocks": clocks, "gpu_launches": 4 * args.steps, "impl": "ours"}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- side steps of a round
def op_inputs(op: str, B: int):
    """Seeded inputs of one --op call at the pages' tree shape (depth 8, top-10,
    60 draft nodes): per-step top-k children for tree construction; accepted
    paths of random 60-node trees and the rows' hidden states (d = 2560) for
    the kept rows.  Host-side structure only (no arithmetic of the method)."""
    from speculative_decoding_verify_lm_gb300 import synth
    rng = np.random.default_rng(20261202 + 3000 + (0 if op == "build_tree" else 1))
    if op == "build_tree":
        D, k, N = 8, 10, 60
        tid = rng.integers(0, 32000, (B, D, k, k)).astype(np.int32)
        lp = np.log(rng.dirichlet(np.ones(k) * 0.7, (B, D, k))).astype(np.float32)
        lp[lp < -60] = -60.0
        return dict(tid=tid, lp=lp, N=N)
    n_nodes, depth, d = 60, 8, 2560
    n = np.zeros(B, np.int32)
    path = np.full((B, depth), -1, np.int32)
    for b in range(B):
        parent, node_depth = synth.random_tree(rng, n_nodes, depth, 10)
        acc = int(rng.integers(0, depth + 1))
        n[b] = acc
        if acc:
            node = int(rng.choice(np.nonzero(node_depth == acc)[0]))
            chain = []
            while node >= 0:
                chain.append(node)
                node = int(parent[node])
            path[b, :acc] = chain[::-1]
    pos_off = (np.arange(B + 1) * (n_nodes + 1)).astype(np.int32)
    hidden = synth.normal_bf16(20261202 + 3001, 1, B * (n_nodes + 1), d, 1.0)
    return dict(n=n, path=path, pos_off=pos_off, hidden=hidden)


def op_oracle(op: str, x: dict):
    import oracle
    o = oracle.default()
    if op == "build_tree":
        return o.build_tree(x["tid"], x["lp"], x["N"])
    rows, off = o.accepted_rows(x["n"], x["path"], x["pos_off"])
    kept = np.concatenate([rows[b][:x["n"][b] + 1] for b in range(len(x["n"]))])
    return rows, off, x["hidden"][kept]


def op_config(op: str, B: int) -> dict:
    """The workload keys of a side step's JSON line, the same for both arms."""
    return {"workload": op_names(op, B)[0], "B": B, "l2": "L2 flushed (256 MB write) before every call"}


def op_names(op: str, B: int):
    if op == "build_tree":
        return (f"eagle3_tree_build_b{B}_d8_k10_n60", "EAGLE-3 draft-tree construction: trees built per second",
                "trees/s")
    return (f"kept_rows_b{B}_n60_d2560", "kept rows of the accepted paths: committed rows gathered per second",
            "rows/s")


def run_op_reference(args):
    """The oracle's side step on the host cores (the reference arm of --op)."""
    import oracle
    x = op_inputs(args.op, args.op_batch)
    name, metric, unit = op_names(args.op, args.op_batch)
    units = args.op_batch if args.op == "build_tree" else int(np.sum(x["n"] + 1))
    for _ in range(args.warmup):
        op_oracle(args.op, x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        op_oracle(args.op, x)
    dt = time.perf_counter() - t0
    val = units * args.steps / dt
    print(json.dumps({"impl": "reference", "metric": metric, "value": val, "unit": unit, "n_gpus": args.gpus,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic", "config": op_config(args.op, args.op_batch),
                      "cpu_baseline": {"value": val, "unit": unit, "cores": oracle.threads(), "kind": "oracle",
                                       "sample": "whole oracle calls of this workload"},
                      "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
          flush=True)


def run_op(args, rank, local, pg):
    import torch
    from speculative_decoding_verify_lm_gb300 import wf
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    B = args.op_batch
    x = op_inputs(args.op, B)
    name, metric, unit = op_names(args.op, B)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16  # noqa: E731
                                   else np.ascontiguousarray(a)).to(device)
    stream = torch.cuda.current_stream(device)
    ws = wf.Workspace(1, device=device)
    if args.op == "build_tree":
        N = x["N"]
        ins = [t(x["tid"]), t(x["lp"])]
        outs = [torch.empty((B, N), dtype=torch.int32, device=device), torch.empty((B, N), dtype=torch.int32,
                device=device), torch.empty((B, N), dtype=torch.float32, device=device),
                torch.empty((B, N), dtype=torch.int32, device=device)]
        D, k = x["tid"].shape[1], x["tid"].shape[2]

        def call():
            st = wf.lib().wf_build_tree(ins[0].data_ptr(), ins[1].data_ptr(), B, D, k, N,
                                        *(o_.data_ptr() for o_ in outs), ws.ptr, ws.nbytes, stream.cuda_stream)
            if st != 0:
                raise RuntimeError(f"wf_build_tree: status {st}")
        units = B
        nbytes = sum(a.numel() * a.element_size() for a in ins + outs)
        launches = 1
    else:
        d = x["hidden"].shape[1]
        total = int(np.sum(x["n"] + 1))
        ins = [t(x["n"]), t(x["path"]), t(x["pos_off"]), t(x["hidden"])]
        ps = x["path"].shape[1]
        outs = [torch.empty((B, ps + 1), dtype=torch.int32, device=device),
                torch.empty(B + 1, dtype=torch.int32, device=device),
                torch.empty((total, d), dtype=torch.int16, device=device)]

        def call():
            st = wf.lib().wf_accepted_rows(ins[0].data_ptr(), ins[1].data_ptr(), ps, ins[2].data_ptr(), B,
                                           outs[0].data_ptr(), outs[1].data_ptr(), ins[3].data_ptr(), d,
                                           outs[2].data_ptr(), stream.cuda_stream)
            if st != 0:
                raise RuntimeError(f"wf_accepted_rows: status {st}")
        units = total
        # the kept rows' hidden states are read and written once; the rest is small
        nbytes = 2 * total * d * 2 + sum(a.numel() * a.element_size() for a in ins[:3] + outs[:2])
        launches = 2
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(device)
    ref = op_oracle(args.op, x)   # the timed outputs are the oracle's
    got = [o_.cpu().numpy() for o_ in outs]
    if args.op == "build_tree":
        ok = all(np.array_equal(a, e) for a, e in zip(got, ref[:4]))
    else:
        ok = np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]) and \
            np.array_equal(got[2].view(np.uint16), ref[2])
    if not ok:
        raise RuntimeError(f"--op {args.op}: outputs disagree with the oracle")
    step = call
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        step = g.replay
        step()
    torch.cuda.synchronize(device)
    l2buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        l2buf.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    sampler.wait(ev[-1][1])
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_mean = statistics.mean(ms)
    hbm_peak, _, _, peak_src = measured_peaks()
    achieved = nbytes / (ms_mean / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": None, "kernel": "build_tree_kernel" if args.op == "build_tree"
            else "accepted_rows_kernel + gather_kept_kernel",
            "algorithmic_per_launch": nbytes, "launch_ms": ms_mean, "peak_source": f"{peak_src} (hbm_gbs, burst)"}
    # end to end: the inputs in from pinned host memory, every output back
    h_in = [torch.empty(a.shape, dtype=a.dtype, pin_memory=True) for a in ins]
    for h_, a in zip(h_in, ins):
        h_.copy_(a)
    h_out = [torch.empty(a.shape, dtype=a.dtype, pin_memory=True) for a in outs]
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def host_step():
        for a, h_ in zip(ins, h_in):
            a.copy_(h_, non_blocking=True)
        step()
        for h_, a in zip(h_out, outs):
            h_.copy_(a, non_blocking=True)
    host_step()
    torch.cuda.synchronize(device)
    e2e_ev[0].record(stream)
    for _ in range(args.steps):
        host_step()
    e2e_ev[1].record(stream)
    torch.cuda.synchronize(device)
    e2e_s = e2e_ev[0].elapsed_time(e2e_ev[1]) / 1e3
    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        import oracle
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0) or reps == 0:
            op_oracle(args.op, x)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": units * reps / dt, "unit": unit, "cores": oracle.threads(), "kind": "oracle",
               "sample": f"{reps} whole oracle call(s) of this workload"}
    line = {"metric": metric, "value": units * args.steps / (sum(ms) / 1e3), "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_mean, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32" if args.op == "build_tree" else "bf16",
            "data": "synthetic",
            "config": op_config(args.op, B),
            "launch": "captured in a CUDA graph" if not args.no_graph else "direct calls",
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": units * args.steps / e2e_s, "unit": unit,
                    "h2d_bytes_per_step": int(sum(a.numel() * a.element_size() for a in ins)),
                    "d2h_bytes_per_step": int(sum(a.numel() * a.element_size() for a in outs))},
            "clocks": clocks, "gpu_launches": launches * args.steps, "impl": "ours"}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def main():
    args = parse()
    world, rank, local, pg = dist_setup(args)
    if args.op is not None:
        if args.impl == "reference":
            if rank == 0:
                run_op_reference(args)
            return
        run_op(args, rank, local, pg)
        return
    if args.catchup is not None:
        if args.impl == "reference":
            if rank == 0:
                run_catchup_reference(args)
            return
        run_catchup(args, rank, local, pg)
        return
    from speculative_decoding_verify_lm_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    cfg_name = cfg.name if args.router_width is None else f"{cfg.name}_m{args.router_width}"
    entropy = args.router == "entropy"
    if entropy:
        cfg_name += "_entropy"
    # both arms: the inputs the oracle's stored answers were computed on
    wl = load_workload(args.config, m=args.router_width)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg_name, cfg, wl, world)
        return

    import torch
    from speculative_decoding_verify_lm_gb300 import wf
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wf.lib()

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16  # noqa: E731
                                   else np.ascontiguousarray(a)).to(device)
    Wdev = t(wl.W)
    draft = wl.Wd is not None
    r = wf.Round(t(wl.hidden), Wdev, t(wl.pos_off), t(wl.node_off), t(wl.tok), t(wl.W1), t(wl.b1), t(wl.w2),
                 wl.b2, wl.tau, kind=t(wl.kind), parent=t(wl.parent), path_stride=wl.max_depth,
                 x=t(wl.x) if draft else None, Wd=t(wl.Wd) if draft else None, d2t=t(wl.d2t) if draft else None,
                 k=wl.topk if draft else 0, router_kind=wf.WF_ROUTER_ENTROPY if entropy else wf.WF_ROUTER_NEURAL)
    P, B, d, V = wl.P, wl.B, cfg.d, cfg.V
    weight_bytes = V * d * 2 + (wl.Wd.nbytes if draft else 0) + wl.W1.nbytes
    flush = flush_l2(weight_bytes)
    l2buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if flush else None
    stream = torch.cuda.current_stream(device)

    for _ in range(max(args.warmup, 3)):
        r()
    torch.cuda.synchronize(device)
    code, info = r.ws.device_error()
    if code:
        raise RuntimeError(f"device error {code} (info {info}) during warm-up")
    # the round's launches captured once in a CUDA graph and replayed per step
    step = r
    if not args.no_graph:
        ref_ids = r.out["ids"].clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            r()
        step = g.replay
        for _ in range(2):
            step()
        torch.cuda.synchronize(device)
        if not torch.equal(ref_ids, r.out["ids"]):
            raise RuntimeError("graph replay disagrees with a direct wf_round call")

    # ---- the dominant kernel on its own: the shared sweep of both heads
    # (timed with its top-k merge) or the LM head alone (with the entropy
    # statistics under entropy routing, when one sweep yields them)
    shared = draft and (B <= 128 if P <= 128 else B <= 256) and not (entropy and P <= 128)
    ent_fused = entropy and P <= 128
    hbm_peak, tc_peak, tc_sus, peak_src = measured_peaks()
    ids_buf = torch.empty(P, dtype=torch.int32, device=device)
    hdev = r.inputs["hidden"]
    if shared:
        k = wl.topk
        ws1 = wf.Workspace(P, B, 1, wl.Wd.shape[0], k, device=device, d=d)
        xdev, Wddev, d2tdev = r.inputs["x"], r.inputs["Wd"], r.inputs["d2t"]
        dbufs = dict(draft_ids=torch.empty((B, k), dtype=torch.int32, device=device),
                     tids=torch.empty((B, k), dtype=torch.int32, device=device),
                     vals=torch.empty((B, k), dtype=torch.float32, device=device))
        kernel_call = lambda: wf.wf_lmhead_draft_topk(hdev, Wdev, xdev, Wddev, d2tdev, k, ws1,  # noqa: E731
                                                      ids=ids_buf, **dbufs)
        Vd = wl.Wd.shape[0]
        alg_bytes = (V + Vd) * d * 2 + (P + B) * d * 2 + Vd * 4 + P * 4 + B * k * 12
        alg_flops = 2.0 * d * (P * V + B * Vd)
        # several activation tiles: the paired-CTA sweep
        kernel_name, kernel_launches = f"gemm_select_kernel<1,0,1,{int(P > 128)}>", 2
    elif ent_fused:
        ws1 = wf.Workspace(P, P, d=d, device=device)
        Hbuf = torch.empty(P, dtype=torch.float32, device=device)
        rbuf = torch.empty(P, dtype=torch.int32, device=device)
        kernel_call = lambda: wf.wf_lmhead_entropy(hdev, Wdev, wl.tau, ws1, H=Hbuf, route=rbuf)  # noqa: E731
        alg_bytes = V * d * 2 + P * d * 2 + P * 8
        alg_flops = 2.0 * P * V * d
        kernel_name, kernel_launches = "gemm_select_kernel<1,1,0,0>", 1
    else:
        ws1 = wf.Workspace(P, device=device)
        kernel_call = lambda: wf.wf_lmhead_argmax(hdev, Wdev, ws1, ids=ids_buf)  # noqa: E731
        alg_bytes = V * d * 2 + P * d * 2 + P * 4
        alg_flops = 2.0 * P * V * d
        # several activation tiles: the paired-CTA sweep
        kernel_name, kernel_launches = f"gemm_select_kernel<1,0,0,{int(P > 128)}>", 1
    for _ in range(3):
        kernel_call()
    if not args.no_graph:   # replayed from a CUDA graph: host argument checks stay out of the events
        kg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kg):
            kernel_call()
        kernel_call = kg.replay
        kernel_call()
    torch.cuda.synchronize(device)

    # ---- timed region: K steps.  Each step is one whole round, then the
    # dominant kernel alone, both on this stream between CUDA events (after an
    # L2 flush when the weights would fit in L2), so both see the same clocks
    # and power state.  Every step is queued before the first one ends (an
    # idle GPU would put the host's launch latency between the events); the
    # host then reads the SM clock while it waits for each step to end.
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize(device)
    try:   # the physical GPU behind this rank's device (CUDA_VISIBLE_DEVICES may renumber)
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk(), mk(), mk()) for _ in range(args.steps)]
    step_mhz = []

    def wait_step(j):
        n0 = len(sampler.sm)
        sampler.wait(ev[j][3])
        step_mhz.append(statistics.median(sampler.sm[n0:]) if len(sampler.sm) > n0 else None)

    for i in range(args.steps):
        if flush:
            l2buf.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        if flush:
            l2buf.zero_()
        ev[i][2].record(stream)
        kernel_call()
        ev[i][3].record(stream)
    for i in range(args.steps):
        wait_step(i)
    torch.cuda.synchronize(device)
    if pg is not None:
        pg.barrier()
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    k_ms_all = [e[2].elapsed_time(e[3]) for e in ev]
    dev_s = sum(step_ms) / 1e3
    out = {k_: (v.cpu().numpy() if v is not None else None) for k_, v in r.out.items()}
    accepted = int((out["n_accept"] + 1).sum())
    max_s = allreduce_max(pg, dev_s, device)
    tot_rows = allreduce_sum(pg, P * args.steps, device)
    tot_acc = allreduce_sum(pg, accepted * args.steps, device)
    value = tot_rows / max_s
    launches_per_round = round_launches(P, B, draft, entropy)

    k_ms = statistics.mean(k_ms_all)
    k_med = statistics.median(k_ms_all)
    hbm_bound = alg_flops / alg_bytes < (tc_peak * 1e12) / (hbm_peak * 1e9)
    if hbm_bound:
        achieved = alg_bytes / (k_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "frac_of_median_launch": alg_bytes / (k_med / 1e3) / 1e9 / hbm_peak}
    else:
        achieved = alg_flops / (k_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "frac_of_median_launch": alg_flops / (k_med / 1e3) / 1e12 / tc_peak,
                "peak_sustained": tc_sus, "frac_sustained": achieved / tc_sus}
    roof.update({"traffic": traffic_for(kernel_name, cfg_name), "kernel": kernel_name,
                 "algorithmic_per_launch": alg_bytes if hbm_bound else alg_flops, "launch_ms": k_ms,
                 "launch_ms_median": k_med,
                 "peak_source": f"{peak_src} ({'hbm_gbs' if hbm_bound else 'bf16_tflops'}, burst)"})

    # ---- end to end through the public API: every step copies the round's inputs
    # (hidden states, drafts, trees, offsets, drafter states) from one pinned host
    # buffer, runs wf_round and reads every output back into one pinned buffer
    host_in = r.pinned_inputs()
    host_out = r.pinned_outputs()
    h2d, d2h = host_in.numel(), host_out.numel()
    for _ in range(2):
        r.upload(host_in)
        r()
        r.download(host_out)
        torch.cuda.synchronize(device)
    if not args.no_graph:   # the step (copy in, round, copy out) replayed as one CUDA graph
        r.capture_host_step(host_in, host_out)
        run_step = r.replay_host_step
    else:
        def run_step():
            r.upload(host_in)
            r()
            r.download(host_out)
    for _ in range(2):
        run_step()
        torch.cuda.synchronize(device)
    if pg is not None:
        pg.barrier()
    e2e_s = 0.0   # per-step wall clock: copy in, round, copy out, synchronise (L2 flush excluded)
    for i in range(args.steps):
        if flush:
            l2buf.zero_()
        torch.cuda.synchronize(device)
        t1 = time.perf_counter()
        run_step()
        torch.cuda.synchronize(device)
        e2e_s += time.perf_counter() - t1
    got = r.host_views(host_out)
    if not np.array_equal(got["n_accept"].numpy(), r.out["n_accept"].cpu().numpy()):
        raise RuntimeError("end-to-end outputs disagree with the device outputs")
    e2e_max = allreduce_max(pg, e2e_s, device)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        v, sample, cores, _, _ = cpu_sample(wl, args.cpu_seconds, entropy)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": sum(step_ms) / len(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": round_config(cfg_name, cfg, wl, entropy, world),
        "launch": "direct wf_round calls" if args.no_graph else "wf_round captured in a CUDA graph",
        "ms_per_step_median": statistics.median(step_ms),
        "accepted_tokens_per_s": tot_acc / max_s,
        "mean_acceptance_length": accepted / B,
        "roofline": roof,
        "samples": [{"round_ms": round(a, 5), "kernel_ms": round(b, 5), "sm_mhz": c}
                    for a, b, c in zip(step_ms, k_ms_all, step_mhz)],
        "cpu_baseline": cpu,
        "e2e": {"value": tot_rows / e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        # the round's launches and the dominant kernel's own, every step of the timed region
        "gpu_launches": (launches_per_round + kernel_launches) * args.steps,
        "impl": "ours",
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
