"""Benchmark of the verification step on GB300.

Default workload: batched mentored speculative sampling, B=64 requests,
K=8 drafts, V=152064, bf16 logits (330.9 MB of logits per step, larger than
the 129 MB L2; two input copies alternate between steps).  One step = one
``spec_verify_sample`` call over the whole batch.

Prints one JSON line:
  value      verified requests per second (all ranks), inputs resident in HBM
  e2e        the same through the C ABI with pinned host buffers: the step's
             inputs copied host->device and tokens/accepted copied back inside
             the timed region
  roofline   the sampling kernel against the measured HBM copy peak
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

``--impl reference`` times the CPU oracle itself (one bounded sample per
step) and prints its line with "impl": "reference".  ``--profile`` runs the
ncu launch list and one capture of the sampling kernel and writes
profiles/seg_verify_kernel_batched.json.  ``--gpus N`` outside torchrun
starts N ranks itself (or refuses when fewer GPUs are visible).

Multi-GPU: one process per GPU under torchrun; requests are independent, so
each rank verifies its own batch (weak scaling, no data-path collective; a
barrier and a max-reduce of the elapsed time only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

KERNEL_SOURCES = ["speculative_decoding_verification_23_gb300/csrc/seg_verify.cu",
                  "speculative_decoding_verification_23_gb300/csrc/seg_internal.h",
                  "speculative_decoding_verification_23_gb300/csrc/stream_common.cuh",
                  "speculative_decoding_verification_23_gb300/csrc/common.cuh",
                  "speculative_decoding_verification_23_gb300/csrc/spec_internal.h"]
KERNEL = "seg_verify_kernel"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "seg_verify_kernel_batched.json")
WORKLOAD = "batched B=64 K=8 V=152064 bf16 logits"
CLOCK_WINDOW_S = 0.2           # the K-step window repeats until this much time has passed
METRIC = "spec-verify rows/s and logits HBM GB/s (% of GB300 peak) at B=64 K=8 V=152064"


TOPP_SOURCES = ["speculative_decoding_verification_23_gb300/csrc/topp_verify.cu",
                "speculative_decoding_verification_23_gb300/csrc/topp_internal.h",
                "speculative_decoding_verification_23_gb300/csrc/common.cuh"]
TOPP_SUMMARY = os.path.join(ROOT, "profiles", "topp_kernels_ragged.json")


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed
    region.  Reads NVML through ctypes every millisecond (read-only queries;
    nothing is set), so that even a timed region of a few milliseconds gets
    samples; falls back to ``nvidia-smi -lms 100`` when NVML cannot load."""

    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.device = device
        self.samples = []           # (sm_mhz, max_mhz, reasons_mask)
        self.stop = threading.Event()
        self.proc = None
        self.thread = None
        self.source = None

    def _nvml_handle(self):
        import ctypes

        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        import torch

        pr = torch.cuda.get_device_properties(self.device)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if nvml.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle for " + bus.decode())
        reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        return nvml, h, reasons

    def _poll_nvml(self, nvml, h, reasons):
        import ctypes

        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))          # NVML_CLOCK_SM = 1
        while True:
            if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), float(mx.value), int(rs.value)))
            if self.stop.wait(0.001):
                break

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            mask = 0
            for bit, v in zip((0x8, 0x40, 0x20, 0x4), parts[5:9]):
                if v.lower().startswith("active"):
                    mask |= bit
            self.samples.append((sm, mx, mask))

    def __enter__(self):
        try:
            nvml, h, reasons = self._nvml_handle()
            self.thread = threading.Thread(target=self._poll_nvml, args=(nvml, h, reasons), daemon=True)
            self.source = "nvml 1 ms"
        except (OSError, AttributeError):
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.device.index}", f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "100"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.thread = threading.Thread(target=self._read_smi, daemon=True)
                self.source = "nvidia-smi 100 ms"
            except FileNotFoundError:
                return self
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        mask = 0
        for _, _, m in self.samples:
            mask |= m
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples),
                "reasons": sorted(n for b, n in self.REASONS.items() if mask & b),
                "samples": len(self.samples), "source": self.source}


def oracle_baseline(batch, budget_s: float, results=None):
    """Requests/s of the CPU oracle on a bounded sample: whole requests of the
    batch in order, cycling through the batch until `budget_s` has passed.
    With `results` (a dict), each request's oracle outputs are kept there."""
    import oracle

    t0 = time.perf_counter()
    n = 0
    while True:
        b = n % batch.B
        r = oracle.verify_batch(batch, [b])
        if results is not None and b not in results:
            off = int(batch.cu_draft[b]) + b
            results[b] = (r["tokens"][off:off + batch.k(b) + 1].copy(), int(r["accepted"][b]),
                          int(r["status"][b]), bool(r["near_tie"][b]))
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def _oracle_worker(args):
    round_, first, budget_s = args
    import oracle

    batch = make_workload(round_)
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < budget_s:
        oracle.verify_batch(batch, [(first + n) % batch.B])
        n += 1
    return n, time.perf_counter() - t0


def oracle_all_cores(round_: int, budget_s: float):
    """The same oracle on every host core at once (one process per core,
    started with spawn): requests/s summed over the workers, and the cores."""
    import multiprocessing as mp

    cores = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(round_, i, budget_s) for i in range(cores)])
    return sum(n / dt for n, dt in res), cores


def parity_sample(got, results, batch):
    """GPU outputs against the oracle's on the requests the CPU sample ran:
    (requests compared, mismatches, near ties)."""
    tok, acc, st = got
    bad = near = 0
    for b, (rt, ra, rs, nt) in results.items():
        if nt:
            near += 1
            continue
        off = int(batch.cu_draft[b]) + b
        if not (np.array_equal(tok[off:off + batch.k(b) + 1], rt) and acc[b] == ra and st[b] == rs):
            bad += 1
    return len(results), bad, near


def reduce_max(x: float, dist, device) -> float:
    """The largest value of `x` over all ranks (the job takes as long as its
    slowest rank); `x` itself without a process group."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, steps: int, elapsed_max: float) -> float:
    """Whole-job units per second: every rank processes `units_per_rank` per
    step (weak scaling), the job lasts the slowest rank's time."""
    return world * units_per_rank * steps / elapsed_max


def make_workload(rank: int):
    from speculative_decoding_verification_23_gb300 import workload as W

    return W.batched(round_=rank)


def bench_config(world: int) -> dict:
    """The workload the line is quoted on (the same for both arms)."""
    return {"workload": WORKLOAD, "B": 64, "K": 8, "V": 152064, "logit_bytes_per_step": 330891264,
            "parallelism": f"replicas x{world}",
            "l2": "inputs 330.9 MB > 129 MB L2; two input copies alternate"}


def bench_reference(args, rank, world):
    batch = make_workload(rank)
    per_step_budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_baseline(batch, min(per_step_budget, 2.0))
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, n, dt = oracle_baseline(batch, per_step_budget)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "requests/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(world),
        "cpu_baseline": {"value": value, "unit": "requests/s", "cores": 1, "kind": "oracle",
                         "sample": f"whole requests of the B=64 batch, ~{per_step_budget:.1f} s of CPU per step"},
        "e2e": {"value": value, "unit": "requests/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_gpu(args, rank, world, dist):
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library()
    batch = make_workload(rank)
    copies = [to_device(batch, dev) for _ in range(2)]
    ws = sv.make_workspace(batch.B, batch.total_drafts, batch.V, dev)
    outs = [torch.empty(batch.total_drafts + batch.B, dtype=torch.int32, device=dev),
            torch.empty(batch.B, dtype=torch.int32, device=dev),
            torch.empty(batch.B, dtype=torch.int32, device=dev)]
    argv = [c.args() for c in copies]
    stream = torch.cuda.current_stream(dev)

    def step(k):
        sv.spec_verify_sample(argv[k % 2], device=dev, workspace=ws, out_tokens=outs[0], out_accepted=outs[1],
                              out_status=outs[2], stream=stream)

    warm = max(3, args.warmup)
    for k in range(warm):
        step(k)
    torch.cuda.synchronize()
    assert int(outs[2].max().item()) == 0, "bench inputs flagged invalid"

    # ---- timed windows of exactly K steps, repeated (the same count on
    # every rank) until CLOCK_WINDOW_S of wall time has passed, clocks
    # sampled throughout
    per_launch, win_s = [], []
    n_win = 0
    t_wall = time.perf_counter()
    torch.cuda.nvtx.range_push("bench: timed windows")
    with ClockSampler(dev) as clk:
        while n_win == 0 or reduce_max(float(time.perf_counter() - t_wall < CLOCK_WINDOW_S), dist, dev) > 0:
            n_win += 1
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for k in range(args.steps):
                ev[k][0].record(stream)
                step(k)
                ev[k][1].record(stream)
            t_end.record(stream)
            torch.cuda.synchronize()
            win_s.append(reduce_max(t_start.elapsed_time(t_end) / 1000.0, dist, dev))
            per_launch += [x.elapsed_time(y) / 1000.0 for x, y in ev]
    torch.cuda.nvtx.range_pop()
    elapsed = float(np.median(win_s))
    if dist:
        dist.barrier()
    value = job_throughput(batch.B, world, args.steps, elapsed)
    ms = 1000.0 * elapsed / args.steps
    got = [t.cpu().numpy() for t in outs]

    # ---- end to end over the same K steps: pinned host inputs -> device ->
    # call -> tokens and accepted counts back
    host = {
        "target": copies[0].target.cpu().pin_memory(), "draft": copies[0].draft.cpu().pin_memory(),
        "small": [t.cpu().pin_memory() for t in (copies[0].cu_draft, copies[0].draft_tokens, copies[0].cu_hist,
                                                 copies[0].hist, copies[0].temperature, copies[0].rep_penalty,
                                                 copies[0].tv_budget, copies[0].uniforms)],
    }
    dstc = copies[1]
    dsmall = [dstc.cu_draft, dstc.draft_tokens, dstc.cu_hist, dstc.hist, dstc.temperature, dstc.rep_penalty,
              dstc.tv_budget, dstc.uniforms]
    out_host = [torch.empty_like(outs[0], device="cpu").pin_memory(),
                torch.empty_like(outs[1], device="cpu").pin_memory()]
    h2d = host["target"].numel() * host["target"].element_size() + host["draft"].numel() * host["draft"].element_size()
    h2d += sum(t.numel() * t.element_size() for t in host["small"])
    d2h = sum(t.numel() * t.element_size() for t in out_host)

    def e2e_step():
        dstc.target.copy_(host["target"], non_blocking=True)
        dstc.draft.copy_(host["draft"], non_blocking=True)
        for d, h in zip(dsmall, host["small"]):
            d.copy_(h, non_blocking=True)
        sv.spec_verify_sample(argv[1], device=dev, workspace=ws, out_tokens=outs[0], out_accepted=outs[1],
                              out_status=outs[2], stream=stream)
        out_host[0].copy_(outs[0], non_blocking=True)
        out_host[1].copy_(outs[1], non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("bench: end to end")
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    e2e_value = job_throughput(batch.B, world, args.steps, reduce_max(a.elapsed_time(b) / 1000.0, dist, dev))

    # ---- roofline of the sampling kernel (one launch per step, after the
    # call's clear of its counters)
    peak, peak_kind = measured_peak()
    alg_bytes = batch.logit_bytes() + 4 * (batch.total_drafts + batch.B) * 2 + 4 * int(batch.hist.size) + 4 * 4 * batch.B
    launch_s = float(np.mean(per_launch))
    achieved = alg_bytes / launch_s / 1e9
    traffic = None
    if os.path.exists(PROFILE_SUMMARY):
        with open(PROFILE_SUMMARY) as f:
            prof = json.load(f)
        if prof.get("kernel_hash") == kernel_hash():
            traffic = prof.get("dram_bytes_per_launch")

    line = {
        "metric": METRIC, "value": value, "unit": "requests/s", "n_gpus": world, "steps": args.steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": bench_config(world),
        "windows": {"count": n_win, "ms_per_step": [round(1000.0 * w / args.steps, 4) for w in win_s],
                    "value_from": "median window"},
        "logit_rows_per_s": value * (2 * 8 + 1),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": peak_kind, "kernel": KERNEL,
                     "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": 1000 * launch_s,
                     "launch_timing": "CUDA events around each call on its stream (one kernel launch)"},
        "e2e": {"value": e2e_value, "unit": "requests/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": args.steps},
        "gpu_launches": args.steps * n_win,
        "clocks": clk.summary(),
    }
    if rank == 0 and args.extras:
        line["extras"] = bench_extras(dev, peak, args.cpu_seconds)
    if rank == 0 and not args.no_cpu_baseline:
        results = {}
        v, n, dt = oracle_baseline(batch, args.cpu_seconds, results)
        v_all, cores = oracle_all_cores(rank, max(2.0, args.cpu_seconds / 3))
        line["cpu_baseline"] = {"value": v, "unit": "requests/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} whole requests cycled through the B=64 batch ({dt:.1f} s, one thread)",
                                "all_cores": {"value": v_all, "cores": cores,
                                              "sample": "one spawned process per core, each cycling through the batch"}}
        checked, bad, near = parity_sample(got, results, batch)
        line["parity"] = {"requests_checked": checked, "mismatches": bad, "near_ties": near,
                          "rule": "tokens, accepted and status equal to the oracle's for every request "
                                  "not within 1e-6 of a decision threshold"}
        line["near_ties"] = near
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_extras(dev, peak: float, cpu_seconds: float) -> dict:
    """The other configurations and entry points, one call at a time with
    L2 flushed before each (a 256 MB write), CUDA events around the call:
    the Qwen2.5-shaped single request (B=1, K=8, resident cluster kernel),
    greedy verification (B=1, K in 1/2/4/8), the ragged top-p batch (B=256,
    fp32, cluster kernel with top-p), and spec_tv_budget and
    spec_draft_confidence on the batched workload.  Each with algorithmic bytes, achieved GB/s against the
    measured peak, and the oracle's requests/s on a bounded sample."""
    import torch

    import oracle
    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300 import workload as W
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(call, iters=20):
        for _ in range(3):
            call()
        ts = []
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) / 1000.0)
        return float(np.median(ts))

    def oracle_rate(fn, batch, budget):
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < budget:
            fn(batch, [n % batch.B])
            n += 1
        return n / (time.perf_counter() - t0)

    def line(name, bytes_, sec, rate, kernel):
        ach = bytes_ / sec / 1e9
        return {"ms": 1000.0 * sec, "bytes": int(bytes_), "achieved_gbs": ach, "frac": ach / peak,
                "kernel": kernel, "oracle_requests_per_s": rate}

    out = {}
    budget = max(1.0, cpu_seconds / 6)
    small = 4 * (2 * 9 + 1) + 4 * 256 + 16
    b1 = W.qwen25_single(0.5)
    d1 = to_device(b1, dev)
    ws1 = sv.make_workspace(b1.B, b1.total_drafts, b1.V, dev)
    a1 = d1.args()
    sec = timed(lambda: sv.spec_verify_sample(a1, device=dev, workspace=ws1, stream=stream))
    out["qwen25_single_B1_K8"] = line("qwen", b1.logit_bytes() + small, sec,
                                      oracle_rate(oracle.verify_batch, b1, budget), "sample_verify_kernel (resident)")
    a1s = d1.args(flags=8)
    calls = [("resident (default)", lambda: sv.spec_verify_sample(a1, device=dev, workspace=ws1, stream=stream)),
             ("split", lambda: sv.spec_verify_sample(a1s, device=dev, workspace=ws1, stream=stream))]
    bg8 = W.greedy_single(8)
    dg8 = to_device(bg8, dev)
    wsg8 = sv.make_workspace(bg8.B, bg8.total_drafts, bg8.V, dev)
    ag8 = dg8.args()
    calls.append(("greedy K=8", lambda: sv.spec_verify_greedy(ag8, device=dev, workspace=wsg8, stream=stream)))
    out["B1_breakdown"] = small_batch_breakdown(dev, calls, stream)
    del dg8, wsg8
    for K in (1, 2, 4, 8):
        bg = W.greedy_single(K)
        dg = to_device(bg, dev)
        wsg = sv.make_workspace(bg.B, bg.total_drafts, bg.V, dev)
        ag = dg.args()
        sec = timed(lambda: sv.spec_verify_greedy(ag, device=dev, workspace=wsg, stream=stream))
        gbytes = (K + 1) * bg.V * 2 + 4 * (2 * K + 2)
        out[f"greedy_B1_K{K}"] = line("greedy", gbytes, sec, oracle_rate(oracle.greedy_batch, bg, budget / 2),
                                      "greedy_verify_kernel")
        del dg, wsg
    br = W.ragged_top_p(0)
    dr = to_device(br, dev)
    wsr = sv.make_workspace(br.B, br.total_drafts, br.V, dev)
    ar = dr.args()
    sec = timed(lambda: sv.spec_verify_sample(ar, device=dev, workspace=wsr, stream=stream), iters=10)
    out["ragged_top_p_B256_fp32"] = line("ragged", br.logit_bytes() + 8 * (br.total_drafts + br.B) + 16 * br.B,
                                         sec, oracle_rate(oracle.verify_batch, br, budget),
                                         "topp_cut_kernel + topp_finish_kernel")
    del dr, wsr
    bb = make_workload(0)
    db = to_device(bb, dev)
    wsb = sv.make_workspace(bb.B, bb.total_drafts, bb.V, dev)
    ab = db.args()
    sec = timed(lambda: sv.spec_tv_budget(ab, device=dev, workspace=wsb, stream=stream))
    tvbytes = 2 * bb.total_drafts * bb.V * 2 + 4 * int(bb.hist.size) + 16 * bb.total_drafts
    out["tv_budget_batched_B64_K8"] = line("tv", tvbytes, sec, None, "pipe_verify_kernel (TV only)")
    sec = timed(lambda: sv.spec_draft_confidence(ab, 0.6, device=dev, workspace=wsb, stream=stream))
    cbytes = bb.total_drafts * bb.V * 2 + 4 * int(bb.hist.size) + 8 * bb.total_drafts
    rate = oracle_rate(lambda batch, reqs: oracle.draft_confidence_batch(batch, 0.6, reqs), bb, budget)
    out["draft_confidence_batched_B64_K8"] = line("conf", cbytes, sec, rate, "conf_pipe_kernel (pipelined)")
    del db, wsb
    out["acceptance_qwen25_K8"] = acceptance_sweep(dev)
    return out


def small_batch_breakdown(dev, calls, stream, iters: int = 200) -> dict:
    """Where a B=1 call's time goes, for each (name, call) given: the host's
    time to check the arguments and enqueue the work (no synchronisation),
    the GPU span of one call (CUDA events around it, L2 warm), the GPU span
    of the same calls issued back to back (launches overlap the host), and
    the span of an empty device operation on the stream (the floor any
    launch pays).  Every call is one kernel launch."""
    import torch

    res = {}
    for name, call in calls:
        for _ in range(10):
            call()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(iters):
            call()
        host_us = 1e6 * (time.perf_counter() - t0) / iters
        torch.cuda.synchronize()
        spans = []
        for _ in range(50):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            spans.append(a.elapsed_time(b) * 1000.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            call()
        b.record(stream)
        b.synchronize()
        res[name] = {"host_enqueue_us": round(host_us, 2), "gpu_span_us": round(float(np.median(spans)), 2),
                     "back_to_back_us": round(a.elapsed_time(b) * 1000.0 / iters, 2),
                     "launches_per_call": 1}
    x = torch.empty(1, device=dev)
    spans = []
    for _ in range(50):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x.zero_()
        b.record(stream)
        b.synchronize()
        spans.append(a.elapsed_time(b) * 1000.0)
    res["empty_operation_us"] = round(float(np.median(spans)), 2)
    return res


def acceptance_sweep(dev, batches: int = 8, per: int = 32) -> dict:
    """Acceptance statistics of the GPU path on the Qwen2.5-shaped rows
    (V=152064, bf16, K=8, rho=0.9, T=0.7, no repetition penalty so that the
    drafts are draws from q): for each TV budget D, batches * per rounds over
    the same rows with fresh drafts and uniforms; per position the observed
    acceptance rate against 1 - max(0, d_i - D) (d_i from spec_tv_budget),
    and per K' in 1/2/4/8 the accepted and emitted tokens per round, with and
    without the bonus."""
    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300 import acceptance as A
    from speculative_decoding_verification_23_gb300 import workload as W
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    res = {}
    for D in (0.0, 0.5, 0.75, 1.0):
        one = to_device(W.acceptance_trials(D, 1), dev)
        d = sv.spec_tv_budget(one.args(), device=dev)[0].cpu().numpy().astype(np.float64)
        accs = []
        for t in range(batches):
            db = to_device(W.acceptance_trials(D, per, draws=1 + t), dev)
            _, acc, st = sv.spec_verify_sample(db.args(), device=dev)
            assert int(st.abs().max()) == 0
            accs.append(acc.cpu().numpy())
            del db
        rep = A.acceptance_report(np.concatenate(accs), d, D)
        res[f"D{D}"] = {
            "rounds": rep["rounds"],
            "d": [round(x, 5) for x in rep["d"]],
            "rate": [round(p["rate"], 4) for p in rep["positions"]],
            "expected": [round(p["expected"], 4) for p in rep["positions"]],
            "max_abs_z": round(max((abs(p["z"]) for p in rep["positions"] if p["z"] == p["z"]), default=0.0), 2),
            "k_sweep": [{k: (round(v, 4) if isinstance(v, float) else v) for k, v in s.items()} for s in rep["k_sweep"]],
        }
    return res


def relaunch(args) -> int:
    """`--gpus N` outside torchrun: run N ranks of this script, one per GPU
    (torch.distributed.run on 127.0.0.1), or refuse when there are fewer
    GPUs.  Returns the exit code."""
    import torch

    have = torch.cuda.device_count()
    if have < args.gpus:
        print(json.dumps({"error": f"--gpus {args.gpus} asked for, {have} GPU(s) visible; refusing"}), flush=True)
        return 2
    import socket

    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def profile(args) -> int:
    """`--profile`: the launch list of a short bench run and one full capture
    of the sampling kernel under ncu (clocks left alone), summarised into
    profiles/<kernel>_batched.json (DRAM bytes per launch, duration, the
    kernel's share of the launches) with the kernel sources' hash.  Run
    only where the same command has run cleanly without ncu."""
    import csv

    os.makedirs(os.path.join(ROOT, "gpurun_out"), exist_ok=True)
    base = [sys.executable, os.path.abspath(__file__), "--steps", "3", "--warmup", "3", "--no-cpu-baseline"]
    if subprocess.call(base, stdout=subprocess.DEVNULL) != 0:
        print("plain run failed; not profiling", file=sys.stderr)
        return 1
    launches = os.path.join(ROOT, "gpurun_out", "launches.csv")
    rc = subprocess.call(["ncu", "--metrics", "gpu__time_duration.sum", "--clock-control", "none", "-c", "400",
                          "--csv", "--log-file", launches] + base, stdout=subprocess.DEVNULL)
    if rc:
        return rc
    rep = os.path.join(ROOT, "gpurun_out", "prof_" + KERNEL)
    rc = subprocess.call(["ncu", "--set", "full", "--clock-control", "none", "-k", "regex:" + KERNEL, "-s", "4",
                          "-c", "1", "-f", "-o", rep] + base, stdout=subprocess.DEVNULL)
    if rc:
        return rc
    raw = subprocess.run(["ncu", "-i", rep + ".ncu-rep", "--page", "raw", "--csv"], capture_output=True,
                         text=True).stdout
    rows = list(csv.reader(raw.splitlines()))
    hdr, vals = rows[0], rows[2]
    get = lambda k: float(vals[hdr.index(k)].replace(",", ""))
    names, times = [], []
    per_ns = {"nsecond": 1.0, "ns": 1.0, "usecond": 1e3, "us": 1e3, "msecond": 1e6, "ms": 1e6, "second": 1e9,
              "s": 1e9}
    with open(launches) as f:
        lines = [l for l in f if l.startswith('"')]
    for r in csv.DictReader(lines):
        if r.get("Metric Name") == "gpu__time_duration.sum":
            names.append(r["Kernel Name"])
            times.append(float(r["Metric Value"].replace(",", "")) * per_ns.get(r.get("Metric Unit", ""), 1.0))
    tot = sum(times) or 1.0
    mine = [t for n, t in zip(names, times) if KERNEL in n]
    rd, wr = get("dram__bytes_read.sum"), get("dram__bytes_write.sum")
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(rows[1][hdr.index("dram__bytes_read.sum")], 1)
    dur = get("gpu__time_duration.sum") * per_ns.get(rows[1][hdr.index("gpu__time_duration.sum")], 1.0) / 1e3
    out = {"kernel": KERNEL, "workload": WORKLOAD, "kernel_hash": kernel_hash(),
           "dram_bytes_per_launch": int((rd + wr) * scale), "dram_read_bytes": int(rd * scale),
           "dram_write_bytes": int(wr * scale),
           "duration_us_under_ncu": dur,
           "launch_list": {"launches": len(names), "kernel_launches": len(mine), "kernel_share": sum(mine) / tot},
           "command": "python bench.py --profile"}
    for path in (PROFILE_SUMMARY, os.path.join(ROOT, "gpurun_out", os.path.basename(PROFILE_SUMMARY))):
        with open(path, "w") as f:
            json.dump(out, f, indent=2)
    print(json.dumps(out), flush=True)
    return 0


def topp_run() -> int:
    """`--topp-run`: three top-p calls on the ragged workload (B=256, K 1..8,
    V=152064, fp32), the command the top-p kernels' ncu capture runs."""
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300 import workload as W
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    b = W.ragged_top_p(0)
    db = to_device(b)
    ws = sv.make_workspace(b.B, b.total_drafts, b.V)
    a = db.args()
    for _ in range(3):
        sv.spec_verify_sample(a, workspace=ws)
    torch.cuda.synchronize()
    return 0


def profile_topp() -> int:
    """The top-p kernels on the ragged workload: duration and DRAM bytes of
    each kernel's last launch (three metrics, a few passes, 1.6 GB of
    inputs on the device), against the algorithmic bytes of the workload."""
    import csv

    base = [sys.executable, os.path.abspath(__file__), "--topp-run"]
    if subprocess.call(base, stdout=subprocess.DEVNULL) != 0:
        print("plain top-p run failed; not profiling", file=sys.stderr)
        return 1
    log = os.path.join(ROOT, "gpurun_out", "topp_prof.csv")
    rc = subprocess.call(["ncu", "--metrics", "gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum",
                          "--clock-control", "none", "-k", "regex:topp_", "-c", "6", "--csv", "--log-file", log] + base,
                         stdout=subprocess.DEVNULL)
    if rc:
        return rc
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3,
             "ns": 1e-3, "us": 1.0, "ms": 1e3}
    per = {}
    with open(log) as f:
        lines = [l for l in f if l.startswith('"')]
    for r in csv.DictReader(lines):
        name = "topp_cut_kernel" if "topp_cut" in r["Kernel Name"] else "topp_finish_kernel"
        v = float(r["Metric Value"].replace(",", "")) * scale.get(r.get("Metric Unit", ""), 1.0)
        per.setdefault(name, {})[r["Metric Name"]] = v      # the last launch wins
    algo = 1574182000
    out = {"kernels": {}, "workload": "ragged top-p B=256 K 1..8 V=152064 fp32", "algorithmic_bytes": algo,
           "kernel_hash": kernel_hash(TOPP_SOURCES), "command": "python bench.py --profile"}
    for name, m in per.items():
        out["kernels"][name] = {"duration_us_under_ncu": m.get("gpu__time_duration.sum"),
                                "dram_read_bytes": int(m.get("dram__bytes_read.sum", 0)),
                                "dram_write_bytes": int(m.get("dram__bytes_write.sum", 0))}
    cut = out["kernels"].get("topp_cut_kernel", {})
    if cut:
        out["cut_traffic_over_algorithmic"] = (cut["dram_read_bytes"] + cut["dram_write_bytes"]) / algo
    for path in (TOPP_SUMMARY, os.path.join(ROOT, "gpurun_out", os.path.basename(TOPP_SUMMARY))):
        with open(path, "w") as f:
            json.dump(out, f, indent=2)
    print(json.dumps(out), flush=True)
    return 0


SMALL_RUNS = {
    # name: (kernel regex, workload, algorithmic bytes, profile file)
    "greedy": ("greedy_verify_kernel", "greedy B=1 K=8 V=151936 bf16", 9 * 151936 * 2 + 4 * 18,
               "greedy_verify_kernel_B1_K8.json"),
    "resident": ("sample_verify_kernel", "Qwen2.5-shaped B=1 K=8 V=152064 bf16 D=0.5", 5171292,
                 "sample_verify_kernel_resident_B1_K8.json"),
    "confidence": ("conf_pipe_kernel", "batched B=64 K=8 V=152064 bf16, threshold 0.6", 155848704,
                   "conf_pipe_kernel_batched.json"),
}


def small_run(name: str) -> int:
    """`--small-run NAME`: five calls of one small entry point (the command
    the small kernels' ncu captures run)."""
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300 import workload as W
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    b = {"greedy": lambda: W.greedy_single(8), "resident": lambda: W.qwen25_single(0.5),
         "confidence": lambda: make_workload(0)}[name]()
    db = to_device(b)
    ws = sv.make_workspace(b.B, b.total_drafts, b.V)
    a = db.args()
    for _ in range(5):
        if name == "greedy":
            sv.spec_verify_greedy(a, workspace=ws)
        elif name == "resident":
            sv.spec_verify_sample(a, workspace=ws)
        else:
            sv.spec_draft_confidence(a, 0.6, workspace=ws)
    torch.cuda.synchronize()
    return 0


def profile_small() -> int:
    """`--profile-small`: duration and DRAM bytes of the greedy, resident
    cluster and confidence kernels on their own workloads (three metrics,
    the last of three captured launches), with the algorithmic bytes."""
    import csv

    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3,
             "ns": 1e-3, "us": 1.0, "ms": 1e3}
    for name, (kern, workload, algo, fname) in SMALL_RUNS.items():
        base = [sys.executable, os.path.abspath(__file__), "--small-run", name]
        if subprocess.call(base, stdout=subprocess.DEVNULL) != 0:
            print(f"plain {name} run failed; not profiling", file=sys.stderr)
            return 1
        log = os.path.join(ROOT, "gpurun_out", f"small_{name}.csv")
        rc = subprocess.call(["ncu", "--metrics", "gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum",
                              "--clock-control", "none", "-k", "regex:" + kern, "-s", "2", "-c", "3", "--csv",
                              "--log-file", log] + base, stdout=subprocess.DEVNULL)
        if rc:
            return rc
        m = {}
        with open(log) as f:
            lines = [l for l in f if l.startswith('"')]
        for r in csv.DictReader(lines):
            m[r["Metric Name"]] = float(r["Metric Value"].replace(",", "")) * scale.get(r.get("Metric Unit", ""), 1.0)
        rd, wr = int(m.get("dram__bytes_read.sum", 0)), int(m.get("dram__bytes_write.sum", 0))
        out = {"kernel": kern, "workload": workload, "algorithmic_bytes": algo,
               "duration_us_under_ncu": m.get("gpu__time_duration.sum"), "dram_read_bytes": rd,
               "dram_write_bytes": wr, "traffic_over_algorithmic": (rd + wr) / algo,
               "note": "cold-cache, serialised launch under ncu: compare bytes, not the duration",
               "command": "python bench.py --profile-small"}
        for path in (os.path.join(ROOT, "profiles", fname), os.path.join(ROOT, "gpurun_out", fname)):
            with open(path, "w") as f:
                json.dump(out, f, indent=2)
        print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", action="store_true",
                    help="also time the other configurations and entry points (adds about a minute)")
    ap.add_argument("--profile", action="store_true",
                    help="ncu launch list and one capture of the sampling kernel, and the top-p kernels' "
                         "durations and DRAM bytes -> profiles/")
    ap.add_argument("--topp-run", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--profile-small", action="store_true",
                    help="ncu durations and DRAM bytes of the greedy, resident cluster and confidence kernels")
    ap.add_argument("--small-run", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.topp_run:
        sys.exit(topp_run())
    if args.small_run:
        sys.exit(small_run(args.small_run))
    if args.profile_small:
        sys.exit(profile_small())
    if args.profile:
        rc = profile(args)
        sys.exit(rc or profile_topp())
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch(args))
    if args.impl == "reference":
        if rank == 0:
            bench_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
        dist = tdist
    try:
        bench_gpu(args, rank, world, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
