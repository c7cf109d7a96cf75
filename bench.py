#!/usr/bin/env python
"""MXFP4 MLA decode benchmark on GB300: µs per call and achieved HBM GB/s.

One step = one decode call (partition + split-KV attention + merge) over the
whole batch of the workload.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload uniform]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Bytes counted per call (the algorithmic bytes): Q (bf16) + packed KV + E8M0
scales + bf16 output.  Partial buffers and the work list are not counted.
Inputs are synthetic (seeded generator), resident in HBM before timing; the
timed calls rotate over enough input copies that the working set exceeds L2.
Under torchrun each rank decodes its own replica of the workload (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def kernel_source_sha1():
    h = hashlib.sha1()
    for f in ("mla_kernels.cuh", "ptx.cuh", "mla_api.cu"):
        with open(os.path.join(ROOT, "mla_decode_attention_mxfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic_per_launch(workload):
    """DRAM bytes per launch of the split kernel from the committed ncu summary,
    only if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("mla_split_kernel", {}).get(workload)
    if not e or e.get("source_sha1") != kernel_source_sha1():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", self.gpu_id], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append(dict(ts=ts, sm=float(parts[2]), sm_max=float(parts[3]), reasons=parts[5],
                                     hw=parts[6], hw_thermal=parts[7], sw_thermal=parts[8], sw_power=parts[9]))
                except ValueError:
                    continue
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [r for r in rows if t0 <= r["ts"] <= t1]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling period: use the load window
            inside = rows
            window = "warm-up + timed load window"
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in inside):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["sm_max"] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def _gpu_id(dev_index):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


def _workload_desc(name, d):
    import mla_inputs as MI
    w = MI.WORKLOADS[name]
    lens = (d.kv_indptr[1:] - d.kv_indptr[:-1])
    return {"workload": f"{name}: {w.note}", "batch": d.batch, "tokens": d.total_kv,
            "kv_len": w.kv_len if w.kv_len else f"U[1,{w.ragged_max}] (min {int(lens.min())}, max {int(lens.max())})",
            "heads": 16, "qk_dim": 576, "v_dim": 512, "kv_format": "MXFP4 (e2m1 + E8M0 per 32)",
            "bytes_per_call": d.algorithmic_bytes(), "seed": w.seed}


def cpu_baseline(d, budget_s=10.0):
    """The fp64 oracle, as it stands, on a bounded sample of whole sequences."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    done_tokens, done_seqs, done_bytes = 0, 0, 0
    B = d.batch
    while done_seqs < B and time.perf_counter() - t0 < budget_s:
        b = done_seqs
        oracle.decode_one(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, b)
        n = int(d.kv_indptr[b + 1] - d.kv_indptr[b])
        done_tokens += n
        done_bytes += 18432 + n * 306 + 16384
        done_seqs += 1
    el = time.perf_counter() - t0
    full_s = el * d.algorithmic_bytes() / done_bytes
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "us_per_call": full_s * 1e6,
            "sample": f"{done_seqs} of {B} sequences ({done_tokens} tokens) decoded by the single-threaded "
                      f"fp64 C oracle in {el:.2f} s; us_per_call extrapolated by bytes"}


def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import torch

    import mla_inputs as MI
    import oracle
    oracle.build()
    d = MI.make_inputs(args.workload)
    # calibrate a per-step sample so the whole run stays within ~2 minutes
    n0 = int(d.kv_indptr[1] - d.kv_indptr[0])
    t = time.perf_counter()
    oracle.decode_one(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, 0)
    per_token = (time.perf_counter() - t) / max(n0, 1)
    steps_total = args.steps + args.warmup
    tok_budget = max(16, min(n0, int(120.0 / steps_total / per_token)))
    ip = torch.tensor([0, tok_budget], dtype=torch.int32)
    times = []
    for i in range(steps_total):
        bb = i % d.batch
        r0 = int(d.kv_indptr[bb])
        n = min(tok_budget, int(d.kv_indptr[bb + 1]) - r0)
        ipb = torch.tensor([0, n], dtype=torch.int32) if n != tok_budget else ip
        kv, sc = d.kv_packed[r0:r0 + n], d.kv_scale[r0:r0 + n]
        t = time.perf_counter()
        oracle.decode(d.q[bb:bb + 1], kv, sc, ipb, d.sm_scale)
        if i >= args.warmup:
            times.append((time.perf_counter() - t, 18432 + n * 306 + 16384))
    step_s = sum(x for x, _ in times) / len(times)
    val = sum(b for _, b in times) / sum(x for x, _ in times) / 1e9
    line = {"impl": "reference", "metric": "MLA decode achieved HBM GB/s (and us/call)", "value": val,
            "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": _workload_desc(args.workload, d),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: sequence (step mod batch), first {tok_budget} tokens, "
                                       "single-threaded fp64 C oracle"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reduce_max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group (the slowest
    rank's time); the values themselves on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_gbps(world, nbytes_per_rank, ms):
    """Whole-job GB/s: the bytes every rank processed in one step over the slowest rank's step time."""
    return world * nbytes_per_rank / (ms * 1e-3) / 1e9


def run_native(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import mla_inputs as MI
    from mla_decode_attention_mxfp4_gb300 import HostDecoder, _lib, alloc_workspace

    d = MI.make_inputs(args.workload)
    nbytes = d.algorithmic_bytes()
    in_bytes = d.q.numel() * 2 + d.kv_packed.numel() + d.kv_scale.numel()
    copies = max(2, min(8, math.ceil(4 * L2_BYTES / in_bytes)))
    stream = torch.cuda.Stream(dev)
    bufs = []
    for _ in range(copies):
        bufs.append((d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev),
                     torch.empty(d.batch, 16, 512, dtype=torch.bfloat16, device=dev)))
    wsb = alloc_workspace(d.batch, dev)
    torch.cuda.synchronize(dev)

    def call(i, ev_b=None, ev_e=None):
        q, kv, sc, ip, out = bufs[i % copies]
        rc = _lib.mla_decode_mxfp4_ws_timed(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), ip.data_ptr(), out.data_ptr(),
                                            d.batch, d.sm_scale, stream.cuda_stream, wsb.data_ptr(), wsb.numel(),
                                            ev_b, ev_e)
        if rc != 0:
            raise RuntimeError(_lib.status_string(rc))

    def barrier():
        if ws > 1:
            dist.barrier()

    sampler = ClockSampler(_gpu_id(local))
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
        # untimed soak (~1 s) so the clock sampler sees the load
        torch.cuda.synchronize(dev)
        t_end = time.time() + 1.0
        i = 0
        while time.time() < t_end:
            for _ in range(200):
                call(i)
                i += 1
            torch.cuda.synchronize(dev)
        # ---- timed region: exactly K steps ----
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.time()
        e0.record(stream)
        for i in range(args.steps):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        wall1 = time.time()
        barrier()
        ms = e0.elapsed_time(e1) / args.steps
        # ---- split-kernel-only timing (same rotation, events around that kernel) ----
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(args.steps, 400))]
        for a, b in evs:  # torch creates the CUDA events lazily, at the first record
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        for i, (a, b) in enumerate(evs):
            call(i, a.cuda_event, b.cuda_event)
        torch.cuda.synchronize(dev)
        split_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows, wall0, wall1)

    # ---- CUDA-graph replay of one rotation (launch overhead removed) ----
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(copies):
                call(i)
        reps = max(1, args.steps // copies)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            g.replay()
            torch.cuda.synchronize(dev)
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(stream)
            for _ in range(reps):
                g.replay()
            gb.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = ga.elapsed_time(gb) / (reps * copies)
    except Exception as exc:  # reported, not fatal
        graph_ms = f"unavailable: {exc}"

    # ---- end to end from pinned host buffers through the public API ----
    hq, hkv, hsc, hip = (d.q.pin_memory(), d.kv_packed.pin_memory(), d.kv_scale.pin_memory(),
                         d.kv_indptr.pin_memory())
    hout = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16).pin_memory()
    hd = HostDecoder(dev)
    for _ in range(2):
        hd(hq, hkv, hsc, hip, d.sm_scale, hout)
    hd.synchronize()
    e2e_steps = max(3, min(args.steps, 30))
    barrier()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(hd.stream)
    for _ in range(e2e_steps):
        hd(hq, hkv, hsc, hip, d.sm_scale, hout)
    eb.record(hd.stream)
    hd.synchronize()
    e2e_ms = ea.elapsed_time(eb) / e2e_steps
    barrier()

    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], dev)
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    peak, peak_src = _peaks()
    achieved = nbytes / (split_ms * 1e-3) / 1e9
    line = {
        "metric": "MLA decode achieved HBM GB/s (and us/call)",
        "value": whole_job_gbps(ws, nbytes, ms),
        "unit": "GB/s",
        "us_per_call": ms * 1e3,
        "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
        "us_per_call_graph": graph_ms * 1e3 if isinstance(graph_ms, float) else graph_ms,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8", "data": "synthetic",
        "config": dict(_workload_desc(args.workload, d),
                       l2=f"timed calls rotate over {copies} input copies "
                          f"({copies * in_bytes / 2**20:.0f} MiB > L2 {L2_BYTES // 2**20} MiB)",
                       parallelism=f"replica per GPU x{ws}" if ws > 1 else "1 GPU"),
        "roofline": {"bound": "hbm", "kernel": "mla_split_kernel", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                     "split_kernel_us": split_ms * 1e3,
                     "traffic": _traffic_per_launch(args.workload)},
        "e2e": {"value": whole_job_gbps(ws, nbytes, e2e_ms), "unit": "GB/s", "us_per_call": e2e_ms * 1e3,
                "h2d_bytes_per_step": in_bytes + d.kv_indptr.numel() * 4,
                "d2h_bytes_per_step": d.batch * 16 * 512 * 2},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="uniform")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
