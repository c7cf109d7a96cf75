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
import tempfile
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
    for f in ("mla_kernels.cuh", "mla_fp8_kernel.cuh", "ptx.cuh", "mla_api.cu"):
        with open(os.path.join(ROOT, "mla_decode_attention_mxfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic_per_launch(workload, kernel="mla_split_kernel"):
    """DRAM bytes per launch of a split kernel from the committed ncu summary,
    only if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
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
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="mla_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
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
            lines = f.readlines()
        os.unlink(self.path)
        if True:
            for line in lines:
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
    """The fp64 oracle, as it stands, on the host cores: the whole call on every core the
    OpenMP runtime offers (its (sequence, head) driver), and beside it the single-threaded
    oracle on a bounded sample of whole sequences."""
    import oracle
    oracle.build()
    nthreads = oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while reps < 1 or (time.perf_counter() - t0 < budget_s / 4 and reps < 5):
        oracle.decode_mt(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, nthreads)
        reps += 1
    mt_s = (time.perf_counter() - t0) / reps
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
    return {"value": d.algorithmic_bytes() / mt_s / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "us_per_call": mt_s * 1e6, "online_cpus": oracle.online_cpus(),
            "sample": f"the whole call ({B} sequences, {d.total_kv} tokens) decoded {reps}x by the fp64 C oracle's "
                      f"OpenMP driver over (sequence, head) on {nthreads} threads",
            "single_thread": {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": 1,
                              "us_per_call": el * d.algorithmic_bytes() / done_bytes * 1e6,
                              "sample": f"{done_seqs} of {B} sequences ({done_tokens} tokens) in {el:.2f} s; "
                                        "us_per_call extrapolated by bytes"}}


def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import mla_inputs as MI
    import oracle
    oracle.build()
    d = MI.make_inputs(args.workload)
    nthreads = oracle.max_threads()
    # calibrate a per-step sample of leading sequences so the whole run stays within ~2 minutes
    steps_total = args.steps + args.warmup
    t = time.perf_counter()
    oracle.decode_mt(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, nthreads)
    full_s = time.perf_counter() - t
    nseq = d.batch
    while nseq > 1 and full_s * nseq / d.batch * steps_total > 120.0:
        nseq = max(1, nseq // 2)
    ip = d.kv_indptr[:nseq + 1]
    rows = int(ip[-1])
    q, kv, sc = d.q[:nseq], d.kv_packed[:rows], d.kv_scale[:rows]
    nbytes = nseq * (18432 + 16384) + rows * 306
    times = []
    for i in range(steps_total):
        t = time.perf_counter()
        oracle.decode_mt(q, kv, sc, ip, d.sm_scale, nthreads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    step_s = sum(times) / len(times)
    val = nbytes / step_s / 1e9
    line = {"impl": "reference", "metric": "MLA decode achieved HBM GB/s (and us/call)", "value": val,
            "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": _workload_desc(args.workload, d),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"each step: the first {nseq} of {d.batch} sequences ({rows} tokens) "
                                       f"decoded by the fp64 C oracle's OpenMP driver on {nthreads} threads"},
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


class DeviceWorkload:
    """One workload's inputs resident in HBM (rotated over enough copies that the working set
    exceeds L2) and one decode call through the C ABI with a caller-owned workspace."""

    def __init__(self, d, dev, stream):
        import torch

        from mla_decode_attention_mxfp4_gb300 import _lib, alloc_workspace
        self.d, self.dev, self.stream, self._lib = d, dev, stream, _lib
        self.nbytes = d.algorithmic_bytes()
        # the split kernel's own algorithmic bytes: every KV row and every query once (the
        # output of split sequences is written by the merge kernel)
        self.split_bytes = d.total_kv * 306 + d.batch * 18432
        self.in_bytes = d.q.numel() * 2 + d.kv_packed.numel() + d.kv_scale.numel()
        self.copies = max(2, min(8, math.ceil(4 * L2_BYTES / self.in_bytes)))
        self.bufs = [(d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev),
                      torch.empty(d.batch, 16, 512, dtype=torch.bfloat16, device=dev)) for _ in range(self.copies)]
        self.ws = alloc_workspace(d.batch, dev)
        torch.cuda.synchronize(dev)

    def l2_note(self):
        return (f"timed calls rotate over {self.copies} input copies "
                f"({self.copies * self.in_bytes / 2**20:.0f} MiB > L2 {L2_BYTES // 2**20} MiB)")

    def call(self, i, ev_b=None, ev_e=None):
        q, kv, sc, ip, out = self.bufs[i % self.copies]
        rc = self._lib.mla_decode_mxfp4_ws_timed(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), ip.data_ptr(),
                                                 out.data_ptr(), self.d.batch, self.d.sm_scale,
                                                 self.stream.cuda_stream, self.ws.data_ptr(), self.ws.numel(),
                                                 ev_b, ev_e)
        if rc != 0:
            raise RuntimeError(self._lib.status_string(rc))

    def time_calls(self, steps):
        """Mean device time of `steps` back-to-back calls (CUDA events on the launching stream)."""
        import torch
        torch.cuda.synchronize(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(steps):
            self.call(i)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / steps

    def time_split_kernel(self, steps):
        """Mean duration of the split kernel alone: events recorded around it by the library,
        on the stream it is launched on, over the same rotation of inputs."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(steps, 400))]
        for a, b in evs:  # torch creates the CUDA events lazily, at the first record
            a.record(self.stream)
            b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        for i, (a, b) in enumerate(evs):
            self.call(i, a.cuda_event, b.cuda_event)
        torch.cuda.synchronize(self.dev)
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    def roofline(self, split_ms, peak, peak_src, workload):
        achieved = self.split_bytes / (split_ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "mla_split_kernel", "achieved": achieved, "peak": peak,
                "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                "split_kernel_us": split_ms * 1e3, "split_kernel_bytes": self.split_bytes,
                "traffic": _traffic_per_launch(workload)}


class GeneralWorkload(DeviceWorkload):
    """A further layout of a workload, timed through its own C entry point: the KV cache as fp8
    with a per-tensor scale ("fp8"), in scattered pages of 64 rows ("paged64"), or with two
    query rows per sequence ("q2")."""

    def __init__(self, name, dev, stream):
        import torch

        import mla_inputs as MI
        from mla_decode_attention_mxfp4_gb300 import _lib, alloc_workspace
        base, form = name.split(":")
        self.name, self.form, self.dev, self.stream, self._lib = name, form, dev, stream, _lib
        if form == "fp8":
            d = MI.make_fp8_inputs(base)
            self.d = d
            self.nbytes = d.algorithmic_bytes()
            self.split_bytes = d.total_kv * 576 + d.q.shape[0] * 18432
            self.in_bytes = d.q.numel() * 2 + d.kv_fp8.numel()
            self.total_q = d.batch
            tensors = lambda: (d.q.to(dev), d.kv_fp8.to(dev), torch.tensor([d.kv_scale], dtype=torch.float32,
                                                                              device=dev), d.kv_indptr.to(dev))
        else:
            d = MI.make_inputs(base)
            self.d = d
            if form == "paged64":
                kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, 64, seed=40, spare_pages=0)
                self.paged = (ix, last, npages)
                tensors = lambda: (d.q.to(dev), kp.to(dev), ks.to(dev), ip.to(dev), ix.to(dev), last.to(dev))
                self.total_q = d.batch
                q_bytes = d.q.numel() * 2
            elif form == "q2":
                q, qo = MI.query_rows([2] * d.batch, seed=41)
                self.qo = qo
                tensors = lambda: (q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev),
                                   qo.to(dev))
                self.total_q = int(qo[-1])
                q_bytes = q.numel() * 2
            else:
                raise ValueError(name)
            kv_bytes = d.kv_packed.numel() + d.kv_scale.numel()
            self.nbytes = q_bytes + kv_bytes + self.total_q * 16 * 512 * 2
            # each query row reads its sequence's KV rows once
            rows_read = d.total_kv * (2 if form == "q2" else 1)
            self.split_bytes = rows_read * 306 + self.total_q * 18432
            self.in_bytes = q_bytes + kv_bytes
        self.copies = max(2, min(8, math.ceil(4 * L2_BYTES / self.in_bytes)))
        self.bufs = []
        for _ in range(self.copies):
            self.bufs.append(tensors() + (torch.empty(self.total_q, 16, 512, dtype=torch.bfloat16, device=dev),))
        self.ws = alloc_workspace(max(self.d.batch, self.total_q), dev)
        torch.cuda.synchronize(dev)

    def call(self, i, ev_b=None, ev_e=None):
        b = self.bufs[i % self.copies]
        L, d = self._lib, self.d
        if self.form == "fp8":
            q, kv, sc, ip, out = b
            rc = L.mla_decode_fp8_ws_timed(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), None, ip.data_ptr(),
                                           kv.shape[0], out.data_ptr(), d.batch, d.batch, d.sm_scale,
                                           self.stream.cuda_stream, self.ws.data_ptr(), self.ws.numel(), ev_b, ev_e)
        elif self.form == "paged64":
            q, kp, ks, ip, ix, last, out = b
            rc = L.mla_decode_mxfp4_paged_ws_timed(q.data_ptr(), kp.data_ptr(), ks.data_ptr(), None, ip.data_ptr(),
                                                   ix.data_ptr(), last.data_ptr(), 64, self.paged[2], out.data_ptr(),
                                                   d.batch, d.batch, d.sm_scale, self.stream.cuda_stream,
                                                   self.ws.data_ptr(), self.ws.numel(), ev_b, ev_e)
        else:
            q, kv, sc, ip, qo, out = b
            rc = L.mla_decode_mxfp4_paged_ws_timed(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), qo.data_ptr(),
                                                   ip.data_ptr(), None, None, 0, 0, out.data_ptr(), d.batch,
                                                   self.total_q, d.sm_scale, self.stream.cuda_stream,
                                                   self.ws.data_ptr(), self.ws.numel(), ev_b, ev_e)
        if rc != 0:
            raise RuntimeError(L.status_string(rc))

    def config(self):
        import mla_inputs as MI
        base = self.name.split(":")[0]
        w = MI.WORKLOADS[base]
        desc = {"workload": f"{self.name}: {w.note}", "batch": self.d.batch, "query_rows": self.total_q,
                "tokens": self.d.total_kv, "bytes_per_call": self.nbytes,
                "kv_format": {"fp8": "fp8 e4m3, one per-tensor scale (576 B per token)",
                              "paged64": "MXFP4 in scattered pages of 64 rows",
                              "q2": "MXFP4, two query rows per sequence (each row reads its sequence's KV)"}[self.form],
                "l2": self.l2_note()}
        return desc

    def roofline(self, split_ms, peak, peak_src, workload):
        r = DeviceWorkload.roofline(self, split_ms, peak, peak_src, workload)
        r["kernel"] = "mla_split_fp8_kernel" if self.form == "fp8" else "mla_split_kernel"
        r["traffic"] = _traffic_per_launch(workload, r["kernel"])
        return r


NUMERICS = ("K/V as e5m2 against a per-tile reference exponent (exact for blocks within 27 binades of "
            "the tile's largest scale), query as two e4m3 terms, P*2^11 as two e5m2 terms, tcgen05 f8f6f4 "
            "MMAs with fp32 accumulation, fp32 softmax and merge, bf16 out")


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
    from mla_decode_attention_mxfp4_gb300 import HostDecoder

    stream = torch.cuda.Stream(dev)
    d = MI.make_inputs(args.workload)
    W = DeviceWorkload(d, dev, stream)

    def barrier():
        if ws > 1:
            dist.barrier()

    sampler = ClockSampler(_gpu_id(local))
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            W.call(i)
        # untimed soak (~1 s) so the clock sampler sees the load
        torch.cuda.synchronize(dev)
        t_end = time.time() + 1.0
        i = 0
        while time.time() < t_end:
            for _ in range(200):
                W.call(i)
                i += 1
            torch.cuda.synchronize(dev)
        # ---- timed region: exactly K steps ----
        barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.time()
        ms = W.time_calls(args.steps)
        wall1 = time.time()
        barrier()
        # ---- split-kernel-only timing (same rotation, events around that kernel) ----
        split_ms = W.time_split_kernel(args.steps)
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows, wall0, wall1)

    # ---- CUDA-graph replay of one rotation (launch overhead removed) ----
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(W.copies):
                W.call(i)
        reps = max(1, args.steps // W.copies)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            g.replay()
            torch.cuda.synchronize(dev)
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(stream)
            for _ in range(reps):
                g.replay()
            gb.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = ga.elapsed_time(gb) / (reps * W.copies)
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

    # ---- the other gated workload(s): device-timed the same way, rank 0 reports them ----
    peak, peak_src = _peaks()
    extra = {}
    for name in args.extra:
        if name == args.workload:
            continue
        if ":" in name:
            X = GeneralWorkload(name, dev, stream)
            with torch.cuda.stream(stream):
                for i in range(max(args.warmup, 10)):
                    X.call(i)
                xs = max(args.steps, 20)
                xms = X.time_calls(xs)
                xsplit = X.time_split_kernel(xs)
            extra[name] = {"config": X.config(), "value": whole_job_gbps(ws, X.nbytes, xms), "unit": "GB/s",
                           "us_per_call": xms * 1e3, "frac_of_hbm_peak": X.nbytes / (xms * 1e-3) / 1e9 / peak,
                           "steps": xs, "roofline": X.roofline(xsplit, peak, peak_src, name)}
            del X
            torch.cuda.empty_cache()
            continue
        dx = MI.make_inputs(name)
        X = DeviceWorkload(dx, dev, stream)
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, 10)):
                X.call(i)
            xs = max(args.steps, 20)
            xms = X.time_calls(xs)
            xsplit = X.time_split_kernel(xs)
        extra[name] = {"config": dict(_workload_desc(name, dx), l2=X.l2_note()),
                       "value": whole_job_gbps(ws, X.nbytes, xms), "unit": "GB/s", "us_per_call": xms * 1e3,
                       "frac_of_hbm_peak": X.nbytes / (xms * 1e-3) / 1e9 / peak, "steps": xs,
                       "roofline": X.roofline(xsplit, peak, peak_src, name)}
        del X
        torch.cuda.empty_cache()

    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], dev)
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": "MLA decode achieved HBM GB/s (and us/call)",
        "value": whole_job_gbps(ws, W.nbytes, ms),
        "unit": "GB/s",
        "us_per_call": ms * 1e3,
        "frac_of_hbm_peak": W.nbytes / (ms * 1e-3) / 1e9 / peak,
        "us_per_call_graph": graph_ms * 1e3 if isinstance(graph_ms, float) else graph_ms,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 operands, fp32 accumulate", "numerics": NUMERICS, "data": "synthetic",
        "config": dict(_workload_desc(args.workload, d), l2=W.l2_note(),
                       parallelism=f"replica per GPU x{ws}" if ws > 1 else "1 GPU"),
        "roofline": W.roofline(split_ms, peak, peak_src, args.workload),
        "e2e": {"value": whole_job_gbps(ws, W.nbytes, e2e_ms), "unit": "GB/s", "us_per_call": e2e_ms * 1e3,
                "h2d_bytes_per_step": W.in_bytes + d.kv_indptr.numel() * 4,
                "d2h_bytes_per_step": d.batch * 16 * 512 * 2,
                "path": "HostDecoder: the kernels read q, kv_packed and kv_scale in place from pinned host "
                        "memory (each byte crosses the host link once); kv_indptr copied in, out copied back"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "extra_workloads": extra,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_profile_workload(args):
    """A fixed number of launches of one workload and nothing else (no soak, no end-to-end leg),
    so that a profiler can address one launch by its index: --warmup calls, then --steps timed
    calls.  Prints one short JSON line."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import mla_inputs as MI
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    name = args.profile_workload
    W = GeneralWorkload(name, dev, stream) if ":" in name else DeviceWorkload(MI.make_inputs(name), dev, stream)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            W.call(i)
        ms = W.time_calls(args.steps)
    print(json.dumps({"profile_workload": name, "launches_of_the_split_kernel": args.warmup + args.steps,
                      "us_per_call": ms * 1e3}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="uniform")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", nargs="*",
                    default=["ragged", "uniform:fp8", "ragged:fp8", "ragged:paged64", "uniform:q2"],
                    help="further workloads measured on the device and reported under extra_workloads")
    ap.add_argument("--profile-workload", default=None,
                    help="only --warmup + --steps calls of this workload (e.g. ragged:paged64), for profilers")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.profile_workload:
        run_profile_workload(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
