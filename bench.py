#!/usr/bin/env python
"""Benchmark of the unified paged varlen attention forward pass on GB300.

One step = one forward call (every stage of the path: work decomposition,
paged K/V gather, scores, score transforms, online softmax, P.V, split
partials and their combine) over one batch of synthetic input already
resident in HBM.  The headline workload is the decode batch (64 sequences,
S_q = 1, S_k ~ U{512..8192}, H 32/8, d = 128, b = 16, 40,000-block pool); the
metric is the K/V bytes the path must read per second.  The same JSON line
also carries the prefill workloads' TFLOPS (``per_config``), the roofline
object of the dominant kernel, the host-buffer end-to-end number, the CPU
oracle baseline and the SM clocks sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank processes its own batch (weak scaling,
no collective on the data path); value = bytes of all ranks / max time.
``--impl reference`` times the fp64 CPU oracle on the same workload and
metric (the host cores' baseline, not a GPU implementation).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill TFLOPS and decode KV-read GB/s on 1×GB300, as % of roofline"
HEADLINE = "decode"
SECONDARY = ["chunked", "long_prefill", "long_prefill_shuffled", "wide_mha_alibi"]
# HBM-bound secondary workloads, reported in GB/s of algorithmic bytes
# ("decode_cold": the headline batch with L2 flushed between steps).
SECONDARY_HBM = ["decode_cold", "decode_d64", "decode_d256", "decode_fp8", "decode_topk"]
L2_FLUSH_BYTES = 256 << 20
# Special-function unit throughput per SM per clock on GB300, measured with a
# dependency-free probe: ex2.approx.f32 32 results, tanh.approx.f32 16.  The
# prefill kernels spend one exponential per (row, key) score, plus one tanh
# with a softcap; on 152 SMs at the maximum SM clock this is a third bound
# beside the tensor and HBM ones.
SFU_EX2_PER_CLK = 32.0
SFU_TANH_PER_CLK = 16.0
NUM_SMS = 152
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "split_kernel": ["ua_split.cu", "ua_ptx.cuh", "ua_common.cuh"],
    "prefill_cta2_kernel": ["ua_prefill_cta2.cu", "ua_prefill_common.cuh", "ua_ptx.cuh", "ua_common.cuh",
                            "ua_tc.cuh"],
    "prefill_pair_kernel": ["ua_prefill_pair.cu", "ua_prefill_common.cuh", "ua_ptx.cuh", "ua_common.cuh",
                            "ua_tc.cuh"],
    "prefill_grid_kernel": ["ua_prefill_grid.cu", "ua_prefill_common.cuh", "ua_ptx.cuh", "ua_common.cuh",
                            "ua_tc.cuh"],
    "decode_tc_kernel": ["ua_decode_tc.cu", "ua_decode_common.cuh", "ua_ptx.cuh", "ua_common.cuh",
                         "ua_tc.cuh"],
    "topk_kernel": ["ua_topk.cu", "ua_decode_common.cuh", "ua_ptx.cuh", "ua_common.cuh", "ua_tc.cuh"],
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, "paged_varlen_flash_gb300", "csrc", name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("workload") != workload:
        return None
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.3 <= t <= t1 + 0.3]
        if not rows and self.samples:
            mid = 0.5 * (t0 + t1)
            rows = [min(self.samples, key=lambda x: abs(x[0] - mid))[1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def aggregate_ranks(local_ms, local_bytes, device):
    """Whole-job timing over ranks: (max of the ranks' timed milliseconds, sum of
    the bytes every rank processed per step).  No data-path collective: each rank
    owns an independent batch; this is the only cross-rank exchange."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(local_ms), int(local_bytes)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([int(local_bytes)], dtype=torch.int64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def dominant_kernel(path):
    """The kernel that carries a forward call's time, from the path name the
    library reports (the combine kernel is ~2% of a split call)."""
    if path.startswith("decode_tc"):
        return "decode_tc_kernel"
    if path.startswith("topk_tc"):
        return "topk_kernel"
    if path.startswith("tensor_core_pair"):
        return "prefill_pair_kernel"
    if path.startswith("tensor_core_grid"):
        return "prefill_grid_kernel"
    if path.startswith("tensor_core_cta2"):
        return "prefill_cta2_kernel"
    return "split_kernel"


def workload_units(w):
    """(algorithmic bytes, algorithmic flops) of one forward pass of w."""
    kv = w.kv_bytes_read()
    qo = 2 * w.total_q * w.hq * w.d * 2
    meta = sum((k + w.b - 1) // w.b for k in w.seqlens_k) * 4 + (2 * w.num_seqs + 1) * 4
    if w.topk_len is not None:
        # the lists and their lengths instead of whole block-table rows
        meta = int(w.topk_len.to("cpu").sum()) * 4 + w.total_q * 4 + (2 * w.num_seqs + 1) * 4
    flops = 4.0 * w.d * w.hq * w.visible_pairs()
    return kv + qo + meta, flops


def time_ours(w, steps, warmup, flush, torch, ua, path=0):
    prob = ua.Problem.for_workload(w, path=path)
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=w.q.device)
    for _ in range(warmup):
        prob.forward_workload(w, out=out)
    torch.cuda.synchronize()
    assert prob.check_device_error() == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for evs in ev:   # torch creates CUDA events lazily: record once so each handle exists
        for x in evs:
            x.record(stream)
    launches = 0
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        if flush:
            flush_buf.zero_()
        s, e, ks, ke = ev[i]
        prob.set_profile_events(ks, ke)
        s.record(stream)
        prob.forward_workload(w, out=out)
        e.record(stream)
        launches += prob.last_launch_count()
    torch.cuda.synchronize()
    t1 = time.time()
    prob.set_profile_events(None, None)
    step_ms = [s.elapsed_time(e) for s, e, _, _ in ev]
    kern_ms = [ks.elapsed_time(ke) for _, _, ks, ke in ev]
    path = prob.last_path()
    err = prob.check_device_error()
    prob.close()
    return dict(step_ms=step_ms, kernel_ms=kern_ms, launches=launches, path=path,
                t0=t0, t1=t1, device_error=err)


def time_e2e(w, steps, warmup, torch, ua):
    """The host-buffer entry point: per-step inputs copied in from pinned host
    memory and the output copied back, all inside the timed call."""
    prob = ua.Problem.for_workload(w)
    flags = ua.flags_of(w.causal, w.softcap, w.alibi_slopes is not None, w.window,
                        w.sinks is not None)
    q_h = w.q.cpu().pin_memory()
    bt_h = w.block_table.cpu().pin_memory()
    cu_h = w.cu_seqlens_q.cpu().pin_memory()
    su_h = w.seqused_k.cpu().pin_memory()
    sk_h = w.sinks.cpu().pin_memory() if w.sinks is not None else None
    al_h = w.alibi_slopes.cpu().pin_memory() if w.alibi_slopes is not None else None
    out_h = torch.empty_like(q_h).pin_memory()
    args = (prob.handle, q_h, w.k_cache, w.v_cache, bt_h, cu_h, su_h, w.num_seqs, w.total_q,
            w.max_seqlen_q, w.max_seqlen_k, flags, sk_h, al_h, out_h)
    for _ in range(warmup):
        assert ua.ua_forward_host(*args) == 0
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        assert ua.ua_forward_host(*args) == 0   # returns after the stream drained
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    h2d = sum(t.numel() * t.element_size() for t in (q_h, cu_h, su_h))
    h2d += w.num_seqs * w.max_blocks_per_seq * 4
    for t in (sk_h, al_h):
        if t is not None:
            h2d += t.numel() * t.element_size()
    d2h = out_h.numel() * out_h.element_size()
    prob.close()
    return statistics.mean(times), h2d, d2h


def cpu_baseline_decode(w_host, budget_s=12.0):
    """The fp64 oracle on the host cores over a bounded sample of the decode
    batch: whole (sequence, kv head) groups, all g query heads of each, so the
    K/V bytes it must read are counted exactly as for the GPU."""
    import numpy as np
    import oracle
    threads = oracle.default_threads()
    order = list(range(w_host.num_seqs))
    done_bytes, done_time, seqs = 0, 0.0, 0
    g = w_host.hq // w_host.hk
    cu = [0]
    for s in w_host.seqlens_q:
        cu.append(cu[-1] + s)
    while done_time < budget_s and seqs < len(order):
        s = order[seqs]
        rows = [tok * w_host.hq + h for tok in range(cu[s], cu[s + 1]) for h in range(w_host.hq)]
        t = time.perf_counter()
        oracle.forward_workload(w_host, row_ids=np.array(rows, dtype=np.int64), nthreads=threads)
        done_time += time.perf_counter() - t
        done_bytes += w_host.seqlens_k[s] * w_host.hk * w_host.d * 2 * 2
        seqs += 1
    return dict(value=done_bytes / done_time / 1e9, unit="GB/s", cores=threads, kind="oracle",
                sample="%d of %d sequences of the decode batch (all %d query heads, g=%d), "
                       "%.1f s" % (seqs, w_host.num_seqs, w_host.hq, g, done_time))


def run_ours(args):
    import torch
    import paged_varlen_flash_gb300 as ua
    from paged_varlen_flash_gb300 import build as ua_build
    from paged_varlen_flash_gb300 import workloads as W

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if rank == 0:
        ua_build.build()
    if world > 1:
        dist.barrier()
    ua.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_src = load_peaks()

    w = W.make(HEADLINE, device=dev)
    nbytes, _ = workload_units(w)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    res = time_ours(w, args.steps, args.warmup, flush=False, torch=torch, ua=ua)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms, total_bytes = aggregate_ranks(sum(res["step_ms"]), nbytes, dev)
    ms_per_step = total_ms / args.steps
    value = total_bytes / (ms_per_step * 1e-3) / 1e9
    kern_ms = statistics.mean(res["kernel_ms"])
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    clocks = sampler.summary(res["t0"], res["t1"])

    # e2e through the host-buffer entry point
    e2e_ms, h2d, d2h = time_e2e(w, max(3, min(args.steps, 20)), 2, torch, ua)

    # prefill / chunked workloads: TFLOPS of the same entry point
    per_config = {}
    if not args.headline_only:
        for name in SECONDARY:
            ws = W.make(name, device=dev)
            b_s, f_s = workload_units(ws)
            r = time_ours(ws, max(3, min(args.steps, 10)), max(3, args.warmup), flush=True,
                          torch=torch, ua=ua)
            ms = statistics.mean(r["step_ms"])
            km = statistics.mean(r["kernel_ms"])
            # The kernel's own roofline: the largest of the tensor-core time
            # of its flops, the HBM time of its bytes (burst peaks: the kernel
            # is timed alone) and the special-function time of its
            # exponentials (and tanh with a softcap).
            scores = f_s / (4.0 * ws.d)
            sfu_clk = scores * (1.0 / SFU_EX2_PER_CLK + (1.0 / SFU_TANH_PER_CLK if ws.softcap else 0.0))
            t_tensor = f_s / (peaks["bf16_tflops"] * 1e12)
            t_hbm = b_s / (peaks["hbm_gbs"] * 1e9)
            t_sfu = sfu_clk / (NUM_SMS * peaks["sm_max_mhz"] * 1e6)
            t_bound = max(t_tensor, t_hbm, t_sfu)
            per_config[name] = {
                "ms_per_step": round(ms, 4), "tflops": round(f_s / (ms * 1e-3) / 1e12, 2),
                "kernel_tflops": round(f_s / (km * 1e-3) / 1e12, 2),
                "frac_of_bf16_peak": round(f_s / (km * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                "roofline_bound": ("tensor", "hbm", "sfu")[[t_tensor, t_hbm, t_sfu].index(t_bound)],
                "roofline_us": round(t_bound * 1e6, 2),
                "bounds_us": {"tensor": round(t_tensor * 1e6, 2), "hbm": round(t_hbm * 1e6, 2),
                              "sfu": round(t_sfu * 1e6, 2)},
                "frac_of_roofline": round(t_bound / (km * 1e-3), 4),
                "path": r["path"], "launches_per_step": r["launches"] // max(1, len(r["step_ms"])),
                "flops": f_s, "bytes": b_s, "device_error": r["device_error"]}
            del ws
            torch.cuda.empty_cache()
        for name in SECONDARY_HBM:
            ws = w if name == "decode_cold" else W.make(name, device=dev)
            b_s, f_s = workload_units(ws)
            # decode_topk touches 0.27 GB per step, only twice L2: flush between
            # steps; decode_cold flushes too (the headline runs warm).
            r = time_ours(ws, max(3, min(args.steps, 20)), max(3, args.warmup),
                          flush=ws.topk_len is not None or name == "decode_cold", torch=torch, ua=ua)
            ms = statistics.mean(r["step_ms"])
            km = statistics.mean(r["kernel_ms"])
            per_config[name] = {
                "ms_per_step": round(ms, 4), "gbs": round(b_s / (ms * 1e-3) / 1e9, 1),
                "kernel_gbs": round(b_s / (km * 1e-3) / 1e9, 1),
                "frac_of_hbm_peak": round(b_s / (km * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "kv_tokens_per_s": round((sum(ws.seqlens_k) if ws.topk_len is None else
                                          int(ws.topk_len.to("cpu").sum())) / (ms * 1e-3), 1),
                "path": r["path"], "launches_per_step": r["launches"] // max(1, len(r["step_ms"])),
                "bytes": b_s, "device_error": r["device_error"],
                "l2": "flushed (256 MiB write) between steps" if (ws.topk_len is not None or
                                                                 name == "decode_cold") else
                      "inputs larger than L2, no flush"}
            if ws is not w:
                del ws
            torch.cuda.empty_cache()
    sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(w.to("cpu"))

    dominant = dominant_kernel(res["path"])
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 values, seeded lengths and block tables)",
            "config": {
                "workload": "decode: 64 seqs, S_q=1, S_k~U[512,8192], H_q/H_k=32/8, d=128, "
                            "b=16, 40000-block pool, causal",
                "num_seqs": w.num_seqs, "total_kv_tokens": int(sum(w.seqlens_k)),
                "algorithmic_bytes_per_step": nbytes, "path": res["path"],
                "l2": "inputs larger than L2 (1.1 GB of K/V per step), no flush",
                "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": recorded_traffic(dominant, HEADLINE),
                         "peak_source": peak_src, "kernel_ms": round(kern_ms, 5)},
            "e2e": {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": res["launches"],
            "clocks": clocks,
            "cpu_baseline": cpu,
            "per_config": per_config,
            "device_error": res["device_error"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_single(args):
    """One named workload, timed alone (device-resident inputs, L2 flushed
    between steps); prints bytes/s and FLOP/s of the whole step and of the
    dominant kernel."""
    import torch
    import paged_varlen_flash_gb300 as ua
    from paged_varlen_flash_gb300 import build as ua_build
    from paged_varlen_flash_gb300 import workloads as W
    torch.cuda.set_device(0)
    ua_build.build()
    ua.load_library()
    peaks, peak_src = load_peaks()
    w = W.make(args.workload, device="cuda")
    nbytes, flops = workload_units(w)
    path = {"auto": ua.UA_PATH_AUTO, "split": ua.UA_PATH_SPLIT_KV,
            "tensor": ua.UA_PATH_TENSOR_CORE, "decode": ua.UA_PATH_DECODE_TC}[args.path]
    r = time_ours(w, args.steps, args.warmup, flush=True, torch=torch, ua=ua, path=path)
    ms = statistics.mean(r["step_ms"])
    km = statistics.mean(r["kernel_ms"])
    print(json.dumps({
        "workload": args.workload, "path": r["path"], "steps": args.steps,
        "ms_per_step": round(ms, 5), "kernel_ms": round(km, 5),
        "gbs": round(nbytes / (ms * 1e-3) / 1e9, 2),
        "kernel_gbs": round(nbytes / (km * 1e-3) / 1e9, 2),
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "kernel_tflops": round(flops / (km * 1e-3) / 1e12, 2),
        "frac_hbm": round(nbytes / (km * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "frac_bf16": round(flops / (km * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
        "peak_source": peak_src, "launches": r["launches"], "device_error": r["device_error"],
        "bytes": nbytes, "flops": flops}), flush=True)


def run_reference(args):
    """The fp64 CPU oracle as the reference arm, on the same workload/metric."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from paged_varlen_flash_gb300 import workloads as W
    w = W.make(HEADLINE, device="cpu")
    threads = oracle.default_threads()
    # Each step: a bounded sample of whole sequences (all heads), ~1-2 s.
    g = w.hq // w.hk
    rng = np.random.default_rng(0)
    seqs = rng.choice(w.num_seqs, size=4, replace=False)
    cu = np.concatenate([[0], np.cumsum(w.seqlens_q)])
    rows = np.array([tok * w.hq + h for s in seqs for tok in range(cu[s], cu[s + 1])
                     for h in range(w.hq)], dtype=np.int64)
    nbytes = int(sum(w.seqlens_k[s] for s in seqs)) * w.hk * w.d * 2 * 2
    for _ in range(args.warmup):
        oracle.forward_workload(w, row_ids=rows, nthreads=threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward_workload(w, row_ids=rows, nthreads=threads)
    el = time.perf_counter() - t
    ms = el * 1e3 / args.steps
    value = nbytes / (ms * 1e-3) / 1e9
    sample = "4 of 64 decode sequences per step (all %d query heads, g=%d)" % (w.hq, g)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode: 64 seqs, S_q=1, S_k~U[512,8192], H_q/H_k=32/8, "
                               "d=128, b=16, 40000-block pool, causal",
                   "sample_bytes_per_step": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the prefill / chunked workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None,
                    choices=["tiny", "decode", "chunked", "long_prefill", "long_prefill_shuffled",
                             "wide_mha_alibi", "decode_fp8", "decode_topk", "decode_d64",
                             "decode_d256"],
                    help="time only this workload and print its own short JSON line "
                         "(for profiling); the default is the full headline run")
    ap.add_argument("--path", default="auto", choices=["auto", "split", "tensor", "decode"],
                    help="kernel family for --workload (default: the library's choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3")
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload:
        run_single(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
