#!/usr/bin/env python
"""Benchmark of absorbed MLA decode on GB300: prints ONE JSON line on rank 0.

A step is one pass of the whole hot path over one batch: the split-KV plan from the
device seq_lens, the decode kernel and the log-sum-exp merge of split partials
(mla_decode_plan + mla_decode, or mla_decode_sparse).  Inputs are seeded synthetic data
already resident in HBM when the timed region starts; L2 is flushed (a 2 x L2-size write)
before every timed step and each step is timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs under torch.distributed.run: every rank decodes its own full batch (requests are
independent, no collective on the data path), value = all ranks' FLOPs / max rank time.
--impl reference times the CPU oracle on a bounded sample of the same workload.

The top-level keys describe the headline workload (--workload, by default the
DeepSeek-V3-shaped dense batch: B=64, H=128, lengths uniform in [1024, 8192]).  `workloads`
holds the same measurements for the other four workloads (tiny, long-context 128K, FP8
ragged, DSA sparse): step and decode-call times (mean, median, min), TFLOP/s, GB/s, the
roofline fraction of the decode call, the end-to-end rate through the public API with host
buffers, and the oracle's CPU baseline.

Beside the step, the line reports the kernels around the decode, each timed alone with the
same flush and events (outside the step's timed region): `append` (one new token per
request into the cache), `absorb` (q~ = q^C W^UK) and `project` (y = W^UV out) for the
workload's B and H, `topk` (DSA selection, k = 2048, over synthetic scores of the
workload's lengths) and `prefill` (decompression + causal attention of one 4,096-token
sequence with the workload's head count).  --only skips the other workloads and these.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOPS & HBM GB/s (B=64,H=128,L≤8K) and % of roofline, 1×GB300"
DEFAULT_WORKLOAD = "dsv3_dense_b64_h128_l1k_8k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# the sources of the decode call (plan, decode kernel, split merge) whose DRAM traffic
# profiles/traffic.json records
DECODE_SOURCES = ("api.cu", "common.cuh", "decode_sm103.cu", "launch.h", "plan.h", "sm103_ptx.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "mla_latent_kv_17_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def time_alone(fn, steps, flush, stream):
    """Mean CUDA-event time (ms) of fn() on `stream`, after 3 warm-up calls, with L2 flushed
    before every timed call."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ms = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        fn()
        eb.record(stream)
        eb.synchronize()
        ms.append(ea.elapsed_time(eb))
    return sum(ms) / len(ms)


def dram_traffic(workload: str):
    """DRAM bytes per decode call from the committed ncu summary, if it matches the source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_call")


class Clocks:
    """Samples the SM clock and the clock-event (throttle) reasons while the timed region runs.

    Reads NVML directly (libnvidia-ml through ctypes) from a background thread every half
    millisecond, so that even a timed region of a few milliseconds gets samples; the GPU is
    matched by UUID (NVML does not see CUDA_VISIBLE_DEVICES).  Only reads settings."""

    # clock-event reason bits of the NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.device_index = device_index
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.error = None
        self.nvml = None
        self.thread = None
        self.stop = threading.Event()

    def _open(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.device_index)
        uuid = getattr(props, "uuid", None)
        rc = -1
        if uuid is not None:
            rc = nv.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(handle))
        if rc != 0:
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle))
        if rc != 0:
            raise RuntimeError("no NVML handle for this GPU")
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:  # 1: SM clock
            self.max_mhz = float(mx.value)
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self.nvml = (nv, handle, reasons_fn)

    def _run(self):
        import ctypes
        nv, handle, reasons_fn = self.nvml
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(mhz)) == 0 and \
                    reasons_fn(handle, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            self._open()
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception as e:  # no NVML on this machine
            self.error = str(e)
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)

    def summary(self):
        if self.error is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"clock sampling unavailable: {self.error}"]}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no clock samples"]}
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def oracle_sample_time(case, budget_s=15.0):
    """Times the oracle on whole requests of `case` until ~budget_s of wall time is used;
    returns (flops_done, seconds, threads, description)."""
    import oracle
    import torch
    from mla_latent_kv_17_gb300 import metrics
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle_ref import oracle_for

    threads = oracle.default_threads()
    toks = metrics.attended_tokens(case)
    done_flops, spent, nreq = 0, 0.0, 0
    b = 0
    group = max(1, threads)
    while b < case.B and spent < budget_s:
        bs = list(range(b, min(case.B, b + group)))
        t0 = time.perf_counter()
        oracle_for(case, bs, None, nthreads=threads)
        spent += time.perf_counter() - t0
        done_flops += sum(toks[i] for i in bs) * 2 * 1088 * case.H
        nreq += len(bs)
        b += group
    desc = f"{nreq} of {case.B} requests (all {case.H} heads), fp64 oracle, {threads} threads"
    return done_flops, spent, threads, desc


def run_reference(args, ws_n, rank):
    if rank != 0:
        return
    import torch
    from mla_latent_kv_17_gb300 import inputs
    case = inputs.make_workload(args.workload, device="cpu")
    per_step = []
    flops_tot = 0
    threads, desc = 0, ""
    for i in range(args.warmup + args.steps):
        f, s, threads, desc = oracle_sample_time(case, budget_s=args.ref_budget)
        if i >= args.warmup:
            per_step.append(s)
            flops_tot += f
    secs = sum(per_step)
    val = flops_tot / secs / 1e12
    from mla_latent_kv_17_gb300 import metrics
    alg = metrics.algorithmic(case)
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "impl": "reference",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": case.B, "H": case.H,
                       "tokens": alg["tokens"], "kv": case.kv_dtype,
                       "l2": "flushed before every step (2x L2 write); step = plan + decode + merge",
                       "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def stats(ms):
    return {"mean": sum(ms) / len(ms), "median": statistics.median(ms), "min": min(ms)}


def measure_workload(name, args, dev, stream, flush, pk, pk_kind, pg, ws_n, clocks=False):
    """Times one workload: the step (plan + decode call, back to back), the decode call alone
    (decode kernel + split merge, the roofline unit) and the end-to-end call through the
    public API with host buffers; returns (summary dict, case, out) plus the clock sampler."""
    import torch
    from mla_latent_kv_17_gb300 import inputs, metrics, ops

    case = inputs.make_workload(name, device=dev)
    alg = metrics.algorithmic(case)
    sparse = case.indices is not None
    topk = case.indices.shape[1] if sparse else 0
    wsp = ops.Workspace(case.B, case.H, device=dev)
    out = torch.empty((case.B, case.H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((case.B, case.H), dtype=torch.float32, device=dev)

    def decode_call():
        if sparse:
            ops.decode_sparse(wsp, case.q_nope, case.q_rope, case.cache, case.block_table,
                              case.seq_lens, case.indices, case.scale, out, lse, stream)
        else:
            ops.decode(wsp, case.q_nope, case.q_rope, case.cache, case.block_table,
                       case.seq_lens, case.scale, out, lse, stream)

    def step():
        ops.plan(wsp, None if sparse else case.seq_lens, topk=topk, stream=stream, kv_dtype=case.kv_dtype)
        decode_call()

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    st = ops.status(wsp, stream)
    if st != 0:
        raise RuntimeError(f"{name}: device status {ops.STATUS_NAMES.get(st, st)} during warm-up")

    # a step is plan + decode call, back to back on the stream (no event between them: the
    # decode launches while the plan finishes)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clk = Clocks(torch.cuda.current_device()) if clocks else None
    if clk:
        clk.__enter__()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if clk:
        clk.__exit__(None, None, None)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    st = ops.status(wsp, stream)
    if st != 0:
        raise RuntimeError(f"{name}: device status {ops.STATUS_NAMES.get(st, st)} in timed region")
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    # the decode call alone (decode kernel + split-KV merge) for the roofline, on the plan
    # of the last step, with the same L2 flush before every call
    dec_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        decode_call()
        b_.record(stream)
        b_.synchronize()
        dec_ms.append(a_.elapsed_time(b_))
    st = ops.status(wsp, stream)
    if st != 0:
        raise RuntimeError(f"{name}: device status {ops.STATUS_NAMES.get(st, st)} in the call timing")
    tot_ms = metrics.max_over_ranks(sum(step_ms), pg, dev)
    ms_per_step = tot_ms / args.steps
    dec_avg_ms = sum(dec_ms) / len(dec_ms)

    # ---- end to end through the public API with host buffers -------------------------
    pin = lambda t: t.cpu().pin_memory()
    h_q_nope, h_q_rope = pin(case.q_nope), pin(case.q_rope)
    h_bt, h_sl = pin(case.block_table), pin(case.seq_lens)
    h_idx = pin(case.indices) if sparse else None
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_q_nope, d_q_rope = torch.empty_like(case.q_nope), torch.empty_like(case.q_rope)
    d_bt, d_sl = torch.empty_like(case.block_table), torch.empty_like(case.seq_lens)
    d_idx = torch.empty_like(case.indices) if sparse else None
    h2d = sum(t.numel() * t.element_size() for t in (h_q_nope, h_q_rope, h_bt, h_sl)) + (
        h_idx.numel() * 4 if sparse else 0)
    d2h = h_out.numel() * 4 + h_lse.numel() * 4

    def e2e_step():
        d_q_nope.copy_(h_q_nope, non_blocking=True)
        d_q_rope.copy_(h_q_rope, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        if sparse:
            d_idx.copy_(h_idx, non_blocking=True)
        ops.plan(wsp, None if sparse else d_sl, topk=topk, stream=stream, kv_dtype=case.kv_dtype)
        if sparse:
            ops.decode_sparse(wsp, d_q_nope, d_q_rope, case.cache, d_bt, d_sl, d_idx, case.scale,
                              out, lse, stream)
        else:
            ops.decode(wsp, d_q_nope, d_q_rope, case.cache, d_bt, d_sl, case.scale, out, lse,
                       stream)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(3):
        flush.fill_(2)
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_ms = metrics.max_over_ranks(sum(e_ms) / len(e_ms), pg, dev)

    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    bound = "hbm" if alg["ai"] < ridge else "tensor"
    dec_s = dec_avg_ms * 1e-3
    if bound == "hbm":
        achieved, peak, unit = alg["bytes"] / dec_s / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = alg["flops"] / dec_s / 1e12, pk["bf16_tflops"], "TFLOP/s"
    roof_s = metrics.roofline_seconds(alg["flops"], alg["bytes"], pk["bf16_tflops"], pk["hbm_gbs"])
    summary = {
        "B": case.B, "H": case.H, "kv": case.kv_dtype, "tokens": alg["tokens"],
        "value": metrics.whole_job_rate(alg["flops"], ws_n, ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s",
        "ms_per_step": ms_per_step, "step_ms": stats(step_ms), "call_ms": stats(dec_ms),
        "hbm_gbs": alg["bytes"] / (ms_per_step * 1e-3) / 1e9,
        "tflops_decode_call": alg["flops"] / dec_s / 1e12,
        "pct_roofline": roof_s / (ms_per_step * 1e-3),
        "roofline": {"kernel": "mla_decode call (decode kernel + split-KV merge)", "bound": bound,
                     "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": dram_traffic(name), "peak_source": pk_kind,
                     "ai_flop_per_byte": alg["ai"], "alg_bytes_per_call": alg["bytes"],
                     "alg_flops_per_call": alg["flops"], "call_ms": dec_avg_ms},
        "e2e": {"value": metrics.whole_job_rate(alg["flops"], ws_n, e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "wall_s_timed_region": t_wall,
    }
    return summary, case, clk


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--only", action="store_true",
                    help="measure --workload alone (no other workloads, no side kernels)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=8.0,
                    help="seconds of oracle work per reference step")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    ws_n, rank, local = dist_env()
    import torch
    pg = None
    if ws_n > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    if args.impl == "reference":
        run_reference(args, ws_n, rank)
        if pg:
            pg.destroy_process_group()
        return

    from mla_latent_kv_17_gb300 import build as mbuild
    mbuild.build()
    from mla_latent_kv_17_gb300 import inputs, ops

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    pk, pk_kind = peaks()

    head, case, clk = measure_workload(args.workload, args, dev, stream, flush, pk, pk_kind, pg, ws_n,
                                       clocks=True)
    do_cpu = rank == 0 and ws_n == 1 and not args.no_cpu_baseline
    threads = 0
    if do_cpu:
        f, s_, threads, desc = oracle_sample_time(case, budget_s=12.0)
        head["cpu_baseline"] = {"value": f / s_ / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "cpu_model": cpu_model(), "kind": "oracle", "sample": desc, "seconds": s_}

    # ---- the kernels around the decode, for the headline workload's B and H ------------
    side = {} if args.only else side_kernels(case, args, dev, stream, flush, pk)
    del case
    torch.cuda.empty_cache()

    # ---- the other workloads: same measurements, each its own line item ----------------
    others = {}
    if not args.only:
        for name in inputs.WORKLOADS:
            if name == args.workload:
                continue
            summ, c2, _ = measure_workload(name, args, dev, stream, flush, pk, pk_kind, pg, ws_n)
            if do_cpu:
                f, s_, th, desc = oracle_sample_time(c2, budget_s=8.0)
                summ["cpu_baseline"] = {"value": f / s_ / 1e12, "unit": "TFLOP/s", "cores": th,
                                        "cpu_model": cpu_model(), "kind": "oracle", "sample": desc,
                                        "seconds": s_}
            others[name] = summ
            del c2
            torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": head["B"], "H": head["H"],
                   "tokens": head["tokens"], "kv": head["kv"],
                   "l2": "flushed before every step (2x L2 write); step = plan + decode + merge",
                   "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU"},
        "step_ms": head["step_ms"], "call_ms": head["call_ms"],
        "hbm_gbs": head["hbm_gbs"], "tflops_decode_call": head["tflops_decode_call"],
        "pct_roofline": head["pct_roofline"], "roofline": head["roofline"], "e2e": head["e2e"],
        "gpu_launches": 3 * args.steps,
        **side,
        "workloads": others,
        "clocks": clk.summary(),
        "wall_s_timed_region": head["wall_s_timed_region"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def side_kernels(case, args, dev, stream, flush, pk):
    """Times the kernels around the decode for `case`'s B and H, each alone with the same
    flush and events: the cache append, query absorption, value projection, top-k selection
    and a 4,096-token prefill."""
    import torch
    from mla_latent_kv_17_gb300 import inputs, ops

    # ---- cache append (the step after decode): one token per request, timed alone -------
    # (written at each request's last position, inside its block table; after every decode
    # measurement, since it changes the cache)
    g_app = torch.Generator().manual_seed(7)
    a_lat = torch.randn(case.B, 512, generator=g_app).to(torch.bfloat16).to(dev)
    a_rope = torch.randn(case.B, 64, generator=g_app).to(torch.bfloat16).to(dev)
    a_pos = (case.seq_lens - 1).clamp(min=-1).to(torch.int32).contiguous()
    app_ms = time_alone(lambda: ops.cache_append(case.cache, case.block_table, a_pos, a_lat, a_rope,
                                                 stream=stream), args.steps, flush, stream)
    rec_bytes = 656 if case.kv_dtype == "fp8" else 1152
    n_app = int((a_pos >= 0).sum().item())
    app_bytes = n_app * (rec_bytes + 1024 + 128 + 4 + 4)  # record out; latent, rope, position, page id in

    # ---- query absorption before and value projection after the decode (random weights of
    # the workload's head count; q^C and the latent output of its batch), each timed alone
    q_c, w_uk, w_uv, lat_out = inputs.projection_inputs(case.B, case.H, seed=8, device=dev)
    q_abs = torch.empty(case.B, case.H, 512, dtype=torch.bfloat16, device=dev)
    y_prj = torch.empty(case.B, case.H, 128, dtype=torch.float32, device=dev)
    ab_ms = time_alone(lambda: ops.absorb_query(q_c, w_uk, q_nope=q_abs, stream=stream), args.steps, flush, stream)
    pj_ms = time_alone(lambda: ops.project_output(lat_out, w_uv, y=y_prj, stream=stream), args.steps, flush, stream)
    # DSA top-k selection over synthetic indexer scores of the workload's lengths (k = 2048)
    tk_k = 2048
    tk_lmax = (int(case.seq_lens.max().item()) + 3) // 4 * 4
    tk_scores = torch.randn(case.B, tk_lmax, generator=torch.Generator(device=dev).manual_seed(9), device=dev)
    tk_idx = torch.empty(case.B, tk_k, dtype=torch.int32, device=dev)
    tk_ms = time_alone(lambda: ops.topk_select(tk_scores, case.seq_lens, tk_k, indices=tk_idx, stream=stream),
                       args.steps, flush, stream)
    tk_bytes = int(case.seq_lens.sum().item()) * 4 + case.B * (tk_k + 1) * 4  # scores, lengths in; indices out
    # non-absorbed prefill of one 4096-token sequence with the workload's head count:
    # decompression (K, V with W^UK, W^UV) + causal attention, timed together
    pf_L = 4096
    gpf = torch.Generator(device=dev).manual_seed(10)
    pf_e = torch.randn(pf_L, 576, generator=gpf, device=dev).to(torch.bfloat16)
    pf_qn = torch.randn(pf_L, case.H, 128, generator=gpf, device=dev).to(torch.bfloat16)
    pf_qr = torch.randn(pf_L, case.H, 64, generator=gpf, device=dev).to(torch.bfloat16)
    pf_k = torch.empty(case.H, pf_L, 128, dtype=torch.bfloat16, device=dev)
    pf_v = torch.empty_like(pf_k)
    pf_o = torch.empty(pf_L, case.H, 128, dtype=torch.float32, device=dev)
    pf_l = torch.empty(pf_L, case.H, dtype=torch.float32, device=dev)

    def prefill_call():
        ops.prefill_decompress(pf_e, w_uk, w_uv, k_nope=pf_k, v=pf_v, stream=stream)
        ops.prefill_attention(pf_qn, pf_qr, pf_e, pf_k, pf_v, case.scale, out=pf_o, lse=pf_l, stream=stream)

    pf_ms = time_alone(prefill_call, args.steps, flush, stream)
    pf_dc_ms = time_alone(lambda: ops.prefill_decompress(pf_e, w_uk, w_uv, k_nope=pf_k, v=pf_v, stream=stream),
                          args.steps, flush, stream)
    pf_dc_flops = 2 * 2 * pf_L * 512 * 128 * case.H
    pf_at_flops = 2 * case.H * (pf_L * (pf_L + 1) // 2) * (192 + 128)
    BH = case.B * case.H
    ab_bytes = case.H * 128 * 512 * 2 + BH * 128 * 2 + BH * 512 * 2  # W^UK, q^C in; q~ out
    pj_bytes = case.H * 128 * 512 * 2 + BH * 512 * 4 + BH * 128 * 4  # W^UV, latent out in; y out
    return {
        "append": {"kernel": "cache append (mla_cache_append), one token per request", "requests": n_app,
                   "kv": case.kv_dtype, "us": app_ms * 1e3, "bytes": app_bytes,
                   "gbs": app_bytes / (app_ms * 1e-3) / 1e9},
        "absorb": {"kernel": "query absorption q~ = q^C W^UK (mla_absorb_query)", "us": ab_ms * 1e3,
                   "bytes": ab_bytes, "gbs": ab_bytes / (ab_ms * 1e-3) / 1e9,
                   "frac_hbm": ab_bytes / (ab_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "project": {"kernel": "value projection y = W^UV out (mla_project_output)", "us": pj_ms * 1e3,
                    "bytes": pj_bytes, "gbs": pj_bytes / (pj_ms * 1e-3) / 1e9,
                    "frac_hbm": pj_bytes / (pj_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "topk": {"kernel": "DSA top-k selection (mla_topk_select), k = 2048 per request", "us": tk_ms * 1e3,
                 "bytes": tk_bytes, "gbs": tk_bytes / (tk_ms * 1e-3) / 1e9,
                 "frac_hbm": tk_bytes / (tk_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "prefill": {"kernel": "non-absorbed prefill (mla_prefill_decompress + mla_prefill_attention), causal",
                    "tokens": pf_L, "heads": case.H, "us": pf_ms * 1e3, "decompress_us": pf_dc_ms * 1e3,
                    "decompress_tflops": pf_dc_flops / (pf_dc_ms * 1e-3) / 1e12,
                    "flops": pf_dc_flops + pf_at_flops,
                    "tflops": (pf_dc_flops + pf_at_flops) / (pf_ms * 1e-3) / 1e12,
                    "frac_bf16": (pf_dc_flops + pf_at_flops) / (pf_ms * 1e-3) / 1e12 / pk["bf16_tflops"]},
    }


if __name__ == "__main__":
    main()
