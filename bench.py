"""Benchmark of the stochastic verification step on GB300.

One step = one pass of the verification hot path over one batch: the fused
max / log-sum-exp / argmax row reduction, the temperature / top-k / top-p /
min-p filtered Gumbel-max sampler, the point-mass rejection chain with
replacement / bonus tokens, and the fused per-position prefix-acceptance
counters -- one spec_verify_sample call on the mixed-temperature workload
B=128 requests, k=4 draft tokens (640 packed rows), V=152064, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank verifies its own
batch (independent requests: weak scaling, no data-path collective).
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import re
import json
import os
import platform
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verified rows/s and achieved HBM GB/s (% of peak) at B=128,k=4,V=152064 bf16"
WORKLOAD = ("stochastic verify: B=128, k=4 (640 packed rows), V=152064, bf16 logits ~N(0,3); "
            "per-request T in {0,0.5,1}, top_k in {0,20,50}, top_p in {1,0.9}, min_p in {0,0.05}; "
            "Philox seed per request; point-mass draft")
B, K, V = 128, 4, W.QWEN_VOCAB
R = B * (K + 1)
KERNEL_SOURCES = ["speculative_decoding_verification_ragged_gb300/csrc/verify.cu",
                  "speculative_decoding_verification_ragged_gb300/csrc/rowkit.cuh",
                  "speculative_decoding_verification_ragged_gb300/csrc/common.cuh"]


# kernels one spec_verify_sample call launches: the row records, stream and
# finish kernels
LAUNCHES_PER_CALL = 3


def _code_only(text: str) -> str:
    """The source without // and /* */ comments or blank lines (comment edits
    do not change a kernel, so they do not invalidate its counters)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def traffic_record():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "verify_sample_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_sources_sha256_16") != kernel_digest():
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------- clocks -----

class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (read-only) in a
    background thread while the timed region runs."""
    HW_SLOWDOWN, HW_THERMAL, SW_THERMAL, SW_POWER = 0x8, 0x40, 0x20, 0x4

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._period = period_s
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self._period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self) -> dict:
        names = []
        for bit, n in [(self.HW_SLOWDOWN, "hw_slowdown"), (self.HW_THERMAL, "hw_thermal_slowdown"),
                       (self.SW_THERMAL, "sw_thermal_slowdown"), (self.SW_POWER, "sw_power_cap")]:
            if self.reasons & bit:
                names.append(n)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples),
                "source": "nvml" if self.ok else "unavailable"}


# ------------------------------------------------------------ our arm -----

# Row classes for profiling the sampler one filter kind at a time (every
# request given the same filters); "mix" is the benchmark's workload.
ROW_CLASSES = {
    "mix": {},
    "greedy": dict(temperatures=(0.0,)),
    "topk": dict(temperatures=(1.0,), top_ks=(50,), top_ps=(1.0,), min_ps=(0.0,)),
    "minp": dict(temperatures=(1.0,), top_ks=(0,), top_ps=(1.0,), min_ps=(0.05,)),
    "topp1": dict(temperatures=(1.0,), top_ks=(0,), top_ps=(0.9,), min_ps=(0.0,)),
    "topp05": dict(temperatures=(0.5,), top_ks=(0,), top_ps=(0.9,), min_ps=(0.0,)),
    "unfiltered": dict(temperatures=(1.0,), top_ks=(0,), top_ps=(1.0,), min_ps=(0.0,)),
}
ROW_CLASS = "mix"


def workload_name() -> str:
    if ROW_CLASS == "mix":
        return WORKLOAD
    return WORKLOAD + " -- profiling variant: every request " + ROW_CLASS


def make_inputs(seed: int):
    vb, p = W.stochastic(seed=seed, **ROW_CLASSES[ROW_CLASS])
    return vb, p


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import speculative_decoding_verification_ragged_gb300 as sv
    import speculative_decoding_verification_ragged_gb300.binding  # noqa: F401
    from speculative_decoding_verification_ragged_gb300 import shard
    sv.build()

    vb, p = make_inputs(W.data_seed(3) + rank)
    logits_host = torch.from_numpy(vb.logits.view(np.int16)).view(torch.bfloat16)
    nsets = args.sets
    sets = [logits_host.to(dev) for _ in range(nsets)]          # rotating copies > L2
    cu = torch.from_numpy(vb.cu_rows).to(dev)
    dr = torch.from_numpy(vb.draft_ids).to(dev)
    tt = torch.from_numpy(p.temperature).to(dev)
    tk = torch.from_numpy(p.top_k).to(dev)
    tp = torch.from_numpy(p.top_p).to(dev)
    mp = torch.from_numpy(p.min_p).to(dev)
    sd = torch.from_numpy(p.seed.view(np.int64)).to(dev)
    rid = torch.from_numpy(p.request_id.view(np.int32)).to(dev)
    ws = sv.new_workspace(R, B, V, torch.bfloat16, dev, sampling=True)
    acc = torch.zeros(K, dtype=torch.int64, device=dev)
    ver = torch.zeros(K, dtype=torch.int64, device=dev)
    hist = torch.zeros(K + 1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    call = sv.binding.PreparedSample(sets[0], cu, dr, tt, tk, tp, mp, sd, rid, V=V, B=B, k_max=K,
                                     R_cap=R, workspace=ws, rows=True, stats=(acc, ver, hist),
                                     stream=stream)

    def step(i):
        return call(sets[i % nsets], i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # The timed region: K calls back to back on the launching stream, one
    # event pair around all of them (a call's first kernel overlaps the
    # previous call's last, as in a serving loop).  Then the same K calls
    # again, each bracketed by its own events, for the spread of one
    # isolated call (the events keep neighbouring calls from overlapping).
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        torch.cuda._sleep(50_000_000)   # queue ahead of the device (outside the timed region)
        t0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    mean_launch_ms = total_ms / args.steps
    total_ms = shard.max_over_ranks(total_ms, dev)          # the job's time: its slowest rank
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda._sleep(50_000_000)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step(args.warmup + args.steps + i)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    launch_ms = [a.elapsed_time(b) for a, b in ev]

    # end to end through the public API with host buffers: H2D of the step's
    # inputs from pinned memory, the call, D2H of the step's results.  As in
    # a serving loop, the next step's inputs (the logits, then the small
    # inputs packed in one buffer) are copied on a second stream into the
    # other of two device slots while this step computes; the copy into a
    # slot waits for the call two steps back, its last reader.  The request
    # outputs and status come back in one copy.  Every step still moves all
    # its bytes, and one link carries them: small copies queued between the
    # large ones on the compute stream would serialise the two.
    pin = logits_host.pin_memory()
    small_np = [np.ascontiguousarray(a) for a in
                [vb.cu_rows, vb.draft_ids, p.temperature, p.top_k, p.top_p, p.min_p,
                 p.seed.view(np.int64), p.request_id.view(np.int32)]]
    small_dt = [torch.int32, torch.int32, torch.float32, torch.int32, torch.float32,
                torch.float32, torch.int64, torch.int32]
    offs, nbytes = [], 0
    for a in small_np:
        nbytes = (nbytes + 15) // 16 * 16
        offs.append(nbytes)
        nbytes += a.nbytes
    small_pin = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    for a, o in zip(small_np, offs):
        small_pin[o:o + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8)))
    slots = [sets[0], sets[1] if nsets > 1 else torch.empty_like(sets[0])]
    small_slots = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    calls = [sv.binding.PreparedSample(
        slots[j], *[small_slots[j][o:o + a.nbytes].view(dt) for a, o, dt in zip(small_np, offs, small_dt)],
        V=V, B=B, k_max=K, R_cap=R, workspace=ws, rows=False, stream=stream) for j in range(2)]
    out_host = torch.empty(calls[0].res["request_block"].numel(), dtype=torch.int32).pin_memory()
    h2d = pin.numel() * 2 + nbytes
    d2h = out_host.numel() * 4
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]

    def e2e_copy(i):
        j = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(used[j])
            slots[j].copy_(pin, non_blocking=True)
            small_slots[j].copy_(small_pin, non_blocking=True)
            copied[j].record(copy_stream)

    def e2e_step(i, n):
        j = i % 2
        if i == 0:
            e2e_copy(0)
        if i + 1 < n:
            e2e_copy(i + 1)
        stream.wait_event(copied[j])
        res = calls[j](slots[j], step=i)
        used[j].record(stream)
        out_host.copy_(res["request_block"], non_blocking=True)

    for i in range(3):
        e2e_step(i, 3)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i, e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = shard.max_over_ranks(e2e_ms, dev)
    # job-wide prefix-acceptance counters (one sum all-reduce, at read time)
    shard.reduce_prefix_stats(acc, ver, hist)

    prefix_acc = [round(float(x), 4) for x in
                  shard.prefix_acceptance(acc.cpu().numpy(), ver.cpu().numpy())]
    entries = time_entry_points(sv, dev, stream, args) if (rank == 0 and not args.no_entries) else None
    entry_errors = None
    if entries is not None:
        # the later entry points run last and cannot cost the line above
        try:
            entries.update(time_more_entry_points(sv, dev, stream, args))
        except Exception as exc:  # noqa: BLE001 -- reported in the JSON line
            entry_errors = "%s: %s" % (type(exc).__name__, exc)

    if rank == 0:
        peaks = measured_peaks()
        bytes_per_launch = (R * V * 2                      # logits, read once
                            + (B + 1) * 4 + R * 4          # cu_rows, draft ids
                            + B * (4 * 4 + 8 + 4)          # per-request parameters
                            + B * 4 * (K + 3)              # request outputs
                            + R * 4 * 4)                   # row outputs
        achieved = bytes_per_launch / (mean_launch_ms * 1e-3) / 1e9
        value = world * R * args.steps / (total_ms * 1e-3)
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_name(), "global_batch": B * world, "rows_per_step": R,
                       "vocab": V, "draft_tokens": K, "parallelism": "replicas" if world > 1 else "1 gpu",
                       "l2": "inputs rotate over %d device copies of %.1f MB each (> 129 MB L2)"
                             % (nsets, R * V * 2 / 1e6)},
            "hbm_gbs": round(achieved, 1),
            "hbm_pct_of_peak": round(100 * achieved / peaks["hbm_gbs"], 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": traffic_record(), "peak_source": peaks["source"],
                         "kernel": "spec_verify_sample call (sample_records + stream_chunks + "
                                   "finish_rows kernels, bf16)",
                         "algorithmic_bytes_per_launch": bytes_per_launch,
                         "mean_launch_us": round(mean_launch_ms * 1e3, 3),
                         "isolated_call_us_mean": round(sum(launch_ms) / len(launch_ms) * 1e3, 3),
                         "isolated_call_us_p10_median_p90": [
                             round(float(np.percentile(launch_ms, q)) * 1e3, 3)
                             for q in (10, 50, 90)]},
            "e2e": {"value": round(world * R * e2e_steps / (e2e_ms * 1e-3), 1), "unit": "rows/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": LAUNCHES_PER_CALL * args.steps,
            "prefix_acceptance": prefix_acc,
            "clocks": clocks.summary(),
        }
        if entries is not None:
            for e in entries.values():
                if "hbm_gbs" in e:
                    e["pct_of_peak"] = round(100 * e["hbm_gbs"] / peaks["hbm_gbs"], 1)
            line["entry_points"] = entries
            if entry_errors:
                line["entry_point_errors"] = entry_errors
            line["step_controller"] = time_step_controller(sv)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(vb, p)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _time_launches(fn, n: int, stream) -> float:
    """Mean device time (ms) of fn(i) over n back-to-back launches: the GPU
    is kept busy while the host queues them, then one pair of events on
    `stream` brackets the n calls."""
    import torch
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(100_000_000)
    t0.record(stream)
    for i in range(n):
        fn(i)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def time_entry_points(sv, dev, stream, args) -> dict:
    """Device time of the other entry points at their workload shapes
    (inputs rotate over device copies larger than L2).  Arguments are
    marshalled once; each timed launch is one C-ABI call."""
    import ctypes as C
    import torch
    from speculative_decoding_verification_ragged_gb300 import binding as Bd

    L = Bd.load_library()
    s = stream.cuda_stream

    def bf(x):
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)

    def ok(rc):
        if rc:
            raise RuntimeError("entry point returned %d" % rc)

    out = {}
    n = args.entry_launches
    # greedy verification, Qwen2.5-14B-shaped (B=128, k=4, V=152064, planted peaks)
    vb = W.planted_greedy()
    sets = [bf(vb.logits) for _ in range(args.sets)]
    cu, dr = torch.from_numpy(vb.cu_rows).to(dev), torch.from_numpy(vb.draft_ids).to(dev)
    ws = sv.new_workspace(vb.R, vb.B, vb.V, torch.bfloat16, dev)
    b = Bd._batch(sets[0], vb.V, vb.B, vb.k_max, vb.R, cu, dr)
    o, _ = Bd._outputs(vb.B, vb.k_max, vb.R, dev, True, None)

    def greedy(i):
        b.logits = sets[i % len(sets)].data_ptr()
        ok(L.spec_verify_greedy(C.byref(b), C.byref(o), ws.data_ptr(), ws.numel(), s))
    for i in range(5):
        greedy(i)
    ms = _time_launches(greedy, n, stream)
    out["spec_verify_greedy"] = {"workload": "B=128 k=4 V=152064 bf16 planted, with row max/LSE/argmax",
                                 "rows": vb.R, "us": round(ms * 1e3, 2),
                                 "hbm_gbs": round(vb.R * vb.V * 2 / (ms * 1e-3) / 1e9, 1)}
    # the same rows with the 5.25 confidence margin, positions from 1, and 16
    # protected token ids
    mg = torch.full((vb.B,), 5.25, dtype=torch.float32, device=dev)
    prot = torch.arange(151_643, 151_659, dtype=torch.int32, device=dev)
    m = Bd.Margin(mg.data_ptr(), None, prot.data_ptr(), prot.numel(), 1, 0)

    def margin(i):
        b.logits = sets[i % len(sets)].data_ptr()
        ok(L.spec_verify_greedy_margin(C.byref(b), C.byref(m), C.byref(o), ws.data_ptr(),
                                       ws.numel(), s))
    for i in range(5):
        margin(i)
    ms = _time_launches(margin, n, stream)
    out["spec_verify_greedy_margin"] = {
        "workload": "B=128 k=4 V=152064 bf16 planted, margin 5.25 from position 1, 16 protected ids",
        "rows": vb.R, "us": round(ms * 1e3, 2),
        "hbm_gbs": round(vb.R * vb.V * 2 / (ms * 1e-3) / 1e9, 1)}
    del sets
    # relaxed top-K (EAGLE-relaxed, B=256, k=5, V=152064, K=4)
    vb = W.relaxed_planted()
    sets = [bf(vb.logits) for _ in range(2)]
    cu, dr = torch.from_numpy(vb.cu_rows).to(dev), torch.from_numpy(vb.draft_ids).to(dev)
    K = torch.from_numpy(vb.extra["relaxed_k"]).to(dev)
    ws = sv.new_workspace(vb.R, vb.B, vb.V, torch.bfloat16, dev)
    acc = torch.zeros(vb.k_max, dtype=torch.int64, device=dev)
    ver, hist = acc.clone(), torch.zeros(vb.k_max + 1, dtype=torch.int64, device=dev)
    b = Bd._batch(sets[0], vb.V, vb.B, vb.k_max, vb.R, cu, dr)
    o, _ = Bd._outputs(vb.B, vb.k_max, vb.R, dev, True, (acc, ver, hist))

    def relaxed(i):
        b.logits = sets[i % 2].data_ptr()
        ok(L.spec_verify_relaxed_topk(C.byref(b), K.data_ptr(), C.byref(o), ws.data_ptr(),
                                      ws.numel(), s))
    for i in range(5):
        relaxed(i)
    ms = _time_launches(relaxed, n, stream)
    out["spec_verify_relaxed_topk"] = {"workload": "B=256 k=5 V=152064 bf16 K=4 + fused stats",
                                       "rows": vb.R, "us": round(ms * 1e3, 2),
                                       "hbm_gbs": round(vb.R * vb.V * 2 / (ms * 1e-3) / 1e9, 1)}
    del sets
    # draft confidence + allocation (MTP/DSpark-shaped, B=16, k=7, V=151552)
    db = W.mtp_adaptive(planted_draft=True)
    dsets = [bf(db.draft_logits) for _ in range(8)]
    dws = Bd.new_draft_workspace(db.B, db.k, db.V, torch.bfloat16, dev)
    d = Bd.Draft(dsets[0].data_ptr(), Bd.SPEC_BF16, db.V, dsets[0].stride(0), db.B, db.k, None,
                 0.3, 0)
    cap = db.B * (db.k + 1)
    bufs = [torch.empty(db.B * db.k, dtype=torch.float32, device=dev)] + \
           [torch.empty(x, dtype=torch.int32, device=dev)
            for x in [db.B * db.k, db.B, db.B + 1, cap, cap, cap, 1, 1]]
    a = Bd.Allocation(*[t.data_ptr() for t in bufs])

    def conf(i):
        d.draft_logits = dsets[i % 8].data_ptr()
        ok(L.spec_draft_confidence(C.byref(d), C.byref(a), dws.data_ptr(), dws.numel(), s))
    for i in range(5):
        conf(i)
    ms = _time_launches(conf, n, stream)
    rows = db.B * db.k
    out["spec_draft_confidence"] = {"workload": "B=16 k=7 V=151552 bf16, threshold 0.3",
                                    "rows": rows, "us": round(ms * 1e3, 2),
                                    "hbm_gbs": round(rows * db.V * 2 / (ms * 1e-3) / 1e9, 1)}
    # the adaptive pipeline on the device: confidence -> allocation -> packed
    # greedy verification of the allocated rows (target logits B*(k+1) x V)
    tsets = [bf(db.target_logits) for _ in range(8)]
    tws = sv.new_workspace(cap, db.B, db.V, torch.bfloat16, dev)
    tb = Bd.Batch(tsets[0].data_ptr(), Bd.SPEC_BF16, db.V, tsets[0].stride(0), db.B, db.k, cap,
                  bufs[3].data_ptr(), bufs[6].data_ptr())
    to, tres = Bd._outputs(db.B, db.k, cap, dev, False, None)

    def pipeline(i):
        d.draft_logits = dsets[i % 8].data_ptr()
        ok(L.spec_draft_confidence(C.byref(d), C.byref(a), dws.data_ptr(), dws.numel(), s))
        tb.logits = tsets[i % 8].data_ptr()
        ok(L.spec_verify_greedy(C.byref(tb), C.byref(to), tws.data_ptr(), tws.numel(), s))
    for i in range(5):
        pipeline(i)
    ms = _time_launches(pipeline, n, stream)
    vrows = int(bufs[7].cpu()[0])
    out["adaptive_pipeline"] = {
        "workload": "B=16 k=7 V=151552 bf16: spec_draft_confidence (threshold 0.3) then "
                    "spec_verify_greedy over the allocated packed rows",
        "draft_rows": rows, "verified_rows": vrows, "us": round(ms * 1e3, 2),
        "hbm_gbs": round((rows + vrows) * db.V * 2 / (ms * 1e-3) / 1e9, 1),
        "mean_accepted": round(float(tres["accepted_len"].float().mean()), 3)}
    del dsets, tsets
    # tiny greedy verification: 4 requests, k=4, vocab 1024, fp32 (launch-
    # and latency-bound; the 80 KB input stays in L2)
    vt = W.tiny_greedy()
    lt = torch.from_numpy(vt.logits).to(dev)
    cu, dr = torch.from_numpy(vt.cu_rows).to(dev), torch.from_numpy(vt.draft_ids).to(dev)
    ws = sv.new_workspace(vt.R, vt.B, vt.V, torch.float32, dev)
    b = Bd._batch(lt, vt.V, vt.B, vt.k_max, vt.R, cu, dr)
    o, _ = Bd._outputs(vt.B, vt.k_max, vt.R, dev, False, None)

    def tiny(i):
        ok(L.spec_verify_greedy(C.byref(b), C.byref(o), ws.data_ptr(), ws.numel(), s))
    for i in range(5):
        tiny(i)
    ms = _time_launches(tiny, n, stream)
    out["spec_verify_greedy_tiny"] = {"workload": "B=4 k=4 V=1024 fp32 (20 rows), L2-resident",
                                      "rows": vt.R, "us": round(ms * 1e3, 2)}
    # relaxed top-K over 20 seeded steps, the prefix-acceptance counters
    # accumulated on the device by the fused path
    steps = []
    for vb in W.relaxed_steps(20):
        steps.append((bf(vb.logits), torch.from_numpy(vb.cu_rows).to(dev),
                      torch.from_numpy(vb.draft_ids).to(dev)))
    K = torch.from_numpy(vb.extra["relaxed_k"]).to(dev)
    ws = sv.new_workspace(vb.R, vb.B, vb.V, torch.bfloat16, dev)
    acc = torch.zeros(vb.k_max, dtype=torch.int64, device=dev)
    ver, hist = acc.clone(), torch.zeros(vb.k_max + 1, dtype=torch.int64, device=dev)
    o, _ = Bd._outputs(vb.B, vb.k_max, vb.R, dev, False, (acc, ver, hist))
    bs = [Bd._batch(lg, vb.V, vb.B, vb.k_max, vb.R, c_, d_) for lg, c_, d_ in steps]

    def step(i):
        ok(L.spec_verify_relaxed_topk(C.byref(bs[i]), K.data_ptr(), C.byref(o), ws.data_ptr(),
                                      ws.numel(), s))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    for x in (acc, ver, hist):
        x.zero_()
    ms = _time_launches(step, len(steps), stream)
    a_, v_ = acc.cpu().numpy(), ver.cpu().numpy()
    out["relaxed_20_steps"] = {
        "workload": "EAGLE-relaxed B=256 k=5 V=152064 bf16 K=4, 20 seeded steps, fused counters",
        "steps": len(steps), "rows_per_step": vb.R, "us_per_step": round(ms * 1e3, 2),
        "hbm_gbs": round(vb.R * vb.V * 2 / (ms * 1e-3) / 1e9, 1),
        "prefix_acceptance": [round(float(x) / max(float(y), 1.0), 4) for x, y in zip(a_, v_)],
        "accepted_hist": [int(x) for x in hist.cpu().numpy()]}
    del steps, bs
    # standalone prefix statistics
    al = torch.randint(0, 5, (128,), dtype=torch.int32, device=dev)
    cu = torch.arange(0, 129 * 5, 5, dtype=torch.int32, device=dev)
    acc = torch.zeros(4, dtype=torch.int64, device=dev)
    ver, hist = acc.clone(), torch.zeros(5, dtype=torch.int64, device=dev)

    def stats(i):
        ok(L.spec_prefix_stats(al.data_ptr(), cu.data_ptr(), 128, 4, acc.data_ptr(), ver.data_ptr(),
                               hist.data_ptr(), None, s))
    ms = _time_launches(stats, n, stream)
    out["spec_prefix_stats"] = {"workload": "B=128 k=4", "us": round(ms * 1e3, 2), "hbm_gbs": 0.0}
    return out


def time_more_entry_points(sv, dev, stream, args) -> dict:
    """Device time of greedy verification over an active vocabulary and of
    the compact-row restore (inputs rotate over copies larger than L2)."""
    import ctypes as C
    import torch
    from speculative_decoding_verification_ragged_gb300 import binding as Bd

    L = Bd.load_library()
    s = stream.cuda_stream
    n = args.entry_launches
    out = {}

    def ok(rc):
        if rc:
            raise RuntimeError("entry point returned %d" % rc)

    g = torch.Generator(device=dev).manual_seed(21)
    # greedy over 32000 active columns of a 152064-token vocabulary
    B, K, Va, Vfull = 128, 4, 32_000, 152_064
    R = B * (K + 1)
    sets = [(3 * torch.randn(R, Va, device=dev, generator=g)).to(torch.bfloat16)
            for _ in range(4)]
    ids = torch.randperm(Vfull, device=dev, generator=g)[:Va].sort().values.to(torch.int32)
    cu = torch.arange(0, R + 1, K + 1, dtype=torch.int32, device=dev)
    dr = ids[torch.randint(0, Va, (R,), device=dev, generator=g)].contiguous()
    ws = sv.new_workspace(R, B, Va, torch.bfloat16, dev)
    b = Bd._batch(sets[0], Va, B, K, R, cu, dr)
    o, _ = Bd._outputs(B, K, R, dev, True, None)

    def active(i):
        b.logits = sets[i % len(sets)].data_ptr()
        ok(L.spec_verify_greedy_active(C.byref(b), ids.data_ptr(), C.byref(o), ws.data_ptr(),
                                       ws.numel(), s))
    for i in range(5):
        active(i)
    ms = _time_launches(active, n, stream)
    out["spec_verify_greedy_active"] = {
        "workload": "B=128 k=4, 32000 active columns of 152064, bf16 N(0,3), row outputs",
        "rows": R, "us": round(ms * 1e3, 2), "hbm_gbs": round(R * Va * 2 / (ms * 1e-3) / 1e9, 1)}
    del sets
    # hidden states of the compact rows back to their slots: B=128, k=4,
    # H=5120 bf16 (10 KiB rows), every request keeping all its rows
    H = 5120
    # (12 source/destination pairs of 6.6 MB each rotate through more than L2)
    comp = [torch.randn(R, H, device=dev, generator=g).to(torch.bfloat16) for _ in range(12)]
    dst = [torch.empty(R, H, device=dev, dtype=torch.bfloat16) for _ in range(12)]

    def restore(i):
        c, d = comp[i % 12], dst[i % 12]
        ok(L.spec_restore_rows(c.data_ptr(), H * 2, R, cu.data_ptr(), B, K, H * 2, d.data_ptr(),
                               H * 2, None, s))
    for i in range(5):
        restore(i)
    ms = _time_launches(restore, n, stream)
    out["spec_restore_rows"] = {
        "workload": "B=128 k=4 rows of 5120 bf16, every slot restored",
        "rows": R, "us": round(ms * 1e3, 2), "hbm_gbs": round(2 * R * H * 2 / (ms * 1e-3) / 1e9, 1)}
    return out


def time_step_controller(sv, batches: int = 20_000) -> dict:
    """Host time of one spec_step_update (the adaptive draft-step decision)
    with the page's policy (window 20, re-scoring every 5, gain 5 %), k <= 5,
    B = 128 and an SPS cost table, fed the counters of synthetic batches."""
    rng = np.random.default_rng(7)
    ctl = sv.StepController(1, 5, 4)
    cost = sv.step_cost_sps(128, 5, [128, 256, 512, 768], [60.0, 55.0, 45.0, 38.0])
    ver = np.full(5, 128, np.int64)
    accs = [np.sort(rng.integers(0, 129, size=5))[::-1].astype(np.int64) for _ in range(64)]
    t0 = time.perf_counter()
    for i in range(batches):
        ctl.update(accs[i % 64], ver, cost, 128)
    us = (time.perf_counter() - t0) / batches * 1e6
    # the C call alone: arguments marshalled once
    L = sv.load_library()
    st = ctl._state.ctypes.data_as(ctypes.c_void_p)
    pa = [a.ctypes.data_as(ctypes.c_void_p) for a in accs]
    pv, pc, k = ver.ctypes.data_as(ctypes.c_void_p), cost.ctypes.data_as(ctypes.c_void_p), \
        ctypes.c_int32(0)
    kr = ctypes.byref(k)
    fn = L.spec_step_update
    t0 = time.perf_counter()
    for i in range(batches):
        fn(st, pa[i % 64], pv, pc, 128, kr)
    us_c = (time.perf_counter() - t0) / batches * 1e6
    return {"policy": "window 20, every 5 batches, gain 0.05, k in [1, 5], B=128, SPS costs",
            "batches": batches, "us_per_batch_binding": round(us, 3),
            "us_per_batch_c_call": round(us_c, 3), "k_final": int(k.value)}


def cpu_baseline(vb, p, budget_s: float = 10.0) -> dict:
    """The oracle as it stands, on the host cores, over whole batches of the
    same workload, repeated until about budget_s of CPU time has passed."""
    import oracle
    oracle.build()
    cores = oracle.threads(len(os.sched_getaffinity(0)))
    rows = 0
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids, p)
        rows += vb.R
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 20:
            break
    dt = time.perf_counter() - t0
    # one thread, on the first 16 requests of the same batch
    nb = min(16, vb.B)
    r1 = int(vb.cu_rows[nb])
    sub = W.VerifyBatch(vb.logits[:r1], vb.dtype, vb.V, nb, vb.k_max, vb.cu_rows[:nb + 1],
                        vb.draft_ids[:r1])
    ps = W.SampleParams(p.temperature[:nb], p.top_k[:nb], p.top_p[:nb], p.min_p[:nb],
                        p.seed[:nb], p.request_id[:nb], p.step)
    oracle.threads(1)
    t1 = time.perf_counter()
    oracle.verify_sample(sub.logits, sub.dtype, sub.V, sub.B, sub.k_max, sub.cu_rows,
                         sub.draft_ids, ps)
    dt1 = time.perf_counter() - t1
    oracle.threads(cores)
    return {"value": round(rows / dt, 2), "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": "%d full batch(es) of the benchmark workload (%d rows each), fp64 C oracle "
                      "with OpenMP over rows" % (n, vb.R),
            "single_thread": {"value": round(r1 / dt1, 2), "unit": "rows/s",
                              "sample": "the first %d requests (%d rows) of one batch, one thread"
                                        % (nb, r1)},
            "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name (x86 and Arm /proc/cpuinfo layouts)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model Name", "Hardware", "CPU part"):
        m = re.search(r"^%s\s*:\s*(.+)$" % key, info, re.M)
        if m:
            return "%s (%s)" % (m.group(1).strip(), platform.machine())
    return platform.machine()


# ------------------------------------------------------ reference arm -----

def run_reference(args) -> None:
    """The CPU oracle timed on the host cores on this workload: each step is
    one packed row of the batch (cycling), sampled exactly as defined."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.threads(1)
    vb, p = make_inputs(W.data_seed(3))
    vals = W.bf16_bits_to_f32(vb.logits).astype(np.float64)
    owner = np.repeat(np.arange(B), K + 1)

    def step(i):
        r = i % R
        b = int(owner[r])
        oracle.sample_row(vals[r, :V], float(p.temperature[b]), int(p.top_k[b]), float(p.top_p[b]),
                          float(p.min_p[b]), int(p.seed[b]), int(p.request_id[b]), r - b * (K + 1),
                          p.step)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "rows/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_name(), "global_batch": B,
                                        "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": cores,
                         "kind": "oracle",
                         "sample": "one packed row of the benchmark batch per step (cycling)"},
        "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=4, help="rotating device copies of the inputs")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-entries", action="store_true", help="skip the other entry points")
    ap.add_argument("--entry-launches", type=int, default=50)
    ap.add_argument("--row-class", choices=sorted(ROW_CLASSES), default="mix",
                    help="every request's filters alike, for profiling (default: the benchmark's mix)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    global ROW_CLASS
    ROW_CLASS = args.row_class
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
