#!/usr/bin/env python3
"""Benchmark of the quantized-weight matmul hot path on GB300.

One step = one M=1 decode pass over every Q4_K/Q6_K GEMV workload:
  * Llama-3.2-1B-shaped Q4_K projections (2048->2048, 2048->512, 2048->8192,
    8192->2048),
  * the Q6_K lm_head 2048->128256,
  * a Qwen3-14B-shaped Q4_K_M layer (q, k, v[Q6_K], o, gate, up, down[Q6_K]),
each call going through the public C ABI (`qmm`: activation quantiser +
decode GEMV).  `value` is the step's weight bytes / device time (GB/s); the
447 MB of weights per step exceed the 129 MB L2, so every matrix is re-read
from HBM.  The same run also times:
  * every matrix alone over rotating copies (>= 4x L2) -> per-matrix GB/s,
  * the prefill GEMM at M=512 -> TOPS: Q4_K (Mistral-7B MLP up and down),
    Q6_K (the Qwen3-14B-shaped layer's v and down), Q8_0 (Mistral up shape),
  * the value side of attention over a q8_0 KV cache (qmm_t, Qwen3-14B
    shaped: 8 heads x 32768 positions x 128) -> GB/s,
  * the dominant kernel (the Q6_K lm_head GEMV) for the roofline object,
  * the end-to-end step with host buffers (x copied in, y copied out),
  * the CPU oracle on a bounded sample (cpu_baseline).

--impl reference times the CPU oracle (plain C, f64 accumulation) on the host
cores instead, on a bounded sample of the same workload.

Weights and activations are seeded synthetic data with the value
distributions of the workloads (synth.py); no model files are used.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def decode_workload():
    mats = []
    for cfg in (1, 2, 3):
        for idx, (name, qtype, K, N) in enumerate(synth.CONFIGS[cfg]["mats"]):
            mats.append(dict(cfg=cfg, idx=idx, name=f"cfg{cfg}:{name}", qtype=qtype, K=K, N=N,
                             bytes=synth.matrix_bytes(qtype, N, K)))
    return mats


# The decode step's launches: matrices that read the same activations in a
# real layer (q/k/v of attention, gate/up of the MLP) go in one qmm_group
# call; the others are single qmm calls.  Names index decode_workload().
STEP_CALLS = [("cfg1:q", "cfg1:kv"), ("cfg1:gate_up",), ("cfg1:down",), ("cfg2:lm_head",),
              ("cfg3:q", "cfg3:k", "cfg3:v"), ("cfg3:o",), ("cfg3:gate", "cfg3:up"), ("cfg3:down",)]
LAYER_CALLS = [c for c in STEP_CALLS if c[0].startswith("cfg3:")]


def make_calls(mats, calls):
    by = {m["name"]: m for m in mats}
    return [[by[n] for n in c] for c in calls]


def run_call(q, call, stream, W_of=lambda m: m["W"]):
    """One launch of the step: a group of matrices sharing x, or one matrix."""
    if len(call) == 1:
        m = call[0]
        q.qmm(m["qtype"], W_of(m), m["N"], m["K"], m["x"], y=m["y"], stream=stream)
    else:
        q.qmm_group([(m["qtype"], W_of(m), m["N"], m["y"]) for m in call], call[0]["K"], call[0]["x"],
                    stream=stream)


WORKLOAD_NAME = ("decode M=1: Llama-3.2-1B Q4_K projections + Q6_K lm_head 2048x128256 + "
                 "Qwen3-14B Q4_K_M layer (q,k,v,o,gate,up,down)")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d.get("hbm_gbs", 6800.0), bf16=d.get("bf16_tflops", 1900.0),
                    bf16_sust=d.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


TRAFFIC_SUMMARY = os.path.join("profiles", "gemv_q6k_lm_head_k2048_n128256.txt")
# the files whose code makes up the lm_head kernel (qmm_internal.h only
# declares host launchers)
TRAFFIC_SOURCES = ("mat_mul_gb300/csrc/gemv_sb.cuh", "mat_mul_gb300/csrc/qmm_device.cuh")


def sources_sha256(paths):
    """sha256 over the named source files, concatenated in the given order."""
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel's sources changed since the capture."""
    summ = os.path.join(ROOT, TRAFFIC_SUMMARY)
    if not os.path.exists(summ):
        return None
    vals = {}
    with open(summ) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != sources_sha256(TRAFFIC_SOURCES):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.all_rows = []
        self.window_open = False
        self.proc = None

    def start(self):
        """Start sampling and wait (up to 5 s) for the first sample."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
            return self
        t0 = time.time()
        while not self.all_rows and time.time() - t0 < 5:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.all_rows.append((time.time(), parts))
                if self.window_open:
                    self.rows.append(parts)

    def __enter__(self):
        self.window_open = True
        return self

    def stop(self):
        self.__exit__()

    def __exit__(self, *a):
        self.window_open = False
        if not self.rows and self.all_rows:
            # the timed window was shorter than one sampling period: keep the
            # sample closest to it
            self.rows.append(self.all_rows[-1][1])

    def close(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ---------------------------------------------------------------- oracle arm

def _oracle_pass(mats, frac, nthreads, reps=1):
    import oracle
    nbytes, secs = 0, 0.0
    for m in mats:
        rows = max(1, int(m["N"] * frac))
        W = synth.weights(m["qtype"], rows, m["K"], seed=m["cfg"] * 1000 + m["idx"])
        x = synth.config_activations(m["cfg"], 1, m["K"])
        for _ in range(reps):
            t0 = time.perf_counter()
            oracle.qmm(m["qtype"], W, rows, m["K"], x, nthreads=nthreads)
            secs += time.perf_counter() - t0
            nbytes += rows * synth.row_bytes(m["qtype"], m["K"])
    return nbytes, secs


def oracle_rate(mats, seconds, nthreads):
    """Time the CPU oracle on row samples of every matrix, the sample grown
    (then repeated, once it covers every row) until it takes about `seconds`;
    return (GB/s, description of the sample)."""
    import oracle
    oracle.lib()
    frac, reps = 1.0 / 8192, 1
    while True:
        nbytes, secs = _oracle_pass(mats, frac, nthreads, reps)
        if secs >= seconds or reps >= 256:
            break
        grow = 4.0 if secs < seconds / 8 else seconds / max(secs, 1e-6) * 1.05
        if frac < 1.0:
            frac = min(1.0, frac * grow)
        else:
            reps = min(256, max(reps + 1, int(reps * grow)))
    what = f"{frac:.4%} of the rows of every matrix" if frac < 1.0 else (
        f"every row of every matrix, {reps} pass{'es' if reps > 1 else ''}")
    return nbytes / secs / 1e9, f"{what}: {nbytes / 1e6:.1f} MB of weights in {secs:.1f} s, M=1"


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.lib()
    cores = len(os.sched_getaffinity(0))
    mats = decode_workload()
    total = sum(m["bytes"] for m in mats)
    # each step: the oracle over a fixed row sample of every matrix, sized so
    # that warm-up plus timed steps take about two minutes in all
    rate_gbs, _ = oracle_rate(mats, 1.0, cores)
    per_step_s = min(2.0, 120.0 / max(1, args.steps + args.warmup))
    frac = min(1.0, per_step_s * rate_gbs * 1e9 / total)
    samples = []
    for m in mats:
        rows = max(1, int(m["N"] * frac))
        W = synth.weights(m["qtype"], rows, m["K"], seed=m["cfg"] * 1000 + m["idx"])
        x = synth.config_activations(m["cfg"], 1, m["K"])
        samples.append((m, rows, W, x))
    step_bytes = sum(rows * synth.row_bytes(m["qtype"], m["K"]) for m, rows, _, _ in samples)

    def step():
        for m, rows, W, x in samples:
            oracle.qmm(m["qtype"], W, rows, m["K"], x, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = step_bytes / dt / 1e9
    sample = f"{frac:.4%} of the rows of every matrix per step ({step_bytes / 1e6:.2f} MB of weights)"
    line = {
        "impl": "reference", "metric": "Q4_K/Q6_K GEMV weight GB/s at M=1 (decode step)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "M": 1, "weight_bytes_per_full_step": total,
                   "l2": "inputs larger than L2 (sampled rows on CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------ the ranks of a job

def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the job is as slow as its slowest
    rank); the value itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_step, ms_per_step):
    """GB/s of the whole job: each of the world's replicas streams
    bytes_per_step every step (weak scaling)."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# --------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch

    import mat_mul_gb300 as q

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    q.load()
    peaks = load_peaks()
    stream = torch.cuda.Stream()

    mats = decode_workload()
    step_bytes = sum(m["bytes"] for m in mats)
    calls = make_calls(mats, STEP_CALLS)
    # every call's x is a slice of one device buffer and every y a slice of
    # another, so that the end-to-end step moves its inputs in one
    # host-to-device copy and its outputs in one device-to-host copy (a
    # group reads one x: its members' synthetic activations coincide)
    x_len = sum(call[0]["K"] for call in calls)
    y_len = sum(m["N"] for m in mats)
    x_host_all = torch.empty(x_len, dtype=torch.float32).pin_memory()
    y_host_all = torch.empty(y_len, dtype=torch.float32).pin_memory()
    x_dev_all = torch.empty(x_len, dtype=torch.float32, device=dev)
    y_dev_all = torch.empty(y_len, dtype=torch.float32, device=dev)
    xo = yo = 0
    for call in calls:
        xv = torch.from_numpy(synth.config_activations(call[0]["cfg"], 1, call[0]["K"])).reshape(-1)
        for m in call[1:]:
            assert torch.equal(torch.from_numpy(synth.config_activations(m["cfg"], 1, m["K"])).reshape(-1), xv)
        x_host_all[xo:xo + xv.numel()] = xv
        for m in call:
            m["x"] = x_dev_all[xo:xo + xv.numel()].view(1, -1)
        xo += xv.numel()
    x_dev_all.copy_(x_host_all)
    for m in mats:
        m["W"] = torch.from_numpy(synth.config_weights(m["cfg"], m["idx"])).to(dev)
        m["y"] = y_dev_all[yo:yo + m["N"]].view(1, -1)
        yo += m["N"]

    def step():
        for call in calls:
            run_call(q, call, stream)

    def step_e2e():
        x_dev_all.copy_(x_host_all, non_blocking=True)
        for call in calls:
            run_call(q, call, stream)
        y_host_all.copy_(y_dev_all, non_blocking=True)

    def capture(fn):
        with torch.cuda.stream(stream):
            fn()  # allocates the workspace of this stream outside the capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed(graph, steps, warmup, sampler=None):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                graph.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ctx = sampler if sampler else _Null()
        with ctx:
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(steps):
                    graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / steps, dist, dev)

    # kernels of this library launched per decode step, counted by the library
    n0 = q.qmm_launch_count()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    launches_per_step = q.qmm_launch_count() - n0

    # ---- headline: the decode step, weights resident
    g_step = capture(step)
    sampler = ClockSampler(dev.index).start()
    ms = timed(g_step, args.steps, args.warmup, sampler)
    clocks = sampler.summary()
    sampler.close()
    value = job_throughput(world, step_bytes, ms)
    status = q.qmm_device_status(stream)
    assert status == 0, f"device status {status}"

    # ---- end to end: x copied in and y copied out every call
    g_e2e = capture(step_e2e)
    ms_e2e = timed(g_e2e, args.steps, args.warmup)
    h2d = x_host_all.numel() * 4
    d2h = y_host_all.numel() * 4
    e2e_value = job_throughput(world, step_bytes, ms_e2e)
    del g_e2e, g_step

    detail = []
    groups = layer = layer_m = gate_up = kq = kv_line = None
    roof = None
    gemm = None
    cpu = None
    if rank == 0 and not args.quick:
        # ---- every matrix alone, over rotating copies >= 4x L2
        for m in mats:
            ncopy = max(2, -(-4 * L2_BYTES // m["bytes"]))
            ncopy = min(ncopy, 2048)
            copies = [m["W"]] + [m["W"].clone() for _ in range(ncopy - 1)]
            calls = max(ncopy, 64)

            def one(copies=copies, m=m, calls=calls):
                for i in range(calls):
                    q.qmm(m["qtype"], copies[i % len(copies)], m["N"], m["K"], m["x"], y=m["y"],
                          stream=stream)

            g = capture(one)
            reps = max(3, min(20, int(2e9 / (calls * m["bytes"]) + 1)))
            t_ms = timed(g, reps, 2) / calls
            gbs = m["bytes"] / (t_ms * 1e-3) / 1e9
            detail.append({"matrix": m["name"], "type": synth.TYPE_NAMES[m["qtype"]], "K": m["K"],
                           "N": m["N"], "MB": round(m["bytes"] / 1e6, 3), "us": round(t_ms * 1e3, 2),
                           "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm"], 4)})
            if m["name"] == "cfg2:lm_head":
                traffic = load_traffic()
                roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm"],
                        "unit": "GB/s", "frac": round(gbs / peaks["hbm"], 4),
                        "traffic": traffic, "kernel": "gemv_sb_kernel<Q6_K,1> (qmm, lm_head 2048x128256)",
                        "bytes_per_launch": m["bytes"], "us_per_launch": round(t_ms * 1e3, 2),
                        "peak_source": peaks["source"] + " hbm_gbs (copy, burst)"}
            del g, copies
            torch.cuda.empty_cache()

        # ---- the grouped launches alone, and the Qwen3-14B layer as the step
        # runs it (four launches), over rotating copies >= 4x L2
        def rotating(call_list):
            nbytes = sum(m["bytes"] for c in call_list for m in c)
            ncopy = min(64, max(2, -(-4 * L2_BYTES // nbytes)))
            copies = {m["name"]: [m["W"]] + [m["W"].clone() for _ in range(ncopy - 1)]
                      for c in call_list for m in c}
            inner = max(ncopy, 8)

            def fn():
                for i in range(inner):
                    for c in call_list:
                        run_call(q, c, stream, W_of=lambda m, i=i: copies[m["name"]][i % ncopy])

            # kernel launches of one pass, counted by the library (a Q4_K call
            # on the tensor-core decode path is two: the quantiser, the GEMV)
            before = q.qmm_launch_count()
            for c in call_list:
                run_call(q, c, stream)
            launches = q.qmm_launch_count() - before
            g = capture(fn)
            t_ms = timed(g, 5, 2) / inner
            del g, copies
            torch.cuda.empty_cache()
            gbs = nbytes / (t_ms * 1e-3) / 1e9
            return {"matrices": "+".join(m["name"] for c in call_list for m in c), "launches": launches,
                    "MB": round(nbytes / 1e6, 3), "us": round(t_ms * 1e3, 2), "GB/s": round(gbs, 1),
                    "frac_hbm": round(gbs / peaks["hbm"], 4)}

        groups = [rotating([c]) for c in make_calls(mats, STEP_CALLS) if len(c) > 1]

        # ---- the gated MLP product h = silu(gate x) * (up x) of the
        # Qwen3-14B layer in one launch (qmm_gate_up), over rotating copies
        by_name = {m["name"]: m for m in mats}
        mg, mu = by_name["cfg3:gate"], by_name["cfg3:up"]
        gu_bytes = mg["bytes"] + mu["bytes"]
        ncopy = min(64, max(2, -(-4 * L2_BYTES // gu_bytes)))
        cg = [mg["W"]] + [mg["W"].clone() for _ in range(ncopy - 1)]
        cu = [mu["W"]] + [mu["W"].clone() for _ in range(ncopy - 1)]
        h_gu = torch.empty((1, mg["N"]), dtype=torch.float32, device=dev)
        inner = max(ncopy, 8)

        def gu_call():
            for i in range(inner):
                q.qmm_gate_up(mg["qtype"], cg[i % ncopy], mu["qtype"], cu[i % ncopy], mg["N"], mg["K"], mg["x"],
                              h=h_gu, stream=stream)

        before = q.qmm_launch_count()
        q.qmm_gate_up(mg["qtype"], mg["W"], mu["qtype"], mu["W"], mg["N"], mg["K"], mg["x"], h=h_gu, stream=stream)
        gu_launches = q.qmm_launch_count() - before
        g = capture(gu_call)
        t_ms = timed(g, 5, 2) / inner
        del g, cg, cu
        torch.cuda.empty_cache()
        gbs = gu_bytes / (t_ms * 1e-3) / 1e9
        gate_up = {"what": "qmm_gate_up: h = silu(gate x) * (up x), Qwen3-14B 5120->17408 Q4_K pair, M=1",
                   "launches": gu_launches, "MB": round(gu_bytes / 1e6, 3), "us": round(t_ms * 1e3, 2),
                   "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm"], 4)}
        layer = rotating(make_calls(mats, LAYER_CALLS))
        layer["M"] = 1

        # ---- the same layer with M = 2, 4, 8 activation rows (the decode of a
        # few sequences at once): weight bytes per launch are unchanged
        layer_m = []
        saved = {m["name"]: (m["x"], m["y"]) for m in mats}
        for Mb in (2, 4, 8):
            for c in make_calls(mats, LAYER_CALLS):
                xb = torch.from_numpy(synth.config_activations(c[0]["cfg"], Mb, c[0]["K"])).to(dev)
                for m in c:
                    m["x"] = xb
                    m["y"] = torch.empty((Mb, m["N"]), dtype=torch.float32, device=dev)
            r = rotating(make_calls(mats, LAYER_CALLS))
            r["M"] = Mb
            layer_m.append(r)
        for m in mats:
            m["x"], m["y"] = saved[m["name"]]

        # ---- prefill GEMM, M=512
        gemm = []
        # the Q4_K Mistral-7B MLP, the Q6_K matrices of the Qwen3-14B-shaped
        # layer, and Q8_0 weights in the Mistral up shape (cfg 0's Q8_0
        # value distribution), all at M=512
        prefill_cases = [(f"mistral_{name}", qtype, K, N, synth.config_weights(4, idx),
                          synth.config_activations(4, 512, K))
                         for idx, (name, qtype, K, N) in enumerate(synth.CONFIGS[4]["mats"])]
        prefill_cases += [(f"qwen3_14b_{name}", qtype, K, N, synth.config_weights(3, idx),
                           synth.config_activations(4, 512, K))
                          for idx, (name, qtype, K, N) in enumerate(synth.CONFIGS[3]["mats"]) if qtype == synth.Q6_K]
        prefill_cases.append(("q8_0_mistral_up", synth.Q8_0, 4096, 14336,
                              synth.weights(synth.Q8_0, 14336, 4096, seed=4100),
                              synth.config_activations(4, 512, 4096)))
        for name, qtype, K, N, w_np, x_np in prefill_cases:
            # rotating weight copies (>= 4x L2), so every call reads its
            # weights from HBM as a model's layers would
            W = torch.from_numpy(w_np).to(dev)
            ncopy = max(2, -(-4 * L2_BYTES // W.numel()))
            copies = [W] + [W.clone() for _ in range(ncopy - 1)]
            x = torch.from_numpy(x_np).to(dev)
            y = torch.empty((512, N), dtype=torch.float32, device=dev)
            inner = max(ncopy, 8)

            def gcall(copies=copies, x=x, y=y, qtype=qtype, K=K, N=N, inner=inner):
                for i in range(inner):
                    q.qmm(qtype, copies[i % len(copies)], N, K, x, y=y, stream=stream)

            g = capture(gcall)
            t_ms = timed(g, 3, 1) / inner
            del copies
            tops = 2 * 512 * N * K / (t_ms * 1e-3) / 1e12
            gemm.append({"matrix": name, "type": ["Q8_0", "Q4_K", "Q6_K"][qtype], "M": 512, "K": K, "N": N,
                         "us": round(t_ms * 1e3, 1), "TOPS": round(tops, 1)})
            del g
        int8_peak = None
        try:
            a = torch.randint(-127, 127, (8192, 8192), dtype=torch.int8, device=dev)
            b = torch.randint(-127, 127, (8192, 8192), dtype=torch.int8, device=dev).t()
            for _ in range(3):
                torch._int_mm(a, b)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(10):
                torch._int_mm(a, b)
            e1.record()
            torch.cuda.synchronize()
            int8_peak = 2 * 8192 ** 3 / (e0.elapsed_time(e1) / 10 * 1e-3) / 1e12
            del a, b
        except Exception as exc:  # noqa: BLE001
            int8_peak = None
            print(f"int8 peak probe unavailable: {exc}", file=sys.stderr)
        for gm in gemm:
            gm["frac_f16_peak"] = round(gm["TOPS"] / peaks["bf16"], 4)
            gm["frac_int8_peak"] = round(gm["TOPS"] / int8_peak, 4) if int8_peak else None
        gemm = {"kernels": gemm, "int8_peak_tops_torch_int_mm": round(int8_peak, 1) if int8_peak else None,
                "f16_peak_tflops": peaks["bf16"]}

        # ---- the other K-quants: decode at M=1 (Qwen3-14B gate shape,
        # rotating copies) and prefill at M=512 (Mistral-7B up shape)
        kq = []
        for qtype in (synth.Q5_K, synth.Q3_K, synth.Q2_K):
            K, N = 5120, 17408
            W = torch.from_numpy(synth.weights(qtype, N, K, seed=5000 + qtype)).to(dev)
            nbytes = W.numel()
            ncopy = max(2, -(-4 * L2_BYTES // nbytes))
            copies = [W] + [W.clone() for _ in range(ncopy - 1)]
            xk = torch.from_numpy(synth.config_activations(3, 1, K)).to(dev)
            yk = torch.empty((1, N), dtype=torch.float32, device=dev)
            inner = max(ncopy, 16)

            def kcall(copies=copies, xk=xk, yk=yk, qtype=qtype, K=K, N=N, inner=inner):
                for i in range(inner):
                    q.qmm(qtype, copies[i % len(copies)], N, K, xk, y=yk, stream=stream)

            g = capture(kcall)
            t_dec = timed(g, 5, 2) / inner
            del g, copies
            K, N = 4096, 14336
            W = torch.from_numpy(synth.weights(qtype, N, K, seed=6000 + qtype)).to(dev)
            ncopy = max(2, -(-4 * L2_BYTES // W.numel()))
            copies = [W] + [W.clone() for _ in range(ncopy - 1)]
            xp = torch.from_numpy(synth.config_activations(4, 512, K)).to(dev)
            yp = torch.empty((512, N), dtype=torch.float32, device=dev)
            inner = max(ncopy, 8)

            def pcall(copies=copies, xp=xp, yp=yp, qtype=qtype, K=K, N=N, inner=inner):
                for i in range(inner):
                    q.qmm(qtype, copies[i % len(copies)], N, K, xp, y=yp, stream=stream)

            g = capture(pcall)
            t_pre = timed(g, 3, 1) / inner
            del g, copies
            torch.cuda.empty_cache()
            dgbs = nbytes / (t_dec * 1e-3) / 1e9
            tops = 2 * 512 * N * K / (t_pre * 1e-3) / 1e12
            kq.append({"type": synth.TYPE_NAMES[qtype],
                       "decode_M1": {"K": 5120, "N": 17408, "MB": round(nbytes / 1e6, 3), "us": round(t_dec * 1e3, 2),
                                     "GB/s": round(dgbs, 1), "frac_hbm": round(dgbs / peaks["hbm"], 4)},
                       "prefill_M512": {"K": K, "N": N, "us": round(t_pre * 1e3, 1), "TOPS": round(tops, 1),
                                        "kernel": "tcgen05 (fp16 operands)"}})

        # ---- the value side of attention over a q8_0 KV cache (qmm_t):
        # Qwen3-14B-shaped, 8 cache heads x 32768 positions x head_dim 128,
        # 5 probability rows per head; rotating copies of the cache (> L2)
        kv = synth.KV_CACHE
        kvH, kvN, kvK, kvM = kv["H"], kv["N"], kv["K"], kv["M"]
        Wkv = torch.from_numpy(synth.kv_cache(kvH, kvN, kvK, seed=9)).to(dev)
        xkv = torch.from_numpy(synth.attention_probs(kvH, kvM, kvN, seed=9)).to(dev)
        ykv = torch.empty((kvH, kvM, kvK), dtype=torch.float32, device=dev)
        kv_bytes = Wkv.numel()
        kv_copies = [Wkv] + [Wkv.clone() for _ in range(max(1, -(-4 * L2_BYTES // kv_bytes)) - 1)]
        kv_inner = max(len(kv_copies), 8)

        def kvcall():
            for i in range(kv_inner):
                q.qmm_t(synth.Q8_0, kv_copies[i % len(kv_copies)], kvH, kvN, kvK, xkv, y=ykv, stream=stream)

        g = capture(kvcall)
        t_ms = timed(g, 5, 2) / kv_inner
        del g, kv_copies
        torch.cuda.empty_cache()
        kv_gbs = kv_bytes / (t_ms * 1e-3) / 1e9
        kv_line = {"what": "qmm_t, " + kv["name"], "H": kvH, "N": kvN, "K": kvK, "M": kvM,
                   "MB": round(kv_bytes / 1e6, 3), "us": round(t_ms * 1e3, 2), "GB/s": round(kv_gbs, 1),
                   "frac_hbm": round(kv_gbs / peaks["hbm"], 4)}

        # ---- CPU oracle on a bounded sample
        cores = len(os.sched_getaffinity(0))
        rate, sample = oracle_rate(mats, args.cpu_seconds, cores)
        cpu = {"value": round(rate, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {
            "metric": "Q4_K/Q6_K GEMV weight GB/s at M=1 (decode step)",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "M": 1, "matrices": len(mats),
                       "launches_per_step": launches_per_step,
                       "weight_bytes_per_step": step_bytes, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (447 MB of weights per step)",
                       "frac_hbm_step": round(value / world / peaks["hbm"], 4)},
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4),
                    "note": "weights resident (model state); every step: all x in (one pinned H2D copy), "
                            "all y out (one D2H copy)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks, "per_matrix": detail, "groups": groups, "gate_up_fused": gate_up,
            "qwen3_14b_layer": layer,
            "qwen3_14b_layer_M": layer_m,
            "prefill_gemm": gemm, "other_k_quants": kq,
            "kv_value_cache": kv_line,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def run_ncu_case(name, calls=3):
    """A few eager qmm calls of one workload matrix (for ncu captures: graphs
    with programmatic dependent launch cannot be replayed node by node)."""
    import torch

    import mat_mul_gb300 as q
    torch.cuda.set_device(0)
    q.load()
    if name == "kv":  # the value side of attention over the q8_0 KV cache (qmm_t)
        kv = synth.KV_CACHE
        W = torch.from_numpy(synth.kv_cache(kv["H"], kv["N"], kv["K"], seed=9)).cuda()
        x = torch.from_numpy(synth.attention_probs(kv["H"], kv["M"], kv["N"], seed=9)).cuda()
        for _ in range(calls):
            y = q.qmm_t(synth.Q8_0, W, kv["H"], kv["N"], kv["K"], x)
        torch.cuda.synchronize()
        assert q.qmm_device_status() == 0
        print(name, "ok", float(y.abs().sum()))
        return 0
    mats = {m["name"]: m for m in decode_workload()}
    for idx, (nm, qtype, K, N) in enumerate(synth.CONFIGS[4]["mats"]):
        mats[f"cfg4:{nm}"] = dict(cfg=4, idx=idx, name=f"cfg4:{nm}", qtype=qtype, K=K, N=N, M=512)
    name, _, rows = name.partition("@")  # "cfg3:gate@4": the matrix with M = 4 activation rows
    m = mats[name]
    W = torch.from_numpy(synth.config_weights(m["cfg"], m["idx"])).cuda()
    x = torch.from_numpy(synth.config_activations(m["cfg"], int(rows) if rows else m.get("M", 1), m["K"])).cuda()
    for _ in range(calls):
        y = q.qmm(m["qtype"], W, m["N"], m["K"], x)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    print(name, "ok", float(y.abs().sum()))
    return 0


def run_ncu_step(steps):
    """`steps` eager decode steps (the headline workload's calls in order, no
    graphs), for an ncu launch list with one entry per kernel launch."""
    import torch

    import mat_mul_gb300 as q
    torch.cuda.set_device(0)
    q.load()
    mats = decode_workload()
    for m in mats:
        m["W"] = torch.from_numpy(synth.config_weights(m["cfg"], m["idx"])).cuda()
        m["x"] = torch.from_numpy(synth.config_activations(m["cfg"], 1, m["K"])).cuda()
        m["y"] = torch.empty((1, m["N"]), dtype=torch.float32, device="cuda")
    calls = make_calls(mats, STEP_CALLS)
    for call in calls:
        for m in call[1:]:
            m["x"] = call[0]["x"]
    stream = torch.cuda.current_stream()
    for _ in range(steps):
        for call in calls:
            run_call(q, call, stream)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    print("decode steps ok", steps, len(calls), "launches per step")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=25000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--quick", action="store_true", help="headline and e2e only")
    ap.add_argument("--ncu-case", default=None,
                    help="run three eager calls of one matrix (e.g. cfg2:lm_head, cfg3:gate@4 for M = 4; kv for the "
                         "q8_0 value cache) and exit")
    ap.add_argument("--ncu-step", type=int, default=0,
                    help="run this many eager decode steps (for an ncu launch list) and exit")
    args = ap.parse_args()
    if args.ncu_step:
        return run_ncu_step(args.ncu_step)
    if args.ncu_case:
        return run_ncu_case(args.ncu_case)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
