"""Benchmark of the block-quantized weight x activation product on GB300.

Default workload: one decode step of SmolLM2-360M's Q4_0 linears (32 layers x
q/k/v/o/gate/up/down, M=1, a fresh seeded x per linear), i.e. 224 GEMVs and
179.1 MB of algorithmic traffic per step.  A step runs every linear once from
weights already resident in HBM; steps alternate between weight copies whose
total exceeds twice the L2, so every step streams its weights from HBM.

Prints one JSON line (rank 0).  At one GPU the line also carries the same
decode step with each layer's dependencies kept (per layer [q,k,v] -> o ->
[gate,up] -> down, 128 calls) and a `per_config` list timing every other
workload one product at a time (the 960x960 GEMV, TinyLlama Q8_0 / INT8-B64,
the Qwen2.5-3B FFN at M = 1..256, the Q6_K lm_head).  `--impl reference`
times the fp64 CPU oracle on the host cores instead.  `--sweep` prints the
per-workload timings to stderr as well.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_quantized_weight_dot_gb300 import synthetic as syn  # noqa: E402

METRIC = ("Q4_0 GEMV achieved HBM GB/s (% of GB300 peak) and decode-step linears/s, M=1")
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
# a GPU sleep of about 1 ms (at ~2 GHz) ahead of each timed region
HEAD_START_CYCLES = 2_000_000


# ---------------------------------------------------------------- helpers ---

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device=None):
    """Element-wise MAX of per-rank timings over the initialised process group
    (the job's step time is its slowest rank's); the values unchanged on one
    rank or without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(bytes_per_step_per_rank, ms_per_step, world):
    """Whole-job throughput of `world` replicas that each process one step of
    `bytes_per_step_per_rank` in `ms_per_step` (weak scaling)."""
    return bytes_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def measured_bf16():
    """Dense bf16 TFLOP/s measured on this machine (burst: a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return BF16_FALLBACK_TFLOPS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_weight_dot_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag):
    """dram read+write bytes per launch recorded by an ncu capture under
    profiles/, or None when absent or taken on different kernel sources."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    want = kernel_source_hash()
    for f in sorted(os.listdir(prof)):
        if not f.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(prof, f)).read()
        m = re.search(r"traffic_bytes_per_launch\[%s\]:\s*([0-9.eE+]+)\s+source_hash:\s*(\w+)"
                      % re.escape(kernel_tag), text)
        if m and m.group(2) == want:
            return float(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        sel = [r for (t, r) in self.rows if t0 - 0.15 <= t <= t1 + 0.15]
        note = "in timed region"
        if not sel and self.rows:
            # region shorter than the sampling period: nearest samples
            sel = [r for (t, r) in sorted(self.rows, key=lambda tr: abs(tr[0] - (t0 + t1) / 2))[:3]]
            note = "nearest samples (timed region shorter than the 100 ms sampling period)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        sm = [float(r[2]) for r in sel if len(r) > 9 and r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in sel if len(r) > 9 and r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel if len(r) > 9 for i in range(4)
                          if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(sel), "note": note}


# -------------------------------------------------------------- workloads ---

def workload_by_name(name):
    table = {
        "decode_stack": syn.smollm2_360m_decode_stack,
        "gemv_960": syn.q4_0_gemv_960,
        "tinyllama_q8_0": lambda: syn.tinyllama_gemv(syn.Q8_0),
        "tinyllama_i8_b64": lambda: syn.tinyllama_gemv(syn.I8_B64),
        "lm_head_q6_k": syn.qwen25_3b_lm_head,
    }
    for M in syn.QWEN25_3B_FFN_BATCHES:
        table["qwen_ffn_M%d" % M] = (lambda M=M: syn.qwen25_3b_ffn(M))
    return table[name]()


class DeviceWorkload:
    """Packed weights (several copies, > 2x L2 in total), x and y resident in HBM."""

    def __init__(self, wl, device, l2_bytes, copies=None):
        import torch
        from block_quantized_weight_dot_gb300 import lean
        self.wl, self.lean, self.torch = wl, lean, torch
        self.lins = list(wl.linears)
        packed, xs = [], []
        for lin in self.lins:
            W, x = lin.make()
            packed.append(lean.lean_pack(lin.fmt, W, lin.N, lin.K))
            xs.append(x)
        self.canon_x = xs
        per_copy = sum(p.size for p in packed)
        self.packed_sizes = packed
        self.copies = copies or max(2, int(np.ceil(2.2 * l2_bytes / per_copy)))
        self.W = [[torch.from_numpy(p).to(device) for p in packed] for _ in range(self.copies)]
        # one contiguous x buffer and one y buffer (host mirrors for e2e)
        self.x_off, self.y_off = [], []
        xo = yo = 0
        for lin in self.lins:
            self.x_off.append(xo)
            self.y_off.append(yo)
            xo += lin.M * lin.K + (-lin.M * lin.K) % 4   # keep every x 16-byte aligned
            yo += lin.M * lin.N + (-lin.M * lin.N) % 4
        x_host = np.zeros(xo, np.float32)
        for lin, off, x in zip(self.lins, self.x_off, xs):
            x_host[off:off + lin.M * lin.K] = x.reshape(-1)
        self.x_host = torch.from_numpy(x_host).pin_memory()
        self.y_host = torch.empty(yo, dtype=torch.float32).pin_memory()
        self.x = self.x_host.to(device)
        self.y = torch.empty(yo, dtype=torch.float32, device=device)
        self.launches_per_step = None
        self.flags = lean.LEAN_FLAG_EARLY_WEIGHTS
        # one workspace, zeroed once: consecutive calls on the stream share it
        fmt0 = self.lins[0].fmt
        self.batch = None
        self.batch_host = None
        self.planes = False
        if (len(self.lins) > 1 and len(self.lins) <= lean.LEAN_MAX_BATCH
                and all(l.M == 1 and l.fmt == fmt0 for l in self.lins)):
            # with a workspace, integer formats streaming >= 32 MiB of weights
            # get a first kernel that writes x as integer planes
            self.planes = fmt0 != syn.Q6_K and sum(p.nbytes for p in packed) >= 32 << 20

            def problems(c, x_base, y_base):
                return lean.make_problems([(self.W[c][i], x_base + 4 * self.x_off[i],
                                            y_base + 4 * self.y_off[i], l.N, l.K)
                                           for i, l in enumerate(self.lins)])
            self.batch = [problems(c, self.x.data_ptr(), self.y.data_ptr())
                          for c in range(self.copies)]
            if self.planes:
                # the plane path reads x and writes y with plain loads and
                # stores, so the same call can take the pinned host buffers
                # themselves (zero-copy over the host link)
                self.batch_host = [problems(c, self.x_host.data_ptr(), self.y_host.data_ptr())
                                   for c in range(self.copies)]
            self.ws_bytes = lean.lean_batch_workspace_bytes(fmt0, self.batch[0])
        else:
            self.ws_bytes = max(lean.lean_qmatmul_workspace_bytes(l.fmt, l.N, l.K, l.M)
                                for l in self.lins)
        self.ws = torch.zeros(max(256, self.ws_bytes), dtype=torch.uint8, device=device)

    def run_step(self, copy, stream, host=False):
        """One pass over every linear: a single batched launch when all linears
        are M = 1 products of one format, otherwise one call per linear.
        host: the batch whose x and y are the pinned host buffers."""
        lean = self.lean
        if self.batch is not None:
            # host buffers only ever go down the plane path (asked for explicitly)
            flags = self.flags | (lean.LEAN_FLAG_X_PLANES if host else 0)
            lean.lean_qmatmul_batch(self.lins[0].fmt,
                                    (self.batch_host if host else self.batch)[copy],
                                    flags, self.ws, self.ws_bytes, stream)
            self.launches_per_step = 2 if self.planes else 1
            return
        n = 0
        for i, lin in enumerate(self.lins):
            x = self.x.data_ptr() + 4 * self.x_off[i]
            y = self.y.data_ptr() + 4 * self.y_off[i]
            lean.lean_qmatmul_ws(lin.fmt, self.W[copy][i], x, y, lin.N, lin.K, lin.M,
                                 self.flags, self.ws, self.ws_bytes, stream)
            if lin.M == 1:
                planes = lin.fmt != syn.Q6_K and lean.lean_packed_bytes(lin.fmt, lin.N, lin.K) >= 32 << 20
                n += 2 if planes else 1
            elif lin.M < lean.lean_tensor_core_min_m(lin.fmt):
                n += 1                        # CUDA-core kernel
            else:
                n += 2                        # x split + tensor-core product
        self.launches_per_step = n

    def capture(self, stream, host=False):
        torch = self.torch
        graphs = []
        for c in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    self.run_step(c, stream, host)
            graphs.append(g)
        return graphs


# ----------------------------------------------------------------- GPU arm ---

def time_gpu(args, wl):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    dw = DeviceWorkload(wl, device, l2)
    stream = torch.cuda.Stream(device)
    # warm the library (plans, attributes) outside capture
    with torch.cuda.stream(stream):
        dw.run_step(0, stream)
    stream.synchronize()
    graphs = dw.capture(stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    # correctness spot check of the first linear against the oracle (rank 0)
    spot = None
    if rank == 0:
        import oracle
        lin = dw.lins[0]
        graphs[0].replay()
        torch.cuda.synchronize()
        W, x = lin.make()
        y_ref, bound = oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K)
        y = dw.y[dw.y_off[0]:dw.y_off[0] + lin.M * lin.N].cpu().numpy().reshape(lin.M, lin.N)
        spot = bool(np.all(np.abs(y - y_ref) <= 1e-4 * bound + 1e-6))

    for s in range(args.warmup):
        graphs[s % dw.copies].replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        # keep the GPU busy while the host enqueues the timed steps, so that
        # host launch latency does not fall inside the timed region
        torch.cuda._sleep(HEAD_START_CYCLES)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for s in range(args.steps):
            graphs[s % dw.copies].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    # end to end: every step takes x from pinned host memory and leaves y in
    # pinned host memory.  On the plane path the call itself is given the host
    # buffers (the kernels read x and write y across the host link); otherwise
    # x is copied in and y out around the call.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e_steps = max(3, min(args.steps, 200))
    zero_copy = dw.batch_host is not None
    if zero_copy:
        hgraphs = dw.capture(stream, host=True)

    def e2e_step(s):
        if zero_copy:
            hgraphs[s % dw.copies].replay()
        else:
            dw.x.copy_(dw.x_host, non_blocking=True)
            graphs[s % dw.copies].replay()
            dw.y_host.copy_(dw.y, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(2):
            e2e_step(s)
    torch.cuda.synchronize()
    barrier()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HEAD_START_CYCLES)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for s in range(e_steps):
            e2e_step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    e2e_same = None
    if zero_copy:
        # the host-buffer call gives bit for bit what the device-buffer call gives
        with torch.cuda.stream(stream):
            graphs[0].replay()
        torch.cuda.synchronize()
        e2e_same = bool(np.array_equal(dw.y_host.numpy(), dw.y.cpu().numpy()))

    if ws > 1:
        import torch.distributed as dist
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], device)
        dist.destroy_process_group()
    kernel = ("qmm_stream_kernel<%s,%s> (TMA ring, %s)"
              % (syn.FORMAT_NAMES[dw.lins[0].fmt], "batch" if dw.batch is not None else "1",
                 "one launch per step" if dw.batch is not None else "one launch per linear"))
    if dw.batch is not None and dw.launches_per_step == 2:
        kernel = "xprep_kernel (x -> int8 planes) + " + kernel.replace(
            "TMA ring", "TMA ring, dp4a")
    return {"ms": ms, "e2e_ms": e2e_ms, "clocks": clocks, "launches": dw.launches_per_step,
            "kernel": kernel,
            "copies": dw.copies, "spot_ok": spot, "h2d": dw.x_host.numel() * 4,
            "d2h": dw.y_host.numel() * 4, "l2": l2, "e2e_zero_copy": zero_copy,
            "planes": dw.planes,
            "e2e_same": e2e_same}


# ----------------------------------------------------------------- CPU arm ---

def oracle_inputs(wl):
    return [(lin, lin.make()) for lin in wl.linears]


def time_oracle(inputs, n_per_step, budget_s, start=0):
    """The oracle as it stands, all host cores, on a bounded sample of the step:
    whole linears in workload order (from `start`, wrapping) until the time
    budget is spent (at least one)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    done_bytes, elapsed, n_lin = 0, 0.0, 0
    i = start
    while n_lin == 0 or elapsed < budget_s:
        lin, (W, x) = inputs[i % len(inputs)]
        t = time.perf_counter()
        oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K, threads=cores)
        elapsed += time.perf_counter() - t
        done_bytes += lin.algorithmic_bytes
        n_lin += 1
        i += 1
    return {"value": done_bytes / elapsed / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d of the workload's linears (%d per step), fp64 scalar C, %d threads, %.2f s"
                      % (n_lin, n_per_step, cores, elapsed),
            "seconds": elapsed, "linears": n_lin, "next": i}


# ------------------------------------------------------ host quantizer ---

def time_quantizer(reps=5):
    """lean_quantize (host threads, no GPU) on seeded fp32 weights at the
    Qwen2.5-3B FFN shapes: one JSON line per format on stdout."""
    from block_quantized_weight_dot_gb300 import lean
    cores = len(os.sched_getaffinity(0))
    rng = np.random.default_rng((0, 9))
    mats = [(rng.standard_normal((N, K)) * 0.02).astype(np.float32)
            for N, K in syn.QWEN25_3B_FFN_SHAPES]
    for fmt in (syn.Q4_0, syn.Q8_0, syn.I8_B64):
        lean.lean_quantize(fmt, mats[0], *mats[0].shape)  # first-touch of the output pages
        best = None
        for _ in range(reps):
            t = time.perf_counter()
            for w in mats:
                lean.lean_quantize(fmt, w, *w.shape)
            dt = time.perf_counter() - t
            best = dt if best is None else min(best, dt)
        params = sum(w.size for w in mats)
        print(json.dumps({"quantizer": syn.FORMAT_NAMES[fmt], "params": params,
                          "seconds": best, "params_per_s": params / best,
                          "input_gb_per_s": 4 * params / best / 1e9, "threads": cores,
                          "shapes": [list(w.shape) for w in mats],
                          "timing": "best of %d, host wall clock" % reps}), flush=True)


# -------------------------------------------------------------------- main ---

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lean", choices=["lean", "reference"])
    ap.add_argument("--workload", default="decode_stack")
    ap.add_argument("--sweep", action="store_true", help="also time every workload (stderr)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload timings and the layer-order decode step")
    ap.add_argument("--quantize", action="store_true",
                    help="time the host quantizer lean_quantize instead (no GPU)")
    args = ap.parse_args()
    if args.quantize:
        time_quantizer()
        return
    ws, rank, local = dist_env()
    wl = workload_by_name(args.workload)
    peak, peak_kind = measured_peaks()
    alg_bytes = wl.algorithmic_bytes
    n_lin = len(wl.linears)
    config = {"workload": wl.name, "linears_per_step": n_lin, "M": wl.linears[0].M,
              "algorithmic_bytes_per_step": alg_bytes, "weight_bytes_per_step": wl.weight_bytes,
              "inputs": "seeded synthetic, resident in HBM", "n_gpus": args.gpus}

    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.time()
        inputs = oracle_inputs(wl)
        per, nxt = [], 0
        for s in range(args.warmup + args.steps):
            r = time_oracle(inputs, n_lin, args.cpu_budget / max(1, args.steps), nxt)
            nxt = r["next"]
            if s >= args.warmup:
                per.append(r)
        gbs = float(np.mean([r["value"] for r in per]))
        ms_step = alg_bytes / (gbs * 1e9) * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": per[0]["cores"],
                                 "kind": "oracle", "sample": per[0]["sample"] + " per step"},
                "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "wall_s": time.time() - t0}
        print(json.dumps(line), flush=True)
        return

    r = time_gpu(args, wl)
    if rank != 0:
        return
    s_step = r["ms"] * 1e-3
    gbs = job_gbs(alg_bytes, r["ms"], ws)
    linears_per_s = n_lin / s_step * ws
    # the stream kernel moves every algorithmic byte of the step; its duration
    # is taken as the whole step (with the x-plane kernel, which only reads x,
    # when there is one), so `achieved` is a lower bound for it
    achieved = alg_bytes / s_step / 1e9
    tag = "qmm_stream:" + wl.name
    traffic = profiled_traffic(tag)
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = time_oracle(oracle_inputs(wl), n_lin, args.cpu_budget)
        for k in ("seconds", "linears", "next"):
            cpu.pop(k, None)
    config.update({"l2_defeat": "weights rotate over %d copies (%.0f MB > 2x L2 of %.0f MB)"
                   % (r["copies"], r["copies"] * wl.weight_bytes / 1e6, r["l2"] / 1e6),
                   "graph": "one CUDA graph per weight copy; a step = one graph replay",
                   "timing": "CUDA events on the launching stream; a ~1 ms GPU sleep precedes "
                             "the first event so the host has enqueued the timed steps",
                   "parallelism": "replicas" if ws > 1 else "single GPU"})
    per_config = dependent = x_int8 = None
    if ws == 1 and not args.no_per_config and args.workload == "decode_stack":
        import torch
        device = torch.device("cuda", local)
        stream = torch.cuda.Stream(device)
        dependent = time_dependent_step(device, r["l2"], stream, min(args.steps, 200),
                                        max(3, min(args.warmup, 20)))
        x_int8 = time_step_x_int8(device, r["l2"], stream, min(args.steps, 1000),
                                  max(3, min(args.warmup, 20)))
        per_config = time_per_config(device, r["l2"], stream)
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        # the x-plane path sums integer products in int32 (dp4a) and combines them in fp32
        "dtype": "int32+fp32" if r["planes"] else "fp32", "data": "synthetic",
        "config": config,
        "linears_per_s": linears_per_s,
        "frac_of_hbm_peak": gbs / ws / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": r["kernel"], "launches_per_step": r["launches"],
                     "duration": "whole step (all launches of the step), a lower bound for "
                                 "the stream kernel alone"},
        "cpu_baseline": cpu,
        "e2e": {"value": job_gbs(alg_bytes, r["e2e_ms"], ws), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": r["e2e_ms"],
                "transfer": ("the call takes the pinned host x and y buffers; its kernels read "
                             "x and write y across the host link (zero-copy)"
                             if r["e2e_zero_copy"] else
                             "cudaMemcpyAsync of x in and y out around the call, every step"),
                "matches_device_buffers": r["e2e_same"]},
        "gpu_launches": r["launches"] * args.steps,
        "clocks": r["clocks"],
        "spot_check_vs_oracle": r["spot_ok"],
        # the same decode step with each layer's dependencies kept (128 calls)
        "decode_step_layer_order": dependent,
        # the same step with x quantized to int8 (an approximate product)
        "decode_step_x_int8": x_int8,
        # every other workload, one product at a time (CUDA events, weights
        # rotating beyond L2); frac against the measured HBM peak
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)

    if args.sweep:
        sweep(args)


def linear_path(lin, tc_min):
    if lin.M == 1:
        return "m1"  # one-wave kernel when the rows fit the GPU at once, else streaming
    return "cuda_cores" if lin.M < tc_min else "mma"


def mma_issued_flops(lin):
    """bf16 MMA work the tensor-core kernels issue for one product, for every
    128-row weight tile and K padded to 64.  Up to 64 rows of x: the integer
    codes times x_hi and x_lo (two MMAs per 16-wide K step; Q6_K's codes in two
    parts, three), x rows padded to 16.  More rows (Q6_K and Q8_0: more than
    32): split weights times split x (three MMAs per step) in 256-row tiles of
    x, each padded to 16."""
    kp = -(-lin.K // 64) * 64
    tiles = -(-lin.N // 128)
    wide_from = 32 if lin.fmt in (syn.Q6_K, syn.Q8_0) else 64
    if lin.M <= wide_from:
        per_step = 3 if lin.fmt == syn.Q6_K else 2
        mp = -(-lin.M // 16) * 16
    else:
        per_step = 3
        mp = 0
        for m0 in range(0, lin.M, 256):
            mp += -(-min(256, lin.M - m0) // 16) * 16
    return per_step * 2 * 128 * tiles * mp * kp


def time_linear(lin, device, l2, stream, reps=20):
    """One product timed alone: a CUDA graph of one call per weight copy (the
    copies together larger than 2.2x L2, so every call streams from HBM)."""
    import torch
    peak, peak_kind = measured_peaks()
    bf16_peak, bf16_kind = measured_bf16()
    one = syn.Workload(lin.name, (lin,))
    dw = DeviceWorkload(one, device, l2)
    with torch.cuda.stream(stream):
        dw.run_step(0, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for c in range(dw.copies):
                dw.run_step(c, stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HEAD_START_CYCLES)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t = ev0.elapsed_time(ev1) / reps / dw.copies * 1e-3
    gbs = lin.algorithmic_bytes / t / 1e9
    path = linear_path(lin, dw.lean.lean_tensor_core_min_m(lin.fmt))
    r = {"linear": lin.name, "fmt": syn.FORMAT_NAMES[lin.fmt], "N": lin.N, "K": lin.K,
         "M": lin.M, "path": path, "us": round(t * 1e6, 3), "GB/s": round(gbs, 1),
         "frac": round(gbs / peak, 4), "useful_TFLOP/s": round(lin.flops / t / 1e12, 3),
         "launches": dw.launches_per_step, "copies": dw.copies}
    if path == "mma":
        issued = mma_issued_flops(lin) / t / 1e12
        r["tensor_pipe"] = {"issued_bf16_TFLOP/s": round(issued, 1),
                            "frac_of_bf16_peak": round(issued / bf16_peak, 4),
                            "peak": bf16_peak, "peak_source": bf16_kind,
                            "basis": "bf16 MMA work the kernels issue (per 16-wide K step 2 MMAs "
                                     "up to 64 rows of x (Q6_K 3; Q6_K and Q8_0 up to 32); 3 "
                                     "above; x rows padded to 16, K to 64) over CUDA-event time"}
    del dw, g
    torch.cuda.empty_cache()
    return r


PER_CONFIG = [("q4_0_gemv_960x960", "gemv_960"), ("tinyllama_1.1b_q8_0", "tinyllama_q8_0"),
              ("tinyllama_1.1b_i8_b64", "tinyllama_i8_b64")] + \
             [("qwen2.5_3b_ffn_q4_0_M%d" % M, "qwen_ffn_M%d" % M) for M in syn.QWEN25_3B_FFN_BATCHES] + \
             [("qwen2.5_3b_lm_head_q6_k", "lm_head_q6_k")]


def time_per_config(device, l2, stream):
    """Every other workload, one product at a time (each a list entry)."""
    out = []
    for cfg, name in PER_CONFIG:
        for lin in workload_by_name(name).linears:
            r = time_linear(lin, device, l2, stream)
            r["config"] = cfg
            out.append(r)
    return out


def time_dependent_step(device, l2, stream, steps, warmup):
    """The SmolLM2-360M decode step with the dependencies of a real layer kept:
    per layer [q, k, v] (one batch call) -> o -> gate / up with the SiLU(gate)
    * up epilogue (lean_qmatmul_swiglu) -> down, which reads that h; 128 calls
    per step in stream order with programmatic dependent launch, one CUDA
    graph per weight copy (the copies larger than 2x L2)."""
    import torch
    from block_quantized_weight_dot_gb300 import lean
    wl = syn.smollm2_360m_decode_stack()
    dw = DeviceWorkload(wl, device, l2)
    lins = dw.lins
    fmt = lins[0].fmt
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS
    layers = len(lins) // 7
    hbuf = torch.empty((layers, lins[4].N), dtype=torch.float32, device=device)
    xp = lambda i: dw.x.data_ptr() + 4 * dw.x_off[i]
    yp = lambda i: dw.y.data_ptr() + 4 * dw.y_off[i]

    def plan(c):
        out = []
        for l in range(layers):
            i = 7 * l
            qkv = lean.make_problems([(dw.W[c][i + j], xp(i + j), yp(i + j), lins[i + j].N,
                                       lins[i + j].K) for j in (0, 1, 2)])
            o = lean.make_problems([(dw.W[c][i + 3], xp(i + 3), yp(i + 3), lins[i + 3].N,
                                     lins[i + 3].K)])
            # gate (i + 4) and up (i + 5) read the gate linear's x; down reads h
            gu = (dw.W[c][i + 4], dw.W[c][i + 5], xp(i + 4), hbuf[l].data_ptr(), lins[i + 4].N,
                  lins[i + 4].K)
            down = lean.make_problems([(dw.W[c][i + 6], hbuf[l].data_ptr(), yp(i + 6),
                                        lins[i + 6].N, lins[i + 6].K)])
            out.append((qkv, o, gu, down))
        return out

    plans = [plan(c) for c in range(dw.copies)]
    wsb = max(max(lean.lean_batch_workspace_bytes(fmt, p) for p in (qkv, o, down))
              for qkv, o, _, down in plans[0])
    ws = torch.zeros(max(256, wsb), dtype=torch.uint8, device=device)

    def step(c):
        for qkv, o, gu, down in plans[c]:
            lean.lean_qmatmul_batch(fmt, qkv, flags, ws, wsb, stream)
            lean.lean_qmatmul_batch(fmt, o, flags, ws, wsb, stream)
            lean.lean_qmatmul_swiglu(fmt, *gu, flags, stream)
            lean.lean_qmatmul_batch(fmt, down, flags, ws, wsb, stream)

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    graphs = []
    for c in range(dw.copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                step(c)
        graphs.append(g)
    for s in range(warmup):
        graphs[s % dw.copies].replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HEAD_START_CYCLES)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for s in range(steps):
            graphs[s % dw.copies].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    peak, _ = measured_peaks()
    # bytes: the step's weights, each call's x once and y once (h counted as
    # the swiglu output and the down input)
    alg = wl.algorithmic_bytes - 4 * layers * lins[5].K
    gbs = alg / (ms * 1e-3) / 1e9
    calls_per_step = 4 * layers
    del dw, graphs
    torch.cuda.empty_cache()
    return {"workload": wl.name + "_layer_order",
            "order": "per layer: [q,k,v] batch -> o -> gate/up with the SiLU(gate)*up epilogue "
                     "(lean_qmatmul_swiglu) -> down reading that h (stream order, programmatic "
                     "dependent launch)",
            "calls_per_step": calls_per_step, "launches_per_step": calls_per_step,
            "ms_per_step": ms, "algorithmic_bytes_per_step": alg, "GB/s": gbs, "frac": gbs / peak,
            "linears_per_s": len(lins) / (ms * 1e-3), "steps": steps, "warmup": warmup}


def time_step_x_int8(device, l2, stream, steps, warmup):
    """The SmolLM2-360M decode step as one batch call with x quantized to int8
    per 32 elements (LEAN_FLAG_X_INT8, the "oxinfer" page's activation
    quantization): a different, approximate product, timed beside the exact
    one."""
    import torch
    from block_quantized_weight_dot_gb300 import lean
    wl = syn.smollm2_360m_decode_stack()
    dw = DeviceWorkload(wl, device, l2)
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS | lean.LEAN_FLAG_X_INT8

    def step(c):
        lean.lean_qmatmul_batch(dw.lins[0].fmt, dw.batch[c], flags, dw.ws, dw.ws_bytes, stream)

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    graphs = []
    for c in range(dw.copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                step(c)
        graphs.append(g)
    for s in range(warmup):
        graphs[s % dw.copies].replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HEAD_START_CYCLES)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for s in range(steps):
            graphs[s % dw.copies].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    peak, _ = measured_peaks()
    gbs = wl.algorithmic_bytes / (ms * 1e-3) / 1e9
    del dw, graphs
    torch.cuda.empty_cache()
    return {"workload": wl.name + "_x_int8", "ms_per_step": ms, "GB/s": gbs, "frac": gbs / peak,
            "launches_per_step": 2, "steps": steps, "warmup": warmup,
            "numerics": "x quantized to int8 per 32 elements (s = max|x|/127); not the exact "
                        "product"}


def sweep(args):
    """--sweep: every other workload, one line per product on stderr."""
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    stream = torch.cuda.Stream()
    for r in time_per_config(torch.device("cuda"), l2, stream):
        print(json.dumps(dict(sweep=r.pop("config"), **r)), file=sys.stderr, flush=True)


if __name__ == "__main__":
    main()
