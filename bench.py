"""Benchmark: verified draft positions per second on GB300.

One step = one spec_verify call (all of the standard path: temperature softmax of both rows, accept test,
chain length, residual or bonus draw) over one batch of the standard-verification workload at the Llama-3
vocabulary (B = 64 sequences, K = 5 draft positions, V = 128256, bf16 logits). Steps cycle through a ring of
distinct input batches whose total size is several times the 129 MB L2, so no step reads the previous
step's logits from L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Multi-GPU (torchrun): sequences are independent, so every rank verifies its own batches (weak scaling) with
no collective on the data path; rank 0 reports total positions / max-over-ranks time.

--impl reference times the fp64 CPU oracle (the only other implementation) on the host cores, on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "verified draft positions/sec"
UNIT = "positions/s"
DEFAULT_WORKLOAD = "sps_llama3_b64_k5"
L2_BYTES = 129 * 1024 * 1024


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes: read-only queries)
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
               0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle", 0x2: "applications_clocks_setting"}

    def __init__(self, index=0, period_s=0.002):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period = period_s
        self._stop = threading.Event()
        self._thr = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            self.nvml.nvmlInit_v2()
            self.dev = ctypes.c_void_p()
            self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev))
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError:
            self.nvml = None

    def _sample(self):
        clk = ctypes.c_uint()
        if self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk)) == 0:
            self.samples.append(clk.value)
        r = ctypes.c_ulonglong()
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        if fn(self.dev, ctypes.byref(r)) == 0:
            for bit, name in self.REASONS.items():
                if r.value & bit and name != "gpu_idle":
                    self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self.nvml:
            self._sample()
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()

    def stop(self):
        if self.nvml:
            self._stop.set()
            self._thr.join()
            self._sample()

    def summary(self):
        if not self.nvml:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ------------------------------------------------------------------------------------------------
# distributed plumbing
# ------------------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg, torch):
    if pg is not None:
        pg.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(pg, torch, v, device):
    if pg is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------------------
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one call (both kernels), from an ncu capture
# of this benchmark's own command (profiles/), keyed by a hash of the kernel sources it was taken with: when
# the sources change the recorded number no longer applies and the JSON line reports null.
RECORDED_TRAFFIC = {
    "12435f7b735a104d": {"sps_llama3_b64_k5": 214668800, "hedgespec_n7_b32_k5": 372430592 + 3307264 + 16286720},
}


def kernel_source_hash():
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "speculative_decoding_verification_target_gb300", "csrc", "*.cu*"))):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kind_of(w):
    """Which entry point a workload exercises: counterfactual gamma (N > 1, fused verify of the selected
    drafter), Cactus (workloads with a delta list; the largest delta is timed) or standard verification."""
    if w.N > 1:
        return "counterfactual"
    if w.deltas:
        return "cactus"
    return "verify"


def time_oracle(w, inp_host, n_seq, repeats=1):
    import oracle
    sel = np.arange(n_seq)
    t = workloads.to_numpy_logits(inp_host["target"][:n_seq])
    tok = inp_host["tokens"][:n_seq].numpy()
    seeds = inp_host["seeds"][:n_seq].numpy().astype(np.uint64)
    kind = kind_of(w)
    if kind == "counterfactual":
        d = workloads.to_numpy_logits(inp_host["drafters"][:, :n_seq])
    else:
        d = workloads.to_numpy_logits(inp_host["draft"][:n_seq])
    oracle.build()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    for _ in range(repeats):
        if kind == "counterfactual":
            oracle.counterfactual(t, d, w.temperature, w.selected, tok, seeds, seq_index=sel, nthreads=cores)
        elif kind == "cactus":
            oracle.cactus(t, d, tok, seeds, max(w.deltas), w.temperature, seq_index=sel, nthreads=cores)
        else:
            oracle.verify(t, d, tok, seeds, w.temperature, seq_index=sel, nthreads=cores)
    dt = (time.perf_counter() - t0) / repeats
    return n_seq * w.K / dt, dt, cores


def run_reference(args, w):
    import torch
    rank, world, local, pg = dist_setup(args.gpus)
    if rank != 0:
        return 0
    n_seq = min(w.B, args.ref_sequences)
    inp = workloads.make(w.scaled(B=n_seq), device="cpu")
    for _ in range(args.warmup):
        time_oracle(w, inp, min(n_seq, 2))
    t0 = time.perf_counter()
    times = []
    for _ in range(args.steps):
        _, dt, cores = time_oracle(w, inp, n_seq)
        times.append(dt)
    total = time.perf_counter() - t0
    value = n_seq * w.K * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "sample_sequences": n_seq},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "%d of %d sequences of one batch per step" % (n_seq, w.B)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    del torch
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    import speculative_decoding_verification_target_gb300 as sv

    rank, world, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load()
    batch_bytes = w.algorithmic_bytes()
    ring = max(2, -(-4 * L2_BYTES // batch_bytes))        # >= 4x L2 in flight across the ring
    ring = min(ring, args.max_ring)
    batches = [workloads.make(w.scaled(gen_seed=w.gen_seed + 101 * i + 7919 * rank), device=dev)
               for i in range(ring)]
    kind = kind_of(w)
    ws = sv.new_workspace(w.B, w.K, w.V, w.N, dev)
    acc = torch.empty(w.B, dtype=torch.int32, device=dev)
    outt = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    gam = torch.empty((w.N, w.B, w.K), dtype=torch.float32, device=dev) if kind == "counterfactual" else None
    stream = torch.cuda.current_stream(dev)
    # kernels per call: the statistics pass (gamma kernel for gamma calls) and the chain-and-draw kernel
    launches_per_call = 2

    def call(bt, s=None):
        if kind == "counterfactual":
            sv.counterfactual_gamma(bt["target"], bt["drafters"], w.temperature, w.selected, bt["tokens"],
                                    bt["seeds"], gamma=gam, want_loss=False, accept_len=acc, out_tokens=outt,
                                    want_diag=False, workspace=ws, stream=s)
        elif kind == "cactus":
            sv.cactus_verify(bt["target"], bt["draft"], bt["tokens"], bt["seeds"], max(w.deltas), w.temperature,
                             accept_len=acc, out_tokens=outt, want_diag=False, workspace=ws, stream=s)
        else:
            sv.verify(bt["target"], bt["draft"], bt["tokens"], bt["seeds"], w.temperature, accept_len=acc,
                      out_tokens=outt, want_diag=False, workspace=ws, stream=s)

    def step(i):
        call(batches[i % ring])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # Host-side marshalling per call (tens of microseconds of Python) would otherwise leave the GPU idle
    # between ~30 us calls: the K timed steps are captured once into a CUDA graph and replayed.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(graph, stream=cap):
        for i in range(args.steps):
            step(args.warmup + i)
    graph.replay()
    torch.cuda.synchronize(dev)
    barrier(pg, torch)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    start.record(stream)
    graph.replay()
    stop.record(stream)
    barrier(pg, torch)
    clocks.stop()
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(pg, torch, elapsed_ms, dev)
    # eager calls through the binding, for reference (includes host marshalling gaps)
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for i in range(args.steps):
        step(i)
    e_stop.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = e_start.elapsed_time(e_stop) / args.steps
    status = sv.read_status(ws)

    # end to end through the public call: pinned host inputs -> device, the call, results -> host
    hb = batches[0]
    in_keys = ("target", "drafters" if kind == "counterfactual" else "draft", "tokens", "seeds")
    host_in = {k: hb[k].to("cpu").pin_memory() for k in in_keys}
    dev_in = {k: torch.empty_like(hb[k]) for k in host_in}
    host_out = {"accept_len": torch.empty(w.B, dtype=torch.int32).pin_memory(),
                "out_tokens": torch.empty((w.B, w.K + 1), dtype=torch.int32).pin_memory()}
    if gam is not None:
        host_out["gamma"] = torch.empty(tuple(gam.shape), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def e2e_step():
        for k in host_in:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        call(dev_in, stream)
        host_out["accept_len"].copy_(acc, non_blocking=True)
        host_out["out_tokens"].copy_(outt, non_blocking=True)
        if gam is not None:
            host_out["gamma"].copy_(gam, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20 if batch_bytes < (2 << 30) else 3))
    for _ in range(2):
        e2e_step()
    barrier(pg, torch)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier(pg, torch)
    e2e_serial_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1), dev)

    # The same steps pipelined: step i + 1's inputs are copied into a second device buffer on a copy stream
    # while step i computes (every step still copies its own inputs in and its results out).
    dev_in2 = [dev_in, {k: torch.empty_like(hb[k]) for k in host_in}]
    cstream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(j):
        with torch.cuda.stream(cstream):
            if j >= 2:
                cstream.wait_event(consumed[j % 2])
            for k in host_in:
                dev_in2[j % 2][k].copy_(host_in[k], non_blocking=True)
            copied[j % 2].record(cstream)

    def e2e_pipelined(n):
        cstream.wait_stream(stream)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(copied[i % 2])
            call(dev_in2[i % 2], stream)
            consumed[i % 2].record(stream)
            host_out["accept_len"].copy_(acc, non_blocking=True)
            host_out["out_tokens"].copy_(outt, non_blocking=True)
            if gam is not None:
                host_out["gamma"].copy_(gam, non_blocking=True)

    e2e_pipelined(2)
    torch.cuda.synchronize(dev)
    barrier(pg, torch)
    e0.record(stream)
    e2e_pipelined(e2e_steps)
    e1.record(stream)
    barrier(pg, torch)
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1), dev)

    if rank != 0:
        return 0
    positions = w.positions * world
    value = positions * args.steps / (elapsed_ms / 1e3)
    # e2e reports the faster of the two ways to run the steps: pipelined for calls whose copy dominates,
    # serial for latency-bound ones (the stream and event bookkeeping costs more than it hides there)
    pipelined = e2e_ms <= e2e_serial_ms
    e2e_best_ms = e2e_ms if pipelined else e2e_serial_ms
    e2e_value = positions * e2e_steps / (e2e_best_ms / 1e3)
    peak, peak_kind = peaks()
    avg_call_s = elapsed_ms / args.steps / 1e3
    achieved = batch_bytes / avg_call_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "N": w.N, "temperature": w.temperature,
                   "positions_per_step_per_gpu": w.positions, "bytes_per_step_per_gpu": batch_bytes,
                   "entry_point": {"verify": "spec_verify", "cactus": "spec_cactus_verify (delta %g)" % max(
                       w.deltas or (0.0,)), "counterfactual": "spec_counterfactual_gamma (N %d, fused verify "
                       "of drafter %d)" % (w.N, w.selected)}[kind],
                   "l2": "inputs larger than L2: ring of %d distinct batches (%.0f MB) > 129 MB L2" % (
                       ring, ring * batch_bytes / 1e6),
                   "parallelism": "replicas over sequences" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": RECORDED_TRAFFIC.get(kernel_source_hash(), {}).get(w.name), "peak_kind": peak_kind,
                     "kernel": "%s + draw_kernel: one whole %s call (both kernels), graph replay timed with CUDA "
                               "events on the launching stream, divided by the steps" % (
                                   "gamma_kernel" if kind == "counterfactual" else "stats_kernel", kind),
                     "avg_call_us": avg_call_s * 1e6, "eager_call_us": eager_ms * 1e3,
                     "frac_of_8tbs_nominal": achieved / 8000.0},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_best_ms / e2e_steps,
                "mode": "pipelined: step i + 1's host-to-device copy overlaps step i's call (two device buffers)"
                        if pipelined else "serial: copy in, call, copy out, one step after another",
                "pipelined_value": positions * e2e_steps / (e2e_ms / 1e3),
                "serial_value": positions * e2e_steps / (e2e_serial_ms / 1e3)},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clocks.summary(),
        "device_status": status,
    }
    if not args.no_cpu_baseline:
        host = {k: batches[0][k].to("cpu") for k in ("target", "drafters" if kind == "counterfactual" else "draft",
                                                       "tokens", "seeds")}
        n_seq = min(w.B, args.cpu_sequences)
        reps, total_dt = 0, 0.0
        while total_dt < args.cpu_seconds and reps < 1000:
            _, dt, cores = time_oracle(w, host, n_seq)
            reps += 1
            total_dt += dt
        line["cpu_baseline"] = {"value": reps * n_seq * w.K / total_dt, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": "%d of %d sequences of one %s batch, repeated %d times (%.1f s)" % (
                                    n_seq, w.B, w.name, reps, total_dt)}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--max-ring", type=int, default=8)
    ap.add_argument("--cpu-sequences", type=int, default=64)
    ap.add_argument("--ref-sequences", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
