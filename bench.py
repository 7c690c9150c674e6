#!/usr/bin/env python3
"""Benchmark of the fused score -> select -> sparse-verify step.

Default workload (--workload batched32k): Qwen2.5-72B-shaped attention, B=16
sequences of L=32768 context, Hq=64, Hkv=8, d=128, gamma=5, budget k=2048
(sinks 16, window 256, m 512), 4 target + 4 draft SRH heads; seeded
synthetic bf16 inputs (see synth/).  The KV caches (2.15 GB) are far larger
than L2, so no flush is needed between steps.

Two more workloads are timed on request:
  --workload sweep32k   B=8, L=32768, the twelve (k, gamma) points
                        k in {512, 1024, 2048, 4096} x gamma in {2, 4, 8},
                        m = k/4, 10 % saliency drift; score, select and verify
                        timed separately at each point, beside dense.
  --workload stack128k  B=4, L=131072, 8 layers (17.2 GB of KV) sharing one
                        I_verify from SRHs on layers 0 and 4, then kv_append
                        of 3 accepted rows per sequence and layer; beside dense
                        verification of all 8 layers.

One JSON line on rank 0.  ``value`` is the algorithmic HBM GB/s of the step
(bytes the method must move / device time per step), summed over ranks;
``ms_per_step`` is the step time.  Per-stage, dense and end-to-end figures are
medians of at least 50 individually timed runs.  ``--impl reference`` times
the fp64 CPU oracle instead, on bounded samples of the headline workload.

Multi-GPU: each rank runs an independent replica of the workload on its own
GPU with its own seed (the sequences are independent, no collective on the
data path); the step time is the max over ranks.  ``--gpus N`` without a
torchrun environment starts the N ranks itself through torch.distributed.run.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse verify step µs & HBM GB/s (score+select+attend), B=16 L=32k k=2048"
METRICS = {
    "batched32k": METRIC,
    "sweep32k": "sparse verify step µs & HBM GB/s (score+select+attend), B=8 L=32k, "
                "k x gamma sweep (12 points)",
    "stack128k": "sparse verify step µs & HBM GB/s (score+select+attend, 8 layers), "
                 "B=4 L=128k k=4096, plus kv_append of 3 rows",
}
WORKLOAD = "batched32k"
FALLBACK_HBM_GBS = 6800.0
MIN_RUNS = 50          # individually timed runs behind every median


# --------------------------------------------------------------------------
# algorithmic bytes (what the method must move; no implementation scratch)
# --------------------------------------------------------------------------

def slabs(wl):
    """Distinct (channel, layer, KV head) slabs read by scoring."""
    out = set()
    for (c, l, h) in wl.srh:
        if c == 0:
            out.add((0, l, h // (wl.Hq_d // wl.Hkv_d)))
        else:
            out.add((1, l, h // (wl.Hq // wl.Hkv)))
    return sorted(out)


def algorithmic_bytes(wl, L=None, B=None):
    L = wl.L if L is None else L
    B = wl.B if B is None else B
    T = wl.gamma + 1
    k_reads = sum(B * L * (wl.d_d if c == 0 else wl.d) * 2 for (c, _, _) in slabs(wl))
    imp = B * 2 * L * 4
    score = k_reads + imp
    select = imp + B * wl.k * 4
    per_layer = (2 * B * wl.Hkv * wl.k * wl.d * 2 + 2 * B * wl.Hkv * T * wl.d * 2
                 + B * T * wl.Hq * wl.d * 2 + B * T * wl.Hq * wl.d * 4)
    verify = wl.n_layers * per_layer + B * wl.k * 4
    dense = wl.n_layers * (2 * B * wl.Hkv * L * wl.d * 2 + 2 * B * wl.Hkv * T * wl.d * 2
                           + B * T * wl.Hq * wl.d * 2 + B * T * wl.Hq * wl.d * 4)
    return dict(score_kernel=k_reads, score=score, select=select, verify=verify,
                step=score + select + verify, dense=dense)


def append_bytes(wl, rows):
    """kv_append of `rows` accepted rows per sequence and layer: the block rows
    read and the cache rows written, K and V, plus seq_len read and written."""
    return wl.n_layers * 2 * 2 * wl.B * wl.Hkv * rows * wl.d * 2 + wl.B * 4 * 2


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "score_stream_kernel.dram_traffic.txt")
TRAFFIC_SOURCES = ("sparse_kv_verify_gb300/csrc/score.cu", "sparse_kv_verify_gb300/csrc/common.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_per_launch(sequences: int):
    """DRAM bytes (read + write) of one stream-kernel launch over `sequences`
    sequences, scaled from the ncu capture recorded in TRAFFIC_FILE; None when
    there is no capture or the kernel source has changed since it was taken."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as fh:
            for ln in fh:
                if "=" in ln and not ln.startswith("#"):
                    k, v = ln.strip().split("=", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256_16") != kernel_source_hash():
            return None
        return float(fields["dram_bytes_per_sequence"]) * sequences
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(x: float, dist, device) -> float:
    """Max of a per-rank scalar over all ranks (the step time of the job)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(wl, rank: int):
    """Rank r's replica of a workload: same shapes, its own seed."""
    return wl.with_(seed_id=wl.seed_id + 1000 * rank) if rank else wl


def free_port() -> int:
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def replica_command(n: int, argv, script=None):
    """torch.distributed.run command that starts `script` (this file by
    default) as n local ranks, one per GPU, rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", f"--master-port={free_port()}",
            script or os.path.abspath(__file__), *argv]


def init_ranks():
    """Process group of a torchrun launch (None for a single process): NCCL
    with one GPU per rank where CUDA is present, gloo on the CPU otherwise."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world == 1:
        return None
    import torch
    import torch.distributed as tdist
    if torch.cuda.is_available():
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
    else:
        tdist.init_process_group("gloo")
    return tdist


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons during the timed region.

    Reads NVML through ctypes (read-only queries) from a background thread
    every ~2 ms; falls back to ``nvidia-smi -lms`` when NVML is unavailable.
    """
    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.stop = False
        self.thread = None
        self.nvml = None
        self.proc = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        return lib, h

    def _loop(self):
        import ctypes
        lib, h = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop:
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0          # NVML_CLOCK_SM
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs))
            if ok:
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        import threading
        try:
            self.nvml = self._nvml_open()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}",
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *a):
        self.stop = True
        if self.thread is not None:
            self.thread.join(timeout=2)

    def collect(self):
        """Ends a fallback nvidia-smi sampler and parses its samples."""
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                out = ""
            self.proc = None
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[0]), float(f[1]), int(f[2], 16)))
                except (ValueError, IndexError):
                    pass
        return self.samples

    def result(self):
        return summarise_clocks(self.collect(), "nvml" if self.nvml is not None else "nvidia-smi")


def summarise_clocks(samples, source):
    """Median SM clock, max clock and the clock-event reasons seen."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    reasons = set()
    for _, _, r in samples:
        for bit, name in ClockSampler.REASONS.items():
            if r & bit:
                reasons.add(name)
    return {"sm_mhz": statistics.median(c for c, _, _ in samples),
            "sm_max_mhz": max(m for _, m, _ in samples),
            "reasons": sorted(reasons), "samples": len(samples), "source": source}


def merge_clocks(samplers):
    """One clock record over several timed regions."""
    samples = [x for sm in samplers for x in sm.collect()]
    src = "nvml" if all(sm.nvml is not None for sm in samplers) else "nvidia-smi"
    return summarise_clocks(samples, src)


# --------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# --------------------------------------------------------------------------

def oracle_steps_worker(n_steps: int, min_seconds: float = 0.0):
    """Times the oracle on one sequence of the workload per step (score,
    select and verify); keeps stepping until ``n_steps`` steps and at least
    ``min_seconds`` are done.  Returns (per-step seconds, bytes per step)."""
    from oracle import dustin_oracle as O
    from synth import WORKLOADS, generate, to_bits
    wl = WORKLOADS[WORKLOAD].with_(B=1)
    x = generate(wl, device="cpu")
    bits = lambda ts: [to_bits(t) for t in ts]
    dq, kd, hq, K = bits(x.draft_q), bits(x.Kd), bits(x.hist_q), bits(x.K)
    Q, V, Kb, Vb = to_bits(x.Q[0]), to_bits(x.V[0]), to_bits(x.Kb[0]), to_bits(x.Vb[0])
    times = []
    t_all = time.perf_counter()
    while len(times) < n_steps or time.perf_counter() - t_all < min_seconds:
        t0 = time.perf_counter()
        imp = O.score(dq, kd, hq, K, wl.srh, x.seq_len, wl.Lcap)
        I, _ = O.select(imp, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
        O.verify(Q, K[0], V, Kb, Vb, I, x.seq_len)
        times.append(time.perf_counter() - t0)
        if len(times) >= 64:
            break
    return times, algorithmic_bytes(wl, B=1)["step"]


def oracle_stages_worker(workload: str, reps: int, dense: bool):
    """Median seconds of each oracle stage on one sequence of `workload`:
    score, select, sparse verify and (if asked, one run) dense verify."""
    from oracle import dustin_oracle as O
    from synth import WORKLOADS, generate, to_bits
    wl = WORKLOADS[workload].with_(B=1)
    x = generate(wl, device="cpu")
    bits = lambda ts: [to_bits(t) for t in ts]
    dq, kd, hq, K = bits(x.draft_q), bits(x.Kd), bits(x.hist_q), bits(x.K)
    Q, V, Kb, Vb = to_bits(x.Q[0]), to_bits(x.V[0]), to_bits(x.Kb[0]), to_bits(x.Vb[0])
    t = {"score": [], "select": [], "verify": []}
    for _ in range(reps):
        t0 = time.perf_counter()
        imp = O.score(dq, kd, hq, K, wl.srh, x.seq_len, wl.Lcap)
        t1 = time.perf_counter()
        I, _ = O.select(imp, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
        t2 = time.perf_counter()
        O.verify(Q, K[0], V, Kb, Vb, I, x.seq_len)
        t3 = time.perf_counter()
        t["score"].append(t1 - t0)
        t["select"].append(t2 - t1)
        t["verify"].append(t3 - t2)
    out = {k: statistics.median(v) for k, v in t.items()}
    out["step"] = out["score"] + out["select"] + out["verify"]
    if dense:
        t0 = time.perf_counter()
        O.dense(Q, K[0], V, Kb, Vb, x.seq_len)
        out["dense"] = time.perf_counter() - t0
    return out


def _oracle_subprocess(call: str, threads: int):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = "import json,sys; sys.path.insert(0, %r); import bench; print(json.dumps(bench.%s))" % (
        ROOT, call)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_oracle_subprocess(n_steps: int, min_seconds: float, threads: int):
    times, nbytes = _oracle_subprocess(f"oracle_steps_worker({n_steps!r}, {min_seconds!r})", threads)
    return times, nbytes


def oracle_stage_report(threads: int):
    """Per-stage oracle seconds per sequence: the headline workload on
    `threads` threads (dense once), and the 8K-position layer on one thread."""
    rep = {"threads": threads,
           "batched32k_per_sequence_s": _oracle_subprocess(
               "oracle_stages_worker('batched32k', 3, True)", threads)}
    rep["layer8k_single_thread_s"] = _oracle_subprocess(
        "oracle_stages_worker('layer8k', 5, True)", 1)
    return rep


ARM_PARTS = {0xd0c: "Neoverse-N1", 0xd40: "Neoverse-V1", 0xd49: "Neoverse-N2",
             0xd4f: "Neoverse-V2", 0xd8e: "Neoverse-N3", 0xd84: "Neoverse-V3"}


def cpu_model():
    """Host CPU model: lscpu's model name, else /proc/cpuinfo's (x86 'model
    name', or the Arm implementer/part codes), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip().lower() == "model name" and val.strip() not in ("", "-"):
                return val.strip()
    except Exception:
        pass
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip().lower()
                if key in ("model name", "cpu implementer", "cpu part") and key not in fields:
                    fields[key] = val.strip()
    except Exception:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        try:
            imp, part = int(fields.get("cpu implementer", "0"), 16), int(fields["cpu part"], 16)
            if imp == 0x41 and part in ARM_PARTS:
                return f"Arm {ARM_PARTS[part]} (implementer 0x41, part {part:#x})"
            return f"Arm implementer {imp:#x}, part {part:#x}"
        except ValueError:
            pass
    import platform
    return platform.machine()


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    if args.workload != WORKLOAD:
        print(json.dumps({"impl": "reference",
                          "unavailable": "the oracle arm times the headline workload only"}))
        return 0
    threads = os.cpu_count() or 1
    times, nbytes = run_oracle_subprocess(args.warmup + args.steps, 0.0, threads)
    times = times[args.warmup:args.warmup + args.steps]
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    sample = f"1 sequence of {WORKLOAD} per step (score+select+verify), fp64 numpy oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3,
            "ms_per_step_is": "per sequence: each reference step scores, selects and verifies "
                              "one sequence of the batch (GB/s is per byte, so it compares "
                              "with the GPU arm's whole-batch steps)",
            "sequences_per_step": 1,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(args, world=args.gpus),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def srh_summary(wl):
    sl = slabs(wl)
    nt = sum(1 for e in wl.srh if e[0] == 1)
    nd = sum(1 for e in wl.srh if e[0] == 0)
    layers = sorted({e[1] for e in wl.srh})
    return (f"{nt} target ({sum(1 for c in sl if c[0] == 1)} KV heads) + {nd} draft "
            f"({sum(1 for c in sl if c[0] == 0)} KV heads)"
            + (f", layers {layers}" if wl.n_layers > 1 else ""))


def config_block(args, wl=None, world=1):
    from synth import WORKLOADS
    wl = wl or WORKLOADS[args.workload]
    kv = 2 * wl.n_layers * wl.B * wl.Hkv * wl.Lcap * wl.d * 2
    c = {"workload": wl.name, "B": wl.B, "L": wl.L, "Lcap": wl.Lcap, "n_layers": wl.n_layers,
         "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "gamma": wl.gamma, "k": wl.k, "sinks": wl.sinks,
         "window": wl.window, "m": wl.m, "srh": srh_summary(wl),
         "draft": f"Hq_d={wl.Hq_d} Hkv_d={wl.Hkv_d} d_d={wl.d_d}",
         "l2": f"inputs larger than L2 (KV {kv / 1e9:.2f} GB), no flush",
         "parallelism": f"replicas x{world}"}
    if args.workload == "sweep32k":
        c.update(k="512..4096", gamma="2,4,8", m="k/4",
                 points="k in {512,1024,2048,4096} x gamma in {2,4,8}", drift=wl.drift)
    if args.workload == "stack128k":
        c["append_rows"] = APPEND_ROWS
    return c


APPEND_ROWS = 3


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_block(fn, n, stream, dev):
    """Milliseconds per call over n back-to-back calls (one event pair)."""
    import torch
    e0, e1 = _events(2)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n


def median_each(fn, n, stream, dev):
    """Median milliseconds of n individually timed calls."""
    import torch
    ev = [_events(2) for _ in range(n)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def stage_medians(call, n, stream, dev, after=None):
    """Median microseconds of each stage over n steps timed with the step's
    stage events (steps apart from the timed region: the events cost a
    little).  `after(event)`: run after each step; it records `event` when
    its own work is queued, timed as the stage "append"."""
    import torch
    ev = [_events(6) for _ in range(n)]
    for e in ev:
        call(stream, events=e[:5])
        if after is not None:
            after(e[5])
    torch.cuda.synchronize(dev)
    st = {"score_stream_group0": [], "score": [], "select": [], "verify": []}
    if after is not None:
        st["append"] = []
    for e in ev:
        st["score_stream_group0"].append(e[0].elapsed_time(e[1]))
        st["score"].append(e[0].elapsed_time(e[2]))
        st["select"].append(e[2].elapsed_time(e[3]))
        st["verify"].append(e[3].elapsed_time(e[4]))
        if after is not None:
            st["append"].append(e[4].elapsed_time(e[5]))
    return {k: statistics.median(v) * 1e3 for k, v in st.items()}


def make_step(wl, dev, n_layers=None):
    import torch
    import sparse_kv_verify_gb300 as dk
    from synth import generate
    x = generate(wl, device=dev)
    p = dk.Params(wl.B, wl.Lcap, wl.gamma, wl.sinks, wl.window, wl.m, wl.k)
    seq = torch.as_tensor(x.seq_len, device=dev)
    layers = [dk.VerifyLayer(x.Q[l], x.K[l], x.V[l], x.Kb[l], x.Vb[l])
              for l in range(n_layers or wl.n_layers)]
    call = dk.StepCall(p, dk.Signal(x.draft_q, x.Kd), dk.Signal(x.hist_q, x.K), wl.srh, layers,
                       seq)
    return x, p, seq, call


def dense_fn(p, x, seq, dev, n_layers, stream):
    """All layers' dense verification on the same inputs (the comparator)."""
    import torch
    import sparse_kv_verify_gb300 as dk
    wl_shape = (x.Q[0].shape[2], x.K[0].shape[1], x.K[0].shape[3], 1)
    ws = dk.workspace(p, verify=wl_shape, device=dev)
    outs = [torch.empty(x.Q[l].shape, dtype=torch.float32, device=dev) for l in range(n_layers)]

    def run():
        for l in range(n_layers):
            dk.dense_verify_attn(p, x.Q[l], x.K[l], x.V[l], x.Kb[l], x.Vb[l], seq, o=outs[l], ws=ws,
                                 stream=stream)
    return run


def roofline_of(stage, wl, group, peak, peak_kind, with_traffic):
    """The dominant kernel (the score stream kernel of the first sequence
    group): its algorithmic bytes over its median event-timed duration."""
    sk_bytes = algorithmic_bytes(wl, B=group)["score_kernel"]
    achieved = sk_bytes / (stage["score_stream_group0"] * 1e-6) / 1e9
    return {"kernel": "score_stream_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic_per_launch(group) if with_traffic else None,
            "algorithmic_bytes_per_launch": sk_bytes, "sequences_per_launch": group}


def gpu_arm(args, rank, world, dist):
    import torch

    import __graft_entry__ as ge

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ge.build()
    if args.workload == "sweep32k":
        return sweep_arm(args, rank, world, dist, dev, local)
    if args.workload == "stack128k":
        return stack_arm(args, rank, world, dist, dev, local)
    return headline_arm(args, rank, world, dist, dev, local)


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def headline_arm(args, rank, world, dist, dev, local):
    import torch

    import sparse_kv_verify_gb300 as dk
    from synth import WORKLOADS

    wl = WORKLOADS[WORKLOAD]
    if args.batch:
        wl = wl.with_(B=args.batch)
    wl = replica_workload(wl, rank)
    x, p, seq, call = make_step(wl, dev)
    stream = torch.cuda.current_stream(dev)
    ab = algorithmic_bytes(wl)
    if args.profile and args.profile != "step":
        return profile_op(args, wl, x, p, seq, call, dev, stream)

    # ---- device-resident timing of exactly `steps` steps
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    flags = dk.check(call.ws)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after warm-up")
    n_launch, group = call.launches()
    _barrier(dist)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.01)
        total_ms = time_block(call, args.steps, stream, dev) * args.steps
    clocks = sampler.result()
    _barrier(dist)
    step_ms = max_over_ranks(total_ms / args.steps, dist, dev)

    if args.profile:
        # profiling run (ncu): warm-up and timed steps only
        if dk.check(call.ws):
            raise RuntimeError("device flags after the profiled steps")
        if rank == 0:
            print(json.dumps({"profile_run": "step", "workload": wl.name, "B": wl.B,
                              "step_us": step_ms * 1e3}), flush=True)
        return 0

    n_med = max(MIN_RUNS, args.steps)
    stage = stage_medians(call, n_med, stream, dev)

    # ---- dense comparator on the same inputs
    dense = dense_fn(p, x, seq, dev, 1, stream)
    for _ in range(2):
        dense()
    dense_ms = median_each(dense, n_med, stream, dev)

    # ---- end to end through the public API: every step copies its inputs from
    # pinned host memory and reads its O back to pinned host memory.  Two sets of
    # device buffers let step i+1's input copies and step i's read-back run on
    # copy streams while step i computes, as a serving loop would.
    def per_layer(ts):
        return [t.cpu().pin_memory() for t in ts]

    host_in = (per_layer([x.Q[0]]) + per_layer(x.hist_q) + per_layer(x.draft_q)
               + per_layer([x.Kb[0], x.Vb[0]]))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    sets = []
    for _ in range(2):
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]
        nh = len(x.hist_q)
        q, hq, dq = dev_in[0], dev_in[1:1 + nh], dev_in[1 + nh:1 + nh + len(x.draft_q)]
        kb, vb = dev_in[-2], dev_in[-1]
        c = dk.StepCall(p, dk.Signal(dq, x.Kd), dk.Signal(hq, x.K), wl.srh,
                        [dk.VerifyLayer(q, x.K[0], x.V[0], kb, vb)], seq)
        out = torch.empty(c.layers[0].o.shape, dtype=torch.float32).pin_memory()
        sets.append((dev_in, c, out))
    d2h = sets[0][2].numel() * sets[0][2].element_size()
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        s_ = i % 2
        with torch.cuda.stream(h2d_stream):
            if i >= 2:
                h2d_stream.wait_event(ev_done[s_])     # step i-2 has read these inputs
            for h, d in zip(host_in, sets[s_][0]):
                d.copy_(h, non_blocking=True)
            ev_in[s_].record(h2d_stream)

    def run_steps(n, start, marks=None):
        h2d_stream.wait_event(start)
        copy_in(0)
        for i in range(n):
            s_ = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(ev_in[s_])
            if i >= 2:
                stream.wait_event(ev_out[s_])          # step i-2's O has been read back
            sets[s_][1](stream)
            ev_done[s_].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_done[s_])
                sets[s_][2].copy_(sets[s_][1].layers[0].o, non_blocking=True)
                ev_out[s_].record(d2h_stream)
                if marks is not None:
                    marks[i].record(d2h_stream)        # step i's result is on the host
        stream.wait_stream(d2h_stream)

    w0 = torch.cuda.Event()
    w0.record(stream)
    run_steps(args.warmup, w0)
    torch.cuda.synchronize(dev)
    _barrier(dist)
    n_e2e = max(MIN_RUNS, args.steps)
    marks = _events(n_e2e)
    e0, e1 = _events(2)
    e0.record(stream)
    run_steps(n_e2e, e0, marks)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, dev)
    e2e_med = statistics.median(marks[i - 1].elapsed_time(marks[i]) for i in range(1, n_e2e))
    if not torch.equal(sets[(n_e2e - 1) % 2][2], sets[(n_e2e - 1) % 2][1].layers[0].o.cpu()):
        raise RuntimeError("end-to-end read-back does not match the device result")
    flags = dk.check(call.ws)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after timing")
    if rank != 0:
        return 0

    peak, peak_kind = peak_hbm()
    value = world * ab["step"] / (step_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_block(args, wl, world),
        "step_us": step_ms * 1e3,
        "stage_us": stage,
        "stage_stat": f"median of {n_med} steps timed with stage events",
        "stage_gbs": {"score": ab["score"] / stage["score"] / 1e3,
                      "select": ab["select"] / stage["select"] / 1e3,
                      "verify": ab["verify"] / stage["verify"] / 1e3},
        "algorithmic_bytes_per_step": ab["step"],
        "verified_tokens_per_s": world * wl.B * (wl.gamma + 1) / (step_ms * 1e-3),
        "step_frac_of_hbm": (ab["step"] / (step_ms * 1e-3) / 1e9) / peak,
        "step_frac_of_nominal_8tbs": (ab["step"] / (step_ms * 1e-3) / 1e9) / 8000.0,
        "dense": {"us": dense_ms * 1e3, "GB/s": ab["dense"] / (dense_ms * 1e-3) / 1e9,
                  "frac_of_hbm": ab["dense"] / (dense_ms * 1e-3) / 1e9 / peak,
                  "stat": f"median of {n_med} calls"},
        "speedup_vs_dense": {"attention_only": dense_ms / (stage["verify"] * 1e-3),
                             "step": dense_ms / step_ms},
        "roofline": roofline_of(stage, wl, group, peak, peak_kind, True),
        "e2e": {"value": world * ab["step"] / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "median_step_interval_ms": e2e_med, "steps": n_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "dustin_verify_step per step; that step's inputs copied from pinned host "
                       "memory and its O read back to pinned host memory inside the timed region, "
                       "double-buffered so copies overlap the neighbouring steps' compute; value "
                       f"over the whole region of {n_e2e} steps, median_step_interval_ms = median "
                       "time between consecutive steps' read-backs"},
        "gpu_launches": n_launch * args.steps,
        "launches_per_step": n_launch,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        try:
            times, nb = run_oracle_subprocess(1, args.cpu_seconds, threads)
            dt, n = sum(times), len(times)
            line["cpu_baseline"] = {"value": nb * n / dt / 1e9, "unit": "GB/s", "cores": threads,
                                    "kind": "oracle", "cpu": cpu_model(),
                                    "sample": f"{n} sequence(s) of {WORKLOAD} through score, "
                                              f"select and verify ({dt:.1f} s, fp64 numpy)"}
            line["cpu_baseline"]["stages"] = oracle_stage_report(threads)
        except Exception as e:  # the GPU number stands without it
            line["cpu_baseline"] = {"value": None, "error": str(e)[-300:]}
    print(json.dumps(line), flush=True)
    return 0


def profile_op(args, wl, x, p, seq, call, dev, stream):
    """warm-up + timed calls of one operation on the step's inputs, for ncu:
    dense verification, the compact-cache copy of one step's selection, or
    kv_append of 3 rows (seq_len put back after each call)."""
    import torch

    import sparse_kv_verify_gb300 as dk
    call()   # importance and I_verify of these inputs
    torch.cuda.synchronize(dev)
    if args.profile == "dense":
        fn = dense_fn(p, x, seq, dev, 1, stream)
    elif args.profile == "compact":
        kc = torch.empty((wl.B, wl.Hkv, wl.k, wl.d), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        slc = torch.empty_like(seq)

        def fn():
            dk.dustin_compact_kv(p, [x.K[0]], [x.V[0]], call.i_verify, seq, [kc], [vc], slc,
                                 ws=call.ws, stream=stream)
    else:
        seq0 = seq.clone()
        n_acc = torch.full((wl.B,), APPEND_ROWS, dtype=torch.int32, device=dev)
        app = dk.AppendCall(p, x.K, x.V, x.Kb, x.Vb, n_acc, seq, ws=call.ws)

        def fn():
            app(stream)
            seq.copy_(seq0, non_blocking=True)
    for _ in range(args.warmup):
        fn()
    ms = time_block(fn, args.steps, stream, dev)
    if dk.check(call.ws):
        raise RuntimeError("device flags after the profiled calls")
    print(json.dumps({"profile_run": args.profile, "workload": wl.name, "B": wl.B,
                      "call_us": ms * 1e3}), flush=True)
    return 0


def sweep_arm(args, rank, world, dist, dev, local):
    """The twelve (k, gamma) points of the B=8, L=32k sweep: step, stages and
    dense comparator at each point."""
    import torch

    import sparse_kv_verify_gb300 as dk
    from synth import WORKLOADS, sweep_points

    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peak_hbm()
    n_med = max(MIN_RUNS, args.steps)
    points, samplers = [], []
    launches = 0
    tot_bytes = tot_ms = 0.0
    roof = None
    for (k, gamma) in sweep_points():
        wl = replica_workload(WORKLOADS["sweep32k"].with_(k=k, gamma=gamma, m=k // 4), rank)
        x, p, seq, call = make_step(wl, dev)
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize(dev)
        n_launch, group = call.launches()
        _barrier(dist)
        sm = ClockSampler(local)
        with sm:
            ms = time_block(call, args.steps, stream, dev)
        samplers.append(sm)
        step_ms = max_over_ranks(ms, dist, dev)
        stage = stage_medians(call, n_med, stream, dev)
        dense = dense_fn(p, x, seq, dev, 1, stream)
        dense()
        dense_ms = median_each(dense, n_med, stream, dev)
        flags = dk.check(call.ws)
        if flags:
            raise RuntimeError(f"device flags {flags:#x} at k={k} gamma={gamma}")
        ab = algorithmic_bytes(wl)
        gbs = lambda b, us: b / us / 1e3
        points.append({
            "k": k, "gamma": gamma, "m": k // 4, "step_us": step_ms * 1e3,
            "step_gbs": gbs(ab["step"], step_ms * 1e3),
            "step_frac_of_hbm": gbs(ab["step"], step_ms * 1e3) / peak,
            "stage_us": {s_: stage[s_] for s_ in ("score", "select", "verify")},
            "stage_gbs": {s_: gbs(ab[s_], stage[s_]) for s_ in ("score", "select", "verify")},
            "stage_frac_of_hbm": {s_: gbs(ab[s_], stage[s_]) / peak
                                  for s_ in ("score", "select", "verify")},
            "dense_us": dense_ms * 1e3, "dense_gbs": gbs(ab["dense"], dense_ms * 1e3),
            "speedup_vs_dense": {"attention_only": dense_ms * 1e3 / stage["verify"],
                                 "step": dense_ms / step_ms},
            "bytes_mb": {s_: ab[s_] / 1e6 for s_ in ("score", "select", "verify", "step", "dense")},
            "launches_per_step": n_launch})
        if (k, gamma) == (2048, 4):
            roof = roofline_of(stage, wl, group, peak, peak_kind, False)
        launches += n_launch * args.steps
        tot_bytes += ab["step"]
        tot_ms += step_ms
        del x, call, dense
        torch.cuda.empty_cache()
    if rank != 0:
        return 0
    line = {
        "metric": METRICS["sweep32k"], "value": world * tot_bytes / (tot_ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_ms / len(points), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(args, WORKLOADS["sweep32k"], world),
        "value_is": "all twelve points' algorithmic bytes over the sum of their step times; "
                    "ms_per_step is the mean step time over the points",
        "points": points, "stage_stat": f"median of {n_med} steps (dense: {n_med} calls)",
        "roofline": roof, "gpu_launches": launches, "clocks": merge_clocks(samplers),
        "e2e": None, "e2e_note": "the end-to-end (host buffers) figure is taken on the "
                                 "headline workload",
    }
    print(json.dumps(line), flush=True)
    return 0


def stack_arm(args, rank, world, dist, dev, local):
    """Eight layers sharing one selection, then kv_append of 3 accepted rows
    per sequence and layer; seq_len is put back after each step so that every
    step appends at the same positions."""
    import torch

    import sparse_kv_verify_gb300 as dk
    from synth import WORKLOADS

    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peak_hbm()
    wl = replica_workload(WORKLOADS["stack128k"], rank)
    x, p, seq, call = make_step(wl, dev)
    seq0 = seq.clone()
    n_acc = torch.full((wl.B,), APPEND_ROWS, dtype=torch.int32, device=dev)
    app = dk.AppendCall(p, x.K, x.V, x.Kb, x.Vb, n_acc, seq, ws=call.ws)

    def step():
        call(stream)
        app(stream)
        seq.copy_(seq0, non_blocking=True)

    def after(ev):
        app(stream)
        ev.record(stream)
        seq.copy_(seq0, non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    flags = dk.check(call.ws)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after warm-up")
    n_launch, group = call.launches()
    _barrier(dist)
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.01)
        ms = time_block(step, args.steps, stream, dev)
    clocks = sampler.result()
    step_ms = max_over_ranks(ms, dist, dev)
    n_med = max(MIN_RUNS, args.steps)
    stage = stage_medians(call, n_med, stream, dev, after=after)
    dense = dense_fn(p, x, seq, dev, wl.n_layers, stream)
    dense()
    dense_ms = median_each(dense, n_med, stream, dev)
    flags = dk.check(call.ws)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after timing")
    if not torch.equal(seq, seq0):
        raise RuntimeError("seq_len was not restored")
    if rank != 0:
        return 0
    ab = algorithmic_bytes(wl)
    apb = append_bytes(wl, APPEND_ROWS)
    gbs = lambda b, us: b / us / 1e3
    line = {
        "metric": METRICS["stack128k"],
        "value": world * (ab["step"] + apb) / (step_ms * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_block(args, wl, world),
        "value_is": "algorithmic bytes of score + select + 8-layer verify + kv_append over the "
                    "step time; the step also restores seq_len (one 16-byte device copy)",
        "step_us": step_ms * 1e3,
        "stage_us": {s_: stage[s_] for s_ in ("score", "select", "verify", "append")},
        "stage_gbs": {"score": gbs(ab["score"], stage["score"]),
                      "select": gbs(ab["select"], stage["select"]),
                      "verify": gbs(ab["verify"], stage["verify"]),
                      "append": gbs(apb, stage["append"])},
        "stage_stat": f"median of {n_med} steps timed with stage events",
        "bytes_mb": {"score": ab["score"] / 1e6, "select": ab["select"] / 1e6,
                     "verify": ab["verify"] / 1e6, "step": ab["step"] / 1e6,
                     "append": apb / 1e6, "dense": ab["dense"] / 1e6},
        "step_frac_of_hbm": gbs(ab["step"] + apb, step_ms * 1e3) / peak,
        "dense": {"us": dense_ms * 1e3, "GB/s": gbs(ab["dense"], dense_ms * 1e3),
                  "frac_of_hbm": gbs(ab["dense"], dense_ms * 1e3) / peak,
                  "stat": f"median of {n_med} runs of all {wl.n_layers} layers"},
        "speedup_vs_dense": {"attention_only": dense_ms * 1e3 / stage["verify"],
                             "step": dense_ms / step_ms},
        "roofline": roofline_of(stage, wl, group, peak, peak_kind, False),
        "gpu_launches": (n_launch + 2) * args.steps, "launches_per_step": n_launch + 2,
        "clocks": clocks,
        "e2e": None, "e2e_note": "the end-to-end (host buffers) figure is taken on the "
                                 "headline workload",
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(METRICS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch size (profiling of smaller cases)")
    ap.add_argument("--profile", nargs="?", const="step", default=None,
                    choices=["step", "dense", "compact", "append"],
                    help="for ncu captures: run only warm-up + timed calls of the step (default) "
                         "or of one other operation on the same inputs, and print no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU, started here as a torchrun launch would
        return subprocess.call(replica_command(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    dist = init_ranks()
    try:
        return gpu_arm(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
