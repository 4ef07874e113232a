"""Benchmark of the GB300 hyper-connection read.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]

One step = the verify-window sweep: 16 reads, T = 1..8 tokens each with and
without a pending write, every read on a different weight set out of a rotation
of 48 sets (630 MB of bf16 weights, larger than the 129 MB L2), so every read
streams its 13 MB of weights from HBM. ``value`` = microseconds per read, device
time from CUDA events around K steps (each step replayed as one CUDA graph;
inputs resident in HBM). ``e2e`` = the same reads through the public call (each
step's 16 calls captured as one CUDA graph) with each step's inputs copied from
pinned host memory and its outputs copied back inside the timed region; the copies
of neighbouring steps run on two copy streams beside the reads. Extra keys carry the 96-read cold round, per-T times and the
8K / 32K-token prefill chunks.

``--impl reference`` times the CPU oracle (float64, single thread) on a bounded
sample of the same sweep: it is the reference arm, not a GPU implementation.

Multi-GPU: the read does not shard (replicas only); with N ranks every rank runs
its own sweep and ``value`` = max-over-ranks time / all reads of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per hc read at 1-8 tokens and ms at 8K/32K; % of GB300 HBM roofline"
WEIGHT_BYTES = 320 * 10240 * 2 + 10240 * 320 * 2 + 4 * 2560 * 2   # 13,127,680
SWEEP = [(T, p) for T in range(1, 9) for p in (False, True)]      # 16 reads per step
N_SETS = 48
EPS = float(np.float32(1e-6))

# DRAM bytes (read + write) that ncu counted for one 4-token read with a pending
# write, both decode kernels together, on the current kernels; None when the
# kernels changed after the last capture. The sweep's traffic is taken as its
# algorithmic bytes times the ratio of this figure to the same read's algorithmic
# bytes. Capture (two reads, 48 rotated weight sets, so the weights come from DRAM):
# down_slice_kernel<4, 0> 6,918,912 B, up_mix_tc_kernel<4> 6,910,848 B, both reads,
# nothing written back to DRAM (the outputs stay in L2).
# GB300's nominal HBM3e bandwidth, GB/s (context beside the measured copy peak)
NOMINAL_HBM_GBS = 7900.0
NCU_TRAFFIC_T4_P = 13_829_376
NCU_TRAFFIC_LAST = "13,829,376 B per T=4 read with P (13,783,296 algorithmic)"


def read_bytes(T: int, with_P: bool) -> int:
    """Algorithmic bytes of one read: weights once, activations in, outputs out."""
    per_tok = 40960 + (40960 if with_P else 0) + 64 + 81920
    return WEIGHT_BYTES + T * per_tok


def prefill_upmix_bytes(T: int) -> int:
    """Algorithmic bytes of the fused up + gate + mix over T tokens (lo, R', Rmix in,
    the three outputs out, W_up once)."""
    return 10240 * 320 * 2 + T * (1280 + 40960 + 64 + 81920)


def prefill_read_bytes(T: int) -> int:
    """Algorithmic bytes of the whole prefill read (down + fused up/mix)."""
    return WEIGHT_BYTES + T * (40960 + 64 + 81920)


def reduce_max(value: float, world: int, device=None) -> float:
    """The largest of the ranks' values, returned on every rank (the slowest rank's
    time is the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def us_per_unit(ms_max: float, units_per_rank: int, world: int) -> float:
    """Whole-job microseconds per unit: the slowest rank's time over the units that
    all ranks processed (every rank runs the same number of units)."""
    return 1e3 * ms_max / (units_per_rank * world)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"hc_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle, single-threaded
# ---------------------------------------------------------------------------

_CPU_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from hyper_connection_residual_read_gb300 import synth
from oracle import hc_oracle as O
budget = float(sys.argv[1]); min_sweeps = int(sys.argv[2])
w = synth.make_weights(0)
cases = [(T, p) for T in range(1, 9) for p in (False, True)]
acts = [synth.make_activations(1 + i, T, p) for i, (T, p) in enumerate(cases)]
sweeps = []; t0 = time.perf_counter()
while len(sweeps) < min_sweeps or time.perf_counter() - t0 < budget:
    t1 = time.perf_counter()
    for a in acts:
        O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], {eps!r})
    sweeps.append(time.perf_counter() - t1)
print(json.dumps({{"sweep_seconds": sweeps, "reads_per_sweep": len(cases)}}))
"""


_CPU_PREFILL_SNIPPET = r"""
import json, multiprocessing as mp, os, sys
sys.path.insert(0, {root!r})
from hyper_connection_residual_read_gb300 import synth
from oracle.timing import timed_read

if __name__ == "__main__":
    n_tok = int(sys.argv[1])
    w = synth.make_weights(0)
    c = synth.make_prefill_chunk(100, n_tok)
    # one thread: the whole sample in one call (tokens are independent, so the time
    # scales linearly to a chunk)
    single = min(timed_read((c["R"], c["Rmix"], w, {eps!r})) for _ in range(2))
    # every core: the same sample split over one single-threaded process a core
    cores = len(os.sched_getaffinity(0))
    pieces = [(c["R"][i::cores].copy(), c["Rmix"][i::cores].copy(), w, {eps!r})
              for i in range(cores)]
    import time
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map_async(timed_read, pieces).get(timeout=300)   # warm-up: imports, first touch
        t0 = time.perf_counter()
        pool.map_async(timed_read, pieces).get(timeout=300)
        wall = time.perf_counter() - t0
    print(json.dumps({{"tokens": n_tok, "single_s": single, "all_cores_s": wall, "cores": cores}}))
"""


def run_oracle_prefill_sample(n_tok: int = 512) -> dict:
    """The oracle on a sample of prefill tokens, one thread and then one single-threaded
    process per host core, in a fresh process (started before nothing on the GPU)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = _CPU_PREFILL_SNIPPET.format(root=ROOT, eps=EPS)
    r = subprocess.run([sys.executable, "-c", code, str(n_tok)], capture_output=True, text=True,
                       env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle prefill sample failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_oracle_sample(budget_s: float, min_sweeps: int) -> dict:
    """Runs the oracle, single-threaded, in a fresh process over whole sweeps until
    both ``min_sweeps`` sweeps and ``budget_s`` seconds are done."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = _CPU_SNIPPET.format(root=ROOT, eps=EPS)
    r = subprocess.run([sys.executable, "-c", code, str(budget_s), str(min_sweeps)],
                       capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def reference_arm(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d = run_oracle_sample(0.0, args.warmup + args.steps)
    per_step = d["sweep_seconds"][args.warmup:]
    us = 1e6 * statistics.mean(per_step) / len(SWEEP)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/read",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(per_step), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config("CPU oracle, float64 numpy, one thread"),
        "cpu_baseline": {"value": us, "unit": "us/read", "cores": 1, "kind": "oracle",
                         "sample": "one verify-window sweep (16 reads, T=1..8 x {no P, P}) "
                                   "per step, one weight set, float64 numpy, 1 thread",
                         "cpu": cpu_model()},
        "e2e": {"value": us, "unit": "us/read", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def workload_config(launch: str = "one CUDA graph per step") -> dict:
    return {"workload": "verify-window sweep: T=1..8 tokens x {no pending write, pending "
                        "write}, 16 reads per step, 4x2560 fp32 residual, 10240->320->10240 "
                        "bf16 weights",
            "weight_sets": N_SETS, "l2": "weights rotated over 48 sets (630 MB > 129 MB L2)",
            "launch": launch}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args) -> None:
    import torch
    import torch.distributed as dist

    import hyper_connection_residual_read_gb300 as hc
    from hyper_connection_residual_read_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hc.hc_read_init(local, 32768, EPS)

    def to_dev(x, dtype=None):
        if x is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x))
        return t.to(dev)

    # weights: 48 sets; activations: one set per sweep case and rotation slot
    sets = []
    for k in range(N_SETS):
        w = synth.make_weights(7000 + 97 * rank + k)
        sets.append({n: to_dev(v) for n, v in w.items()})
    acts = []
    for i in range(N_SETS):
        T, p = SWEEP[i % len(SWEEP)]
        a = synth.make_activations(9000 + 97 * rank + i, T, p)
        acts.append({"T": T, "P": p, "host": a,
                     "R": to_dev(a["R"]), "Pd": to_dev(a["P"]), "M": to_dev(a["Rmix"])})
    outs = [tuple(torch.empty((T, 4, 2560), dtype=dt, device=dev)
                  for dt in (torch.float32, torch.int16, torch.int16))
            for (T, _p) in [(x["T"], x["P"]) for x in acts]]

    stream = torch.cuda.Stream(device=dev)
    n_groups = N_SETS // len(SWEEP)   # 3 steps cover the 48 rotation slots

    def enqueue_step(g: int):
        for j in range(len(SWEEP)):
            i = g * len(SWEEP) + j
            a, W = acts[i], sets[i]
            hc.hc_read(a["T"], a["R"], a["Pd"], W["w_norm"], W["W_down"], W["W_up"], a["M"],
                       *outs[i], stream=stream)

    # one graph per rotation group
    graphs = []
    with torch.cuda.stream(stream):
        for g in range(n_groups):
            enqueue_step(g)
        stream.synchronize()
        for g in range(n_groups):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                enqueue_step(g)
            graphs.append(gr)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, steps, warmup):
        """Device time of `steps` calls of fn on `stream`, after `warmup` calls."""
        with torch.cuda.stream(stream):
            for k in range(warmup):
                fn(k)
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k in range(steps):
                fn(k)
            e1.record(stream)
            barrier()
        return reduce_max(e0.elapsed_time(e1), world, dev)

    # --- main number: graph replays of the sweep ---
    with ClockSampler(local) as clk:
        ms = timed(lambda k: graphs[k % n_groups].replay(), args.steps, args.warmup)
    clocks = clk.summary()
    reads_per_step = len(SWEEP)
    us_per_read = us_per_unit(ms, args.steps * reads_per_step, world)
    step_bytes = sum(read_bytes(T, p) for T, p in SWEEP)

    # --- per-T times (graph of 48 reads of one T over the 48 sets), for each decode path ---
    def per_t_times(path, Ts, with_p=(False, True), warm=False):
        """µs per read at each T, 48 reads per graph: weights rotated over the 48 sets
        (cold, from HBM) or, with ``warm``, one set for every read (L2-resident)."""
        out = {}
        for T in Ts:
            for p in with_p:
                a0 = synth.make_activations(500 + T, T, p)
                R, Pd, M = to_dev(a0["R"]), to_dev(a0["P"]), to_dev(a0["Rmix"])
                o = tuple(torch.empty((T, 4, 2560), dtype=dt, device=dev)
                          for dt in (torch.float32, torch.int16, torch.int16))
                gr = torch.cuda.CUDAGraph()

                def enqueue():
                    for i in range(N_SETS):
                        W = sets[0 if warm else i]
                        hc.hc_read_path(path, T, R, Pd, W["w_norm"], W["W_down"], W["W_up"], M,
                                        *o, stream=stream)
                with torch.cuda.stream(stream):
                    enqueue()
                    stream.synchronize()
                    with torch.cuda.graph(gr, stream=stream):
                        enqueue()
                ms_t = timed(lambda k: gr.replay(), 40, 3)
                us = 1e3 * ms_t / (40 * N_SETS)
                out[f"T{T}{'_P' if p else ''}"] = {
                    "us": us, "gbps": read_bytes(T, p) / (us * 1e-6) / 1e9}
        return out

    per_t = per_t_times(hc.HC_PATH_AUTO, (1, 4, 8))
    # the same reads with one weight set (13 MB, resident in L2): the latency floor of
    # the kernels without the HBM weight stream
    per_t_warm = {k: round(v["us"], 2)
                  for k, v in per_t_times(hc.HC_PATH_DECODE, range(1, 9), (True,), warm=True).items()}
    per_t_paths = {name: {k: round(v["us"], 2) for k, v in per_t_times(path, range(1, 9), (True,)).items()}
                   for name, path in (("two_kernels", hc.HC_PATH_DECODE),
                                      ("one_kernel", hc.HC_PATH_DECODE_ONE_KERNEL))}

    # --- cold round: 96 reads of T=4 with P over the 48 sets ---
    a4 = synth.make_activations(600, 4, True)
    R4, P4, M4 = to_dev(a4["R"]), to_dev(a4["P"]), to_dev(a4["Rmix"])
    o4 = [tuple(torch.empty((4, 4, 2560), dtype=dt, device=dev)
                for dt in (torch.float32, torch.int16, torch.int16)) for _ in range(2)]
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        def round96():
            for i in range(96):
                W = sets[i % N_SETS]
                hc.hc_read(4, R4, P4, W["w_norm"], W["W_down"], W["W_up"], M4, *o4[i % 2],
                           stream=stream)
        round96()
        stream.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            round96()
    ms_r = timed(lambda k: gr.replay(), 20, 3)
    cold_round = {"us_per_round": 1e3 * ms_r / 20, "us_per_read": 1e3 * ms_r / 20 / 96,
                  "gbps": 96 * read_bytes(4, True) / (ms_r / 20 * 1e-3) / 1e9}

    # --- e2e: pinned host inputs -> device, 16 reads via the public call, outputs back.
    #     A step's inputs sit in one pinned buffer and go over in one copy; its outputs
    #     come back in one copy (how a caller would stage them). Two device buffer sets
    #     alternate between steps: step k+1's inputs go over on a copy stream while step
    #     k computes, and step k's outputs come back on another while step k+1 computes.
    #     Each step's reads are one CUDA graph of the public calls. ---
    in_off, out_off = [], []
    n_in = n_out = 0
    for T, p in SWEEP:
        sizes = {"R": T * 10240, "P": T * 10240 if p else 0, "Rmix": T * 16}
        offs = {}
        for key, n in sizes.items():
            offs[key] = (n_in, n) if n else None
            n_in += n
        in_off.append(offs)
        out_off.append((n_out, T))
        n_out += T * 10240
    pin_in = torch.empty(n_in, dtype=torch.float32).pin_memory()
    for j, offs in enumerate(in_off):
        a = acts[j]["host"]
        for key, o in offs.items():
            if o is not None:
                pin_in[o[0]:o[0] + o[1]].copy_(torch.from_numpy(np.ascontiguousarray(a[key]).reshape(-1)))
    pin_out = torch.empty(n_out * 8, dtype=torch.uint8).pin_memory()
    h2d, d2h = n_in * 4, n_out * 8
    dev_in = [torch.empty(n_in, dtype=torch.float32, device=dev) for _ in range(2)]
    # outputs: fp32 region, then the bf16 and fp16 regions, as bytes
    dev_out = [torch.empty(n_out * 8, dtype=torch.uint8, device=dev) for _ in range(2)]

    def step_views(b):
        o32 = dev_out[b][:n_out * 4].view(torch.float32)
        o16b = dev_out[b][n_out * 4:n_out * 6].view(torch.int16)
        o16h = dev_out[b][n_out * 6:].view(torch.int16)
        views = []
        for j, (T, p) in enumerate(SWEEP):
            offs, (oo, _) = in_off[j], out_off[j]
            v = {key: (dev_in[b][o[0]:o[0] + o[1]] if o is not None else None)
                 for key, o in offs.items()}
            views.append((v, o32[oo:oo + T * 10240], o16b[oo:oo + T * 10240],
                          o16h[oo:oo + T * 10240]))
        return views

    e2e_views = [step_views(b) for b in range(2)]

    def enqueue_reads(g, b):
        for j in range(len(SWEEP)):
            v, f32, b16, h16 = e2e_views[b][j]
            W = sets[g * len(SWEEP) + j]
            hc.hc_read(SWEEP[j][0], v["R"], v["P"], W["w_norm"], W["W_down"], W["W_up"],
                       v["Rmix"], f32, b16, h16, stream=stream)

    stream_handle = stream.cuda_stream
    e2e_args = {}
    for g in range(n_groups):
        for b in range(2):
            rows = []
            for j in range(len(SWEEP)):
                v, f32, b16, h16 = e2e_views[b][j]
                W = sets[g * len(SWEEP) + j]
                rows.append((SWEEP[j][0], v["R"], v["P"], W["w_norm"], W["W_down"], W["W_up"],
                             v["Rmix"], f32, b16, h16))
            e2e_args[(g, b)] = rows
    e2e_graphs = {}
    with torch.cuda.stream(stream):
        for g in range(n_groups):
            for b in range(2):
                enqueue_reads(g, b)
        stream.synchronize()
        for g in range(n_groups):
            for b in range(2):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=stream):
                    enqueue_reads(g, b)
                e2e_graphs[(g, b)] = gr
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    ev = {(kind, b): torch.cuda.Event() for kind in ("in", "done", "out") for b in range(2)}
    for b in range(2):   # every buffer starts free
        for kind in ("done", "out"):
            ev[(kind, b)].record(stream)

    def e2e_step(k, graphed=True):
        b = k % 2
        # inputs of this step into buffer b once the step that last read it is done
        h2d_stream.wait_event(ev[("done", b)])
        with torch.cuda.stream(h2d_stream):
            dev_in[b].copy_(pin_in, non_blocking=True)
        ev[("in", b)].record(h2d_stream)
        # the reads, once the inputs are over and buffer b's last outputs have left
        stream.wait_event(ev[("in", b)])
        stream.wait_event(ev[("out", b)])
        if graphed:
            with torch.cuda.stream(stream):   # a graph replays on the current stream
                e2e_graphs[(k % n_groups, b)].replay()
        else:
            # the 16 public calls, launched one by one on the stream they name, with
            # each read's arguments held as a caller holds its tensors
            for args in e2e_args[(k % n_groups, b)]:
                hc.hc_read(*args, stream=stream_handle)
        ev[("done", b)].record(stream)
        # the outputs back while the next step computes
        d2h_stream.wait_event(ev[("done", b)])
        with torch.cuda.stream(d2h_stream):
            pin_out.copy_(dev_out[b], non_blocking=True)
        ev[("out", b)].record(d2h_stream)

    def e2e_run(steps, warmup, graphed=True):
        """Device time of `steps` pipelined steps, from the first copy to the last
        output back on the host, after `warmup` steps."""
        for k in range(warmup):
            e2e_step(k, graphed)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        for k in range(warmup, warmup + steps):
            e2e_step(k, graphed)
        stream.wait_stream(d2h_stream)
        e1.record(stream)
        barrier()
        return reduce_max(e0.elapsed_time(e1), world, dev)

    e2e_steps = max(10, min(args.steps, 500))
    ms_e = e2e_run(e2e_steps, min(args.warmup, 5) + 3)
    # the same pipelined steps with every read a direct call (no CUDA graph): the
    # host's launch work per call is then on the path
    ms_e_direct = e2e_run(e2e_steps, min(args.warmup, 5) + 3, graphed=False)

    def e2e_serial_step(k):
        # the same step with copies and reads in order on one stream: no overlap
        with torch.cuda.stream(stream):
            dev_in[0].copy_(pin_in, non_blocking=True)
            e2e_graphs[(k % n_groups, 0)].replay()
            pin_out.copy_(dev_out[0], non_blocking=True)

    ms_e_serial = timed(e2e_serial_step, e2e_steps, 3)
    e2e_us = us_per_unit(ms_e, e2e_steps * reads_per_step, world)

    # --- prefill chunks: the whole read, and the fused up + gate + mix stage alone
    #     (re-run on the chunk's lo) next to the unfused pair (up GEMM writing gated,
    #     then the mix) in the same build ---
    prefill = {}
    peaks = measured_peaks()
    W0 = sets[0]
    for T in (8192, 32768):
        c = synth.make_prefill_chunk(104 if T == 32768 else 100, T)
        R, M = to_dev(c["R"]), to_dev(c["Rmix"])
        o = tuple(torch.empty((T, 4, 2560), dtype=dt, device=dev)
                  for dt in (torch.float32, torch.int16, torch.int16))

        def chunk(k):
            hc.hc_read(T, R, None, W0["w_norm"], W0["W_down"], W0["W_up"], M, *o,
                       stream=stream)

        def upmix_fused(k):
            hc.hc_read_upmix(hc.HC_PATH_PREFILL, T, R, None, W0["W_up"], M, *o, stream=stream)

        def upmix_pair(k):
            hc.hc_read_upmix(hc.HC_PATH_PREFILL_UNFUSED, T, R, None, W0["W_up"], M, *o,
                             stream=stream)

        def chunk_bf16(k):
            hc.hc_read_path(hc.HC_PATH_PREFILL_BF16_LO, T, R, None, W0["w_norm"], W0["W_down"],
                            W0["W_up"], M, *o, stream=stream)

        def upmix_bf16(k):
            hc.hc_read_upmix(hc.HC_PATH_PREFILL_BF16_LO, T, R, None, W0["W_up"], M, *o,
                             stream=stream)

        reps = 10 if T == 8192 else 4
        ms_read = timed(chunk, reps, 3) / reps          # leaves this chunk's lo in scratch
        ms_fused = timed(upmix_fused, reps, 3) / reps
        ms_pair = timed(upmix_pair, reps, 3) / reps
        oy = tuple(torch.empty((T, 2560), dtype=dt, device=dev)
                   for dt in (torch.float32, torch.int16, torch.int16))

        def chunk_y(k):
            hc.hc_read_y(T, R, None, W0["w_norm"], W0["W_down"], W0["W_up"], *oy, stream=stream)

        ms_read_y = timed(chunk_y, reps, 3) / reps      # the 2560-wide read-out
        del oy
        ms_read16 = timed(chunk_bf16, reps, 3) / reps   # the pages' bf16-lo numerics
        ms_up16 = timed(upmix_bf16, reps, 3) / reps
        fused_gbps = prefill_upmix_bytes(T) / (ms_fused * 1e-3) / 1e9
        # the bf16-lo stage reads lo as one bf16 term (640 B per token instead of 1,280)
        up16_gbps = (prefill_upmix_bytes(T) - 640 * T) / (ms_up16 * 1e-3) / 1e9
        prefill[f"T{T}"] = {
            "read_ms": ms_read, "tokens_per_s": T / (ms_read * 1e-3),
            "read_gbps": prefill_read_bytes(T) / (ms_read * 1e-3) / 1e9,
            "upmix_fused_ms": ms_fused, "upmix_fused_gbps": fused_gbps,
            "upmix_fused_frac": fused_gbps / peaks["hbm_gbs"],
            "upmix_unfused_pair_ms": ms_pair, "fused_speedup": ms_pair / ms_fused,
            "bf16_lo_read_ms": ms_read16, "bf16_lo_upmix_ms": ms_up16,
            "bf16_lo_upmix_frac": up16_gbps / peaks["hbm_gbs"],
            "readout_y_read_ms": ms_read_y,
            "readout_y_read_gbps": (WEIGHT_BYTES + T * (40960 + 20480)) / (ms_read_y * 1e-3) / 1e9}
        del R, M, o

    # --- decode / prefill crossover: both paths on the same reads (one weight set,
    #     pending write, the tokens of one chunk), µs per read ---
    crossover = {}
    c = synth.make_prefill_chunk(105, 256)
    Rc, Mc = to_dev(c["R"]), to_dev(c["Rmix"])
    Pc = to_dev((0.1 * np.random.default_rng(106).standard_normal(c["R"].shape)).astype(np.float32))
    for T in (8, 9, 16, 24, 32, 48, 64, 128, 256):
        o = tuple(torch.empty((T, 4, 2560), dtype=dt, device=dev)
                  for dt in (torch.float32, torch.int16, torch.int16))
        row = {}
        for name, path in (("decode", hc.HC_PATH_DECODE), ("prefill", hc.HC_PATH_PREFILL)):
            # 20 reads per CUDA graph: device time, as an engine that captures its
            # step sees it (without the graph the tile path's host launch cost shows)
            def enqueue(path=path):
                for _ in range(20):
                    hc.hc_read_path(path, T, Rc, Pc, W0["w_norm"], W0["W_down"], W0["W_up"],
                                    Mc, *o, stream=stream)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                enqueue()
                stream.synchronize()
                with torch.cuda.graph(gr, stream=stream):
                    enqueue()
            row[name] = 1e3 * timed(lambda k: gr.replay(), 10, 2) / 200
        crossover[f"T{T}"] = row
    del Rc, Mc, Pc

    achieved = step_bytes / (ms / args.steps * 1e-3) / 1e9
    traffic = (None if NCU_TRAFFIC_T4_P is None
               else step_bytes * NCU_TRAFFIC_T4_P / read_bytes(4, True))
    kernel_launches_per_step = sum(2 * ((T + 7) // 8) for T, _ in SWEEP)

    line = {
        "metric": METRIC, "value": us_per_read, "unit": "us/read", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(),
        "roofline": {"bound": "hbm", "kernel": "decode read (down_slice + up_mix_tc kernels)",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "traffic_basis": ("ncu DRAM bytes of one T=4 read with P, scaled to the "
                                       "sweep by algorithmic bytes" if traffic is not None else
                                       "null: the kernels changed after the last ncu capture; "
                                       "that capture: " + NCU_TRAFFIC_LAST),
                     "peak_source": peaks["source"],
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "bytes_per_step": step_bytes},
        "clocks": clocks,
        "e2e": {"value": e2e_us, "unit": "us/read", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelining": "step k+1's inputs and step k-1's outputs cross on two copy "
                              "streams while step k computes",
                "serial_us": us_per_unit(ms_e_serial, e2e_steps * reads_per_step, world),
                "ungraphed_us": us_per_unit(ms_e_direct, e2e_steps * reads_per_step, world),
                "ungraphed": "the same pipelined steps, each read a direct hc_read call "
                             "(no CUDA graph)"},
        "gpu_launches": kernel_launches_per_step * args.steps,
        "decode_by_T": per_t,
        "decode_paths_us_by_T_with_P": per_t_paths,
        "decode_warm_weights_us_by_T_with_P": per_t_warm,
        "cold_round_96x_T4_P": cold_round,
        "prefill": prefill,
        "crossover_us_per_read": crossover,
    }
    if rank == 0:
        if not args.no_cpu_baseline:
            d = run_oracle_sample(args.cpu_seconds, 1)
            n = len(d["sweep_seconds"]) * d["reads_per_sweep"]
            line["cpu_baseline"] = {
                "value": 1e6 * sum(d["sweep_seconds"]) / n, "unit": "us/read", "cores": 1,
                "kind": "oracle", "cpu": cpu_model(),
                "sample": f"{n} reads ({len(d['sweep_seconds'])} sweeps of T=1..8 x "
                          "{no P, P}, one weight set), float64 numpy, 1 thread"}
            # the prefill chunks: a sample of tokens, extrapolated linearly
            pf = run_oracle_prefill_sample(512)
            per_tok_1, per_tok_n = pf["single_s"] / pf["tokens"], pf["all_cores_s"] / pf["tokens"]
            line["cpu_baseline_prefill"] = {
                "kind": "oracle", "cpu": cpu_model(), "unit": "ms per chunk",
                "T8192": {"single_thread_ms": 1e3 * per_tok_1 * 8192,
                          "all_cores_ms": 1e3 * per_tok_n * 8192},
                "T32768": {"single_thread_ms": 1e3 * per_tok_1 * 32768,
                           "all_cores_ms": 1e3 * per_tok_n * 32768},
                "cores": pf["cores"],
                "sample": f"{pf['tokens']} tokens of a prefill chunk (R ~ N(0,1), no P), float64 "
                          "numpy, timed on one thread and on one single-threaded process per "
                          "core, extrapolated linearly to the chunk (tokens are independent)"}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def profile_decode(args, path=None) -> None:
    """A small fixed decode workload for ncu: 48 rotated weight sets (larger than
    L2), ``--steps`` reads of T=4 tokens with a pending write (``path``: a forced
    HC_PATH_*, else the default choice). No timing."""
    import torch
    import hyper_connection_residual_read_gb300 as hc
    from hyper_connection_residual_read_gb300 import synth
    hc.hc_read_init(0, 64, EPS)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(  # noqa: E731
        x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
    sets = [{k: dev(v) for k, v in synth.make_weights(7000 + k).items()} for k in range(N_SETS)]
    a = synth.make_activations(600, 4, True)
    R, P, M = dev(a["R"]), dev(a["P"]), dev(a["Rmix"])
    o = [torch.empty((4, 4, 2560), dtype=dt, device="cuda")
         for dt in (torch.float32, torch.int16, torch.int16)]
    for i in range(args.steps):
        W = sets[i % N_SETS]
        if path is None:
            hc.hc_read(4, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
        else:
            hc.hc_read_path(path, 4, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    torch.cuda.synchronize()
    rc = hc.hc_read_status()
    print(json.dumps({"profile": "decode", "reads": args.steps, "status": rc}))


def profile_prefill(args) -> None:
    """A fixed prefill workload for ncu: ``--steps`` reads of one 8,192-token chunk
    (fused path), then one read through the unfused pair. No timing."""
    import torch
    import hyper_connection_residual_read_gb300 as hc
    from hyper_connection_residual_read_gb300 import synth
    T = 8192
    hc.hc_read_init(0, T, EPS)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(  # noqa: E731
        x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
    W = {k: dev(v) for k, v in synth.make_weights(0).items()}
    c = synth.make_prefill_chunk(100, T)
    R, M = dev(c["R"]), dev(c["Rmix"])
    o = [torch.empty((T, 4, 2560), dtype=dt, device="cuda")
         for dt in (torch.float32, torch.int16, torch.int16)]
    for _ in range(args.steps):
        hc.hc_read_path(hc.HC_PATH_PREFILL, T, R, None, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    hc.hc_read_path(hc.HC_PATH_PREFILL_UNFUSED, T, R, None, W["w_norm"], W["W_down"], W["W_up"],
                    M, *o)
    torch.cuda.synchronize()
    print(json.dumps({"profile": "prefill", "reads": args.steps, "status": hc.hc_read_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["decode", "decode1", "prefill"], default=None,
                    help="run a small fixed workload for an ncu capture instead of timing")
    args = ap.parse_args()
    if args.profile == "decode":
        profile_decode(args)
    elif args.profile == "decode1":      # the one-kernel decode read
        profile_decode(args, path=4)
    elif args.profile == "prefill":
        profile_prefill(args)
    elif args.impl == "reference":
        # each reference step is a whole 16-read oracle sweep (about a second)
        args.steps = max(1, min(args.steps, 20))
        args.warmup = max(1, min(args.warmup, 3))
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
