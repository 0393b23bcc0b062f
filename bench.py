#!/usr/bin/env python3
"""Benchmark: chunked causal linear attention, forward + backward, on GB300.

One step = the whole hot path over one batch: la_chunked_fwd then la_chunked_bwd on
the Fractus-1B block shape (B=4, levels=2, heads=20 -> G=160 groups, C=128 tokens,
head size D=64, block=64, bf16 inputs, fp32 carry, carry active), synthetic seeded
inputs.  Metric: G*C tokens per second (groups x tokens processed per second).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timed region: W eager warm-up steps, then EXACTLY K steps replayed from CUDA graphs,
bracketed by a barrier and cudaDeviceSynchronize, timed with CUDA events on the
launching stream, max over ranks.  The steps cycle through enough input/output buffer
sets that the working set is over 4x the L2 size, so every step reads HBM.
One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = dict(G=160, C=128, D=64, block=64, dtype="bf16", eps=1e-6)
WORKLOAD_NAME = "fractus1b_block: G=160 (B=4 x 2 levels x 20 heads), C=128, D=64, block=64, bf16, fwd+bwd"
METRIC = "linear-attn tokens·groups/s (G·C/s) fwd and fwd+bwd; % of binding roofline"
UNIT = "G·C tokens/s"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per launch from one ncu capture of each kernel on this workload
# (dram__bytes_read.sum, dram__bytes_write.sum), with the hash of the kernel sources they were
# taken on; reported as null once the sources differ.  A single launch's outputs are still in
# L2 when it ends (they are written back to DRAM later), so the write counter of one launch
# reads ~0: the line carries both counters and says so.
NCU_TRAFFIC = {
    "la_fwd": {"read": 10562560, "write": 0, "l2_write": 7974080, "src": "bb92639dca406800"},
    "la_bwd": {"read": 15877760, "write": 0, "l2_write": 15799488, "src": "82c52753b6c829a2"},
}


# GB300's nominal HBM3e bandwidth (GB/s), reported beside the measured copy rate.
NOMINAL_HBM_GBS = 7900.0


# The headers that make up each timed kernel (its body and everything it includes).
KERNEL_FILES = {
    "la_fwd": ("la_fwd_tile.cuh", "la_fwd_tc.cuh", "la_tc.cuh", "la_device.cuh"),
    "la_bwd": ("la_bwd_tile.cuh", "la_fwd_tc.cuh", "la_tc.cuh", "la_device.cuh"),
}


def kernel_source_hash(kernel):
    """Hash of the sources of one timed kernel: ncu traffic taken from another build of it
    is not reported."""
    import hashlib
    csrc = os.path.join(ROOT, "causal_linear_attention_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_FILES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(G, C, D, esz):
    """Bytes a launch must move at minimum (each input read once, each output written once)."""
    state = (D * D + D) * 4
    fwd = G * (3 * C * D * esz + C * D * esz + 2 * state)            # q,k,v in; o out; carry in + out
    bwd = G * (4 * C * D * esz + 2 * state + 3 * C * D * esz + state)  # q,k,v,dO,S0,z0,dS,dz in; dq,dk,dv,dS0,dz0 out
    return fwd, bwd


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """The dense bf16 GEMM rate of MEASURED_PEAKS.json (burst), TFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measure_chunked_ce(stream):
    """The chunked cross-entropy of the tied head (N = 512 tokens, V = 50257, d = 1280,
    bf16; one chunk of 512 and chunks of 128): device time per call of la_ce_fwd and
    la_ce_bwd, CUDA graphs of 10 calls.  Its binding roofline is the tensor pipe: the GEMM
    FLOPs (2 N V d forward; the recomputed logits plus dh and dW, 6 N V d, backward)
    against the measured bf16 dense rate."""
    import torch

    import causal_linear_attention_gb300 as la
    from causal_linear_attention_gb300.inputs import CE_SHAPE, make_ce_inputs
    dev = stream.device
    N, V, d = CE_SHAPE["N"], CE_SHAPE["V"], CE_SHAPE["d"]
    h, W, y = (t.to(dev) for t in make_ce_inputs(N, V, d, seed=rank_seed(0)))
    peak, src = measured_bf16_peak()
    out = {"N": N, "V": V, "d": d, "dtype": "bf16",
           "api": "la_ce_fwd / la_ce_bwd (logits on this library's tcgen05 kernel with the log-sum-exp or the "
                  "gradient in its epilogue; dh, dW on its persistent tcgen05 GEMM)"}
    for chunk in (512, 128):
        ws = la.ce_workspace(N, V, d, chunk, dev)
        loss = torch.empty((), dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        dh = torch.empty_like(h)
        dW = torch.empty(V, d, dtype=torch.float32, device=dev)
        calls = {
            "fwd": lambda: la.la_ce_fwd(h, W, y, N, V, d, chunk, loss, lse, ws, ws.numel(), stream.cuda_stream),
            "bwd": lambda: la.la_ce_bwd(h, W, y, lse, 1.0, N, V, d, chunk, dh, dW, ws, ws.numel(), stream.cuda_stream),
        }
        entry = {}
        for name, fn in calls.items():
            with torch.cuda.stream(stream):
                for _ in range(3):
                    fn()
            torch.cuda.synchronize()
            n = 10
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                for _ in range(n):
                    fn()
            gph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                gph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / n
            flop = (2 if name == "fwd" else 6) * N * V * d
            tf = flop / us / 1e6
            entry[name] = {"us": round(us, 2), "tflops": round(tf, 1), "frac": round(tf / peak, 4)}
        out[f"ce_chunk={chunk}"] = entry
        del ws, dW
    out["roofline"] = {"bound": "tensor", "peak_tflops": peak, "peak_source": src}
    torch.cuda.empty_cache()
    return out


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(rank):
    """Each rank draws its own groups: weak scaling over independent groups, no collective
    in the data path."""
    return 1000 + rank


def max_over_ranks(x, world, device="cpu"):
    """The slowest rank's time (the job's time); a no-op on one rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_value(world, G, C, steps, secs):
    """Whole-job throughput: the G*C tokens every rank processed in each step / the job time."""
    return world * G * C * steps / secs


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ---------------------------------------------------------------- clocks during the timed region
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        if not rows:
            return None
        t0, t1 = self.window or (rows[0][0], rows[-1][0])
        inside = [p for t, p in rows if t0 - 0.1 <= t <= t1 + 0.1] or [rows[-1][1]]
        sm = [float(p[1]) for p in inside if p[1].replace(".", "", 1).isdigit()]
        smax = [float(p[2]) for p in inside if p[2].replace(".", "", 1).isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in inside for n, val in zip(names, p[5:9]) if val.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------- our arm (GPU)
class StepBuffers:
    """Device inputs and outputs of one step."""

    def __init__(self, src, G, C, D):
        import torch
        self.x = src
        self.o = torch.empty_like(src.q)
        self.S_out = torch.empty(G, D, D, device=src.q.device, dtype=torch.float32)
        self.z_out = torch.empty(G, D, device=src.q.device, dtype=torch.float32)
        self.grads = (torch.empty_like(src.q), torch.empty_like(src.q), torch.empty_like(src.q),
                      torch.empty(G, D, D, device=src.q.device, dtype=torch.float32),
                      torch.empty(G, D, device=src.q.device, dtype=torch.float32))

    def nbytes(self):
        ts = list(self.x.tensors().values()) + [self.o, self.S_out, self.z_out, *self.grads]
        return sum(t.numel() * t.element_size() for t in ts)


def run_ours(args, rank, world, local):
    import torch

    import causal_linear_attention_gb300 as la
    from causal_linear_attention_gb300.inputs import Inputs, make_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    la.build()
    G, C, D, block, eps = (WORKLOAD[k] for k in ("G", "C", "D", "block", "eps"))
    esz = 2
    fwd_bytes, bwd_bytes = algorithmic_bytes(G, C, D, esz)

    # one seeded set of inputs (each rank draws its own groups), replicated into enough
    # buffer sets that the rotation touches > 4x L2 between two uses of a set
    host = make_inputs(G, C, D, dtype="bf16", seed=rank_seed(rank), grads=True)
    base = host.to(dev)
    one = StepBuffers(base, G, C, D)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, -(-4 * l2 // one.nbytes()))
    sets = [one] + [StepBuffers(Inputs(**{k: (None if t is None else t.clone()) for k, t in base.__dict__.items()}),
                                G, C, D) for _ in range(nsets - 1)]

    def fwd(b):
        la.chunked_fwd(b.x.q, b.x.k, b.x.v, b.x.S0, b.x.z0, block=block, eps=eps, o=b.o, S_out=b.S_out,
                       z_out=b.z_out)

    def bwd(b):
        la.chunked_bwd(b.x.q, b.x.k, b.x.v, b.x.S0, b.x.z0, b.x.dO, b.x.dS_out, b.x.dz_out, block=block, eps=eps,
                       out=b.grads)

    def step(b):
        fwd(b)
        bwd(b)

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(sets[i % nsets])
    torch.cuda.synchronize()

    def capture(fn, n, offset=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(sets[(offset + i) % nsets])
        return g

    chunk = min(args.steps, 512)

    def timed(fn, steps):
        """Replay `steps` calls of fn from CUDA graphs; returns device seconds (this rank)."""
        full, rest = divmod(steps, chunk)
        g_full = capture(fn, chunk) if full else None
        g_rest = capture(fn, rest, offset=full * chunk) if rest else None
        if g_full is not None:  # one untimed replay: graph upload / first-launch costs
            g_full.replay()
        torch.cuda.synchronize()
        bar()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(full):
                g_full.replay()
            if g_rest is not None:
                g_rest.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        bar()
        return e0.elapsed_time(e1) / 1e3

    bar = lambda: barrier(world)
    mor = lambda x: max_over_ranks(x, world, dev)

    clocks = ClockSampler(local)
    clocks.start()
    t_wall0 = time.time()
    secs = mor(timed(step, args.steps))
    clocks.mark(t_wall0, time.time())
    clock_info = clocks.stop()

    # per-kernel average launch durations (same rotation, same stream)
    n_k = max(args.steps, 64)
    fwd_secs = mor(timed(fwd, n_k)) / n_k
    bwd_secs = mor(timed(bwd, n_k)) / n_k

    # end to end through the public API: pinned host inputs -> device -> fwd + bwd -> host outputs
    e2e = run_e2e(args, host, G, C, D, block, eps, local, bar, mor)

    value = job_value(world, G, C, args.steps, secs)
    hbm, peak_src = measured_peaks()
    kernels = {
        "la_fwd": {"avg_us": fwd_secs * 1e6, "alg_bytes": fwd_bytes, "gbs": fwd_bytes / fwd_secs / 1e9},
        "la_bwd": {"avg_us": bwd_secs * 1e6, "alg_bytes": bwd_bytes, "gbs": bwd_bytes / bwd_secs / 1e9},
    }
    dom = max(kernels, key=lambda k: kernels[k]["avg_us"])
    src_hash = kernel_source_hash(dom)
    traffic = NCU_TRAFFIC.get(dom)
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(kernels[dom]["gbs"], 1), "peak": hbm,
            "unit": "GB/s", "frac": round(kernels[dom]["gbs"] / hbm, 4), "peak_source": peak_src,
            "traffic": traffic["read"] + traffic["write"] if traffic and traffic["src"] == src_hash else None,
            "traffic_counters": ({"dram__bytes_read.sum": traffic["read"], "dram__bytes_write.sum": traffic["write"],
                                  "lts__t_sectors_op_write.sum_bytes": traffic["l2_write"],
                                  "note": "one ncu-captured launch; its outputs are still in L2 when it ends and "
                                          "reach DRAM later, so the write counter of a single launch reads ~0; "
                                          "the L2 write sectors (x 32 B) show the writes the launch made"}
                                 if traffic and traffic["src"] == src_hash else None),
            "alg_bytes": kernels[dom]["alg_bytes"],
            "frac_of_nominal": round(kernels[dom]["gbs"] / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS}
    for k in kernels:
        kernels[k]["frac"] = round(kernels[k]["gbs"] / hbm, 4)
        kernels[k]["avg_us"] = round(kernels[k]["avg_us"], 3)
        kernels[k]["gbs"] = round(kernels[k]["gbs"], 1)
    fwd_only = job_value(world, G, C, 1, fwd_secs)
    others = measure_other_configs(stream, eps, hbm) if rank == 0 else None
    if others is not None:
        others["chunked_ce_fwdbwd: N=512 tokens, V=50257, d=1280, bf16 (tied head)"] = measure_chunked_ce(stream)

    out = None
    if rank == 0:
        cpu = cpu_baseline(host, G, C, D, eps)
        cpu_torch = cpu_torch_fp32(host, G, C, D, block, eps)
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "G_per_gpu": G, "C": C, "D": D, "block": block, "eps": eps,
                       "step": "la_chunked_fwd + la_chunked_bwd", "parallelism": f"groups sharded, {world} rank(s)",
                       "l2": f"rotating {nsets} buffer sets ({nsets * one.nbytes() / 2**20:.0f} MiB > 4x L2 "
                             f"{l2 / 2**20:.0f} MiB)", "timing": "CUDA graphs, CUDA events, max over ranks"},
            "fwd_only": {"value": fwd_only, "unit": UNIT, "us_per_launch": kernels["la_fwd"]["avg_us"]},
            "roofline": roof, "kernels": kernels, "e2e": e2e, "gpu_launches": 2 * args.steps,
            "clocks": clock_info, "cpu_baseline": cpu, "cpu_torch_fp32": cpu_torch, "other_configs": others,
        }
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


def gpu_local_cpus(local):
    """CPUs of the NUMA node the GPU is attached to (Linux sysfs), intersected with this
    process's allowed CPUs; None when that cannot be determined."""
    import torch
    props = torch.cuda.get_device_properties(local)
    if hasattr(props, "pci_bus_id"):
        bus = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    else:
        try:
            cudart = ctypes.CDLL(os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64",
                                              "libcudart.so"))
        except OSError:
            return None
        buf = ctypes.create_string_buffer(64)
        if cudart.cudaDeviceGetPCIBusId(buf, 64, local) != 0:
            return None
        bus = buf.value.decode().lower()
    try:
        node = int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read().strip())
        if node < 0:
            return None
        cpus = set()
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
    except (OSError, ValueError):
        return None
    cpus &= os.sched_getaffinity(0)
    return cpus or None


# The other workloads (parity cases in tests/), measured the same way as the headline's
# per-kernel numbers, for context: (name, G, C, D, block, directions, implementation).
# "threaded" runs the C tokens as C / 128 launches of 128 tokens each, the carry passed
# from launch to launch in place; its bytes count every launch's carry round trip.
THREAD_CHUNK = 128
OTHER_CONFIGS = (
    ("batch16_fwdbwd: G=640, C=128, D=64, block=64, bf16", 640, 128, 64, 64, ("fwd", "bwd"), "chunked"),
    ("long_stream_fwd: G=160, T=8192 as one C=8192 launch, D=64, bf16", 160, 8192, 64, 64, ("fwd",), "chunked"),
    ("long_stream_threaded_fwd: G=160, T=8192 as 64 launches of C=128, carry threaded in place, D=64, bf16", 160,
     8192, 64, 64, ("fwd",), "threaded"),
    ("wide_heads_fwdbwd: G=320, C=256, D=128, block=64, bf16", 320, 256, 128, 64, ("fwd", "bwd"), "chunked"),
    ("wide_heads_ragged_fwdbwd: G=320, C=200, D=128, block=64, bf16", 320, 200, 128, 64, ("fwd", "bwd"), "chunked"),
    ("wide_heads_block128_fwdbwd: G=320, C=256, D=128, block=128, bf16", 320, 256, 128, 128, ("fwd", "bwd"),
     "chunked"),
    ("cumsum_form_fwdbwd: G=160, C=128, D=64, bf16, token-by-token scan", 160, 128, 64, 64, ("fwd", "bwd"),
     "cumsum"),
    ("few_groups_wide_heads_fwdbwd: G=8, C=8192, D=128, bf16, one CTA per group", 8, 8192, 128, 64,
     ("fwd", "bwd"), "chunked"),
    ("few_groups_wide_heads_split_fwdbwd: G=8, C=8192, D=128, bf16, chunk-parallel (la_chunked_fwd_split, "
     "la_chunked_bwd_split)", 8, 8192, 128, 64, ("fwd", "bwd"), "split"),
)

# The cumsum form runs on the CUDA cores: its bound is fp32 FMA issue, 128 FMA lanes per
# SM at the maximum SM clock (2 FLOP per FMA).
FP32_LANES_PER_SM = 128
MAX_SM_MHZ = 2070.0


def cumsum_flop(G, C, D):
    """Algorithmic FLOP of the cumsum form per launch: each token updates the D x D state
    and reads it out once per sweep (2 D^2 FMA); the forward makes one sweep, the backward
    four (n and den; R with dv; S with dq; R with dk).  The length-D sums (z, q.z, r) are
    left out."""
    per_sweep = 2 * D * D * 2
    return G * C * per_sweep, G * C * 4 * per_sweep


def measure_other_configs(stream, eps, hbm):
    """Per-launch device time of each direction on the other workloads: CUDA graphs of 20
    launches over enough buffer sets that the working set exceeds 4x L2."""
    import torch

    import causal_linear_attention_gb300 as la
    from causal_linear_attention_gb300.inputs import make_inputs
    dev = stream.device
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    props = torch.cuda.get_device_properties(dev)
    alu_peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * MAX_SM_MHZ * 1e6 / 1e12  # TFLOP/s
    for name, G, C, D, block, dirs, impl in OTHER_CONFIGS:
        x = make_inputs(G, C, D, dtype="bf16", seed=rank_seed(0), grads="bwd" in dirs).to(dev)
        fb, bb = algorithmic_bytes(G, C, D, 2)
        if impl == "threaded":
            nch = C // THREAD_CHUNK
            fb = nch * algorithmic_bytes(G, THREAD_CHUNK, D, 2)[0]
        nsets = max(1, min(8, -(-4 * l2 // (fb + (bb if "bwd" in dirs else 0)))))
        sets = []
        for _ in range(nsets):
            d = {k: (None if t is None else t.clone()) for k, t in x.__dict__.items()}
            o = (torch.empty_like(x.q), torch.empty(G, D, D, device=dev), torch.empty(G, D, device=dev))
            gr = (torch.empty_like(x.q), torch.empty_like(x.q), torch.empty_like(x.q), torch.empty(G, D, D, device=dev),
                  torch.empty(G, D, device=dev)) if "bwd" in dirs else None
            ws = None
            if impl == "cumsum" and "bwd" in dirs:
                ws = torch.empty(la.la_cumsum_bwd_workspace_bytes(G, C, D, la.LA_BF16), dtype=torch.uint8, device=dev)
            if impl == "split":  # one workspace serves both directions (the calls are stream-ordered)
                ws = torch.empty(max(1, la.la_fwd_split_workspace_bytes(G, C, D, la.LA_BF16),
                                     la.la_bwd_split_workspace_bytes(G, C, D, la.LA_BF16)), dtype=torch.uint8,
                                 device=dev)
            if impl == "threaded":  # contiguous [G][128][D] pieces of q, k, v; o as 64 pieces
                for key in ("q", "k", "v"):
                    d[key] = [t.contiguous() for t in d[key].split(THREAD_CHUNK, dim=1)]
                o = ([t.contiguous() for t in o[0].split(THREAD_CHUNK, dim=1)], o[1], o[2])
            sets.append((d, o, gr, ws))
        entry = {"G": G, "C": C, "D": D, "block": block, "impl": impl}
        for direction in dirs:
            def call(i, direction=direction):
                d, o, gr, ws = sets[i % nsets]
                if impl == "cumsum" and direction == "fwd":
                    la.cumsum_fwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], eps=eps, o=o[0], S_out=o[1], z_out=o[2])
                elif impl == "threaded":  # the first piece reads S0, z0; the rest the carry in place
                    for c, (qc, kc, vc, oc) in enumerate(zip(d["q"], d["k"], d["v"], o[0])):
                        S_in, z_in = (d["S0"], d["z0"]) if c == 0 else (o[1], o[2])
                        la.chunked_fwd(qc, kc, vc, S_in, z_in, block=block, eps=eps, o=oc, S_out=o[1], z_out=o[2])
                elif impl == "split" and direction == "fwd":
                    la.chunked_fwd_split(d["q"], d["k"], d["v"], d["S0"], d["z0"], block=block, eps=eps, o=o[0],
                                         S_out=o[1], z_out=o[2], workspace=ws)
                elif impl == "split":
                    la.chunked_bwd_split(d["q"], d["k"], d["v"], d["S0"], d["z0"], d["dO"], d["dS_out"], d["dz_out"],
                                         block=block, eps=eps, out=gr, workspace=ws)
                elif impl == "cumsum":
                    la.cumsum_bwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], d["dO"], d["dS_out"], d["dz_out"],
                                  eps=eps, out=gr, workspace=ws)
                elif direction == "fwd":
                    la.chunked_fwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], block=block, eps=eps, o=o[0],
                                   S_out=o[1], z_out=o[2])
                else:
                    la.chunked_bwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], d["dO"], d["dS_out"], d["dz_out"],
                                   block=block, eps=eps, out=gr)
            n = 20
            with torch.cuda.stream(stream):
                for i in range(3):
                    call(i)
            torch.cuda.synchronize()
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                for i in range(n):
                    call(i)
            gph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(3):
                    gph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (3 * n)
            byts = fb if direction == "fwd" else bb
            entry[direction] = {"us": round(us, 2), "gbs": round(byts / us / 1e3, 1),
                                "frac": round(byts / us / 1e3 / hbm, 4)}
            if impl == "cumsum":
                flop = cumsum_flop(G, C, D)[0 if direction == "fwd" else 1]
                tf = flop / us / 1e6
                entry[direction]["alu"] = {"bound": "alu", "alg_flop": flop, "achieved_tflops": round(tf, 2),
                                           "peak_tflops": round(alu_peak, 1), "frac": round(tf / alu_peak, 4),
                                           "peak_source": "SMs x 128 fp32 lanes x 2 x 2070 MHz"}
        secs = sum(entry[d]["us"] for d in dirs) * 1e-6
        entry["value"] = G * C / secs
        entry["unit"] = UNIT + (" (" + "+".join(dirs) + ")")
        out[name] = entry
        del sets, x
        torch.cuda.empty_cache()
    return out


def run_e2e(args, host, G, C, D, block, eps, local, barrier, max_over_ranks, nstreams=8):
    """End to end through the C ABI with HOST buffers: every step copies its inputs from
    pinned host memory into a device workspace, runs forward + backward and copies every
    output back (la_chunked_step_host; with page-locked buffers each direction is one
    copy kernel of the library).  Eight streams with a workspace and an output set each
    let one step's copies overlap the other steps', as a pipelined caller would (six
    streams measured 4 % slower, four 10 %, twelve the same)."""
    import torch

    import causal_linear_attention_gb300 as la
    dev = torch.device("cuda", local)
    old_aff = os.sched_getaffinity(0)
    near = gpu_local_cpus(local)
    if near:
        os.sched_setaffinity(0, near)  # pinned buffers get first-touched next to the GPU
    try:
        pin = {k: (None if t is None else t.pin_memory()) for k, t in host.__dict__.items()}
        q = pin["q"]

        def outs():
            f = lambda *shape: torch.empty(*shape, dtype=torch.float32, pin_memory=True)
            return (torch.empty_like(q, pin_memory=True), f(G, D, D), f(G, D), torch.empty_like(q, pin_memory=True),
                    torch.empty_like(q, pin_memory=True), torch.empty_like(q, pin_memory=True), f(G, D, D), f(G, D))

        sets = [(outs(), la.step_workspace(G, C, D, q.dtype, dev), torch.cuda.Stream(device=dev))
                for _ in range(nstreams)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in sets[0][0])

        def step(i):
            out, ws, s = sets[i % nstreams]
            la.chunked_step_host(pin["q"], pin["k"], pin["v"], pin["S0"], pin["z0"], pin["dO"], pin["dS_out"],
                                 pin["dz_out"], out=out, workspace=ws, block=block, eps=eps, stream=s)

        n = min(args.steps, 2000)
        for i in range(4):
            step(i)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            step(i)
        for _, _, s in sets:
            s.synchronize()
        secs = max_over_ranks(time.perf_counter() - t0)
        barrier()
        # the copies alone, for context: one H2D of the step's input bytes, one D2H of its output bytes
        s = sets[0][2]
        hb = torch.empty(h2d, dtype=torch.uint8, pin_memory=True)
        db = torch.empty(max(h2d, d2h), dtype=torch.uint8, device=dev)
        gbs = {}
        for name, (dst, src, nb) in {"h2d": (db[:h2d], hb, h2d), "d2h": (hb[:d2h], db[:d2h], d2h)}.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                for _ in range(3):
                    dst.copy_(src, non_blocking=True)
                e0.record(s)
                for _ in range(20):
                    dst.copy_(src, non_blocking=True)
                e1.record(s)
            s.synchronize()
            gbs[name] = round(20 * nb / (e0.elapsed_time(e1) / 1e3) / 1e9, 1)
    finally:
        os.sched_setaffinity(0, old_aff)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": job_value(world, G, C, n, secs), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": n, "api": f"la_chunked_step_host (C ABI, pinned host buffers copied by the library's SM-copy "
                   f"kernels), {nstreams} streams",
            "host_cpus": f"{len(near)} cpus of the GPU's NUMA node" if near else "unrestricted",
            "copy_gbs": gbs}


# ---------------------------------------------------------------- the oracle on the host cores
def oracle_step(x, eps):
    import oracle
    oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=eps)
    oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=eps)


def cpu_baseline(host, G, C, D, eps, budget_s=10.0):
    """The fp64 oracle (as it stands) on this host's cores: full fwd+bwd of the same
    workload, repeated until `budget_s` seconds of work have run."""
    import oracle
    oracle.build()
    oracle_step(host, eps)  # warm (page-in, thread pool)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(host, eps)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": G * C * reps / el, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{reps} x full fwd+bwd of the workload (G={G}, C={C}, D={D}) in fp64, {el:.1f} s"}


def cpu_torch_fp32(host, G, C, D, block, eps, reps=5):
    """The page's chunked form as plain PyTorch CPU ops in fp32 (oracle/torch_chunked.py; the
    backward by autograd), the way the page's own CPU micro-benchmark runs it: median of
    `reps` runs of the forward and of forward + backward on the same workload."""
    import statistics

    import torch

    from oracle import torch_chunked
    x = [None if t is None else t.float() for t in (host.q, host.k, host.v, host.S0, host.z0, host.dO,
                                                     host.dS_out, host.dz_out)]
    res = {}
    for name, fn in (("fwd", lambda: torch_chunked.chunked_fwd(*x[:5], block=block, eps=eps)),
                     ("fwdbwd", lambda: torch_chunked.chunked_fwd_bwd(*x, block=block, eps=eps))):
        with torch.no_grad() if name == "fwd" else torch.enable_grad():
            fn()
            times = []
            for _ in range(reps):
                t0 = time.perf_counter()
                fn()
                times.append(time.perf_counter() - t0)
        ms = statistics.median(times) * 1e3
        res[name] = {"value": G * C / (ms / 1e3), "unit": UNIT, "ms": round(ms, 2)}
    res.update({"kind": "torch-CPU fp32 restatement of the chunked form (oracle/torch_chunked.py), autograd backward",
                "threads": torch.get_num_threads(), "cpu": cpu_model(), "torch": torch.__version__,
                "sample": f"median of {reps} runs of the workload (G={G}, C={C}, D={D}, block {block})",
                "page_cpu_table": {"fwd_ms": 23.0, "fwdbwd_ms": 72.4,
                                   "note": "the page's chunked CPU micro-benchmark at G = 160 (torch on a CPU "
                                           "of unstated model and core count): context, not a target"}})
    return res


def run_reference(args, rank, world):
    """Reference arm: the fp64 oracle on the host cores, same workload/metric/unit.
    Under torchrun only rank 0 runs it."""
    if rank != 0:
        return None
    import oracle
    from causal_linear_attention_gb300.inputs import make_inputs
    G, C, D, eps = (WORKLOAD[k] for k in ("G", "C", "D", "eps"))
    oracle.build()
    host = make_inputs(G, C, D, dtype="bf16", seed=rank_seed(0), grads=True)
    # each step: a bounded sample of the workload sized so the whole run takes a few minutes
    t0 = time.perf_counter()
    oracle_step(host, eps)
    one = time.perf_counter() - t0
    budget_per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    g_sample = max(1, min(G, int(G * budget_per_step / max(one, 1e-9))))
    sample = make_inputs(g_sample, C, D, dtype="bf16", seed=rank_seed(0), grads=True)
    for _ in range(args.warmup):
        oracle_step(sample, eps)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample, eps)
    secs = time.perf_counter() - t0
    value = g_sample * C * args.steps / secs
    desc = f"{g_sample} of {G} groups per step (C={C}, D={D}), fp64 fwd+bwd"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "G_per_step": g_sample, "C": C, "D": D, "block": WORKLOAD["block"],
                   "eps": eps, "step": "oracle fwd + bwd (per-token fp64 loop, OpenMP over groups)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "cpu": cpu_model(), "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: CPU seconds the whole run aims at (sizes the bounded sample)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    rank, world, local = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
