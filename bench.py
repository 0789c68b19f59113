"""Benchmark of the MX block quantize / QDQ hot path on GB300.

Default workload (one step): MXFP4 (E2M1) QDQ, group 32, bf16 in / bf16 out, of the weight-like
x[8192, 8192] (Student-t nu=4 * 0.02) and the activation-like x[4096, 8192] (N(0,1), 8 outlier
columns * 100): two kernel launches, 402,653,184 algorithmic bytes (4 B per element). Inputs
(192 MiB) and outputs (192 MiB) are larger than L2 (129 MB), so no flush runs between steps.

Prints one JSON line: metric/value in algorithmic GB/s over the CUDA-event-timed region of K
steps, launched back to back with no event between them (an event at a kernel boundary makes
the stream drain there); after that region, a separate pass brackets each launch of some more
steps with events for the per-launch durations. A roofline object for the kernel (against the
measured HBM copy bandwidth, with the DRAM traffic per launch that an ncu capture recorded in
profiles/mx_stream_qdq_traffic.json while the kernel's sources are unchanged), the CPU oracle timed
on the host cores (cpu_baseline), an end-to-end figure through the same calls with the inputs
copied in from, and the outputs back to, pinned host memory every step (e2e; copies in both
directions pipelined over two buffer sets), SM clocks sampled during the timed region, and
per-workload kernel figures for the other workloads, cold (a 256 MiB buffer is written before
each timed launch; mean of the launches, since event timestamps advance in ~2 us steps) and
steady (launches back to back over copies of the buffers that together exceed 3x L2).

--impl reference times the CPU oracle instead (bounded sample per step, all host cores).
"""

from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MX quant/QDQ HBM GB/s and % of GB300 peak; Gelem/s vs CPU oracle"
WORKLOAD = "mxfp4_qdq: E2M1 QDQ g32 of bf16 x[8192,8192] Student-t(4)*0.02 + x[4096,8192] N(0,1) w/ 8 outlier cols"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "mx_stream_qdq_traffic.json")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--quick", action="store_true",
                   help="main timed loop only (no e2e, CPU baseline, extra workloads)")
    p.add_argument("--case", choices=sorted(CASES), default=None,
                   help="run one other workload only (for profiler captures): warmup + steps "
                        "launches, one JSON line with its kernel-only GB/s")
    p.add_argument("--gemm-shapes", default="o_proj,down_proj,square,decode",
                   help="--case gemm: comma-separated subset of o_proj, down_proj, square, decode")
    p.add_argument("--tiles-per-sm", type=int, default=8,
                   help="rotate_quant_tiles: x[128, 128 * SMs * n] gives exactly n tiles per SM")
    return p.parse_args()


# ---------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; weak scaling, no data-path collective)
# ---------------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("mx_stream.cu", "mx_device.cuh", "mx_launch.h"):
        with open(os.path.join(ROOT, "mx_microscaling_quantize_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu record (read + write,
    --cache-control none), if the kernel's sources are unchanged since it was taken; else
    None."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != kernel_source_hash():
        return None
    return rec


def to_gpu(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (bounded samples)
# ---------------------------------------------------------------------------------------------
def oracle_qdq_rows(parts, threads):
    """Run the oracle's QDQ on row chunks of each (bits) array with a thread pool."""
    import oracle as O
    jobs = []
    for bits in parts:
        step = max(1, bits.shape[0] // (threads * 4))
        for r in range(0, bits.shape[0], step):
            jobs.append(bits[r:r + step])
    with concurrent.futures.ThreadPoolExecutor(threads) as pool:
        list(pool.map(lambda b: O.qdq(b, O.E2M1), jobs))


def time_oracle_for(xw, xa, min_seconds):
    """Oracle QDQ of whole-row samples on all host cores, repeated until min_seconds elapsed
    (at least once); returns (GB/s over algorithmic bytes, seconds, passes, threads)."""
    import oracle as O
    O.build()
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle_qdq_rows([xw, xa], threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    nbytes = 4 * (xw.size + xa.size) * passes
    return nbytes / dt / 1e9, dt, passes, threads


def time_oracle_one_core(xw, min_seconds, rows=256):
    """Oracle QDQ of the weight's first `rows` rows on one host core (one oracle call per pass,
    no thread pool), repeated until min_seconds elapsed (at least once); returns (GB/s over
    algorithmic bytes, seconds, passes, rows)."""
    import oracle as O
    O.build()
    sample = np.ascontiguousarray(xw[:rows])
    t0 = time.perf_counter()
    passes = 0
    while True:
        O.qdq(sample, O.E2M1)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return 4 * sample.size * passes / dt / 1e9, dt, passes, rows


# ---------------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    from mx_microscaling_quantize_gb300 import workloads as W
    xw, xa = W.mxfp4_qdq_weight(), W.mxfp4_qdq_activation()
    # each step: one oracle pass over the whole workload on all host cores (about 0.3 s on
    # 16 Grace cores), so that --steps K --warmup W ends within minutes
    for _ in range(args.warmup):
        time_oracle_for(xw, xa, 0.0)
    total = 0.0
    threads = os.cpu_count() or 1
    for _ in range(args.steps):
        total += time_oracle_for(xw, xa, 0.0)[1]
    nbytes = 4 * (xw.size + xa.size)
    value = nbytes * args.steps / total / 1e9
    sample = "the whole workload (both tensors) per step, row chunks over all host cores"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": 8192,
                   "parallelism": "none (CPU oracle)", "l2": "n/a"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gelem_per_s": value / 4,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def extra_workloads(dev, peak):
    """Kernel-only figures of the other workloads, two ways (CUDA events on the launching
    stream both times):
    - cold: single launches, a 256 MiB buffer written before each so that it starts with a
      cold L2. The launch then also pays for writing back the dirty lines that buffer left,
      up to the whole L2 (129 MB), which stands in for the write-back of its own outputs
      (still in L2 when it ends); for a launch that writes less than L2 this overcharges.
    - steady: launches back to back, cycling over enough copies of the buffers (inputs and
      outputs) that the copies together are at least three times L2, so no launch finds its
      inputs in L2 and each pays for the write-back of what the launch before it wrote, as in
      a stream of such calls; the mean over the loop.
    - graph (calls under 32 MiB of traffic only, which the two above time as launch latency):
      device time per call of 100 calls captured in one CUDA graph and replayed (the small
      buffer copies then partly sit in L2)."""
    import torch
    import mx_microscaling_quantize_gb300 as mxq
    from mx_microscaling_quantize_gb300 import workloads as W

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_bytes = 129 * 10 ** 6
    out = {}

    def timed(fn, iters=30):
        # The event timestamps advance in steps of about 2 us on this GPU, so a single launch
        # reads as a multiple of the step; the mean over launches that start at random phases
        # of the step is unbiased where a median is not.
        times = []
        for i in range(iters + 2):
            flush.fill_(i & 0xFF)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            e.synchronize()
            if i >= 2:
                times.append(s.elapsed_time(e) / 1e3)
        return statistics.fmean(times)

    def steady(fns, iters):
        for fn in fns:
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(iters):
            fns[i % len(fns)]()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / 1e3 / iters

    def graph_time(fns, calls=100):
        """Device time per call of `calls` launches (cycling over fns) captured in one CUDA graph
        and replayed: what a call costs inside a captured serving step, without host launches."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for fn in fns:
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(calls):
                fns[i % len(fns)]()
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(5):
            graph.replay()
        e.record()
        e.synchronize()
        del graph
        return s.elapsed_time(e) / 1e3 / (5 * calls)

    def measure(name, nbytes, elems, make, footprint, iters=30):
        """make(k) -> a launch closure over buffer set k (k = 0: the given buffers, k > 0:
        copies); footprint: bytes of one set's inputs and outputs."""
        fns = [make(0)]
        t_cold = timed(fns[0], iters)
        sets = max(1, min(64, -(-3 * l2_bytes // footprint)))
        fns += [make(k) for k in range(1, sets)]
        t_steady = steady(fns, max(2 * iters, 2 * sets))
        out[name] = {"GB/s": nbytes / t_cold / 1e9, "frac_of_peak": nbytes / t_cold / 1e9 / peak,
                     "Gelem/s": elems / t_cold / 1e9, "us": t_cold * 1e6, "launches": 1,
                     "steady_GB/s": nbytes / t_steady / 1e9,
                     "steady_frac": nbytes / t_steady / 1e9 / peak,
                     "steady_us": t_steady * 1e6, "steady_sets": sets}
        if footprint < (32 << 20):  # small calls: launch-bound above; device time in a graph
            out[name]["graph_us"] = graph_time(fns) * 1e6
        del fns

    def copy_of(t, k):
        return t if k == 0 else t.clone()

    def empty_of(t, k):
        return t if k == 0 else torch.empty_like(t)

    # MXFP8 quantize, linear scales, x[128, 4096]
    x = to_gpu(W.mxfp8_linear_quant(), dev)
    c, s = mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize(xk, mxq.E4M3, mxq.LINEAR, codes=ck, scales=sk)
    nb = 3 * x.numel() + s.numel()
    measure("mxfp8_linear_quant[128,4096]", nb, x.numel(), make, nb)

    # the two QDQ tensors separately, both formats
    for name, bits in (("weight[8192,8192]", W.mxfp4_qdq_weight()),
                       ("activation[4096,8192]", W.mxfp4_qdq_activation())):
        x = to_gpu(bits, dev)
        y = torch.empty_like(x)
        for fmt, fname in ((mxq.E2M1, "mxfp4"), (mxq.E4M3, "mxfp8")):
            def make(k, x=x, y=y, fmt=fmt):
                xk, yk = copy_of(x, k), empty_of(y, k)
                return lambda: mxq.mx_qdq(xk, fmt, y=yk)
            measure(f"{fname}_qdq_{name}", 4 * x.numel(), x.numel(), make, 4 * x.numel())
        del x, y

    # fused rotate + MXFP4 quantize, g = 32 Hadamard, swizzled scales: on the tensor cores
    # (rot_kind ROT_DENSE, any H) and with the Hadamard statement (ROT_HADAMARD: in-register
    # Walsh-Hadamard transform)
    H = to_gpu(W.normalized_hadamard_bf16(32), dev)
    kinds = ((mxq.ROT_DENSE, ""), (mxq.ROT_HADAMARD, "_hadamard"))
    for K in W.ROTATE_QUANT_K:
        for M in W.ROTATE_QUANT_M:
            x = to_gpu(W.rotate_quant_activation(M, K), dev)
            c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED)
            for rk, kname in kinds:
                def make(k, x=x, c=c, s=s, rk=rk):
                    xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
                    return lambda: mxq.mx_rotate_quantize(xk, H, mxq.E2M1, mxq.SWIZZLED, codes=ck,
                                                          scales=sk, rot_kind=rk)
                nb = 2 * x.numel() + c.numel() + s.numel()
                measure(f"rotate_quant_mxfp4_g32{kname}[{M},{K}]", nb, x.numel(), make, nb)
            del x, c, s

    # weight-side rotate + quantize of the 70B layer weights, g = 32, swizzled scales
    for N, K in W.WEIGHT_SHAPES:
        x = to_gpu(W.weight_rotate_quant(N, K), dev)
        for fmt, fname in ((mxq.E2M1, "mxfp4"), (mxq.E4M3, "mxfp8")):
            c, s = mxq.mx_rotate_quantize(x, H, fmt, mxq.SWIZZLED)
            for rk, kname in kinds:
                def make(k, x=x, c=c, s=s, fmt=fmt, rk=rk):
                    xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
                    return lambda: mxq.mx_rotate_quantize(xk, H, fmt, mxq.SWIZZLED, codes=ck,
                                                          scales=sk, rot_kind=rk)
                nb = 2 * x.numel() + c.numel() + s.numel()
                measure(f"weight_rotate_quant_{fname}_g32{kname}[{N},{K}]", nb, x.numel(), make,
                        nb, iters=15)
            del c, s
        del x

    # the Quest-like MXFP4 scale (rounding QUEST): plain quantize and QDQ of the QDQ weight,
    # rotate(g = 32) + quantize of the rotate + quantize activation, both rotation kinds
    x = to_gpu(W.mxfp4_qdq_weight(), dev)
    c, s = mxq.mx_quantize(x, mxq.E2M1, mxq.SWIZZLED, rounding=mxq.QUEST)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize(xk, mxq.E2M1, mxq.SWIZZLED, codes=ck, scales=sk,
                                       rounding=mxq.QUEST)
    nb = 2 * x.numel() + c.numel() + s.numel()
    measure("quest_quant_mxfp4_swizzled[8192,8192]", nb, x.numel(), make, nb)
    y = torch.empty_like(x)

    def make(k, x=x, y=y):
        xk, yk = copy_of(x, k), empty_of(y, k)
        return lambda: mxq.mx_qdq(xk, mxq.E2M1, y=yk, rounding=mxq.QUEST)
    measure("quest_qdq_mxfp4[8192,8192]", 4 * x.numel(), x.numel(), make, 4 * x.numel())
    del x, y, c, s
    for M, K in ((8192, 8192), (8192, 28672)):
        x = to_gpu(W.rotate_quant_activation(M, K), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, rounding=mxq.QUEST)
        for rk, kname in kinds:
            def make(k, x=x, c=c, s=s, rk=rk):
                xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
                return lambda: mxq.mx_rotate_quantize(xk, H, mxq.E2M1, mxq.SWIZZLED, codes=ck,
                                                      scales=sk, rot_kind=rk, rounding=mxq.QUEST)
            nb = 2 * x.numel() + c.numel() + s.numel()
            measure(f"quest_rotate_quant_mxfp4_g32{kname}[{M},{K}]", nb, x.numel(), make, nb)
        del x, c, s

    # dequantize stored codes + scales of the QDQ weight x[8192, 8192]
    x = to_gpu(W.mxfp4_qdq_weight(), dev)
    y = torch.empty_like(x)
    K = x.shape[1]
    for fmt, fname in ((mxq.E2M1, "mxfp4"), (mxq.E4M3, "mxfp8")):
        for layout, lname in ((mxq.LINEAR, "linear"), (mxq.SWIZZLED, "swizzled")):
            c, s = mxq.mx_quantize(x, fmt, layout)

            def make(k, c=c, s=s, fmt=fmt, layout=layout):
                ck, sk, yk = copy_of(c, k), copy_of(s, k), empty_of(y, k)
                return lambda: mxq.mx_dequantize(ck, sk, K, fmt, layout, y=yk)
            nb = c.numel() + x.numel() // 32 + 2 * x.numel()
            measure(f"dequant_{fname}_{lname}[8192,8192]", nb, x.numel(), make, nb)
            del c, s
    del y

    # NVFP4 (16-element blocks, E4M3 scales under a global scale): plain quantize, QDQ and
    # dequantize of the QDQ weight, and rotate(g = 16) + quantize of the largest activation
    gs = torch.tensor([448.0 * 6.0], device=dev) / x.float().abs().max()
    c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_nvfp4(xk, gs, mxq.SWIZZLED, codes=ck, scales=sk)
    nb = 2 * x.numel() + c.numel() + x.numel() // 16
    measure("nvfp4_quant[8192,8192]", nb, x.numel(), make, nb)
    y = torch.empty_like(x)

    def make(k, x=x, y=y):
        xk, yk = copy_of(x, k), empty_of(y, k)
        return lambda: mxq.mx_qdq_nvfp4(xk, gs, y=yk)
    measure("nvfp4_qdq[8192,8192]", 4 * x.numel(), x.numel(), make, 4 * x.numel())

    def make(k, c=c, s=s, y=y):
        ck, sk, yk = copy_of(c, k), copy_of(s, k), empty_of(y, k)
        return lambda: mxq.mx_dequantize_nvfp4(ck, sk, K, gs, mxq.SWIZZLED, y=yk)
    nb = c.numel() + x.numel() // 16 + 2 * x.numel()
    measure("nvfp4_dequant_swizzled[8192,8192]", nb, x.numel(), make, nb)
    del x, y, c, s
    x = to_gpu(W.rotate_quant_activation(8192, 28672), dev)
    H16 = to_gpu(W.normalized_hadamard_bf16(16), dev)
    c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H16)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_nvfp4(xk, gs, mxq.SWIZZLED, H16, codes=ck, scales=sk)
    nb = 2 * x.numel() + c.numel() + x.numel() // 16
    measure("nvfp4_rotate_quant_g16[8192,28672]", nb, x.numel(), make, nb, iters=15)
    del x, c, s

    # MoE grouped quantize, swizzled scales padded per expert: MXFP8, and the same expert
    # inputs in NVFP4 with one global scale per expert
    xb, off = W.moe_quant()
    x = to_gpu(xb, dev)
    offs = torch.from_numpy(off).to(dev)
    c, s = mxq.mx_quantize_grouped(x, offs, mxq.E4M3, mxq.SWIZZLED)
    used_rows = int(sum(-(-int(n) // 128) * 128 for n in np.diff(off)))

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_grouped(xk, offs, mxq.E4M3, mxq.SWIZZLED, codes=ck,
                                               scales=sk)
    nb = 3 * x.numel() + used_rows * s.shape[1]
    measure("moe_quant_mxfp8[16384,2048]x128", nb, x.numel(), make, nb)
    del c, s
    c, s = mxq.mx_quantize_grouped(x, offs, mxq.E4M3, mxq.LINEAR)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_grouped(xk, offs, mxq.E4M3, mxq.LINEAR, codes=ck,
                                               scales=sk)
    nb = 3 * x.numel() + s.numel()
    measure("moe_quant_mxfp8_linear[16384,2048]x128", nb, x.numel(), make, nb)
    del c, s
    gse = torch.stack([448.0 * 6.0 / x[int(off[e]):int(off[e + 1])].float().abs().max()
                       if off[e + 1] > off[e] else torch.ones((), device=dev)
                       for e in range(len(off) - 1)]).float().contiguous()
    c, s = mxq.mx_quantize_nvfp4_grouped(x, offs, gse, mxq.SWIZZLED)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_nvfp4_grouped(xk, offs, gse, mxq.SWIZZLED, codes=ck,
                                                     scales=sk)
    nb = 2 * x.numel() + c.numel() + used_rows * s.shape[1]
    measure("moe_quant_nvfp4[16384,2048]x128", nb, x.numel(), make, nb)
    del x, c, s

    # rotate+quantize with linear scales (the layout of mxfp8_quantize without swizzling)
    x = to_gpu(W.rotate_quant_activation(8192, 28672), dev)
    H32 = to_gpu(W.normalized_hadamard_bf16(32), dev)
    for fmt, fname, cb in ((mxq.E2M1, "mxfp4", 0.5), (mxq.E4M3, "mxfp8", 1.0)):
        c, s = mxq.mx_rotate_quantize(x, H32, fmt, mxq.LINEAR)

        def make(k, x=x, c=c, s=s, fmt=fmt):
            xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
            return lambda: mxq.mx_rotate_quantize(xk, H32, fmt, mxq.LINEAR, codes=ck, scales=sk)
        nb = 2 * x.numel() + c.numel() + s.numel()
        measure(f"rotate_quant_{fname}_g32_linear[8192,28672]", nb, x.numel(), make, nb, iters=15)
        del c, s
    H16 = to_gpu(W.normalized_hadamard_bf16(16), dev)
    gsx = (448.0 * 6.0 / x.float().abs().max()).reshape(1).float().contiguous()
    c, s = mxq.mx_quantize_nvfp4(x, gsx, mxq.LINEAR, H16)

    def make(k, x=x, c=c, s=s):
        xk, ck, sk = copy_of(x, k), empty_of(c, k), empty_of(s, k)
        return lambda: mxq.mx_quantize_nvfp4(xk, gsx, mxq.LINEAR, H16, codes=ck, scales=sk)
    nb = 2 * x.numel() + c.numel() + s.numel()
    measure("nvfp4_rotate_quant_g16_linear[8192,28672]", nb, x.numel(), make, nb, iters=15)
    del x, c, s

    # rotation sweep: rotated QDQ, g in {16,32,64,128} x {MXFP4, MXFP8} on 3 layer inputs
    for lname, M, K in W.ROTATION_SWEEP_LAYERS:
        x = to_gpu(W.rotation_sweep_input(lname), dev)
        y = torch.empty_like(x)
        for g in W.ROTATION_SWEEP_G:
            Hg = to_gpu(W.normalized_hadamard_bf16(g), dev)
            for fmt, fname in ((mxq.E2M1, "mxfp4"), (mxq.E4M3, "mxfp8")):
                # ROT_HADAMARD with g = 128 runs on the tensor cores, as ROT_DENSE
                for rk, kname in (kinds if g <= 64 else kinds[:1]):
                    def make(k, x=x, y=y, Hg=Hg, fmt=fmt, rk=rk):
                        xk, yk = copy_of(x, k), empty_of(y, k)
                        return lambda: mxq.mx_qdq(xk, fmt, Hg, y=yk, rot_kind=rk)
                    measure(f"rotated_qdq_{fname}_g{g}{kname}_{lname}[{M},{K}]", 4 * x.numel(),
                            x.numel(), make, 4 * x.numel(), iters=15)
        del x, y
    return out


CASES = {
    "mxfp8_linear_quant": "E4M3 quantize, linear scales, x[128,4096]",
    "rotate_quant": "E2M1 rotate(g=32 Hadamard)+quantize, swizzled, x[8192,8192]",
    "rotate_quant_hadamard": "the same call with rot_kind ROT_HADAMARD (in-register fast "
                             "Walsh-Hadamard transform on the streaming layout)",
    "rotated_qdq_g128": "E4M3 rotated QDQ g=128, x[4096,28672] Student-t(5)",
    "moe_quant": "E4M3 grouped quantize, swizzled, 128 experts, x[16384,2048]",
    "dequant_mxfp4": "E2M1 dequantize, swizzled scales, codes of the weight x[8192,8192]",
    "weight_rotate_quant": "E4M3 rotate(g=32)+quantize, swizzled, weight [57344,8192]",
    "nvfp4_quant": "NVFP4 quantize, swizzled E4M3 scales, weight x[8192,8192]",
    "nvfp4_rotate_quant": "NVFP4 rotate(g=16)+quantize, swizzled, x[8192,28672]",
    "nvfp4_dequant": "NVFP4 dequantize, swizzled E4M3 scales, codes of the weight x[8192,8192]",
    "rotate_quant_decode": "E2M1 rotate(g=32)+quantize, swizzled, x[16,28672] (FMA kernel)",
    "rotate_quant_quest": "E2M1 rotate(g=32 Hadamard)+quantize under the Quest-like scale, "
                          "swizzled, x[8192,8192] (tensor-core kernel)",
    "qdq_quest": "E2M1 QDQ under the Quest-like scale, weight x[8192,8192] (streaming kernel)",
    "moe_quant_nvfp4": "NVFP4 grouped quantize, swizzled, 128 experts, per-expert scales, x[16384,2048]",
    "qdq_vs_copy": "MXFP4 QDQ of the weight and activation, each followed by an elementwise "
                   "copy of the same bytes (torch.mul(x, 1, out=y)) for profiler comparisons",
    "quant_vs_cast": "MXFP8 quantize and dequantize of the weight x[8192,8192], each followed by "
                     "torch's plain bf16 <-> float8_e4m3fn cast of the same bytes",
    "rotate_quant_tiles": "E2M1 rotate(g=32)+quantize, swizzled, x[128, 128 * SMs * n]: exactly "
                          "n = --tiles-per-sm tiles per SM, launches cycling over input copies",
    "gemm": "block-scaled GEMM consumer C = dequant(A) dequant(B)^T (bf16 out) on the quantized "
            "activation and weight workloads, MXFP4 and MXFP8, swizzled scales, at the o_proj, "
            "down_proj, square and decode shapes; beside it torch.matmul (cuBLAS bf16) of the "
            "dequantized operands, alone and after the two mx_dequantize calls, and for MXFP8 "
            "cuBLAS's block-scaled GEMM (torch._scaled_mm) on the same codes and scales",
    "nonrotated_sweep": "every non-rotated kernel at full workload size (quantize, QDQ, "
                        "dequantize, NVFP4, grouped MoE, the x[128,4096] MXFP8 quantize), each "
                        "launched --steps times back to back over buffer copies that exceed 3x "
                        "L2, in turn (for per-kernel ncu captures; one JSON line with each "
                        "variant's mean us per launch)",
}


def nonrotated_variants(dev):
    """(name, make, algorithmic bytes per launch, bytes of one buffer set) of every non-rotated
    kernel variant at its full workload size; make(k) returns a launch closure over buffer set k
    (k = 0: the workload's own input; k > 0: copies). Outputs are torch.empty buffers and the
    dequantize inputs random code / scale bytes, so that building the variants launches no
    kernel of the library."""
    import torch
    import mx_microscaling_quantize_gb300 as mxq
    from mx_microscaling_quantize_gb300 import workloads as W
    out = []
    xw = to_gpu(W.mxfp4_qdq_weight(), dev)
    xa = to_gpu(W.mxfp4_qdq_activation(), dev)
    n = xw.numel()
    M, K = xw.shape
    gen = torch.Generator(device=dev).manual_seed(7)

    def rnd_bytes(shape):
        return torch.randint(0, 256, shape, dtype=torch.uint8, device=dev, generator=gen)

    def cpy(t, k):
        return t if k == 0 else t.clone()

    for fmt, fname, cb in ((mxq.E2M1, "mxfp4", 0.5), (mxq.E4M3, "mxfp8", 1.0)):
        cshape = (M, mxq.code_bytes_per_row(fmt, K))
        for layout, lname in ((mxq.LINEAR, "linear"), (mxq.SWIZZLED, "swizzled")):
            sshape = mxq.mx_scales_shape(M, K, layout)
            nb = int(2 * n + cb * n + n // 32)

            def make_q(k, fmt=fmt, layout=layout, cshape=cshape, sshape=sshape):
                x = cpy(xw, k)
                c = torch.empty(cshape, dtype=torch.uint8, device=dev)
                s_ = torch.empty(sshape, dtype=torch.uint8, device=dev)
                return lambda: mxq.mx_quantize(x, fmt, layout, codes=c, scales=s_)
            out.append((f"quant_{fname}_{lname}[8192,8192]", make_q, nb, nb))
            codes0, scales0 = rnd_bytes(cshape), rnd_bytes(sshape)

            def make_d(k, fmt=fmt, layout=layout, codes0=codes0, scales0=scales0):
                c, s_ = cpy(codes0, k), cpy(scales0, k)
                y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
                return lambda: mxq.mx_dequantize(c, s_, K, fmt, layout, y=y)
            out.append((f"dequant_{fname}_{lname}[8192,8192]", make_d, nb, nb))
        for x0, tname in ((xw, "weight[8192,8192]"), (xa, "activation[4096,8192]")):
            def make_qdq(k, x0=x0, fmt=fmt):
                x = cpy(x0, k)
                y = torch.empty_like(x)
                return lambda: mxq.mx_qdq(x, fmt, y=y)
            out.append((f"qdq_{fname}_{tname}", make_qdq, 4 * x0.numel(), 4 * x0.numel()))
    gs = torch.tensor([448.0 * 6.0], device=dev) / xw.float().abs().max()
    nb4 = int(2.5 * n + n // 16)
    for layout, lname in ((mxq.LINEAR, "linear"), (mxq.SWIZZLED, "swizzled")):
        sshape = mxq.mx_nvfp4_scales_shape(M, K, layout)

        def make_q4(k, layout=layout, sshape=sshape):
            x = cpy(xw, k)
            c = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
            s_ = torch.empty(sshape, dtype=torch.uint8, device=dev)
            return lambda: mxq.mx_quantize_nvfp4(x, gs, layout, codes=c, scales=s_)
        out.append((f"nvfp4_quant_{lname}[8192,8192]", make_q4, nb4, nb4))
        codes0 = rnd_bytes((M, K // 2))
        scales0 = rnd_bytes(sshape) & 0x77  # finite E4M3 scale bytes

        def make_d4(k, layout=layout, codes0=codes0, scales0=scales0):
            c, s_ = cpy(codes0, k), cpy(scales0, k)
            y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            return lambda: mxq.mx_dequantize_nvfp4(c, s_, K, gs, layout, y=y)
        out.append((f"nvfp4_dequant_{lname}[8192,8192]", make_d4, nb4, nb4))

    def make_qdq4(k):
        x = cpy(xw, k)
        y = torch.empty_like(x)
        return lambda: mxq.mx_qdq_nvfp4(x, gs, y=y)
    out.append(("nvfp4_qdq[8192,8192]", make_qdq4, 4 * n, 4 * n))
    xb, off = W.moe_quant()
    xm = to_gpu(xb, dev)
    offs = torch.from_numpy(off).to(dev)
    E = len(off) - 1
    used = int(sum(-(-int(k) // 128) * 128 for k in np.diff(off)))
    srows, scols = mxq.mx_grouped_scales_shape(xm.shape[0], E, xm.shape[1], mxq.SWIZZLED)
    nb8 = 3 * xm.numel() + used * scols

    def make_moe8(k):
        x = cpy(xm, k)
        c = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        s_ = torch.empty((srows, scols), dtype=torch.uint8, device=dev)
        return lambda: mxq.mx_quantize_grouped(x, offs, mxq.E4M3, mxq.SWIZZLED, codes=c, scales=s_)
    out.append(("moe_quant_mxfp8[16384,2048]x128", make_moe8, nb8, nb8))
    gse = torch.full((E,), 100.0, device=dev)
    srows4, scols4 = mxq.mx_nvfp4_grouped_scales_shape(xm.shape[0], E, xm.shape[1], mxq.SWIZZLED)
    nbm4 = int(2.5 * xm.numel()) + used * scols4

    def make_moe4(k):
        x = cpy(xm, k)
        c = torch.empty((x.shape[0], x.shape[1] // 2), dtype=torch.uint8, device=dev)
        s_ = torch.empty((srows4, scols4), dtype=torch.uint8, device=dev)
        return lambda: mxq.mx_quantize_nvfp4_grouped(x, offs, gse, mxq.SWIZZLED, codes=c,
                                                     scales=s_)
    out.append(("moe_quant_nvfp4[16384,2048]x128", make_moe4, nbm4, nbm4))
    x1 = to_gpu(W.mxfp8_linear_quant(), dev)
    nb1 = 3 * x1.numel() + x1.numel() // 32

    def make_c1(k):
        x = cpy(x1, k)
        c = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        s_ = torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.uint8, device=dev)
        return lambda: mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR, codes=c, scales=s_)
    out.append(("quant_mxfp8_linear[128,4096]", make_c1, nb1, nb1))
    return out


def run_case(args):
    """One workload, `warmup` untimed + `steps` timed launches back to back (no L2 flush)."""
    import torch
    dev = torch.device("cuda", 0)
    import __graft_entry__
    __graft_entry__.build()
    import mx_microscaling_quantize_gb300 as mxq
    from mx_microscaling_quantize_gb300 import workloads as W
    if args.case == "nonrotated_sweep":
        # Each variant: its own buffer sets, together at least three times L2 (so that no launch
        # finds its input in L2), one warm-up launch per set, then --steps launches cycling over
        # the sets. No kernel of the library runs outside these launches, so under a profiler
        # the launches come in this order: every variant's warm-up launches, then its timed ones,
        # variant after variant.
        l2 = 129 * 10 ** 6
        res = {}
        order = []
        for name, make, nbytes, footprint in nonrotated_variants(dev):
            sets = max(1, min(64, -(-3 * l2 // footprint)))
            fns = [make(k) for k in range(sets)]
            for fn in fns:
                fn()
            torch.cuda.synchronize()
            steps = max(1, args.steps)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(steps):
                fns[i % sets]()
            b.record()
            b.synchronize()
            t = a.elapsed_time(b) / 1e3 / steps
            res[name] = {"us_per_launch": t * 1e6, "GB/s": nbytes / t / 1e9,
                         "algorithmic_bytes": nbytes, "warmup_launches": sets,
                         "timed_launches": steps}
            order.append(name)
            del fns
        print(json.dumps({"case": args.case, "what": CASES[args.case], "variants": res,
                          "launch_order": order,
                          "gpu_launches": sum(v["warmup_launches"] + v["timed_launches"]
                                              for v in res.values())}), flush=True)
        return
    if args.case == "gemm":
        run_gemm_case(args, dev)
        return
    if args.case == "mxfp8_linear_quant":
        x = to_gpu(W.mxfp8_linear_quant(), dev)
        c, s = mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR)
        fn = lambda: mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR, codes=c, scales=s)
        nbytes = 3 * x.numel() + s.numel()
    elif args.case == "rotate_quant":
        x = to_gpu(W.rotate_quant_activation(8192, 8192), dev)
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED)
        fn = lambda: mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "rotate_quant_quest":
        x = to_gpu(W.rotate_quant_activation(8192, 8192), dev)
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, rounding=mxq.QUEST)
        fn = lambda: mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s,
                                            rounding=mxq.QUEST)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "qdq_quest":
        x = to_gpu(W.mxfp4_qdq_weight(), dev)
        y = torch.empty_like(x)
        fn = lambda: mxq.mx_qdq(x, mxq.E2M1, y=y, rounding=mxq.QUEST)
        nbytes = 4 * x.numel()
    elif args.case == "rotate_quant_hadamard":
        x = to_gpu(W.rotate_quant_activation(8192, 8192), dev)
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, rot_kind=mxq.ROT_HADAMARD)
        fn = lambda: mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s,
                                            rot_kind=mxq.ROT_HADAMARD)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "rotated_qdq_g128":
        x = to_gpu(W.rotation_sweep_input("down_proj_in"), dev)
        H = to_gpu(W.normalized_hadamard_bf16(128), dev)
        y = torch.empty_like(x)
        fn = lambda: mxq.mx_qdq(x, mxq.E4M3, H, y=y)
        nbytes = 4 * x.numel()
    elif args.case == "dequant_mxfp4":
        x = to_gpu(W.mxfp4_qdq_weight(), dev)
        c, s = mxq.mx_quantize(x, mxq.E2M1, mxq.SWIZZLED)
        y = torch.empty_like(x)
        K = x.shape[1]
        fn = lambda: mxq.mx_dequantize(c, s, K, mxq.E2M1, mxq.SWIZZLED, y=y)
        nbytes = c.numel() + s.numel() + 2 * x.numel()
    elif args.case == "weight_rotate_quant":
        x = to_gpu(W.weight_rotate_quant(57344, 8192), dev)
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E4M3, mxq.SWIZZLED)
        fn = lambda: mxq.mx_rotate_quantize(x, H, mxq.E4M3, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "nvfp4_quant":
        x = to_gpu(W.mxfp4_qdq_weight(), dev)
        gs = torch.tensor([448.0 * 6.0], device=dev) / x.float().abs().max()
        c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED)
        fn = lambda: mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + x.numel() // 16
    elif args.case == "qdq_vs_copy":
        # the reference copy is a torch elementwise kernel (2 bytes in, 2 out per element, like
        # QDQ); it is profiled beside the QDQ launches, never part of the library's path
        xw, xa = to_gpu(W.mxfp4_qdq_weight(), dev), to_gpu(W.mxfp4_qdq_activation(), dev)
        yw, ya, cw, ca = (torch.empty_like(t) for t in (xw, xa, xw, xa))

        def fn():
            mxq.mx_qdq(xw, mxq.E2M1, y=yw)
            torch.mul(xw, 1.0, out=cw)
            mxq.mx_qdq(xa, mxq.E2M1, y=ya)
            torch.mul(xa, 1.0, out=ca)
        nbytes = 8 * (xw.numel() + xa.numel())
    elif args.case == "quant_vs_cast":
        # torch's casts move the same bytes per element as the MXFP8 quantize (2 in, 1 out) and
        # dequantize (1 in, 2 out) without the block scales; profiled beside them only
        x = to_gpu(W.mxfp4_qdq_weight(), dev)
        c, s = mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR)
        y = torch.empty_like(x)
        f8 = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=dev)
        yb = torch.empty_like(x)
        K = x.shape[1]

        def fn():
            mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR, codes=c, scales=s)
            f8.copy_(x)
            mxq.mx_dequantize(c, s, K, mxq.E4M3, mxq.LINEAR, y=y)
            yb.copy_(f8)
        nbytes = 6 * x.numel() + 2 * s.numel()
    elif args.case == "rotate_quant_tiles":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        n = max(1, args.tiles_per_sm)
        M, K = 128, 128 * sms * n
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        copies = max(1, -(-400 // (6 * n * sms // 152)))  # together well above L2
        xs = [to_gpu(W.rotate_quant_activation(M, K, stream=i), dev) for i in range(copies)]
        outs = [mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED) for x in xs]
        calls = [(x, c, s) for x, (c, s) in zip(xs, outs)]
        it = [0]

        def fn():
            x, c, s = calls[it[0] % len(calls)]
            it[0] += 1
            mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * M * K + M * K // 2 + outs[0][1].numel()
    elif args.case == "moe_quant_nvfp4":
        xb, off = W.moe_quant()
        x = to_gpu(xb, dev)
        offs = torch.from_numpy(off).to(dev)
        gse = torch.full((len(off) - 1,), 100.0, device=dev)
        c, s = mxq.mx_quantize_nvfp4_grouped(x, offs, gse, mxq.SWIZZLED)
        fn = lambda: mxq.mx_quantize_nvfp4_grouped(x, offs, gse, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "rotate_quant_decode":
        x = to_gpu(W.rotate_quant_activation(16, 28672), dev)
        H = to_gpu(W.normalized_hadamard_bf16(32), dev)
        c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED)
        fn = lambda: mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + s.numel()
    elif args.case == "nvfp4_dequant":
        x = to_gpu(W.mxfp4_qdq_weight(), dev)
        gs = torch.tensor([448.0 * 6.0], device=dev) / x.float().abs().max()
        c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED)
        y = torch.empty_like(x)
        K = x.shape[1]
        fn = lambda: mxq.mx_dequantize_nvfp4(c, s, K, gs, mxq.SWIZZLED, y=y)
        nbytes = c.numel() + x.numel() // 16 + 2 * x.numel()
    elif args.case == "nvfp4_rotate_quant":
        x = to_gpu(W.rotate_quant_activation(8192, 28672), dev)
        H = to_gpu(W.normalized_hadamard_bf16(16), dev)
        gs = torch.tensor([448.0 * 6.0 / 8.0], device=dev)
        c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H)
        fn = lambda: mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H, codes=c, scales=s)
        nbytes = 2 * x.numel() + c.numel() + x.numel() // 16
    else:
        xb, off = W.moe_quant()
        x = to_gpu(xb, dev)
        offs = torch.from_numpy(off).to(dev)
        c, s = mxq.mx_quantize_grouped(x, offs, mxq.E4M3, mxq.SWIZZLED)
        fn = lambda: mxq.mx_quantize_grouped(x, offs, mxq.E4M3, mxq.SWIZZLED, codes=c, scales=s)
        nbytes = 3 * x.numel() + s.numel()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3 / max(1, args.steps)
    print(json.dumps({"case": args.case, "what": CASES[args.case], "us_per_launch": t * 1e6,
                      "GB/s": nbytes / t / 1e9,
                      "gpu_launches": args.steps * (2 if args.case in ("qdq_vs_copy",
                                                                       "quant_vs_cast") else 1)}),
          flush=True)


def time_oracle_gemm(ca, sa, cw, sw, K, fmt, layout, rows, min_seconds=2.0):
    """The oracle's GEMM (dequantize, then a float64 matmul) of A's first `rows` rows (one
    128-row block of the swizzled scales) against the whole B, repeated until min_seconds."""
    import oracle as O
    O.build()
    a = ca[:rows].cpu().numpy()
    s_a = sa[:128].cpu().numpy() if layout == 1 else sa[:rows].cpu().numpy()
    b, s_b = cw.cpu().numpy(), sw.cpu().numpy()
    N = b.shape[0]
    t0 = time.perf_counter()
    passes = 0
    while True:
        O.gemm(a, s_a, b, s_b, K, fmt, layout)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return {"TFLOP/s": 2.0 * rows * N * K * passes / dt / 1e12, "kind": "oracle",
            "cores": os.cpu_count() or 1,
            "sample": f"C rows 0..{rows - 1} (A[{rows},{K}] x B[{N},{K}]^T), {passes} passes in "
                      f"{dt:.1f} s: C dequantize of both operands + numpy float64 matmul"}


def run_gemm_case(args, dev):
    """TFLOP/s (2 M N K per call) of mx_gemm, launches back to back after --warmup, against the
    measured bf16 tensor peak; the same product through cuBLAS on bf16 operands for context."""
    import torch
    import mx_microscaling_quantize_gb300 as mxq
    from mx_microscaling_quantize_gb300 import workloads as W
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("bf16_tflops", 1900.0)
    shapes = [("o_proj", 4096, 8192, 8192), ("down_proj", 1024, 8192, 28672),
              ("square", 8192, 8192, 8192), ("decode", 16, 8192, 8192)]
    wanted = set(args.gemm_shapes.split(","))
    shapes = [sh for sh in shapes if sh[0] in wanted]
    steps = max(1, args.steps)

    def clock(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) / 1e3 / steps

    res = {}
    launches = 0
    for name, M, N, K in shapes:
        xa = to_gpu(W.mxfp4_qdq_activation(M, K), dev)
        xw = to_gpu(W.weight_rotate_quant(N, K), dev)
        for fmt, fname in ((mxq.E2M1, "mxfp4"), (mxq.E4M3, "mxfp8")):
            ca, sa = mxq.mx_quantize(xa, fmt, mxq.SWIZZLED)
            cw, sw = mxq.mx_quantize(xw, fmt, mxq.SWIZZLED)
            c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            t = clock(lambda: mxq.mx_gemm(ca, sa, cw, sw, K, fmt, mxq.SWIZZLED, c=c))
            da = mxq.mx_dequantize(ca, sa, K, fmt, mxq.SWIZZLED)
            dw = mxq.mx_dequantize(cw, sw, K, fmt, mxq.SWIZZLED)
            t_mm = clock(lambda: torch.matmul(da, dw.t(), out=c))

            def two_step():
                mxq.mx_dequantize(ca, sa, K, fmt, mxq.SWIZZLED, y=da)
                mxq.mx_dequantize(cw, sw, K, fmt, mxq.SWIZZLED, y=dw)
                torch.matmul(da, dw.t(), out=c)
            t_two = clock(two_step)
            launches += 4 + 3 * (max(3, args.warmup) + steps)
            t_bs = None
            if fmt == mxq.E4M3:  # cuBLAS's own MXFP8 block-scaled GEMM on the same bytes
                a8, w8 = ca.view(torch.float8_e4m3fn), cw.view(torch.float8_e4m3fn)
                sa8 = sa.view(torch.float8_e8m0fnu).reshape(-1)
                sw8 = sw.view(torch.float8_e8m0fnu).reshape(-1)
                try:
                    t_bs = clock(lambda: torch._scaled_mm(a8, w8.t(), scale_a=sa8, scale_b=sw8,
                                                          out_dtype=torch.bfloat16))
                except Exception:  # not offered by this torch build on this GPU
                    t_bs = None
            flops = 2.0 * M * N * K
            res[f"{name}_{fname}"] = {
                "M": M, "N": N, "K": K, "us": t * 1e6, "TFLOP/s": flops / t / 1e12,
                "frac_of_bf16_peak": flops / t / 1e12 / peak,
                "cublas_bf16_us": t_mm * 1e6, "cublas_bf16_TFLOP/s": flops / t_mm / 1e12,
                "dequant_then_cublas_us": t_two * 1e6}
            if t_bs is not None:
                res[f"{name}_{fname}"]["cublas_mxfp8_block_scaled_us"] = t_bs * 1e6
                res[f"{name}_{fname}"]["cublas_mxfp8_block_scaled_TFLOP/s"] = flops / t_bs / 1e12
            if name == shapes[0][0]:  # the oracle beside it, on a bounded sample of C's rows
                res[f"{name}_{fname}"]["cpu_baseline"] = time_oracle_gemm(
                    ca, sa, cw, sw, K, fmt, mxq.SWIZZLED, rows=min(M, 128))
            del ca, sa, cw, sw, c, da, dw
        del xa, xw
        torch.cuda.empty_cache()
    print(json.dumps({"case": args.case, "what": CASES[args.case], "bf16_peak_TFLOP/s": peak,
                      "peak_source": "measured bf16_tflops (cuBLAS burst)" if peaks else
                      "fallback", "steps": steps, "shapes": res, "gpu_launches": launches}),
          flush=True)


def end_to_end(mxq, xw_b, xa_b, dev, steps):
    """The same step through the public call with the inputs in pinned host memory and the
    outputs read back to pinned host memory, every step: host-to-device copies on one stream,
    the two QDQ calls on another, device-to-host copies on a third, two device buffer sets so
    that step i+1's inbound copies overlap step i's outbound ones (the host link is full
    duplex). Timed from the first inbound copy to the last outbound one."""
    import torch
    hw = torch.from_numpy(xw_b.view(np.int16)).pin_memory()
    ha = torch.from_numpy(xa_b.view(np.int16)).pin_memory()
    ow = torch.empty_like(hw).pin_memory()
    oa = torch.empty_like(ha).pin_memory()
    bufs = [[torch.empty(t.shape, dtype=torch.int16, device=dev) for t in (hw, ha, hw, ha)]
            for _ in range(2)]
    s_in, s_qdq, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)
    loaded = [ev() for _ in range(2)]
    computed = [ev() for _ in range(2)]
    drained = [ev() for _ in range(2)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(n, timed):
        torch.cuda.synchronize()
        for i in range(n):
            j = i % 2
            xw, xa, yw, ya = bufs[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[j])  # buffer set j no longer read by step i-2
                if timed and i == 0:
                    t0.record(s_in)
                xw.copy_(hw, non_blocking=True)
                xa.copy_(ha, non_blocking=True)
                loaded[j].record(s_in)
            with torch.cuda.stream(s_qdq):
                s_qdq.wait_event(loaded[j])
                if i >= 2:
                    s_qdq.wait_event(drained[j])  # outputs of step i-2 already copied out
                mxq.mx_qdq(xw.view(torch.bfloat16), mxq.E2M1, y=yw.view(torch.bfloat16),
                           stream=s_qdq)
                mxq.mx_qdq(xa.view(torch.bfloat16), mxq.E2M1, y=ya.view(torch.bfloat16),
                           stream=s_qdq)
                computed[j].record(s_qdq)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[j])
                ow.copy_(yw, non_blocking=True)
                oa.copy_(ya, non_blocking=True)
                drained[j].record(s_out)
        if timed:
            t1.record(s_out)
        torch.cuda.synchronize()

    run(3, False)
    run(steps, True)
    sec = t0.elapsed_time(t1) / 1e3 / steps
    elems = hw.numel() + ha.numel()
    return {"value": 4 * elems / sec / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 2 * elems,
            "d2h_bytes_per_step": 2 * elems, "ms_per_step": sec * 1e3,
            "pipeline": "2 buffer sets; H2D, QDQ and D2H on 3 streams"}


def run_ours(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import mx_microscaling_quantize_gb300 as mxq
    from mx_microscaling_quantize_gb300 import workloads as W

    xw_b, xa_b = W.mxfp4_qdq_weight(), W.mxfp4_qdq_activation()
    xw, xa = to_gpu(xw_b, dev), to_gpu(xa_b, dev)
    yw, ya = torch.empty_like(xw), torch.empty_like(xa)
    elems = xw.numel() + xa.numel()
    step_bytes = 4 * elems  # bf16 in + bf16 out
    stream = torch.cuda.current_stream()
    peak, peak_src = hbm_peak()

    def step():
        mxq.mx_qdq(xw, mxq.E2M1, y=yw, stream=stream)
        mxq.mx_qdq(xa, mxq.E2M1, y=ya, stream=stream)

    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sleep = getattr(torch.cuda, "_sleep", None)
    with ClockSampler(local) as clocks:
        # The warm-up runs once the clock sampler is up, right before the timed region, so that
        # the region does not start on a GPU that sat idle while the sampler started.
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        # A short device-side wait (about 50 us) ahead of the region's first event: the host
        # queues the first launches meanwhile, so the region starts with its work already
        # submitted instead of on a host launch.
        if sleep is not None:
            sleep(100_000)
        t_start.record(stream)
        for _ in range(K):
            mxq.mx_qdq(xw, mxq.E2M1, y=yw, stream=stream)
            mxq.mx_qdq(xa, mxq.E2M1, y=ya, stream=stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_per_step = ms_total / K
    # Per-launch durations, after the timed region: each launch of these steps is bracketed by
    # events (which make the stream drain at every kernel boundary, so they read a little longer
    # than the launches of the timed region).
    n_sampled = min(200, max(20, K))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_sampled)]
    for e in ev:
        e[0].record(stream)
        mxq.mx_qdq(xw, mxq.E2M1, y=yw, stream=stream)
        e[1].record(stream)
        e[2].record(stream)
        mxq.mx_qdq(xa, mxq.E2M1, y=ya, stream=stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    t_weight = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_act = statistics.fmean(e[2].elapsed_time(e[3]) for e in ev) / 1e3
    launches = 2 * K
    value = step_bytes * world / (ms_per_step / 1e3) / 1e9
    # Average launch duration of the kernel: the timed region holds nothing but its launches,
    # back to back, so bytes of all launches / region time is the byte-weighted average
    # (kernel boundaries included).
    achieved = step_bytes * K / (ms_total / 1e3) / 1e9
    traffic = recorded_traffic()

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "format": "E2M1 (MXFP4)", "group": 32,
                   "elements_per_step": elems, "algorithmic_bytes_per_step": step_bytes,
                   "global_batch": 1, "seq_len": 8192, "parallelism": f"replicas x{world}",
                   "l2": "inputs+outputs 384 MiB per step > 129 MB L2; no flush"},
        "gelem_per_s": elems * world / (ms_per_step / 1e3) / 1e9,
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "kernel": "mx_stream_kernel<E2M1, QDQ>",
                     "launch_us": {"weight": t_weight * 1e6, "activation": t_act * 1e6,
                                   "region_per_step": ms_per_step * 1e3,
                                   "bracketed_steps": n_sampled,
                                   "note": "event-bracketed launches after the timed region"},
                     "traffic": None if traffic is None else traffic["traffic_bytes_per_launch"],
                     "traffic_detail": None if traffic is None else {
                         "method": traffic["method"], "launches": traffic["launches"]},
                     "algorithmic_bytes_per_launch": (4 * xw.numel() + 4 * xa.numel()) // 2,
                     "algorithmic_bytes_by_tensor": {"weight": 4 * xw.numel(),
                                                     "activation": 4 * xa.numel()}},
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.quick:
        line["e2e"] = end_to_end(mxq, xw_b, xa_b, dev, min(K, 50))
        line["workloads"] = extra_workloads(dev, peak)
        cpu_gbs, cpu_s, passes, threads = time_oracle_for(xw_b, xa_b, 10.0)
        line["cpu_baseline"] = {
            "value": cpu_gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} passes of the whole workload (E2M1 QDQ of x[8192,8192] and "
                      f"x[4096,8192]) in {cpu_s:.1f} s, row chunks on {threads} threads",
            "gelem_per_s": cpu_gbs / 4}
        one_gbs, one_s, one_passes, one_rows = time_oracle_one_core(xw_b, 2.0)
        line["cpu_baseline"]["single_core"] = {
            "value": one_gbs, "unit": "GB/s", "cores": 1,
            "sample": f"{one_passes} passes of the weight's first {one_rows} rows "
                      f"(E2M1 QDQ of x[{one_rows},8192]) in {one_s:.1f} s on one thread"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.case:
        run_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
