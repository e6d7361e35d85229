"""Benchmark of the software-pipelined tiled GEMM (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--stages S] [--no-e2e]

A step is one GEMM of the workload on one set of inputs already resident in
device memory. The default workload is the binary16 4096 x 4096 x 4096
product with a binary16 output; the metric is TFLOPS (TOPS for int8).

L2 policy: the inputs and outputs rotate over several device copies whose
total size is well above the 129 MB L2, so every step reads its operands from
HBM, not from what the previous step left in L2.

`value` is timed with CUDA events on the launching stream around exactly K
steps, between a barrier + synchronize on each side, max over ranks. `e2e`
is the same metric through the public API from pinned host buffers, the
host->device copies of A and B and the device->host copy of C inside the
timed region. `cpu_baseline` is the CPU oracle (fp64 triple loop) timed on the
host cores on a bounded sample of the same workload.

`parity` compares the output of the last timed step with the oracle on the
rows of that sample (all rows when the oracle finishes them in time).

`workloads` adds the other four workloads, each timed on its own in the same
way (its own rotating sets, warm-up, CUDA events; a product whose host issue
time rivals its run time is also replayed as one CUDA graph, and that time is
reported, with the stream-launched one under `launch`), with its roofline, the
oracle on a bounded sample (a few seconds) and a parity verdict on its own
output: every element where the oracle covers all rows, else every element
of the sampled rows plus 4096 random positions. --no-workloads skips them.

--impl reference times that oracle as the reference arm on the same
workload, each step a bounded sample (a block of output rows).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, WORKLOAD_ORDER, TORCH_DTYPE, workload_inputs  # noqa: E402

DEFAULT_WORKLOAD = "f16_4096x4096x4096_f16out"
L2_BYTES = 129 * 10 ** 6
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def metric_for(w):
    if w.in_type == "s8":
        return "int8 GEMM TOPS", "TOPS"
    return "GEMM TFLOPS", "TFLOPS"


def algorithmic_bytes(w):
    isz = 1 if w.in_type == "s8" else 2
    osz = {"f32": 4, "s32": 4, "f16": 2, "bf16": 2}[w.out_type]
    return (w.M * w.K + w.N * w.K) * isz + w.M * w.N * osz


def bound_for(w):
    # arithmetic intensity against the machine balance decides the roof
    peaks, _ = measured_peaks()
    balance = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = w.flops / algorithmic_bytes(w)
    return "tensor" if ai >= balance else "hbm"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                clk = float(f[1])
                mx = float(f[2])
            except ValueError:
                continue
            try:
                power = float(f[3])
            except ValueError:
                power = None
            sm.append(clk)
            pw.append(power)
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        # The median over samples taken under load: those drawing at least half
        # the run's highest power (an idle GPU sits at its maximum clock, so
        # the samples before and after the timed region would otherwise hide a
        # clock the power cap pulled down), else those above 30 % of the
        # maximum clock when no power figure was read.
        known = [p for p in pw if p is not None]
        if known:
            top = max(known)
            loaded = sorted(c for c, p in zip(sm, pw) if p is not None and p >= 0.5 * top)
        else:
            loaded = sorted(c for c in sm if c > 0.3 * (mx or c))
        loaded = loaded or sorted(sm)
        return {"sm_mhz": loaded[len(loaded) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(loaded)}


def sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "software_pipelined_tiled_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(f"{kernel}/{workload}")
        if rec and rec.get("sources") == sources_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------- CPU oracle leg
def oracle_sample(w, A, B, target_s: float = 12.0):
    """Times the CPU oracle on a leading block of output rows (about target_s seconds)."""
    import oracle
    it = {"f16": oracle.IN_F16, "bf16": oracle.IN_BF16}.get(w.in_type)

    def run_rows(r):
        t0 = time.perf_counter()
        if w.in_type == "s8":
            oracle.gemm_s8(A[:r], B)
        else:
            oracle.gemm_float(A[:r], B, it)
        return time.perf_counter() - t0

    probe = min(w.M, max(1, 2 * oracle.threads()))
    run_rows(probe)  # loads the oracle library and warms the caches
    t = run_rows(probe)
    rows = int(min(w.M, max(probe, probe * target_s / max(t, 1e-6))))
    return rows, oracle.threads()


def oracle_rows(w, A, B, rows: int):
    """The oracle on output rows 0..rows-1: (seconds, result); the result is
    (C_ref, sum_k |A_ik B_kj|) in fp64 for float inputs, the int64 C for int8."""
    import oracle
    t0 = time.perf_counter()
    if w.in_type == "s8":
        res = oracle.gemm_s8(A[:rows], B)
    else:
        res = oracle.gemm_float(A[:rows], B, {"f16": oracle.IN_F16, "bf16": oracle.IN_BF16}[w.in_type])
    return time.perf_counter() - t0, res


def cpu_baseline(w, A, B, target_s: float = 12.0):
    """The oracle timed on a leading block of output rows (about target_s
    seconds); returns (cpu_baseline record, rows, oracle result)."""
    rows, cores = oracle_sample(w, A, B, target_s)
    dt, res = oracle_rows(w, A, B, rows)
    _, unit = metric_for(w)
    rec = {"value": 2.0 * rows * w.N * w.K / dt / 1e12, "unit": unit, "cores": cores,
           "kind": "oracle",
           "sample": f"output rows 0..{rows - 1} of {w.M} ({rows}x{w.N}x{w.K}), {dt:.1f} s"}
    return rec, rows, res


# The element-wise bar of the float workloads: |C - C_ref| <= 1e-3 sum_k |A_ik B_kj|
# for the fp32-accumulated sum, plus the round-to-nearest of a 16-bit output
# (unit roundoff u); int8 results must equal the oracle's.
PARITY_TOL = 1e-3
OUT_U = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def parity_verdict(w, C, A, B, rows: int, res, n_random: int = 0):
    """Compares this run's own output C (host tensor) with the oracle: every
    element of rows 0..rows-1 (res is the oracle's result for them) and
    n_random uniformly drawn positions of the whole matrix."""
    import numpy as np
    import oracle
    checked = "every element" if rows == w.M else f"every element of rows 0..{rows - 1}"
    if n_random:
        g = np.random.default_rng(w.seed)
        r = g.integers(0, w.M, n_random).astype(np.int64)
        c = g.integers(0, w.N, n_random).astype(np.int64)
        checked += f" + {n_random} random positions"
    if w.in_type == "s8":
        got = C[:rows].to(torch.int64).numpy()
        bad = int((got != res).sum())
        n = got.size
        if n_random:
            ref_r = oracle.gemm_s8_at(A, B, r, c)
            bad += int((C.to(torch.int64).numpy()[r, c] != ref_r).sum())
            n += n_random
        return {"checked": checked, "elements": int(n), "rule": "bit-exact", "ok": bad == 0,
                "mismatches": bad}
    ref, S = res
    u = OUT_U[w.out_type]
    full = C.to(torch.float64).numpy()
    gots, refs, sums = [full[:rows]], [ref], [S]
    if n_random:
        it = {"f16": oracle.IN_F16, "bf16": oracle.IN_BF16}[w.in_type]
        ref_r, S_r = oracle.gemm_float_at(A, B, it, r, c)
        gots.append(full[r, c])
        refs.append(ref_r)
        sums.append(S_r)
    worst, worst_plain, bad, n = 0.0, 0.0, 0, 0
    tiny = np.finfo(np.float64).tiny
    for got, rf, sm in zip(gots, refs, sums):
        err = np.abs(got - rf)
        bound = PARITY_TOL * sm + u * (np.abs(rf) + PARITY_TOL * sm)
        bad += int((~(err <= bound)).sum())
        n += err.size
        worst = max(worst, float((err / np.maximum(bound, tiny)).max()))
        worst_plain = max(worst_plain, float((err / np.maximum(PARITY_TOL * sm, tiny)).max()))
    return {"checked": checked, "elements": int(n),
            "rule": "|C - C_ref| <= 1e-3 sum|ab| + u (|C_ref| + 1e-3 sum|ab|)", "ok": bad == 0,
            "outside": bad, "max_err_over_bound": worst,
            "max_err_over_1e-3_sum_abs": worst_plain}


# ------------------------------------------------------------- GPU leg
def init_dist(n_gpus, backend: str = "nccl"):
    """One process per GPU (torchrun env); replicas only, no data-path collective."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: every replica's measurement is reduced with MAX."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's time (per ms)."""
    return world * units_per_rank / ms_max


def _page_numa_node(ptr: int):
    """NUMA node of the page holding host address ptr (Linux move_pages query), or None."""
    import ctypes
    import platform
    nr = {"aarch64": 239, "x86_64": 279}.get(platform.machine())
    if nr is None:
        return None
    libc = ctypes.CDLL(None, use_errno=True)
    pages = (ctypes.c_void_p * 1)(ptr)
    status = (ctypes.c_int * 1)(-1)
    if libc.syscall(nr, 0, 1, pages, None, status, 0) != 0:
        return None
    return int(status[0])


def host_link(h_in, h_out, dev, reps: int = 8):
    """Copy rates of the host link with the end-to-end leg's own pinned buffers
    (GB/s, CUDA events): host->device alone, device->host alone, and both at
    once on two streams; plus where the buffers' pages and the GPU sit."""
    import glob
    d_in = torch.empty(h_in.numel() * h_in.element_size(), dtype=torch.uint8, device=dev)
    d_out = torch.empty(h_out.numel() * h_out.element_size(), dtype=torch.uint8, device=dev)
    hi = h_in.view(-1).view(torch.uint8)
    ho = h_out.view(-1).view(torch.uint8)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        e0.record(cur)
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        for _ in range(reps):
            fn()
        cur.wait_stream(s1)
        cur.wait_stream(s2)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    def up():
        with torch.cuda.stream(s1):
            d_in.copy_(hi, non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            ho.copy_(d_out, non_blocking=True)

    def both():
        up()
        down()

    t_up, t_down, t_both = timed(up), timed(down), timed(both)
    nin, nout = d_in.numel(), d_out.numel()
    gpu_node = None
    try:
        pr = torch.cuda.get_device_properties(dev)
        addr = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{addr}/numa_node") as f:
            gpu_node = int(f.read())
    except Exception:
        gpu_node = None
    return {"h2d_gbs": nin * reps / t_up / 1e9, "d2h_gbs": nout * reps / t_down / 1e9,
            "both_gbs": (nin + nout) * reps / t_both / 1e9,
            "numa_nodes": len(glob.glob("/sys/devices/system/node/node[0-9]*")),
            "gpu_numa_node": gpu_node,
            "pinned_in_page_node": _page_numa_node(h_in.data_ptr()),
            "pinned_out_page_node": _page_numa_node(h_out.data_ptr())}


def run_ours(args, w):
    import software_pipelined_tiled_gb300 as sptg

    rank, world, local = init_dist(args.gpus)
    sptg.load()
    metric, unit = metric_for(w)
    A, B = workload_inputs(w)
    out_dtype = TORCH_DTYPE[w.out_type]
    set_bytes = algorithmic_bytes(w)
    n_sets = max(2, -(-3 * L2_BYTES // set_bytes) + 1)  # total well above L2
    dev = torch.device("cuda", local)
    As = [A.to(dev) for _ in range(n_sets)]
    Bs = [B.to(dev) for _ in range(n_sets)]
    Cs = [torch.empty(w.M, w.N, dtype=out_dtype, device=dev) for _ in range(n_sets)]
    cfg = None
    if args.kernel or args.stages or args.bn or args.cta_pair or args.no_overlap or args.stream_k:
        cfg = sptg.Config(args.kernel, args.bn, args.stages, 0, 0, 0, args.cta_pair,
                          int(args.no_overlap))
        cfg.stream_k = args.stream_k
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % n_sets
        sptg.gemm(As[j], Bs[j], C=Cs[j], config=cfg)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if sptg.device_error() != 0:
        raise RuntimeError("kernel reported a timed-out wait during warm-up")
    launches_per_step = int(sptg.last_config().split("launches=")[-1].split()[0])
    kernel_name = sptg.last_config().split()[0].split("=")[1]

    graph = None
    if args.graph:
        # the K timed steps captured once as a CUDA graph on a side stream
        # (warm-up on that stream first, so its scratch exists before capture)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for i in range(args.warmup):
                step(i)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(args.steps):
                step(i)
        torch.cuda.synchronize()
        # replay() launches on the current stream, where the events are recorded

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    ev1.record(stream)
    host_us = (time.perf_counter() - h0) * 1e6 / args.steps
    torch.cuda.synchronize()
    barrier(world)
    if rank == 0:
        sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    value = job_throughput(w.flops, world, ms_per_step) * 1e3 / 1e12
    if sptg.device_error() != 0:
        raise RuntimeError("kernel reported a timed-out wait in the timed region")
    # the output of the last timed step, for the parity verdict
    C_check = Cs[(args.steps - 1) % n_sets].cpu() if rank == 0 else None

    # ---- end to end through the public API from pinned host memory
    # Each step is one sptg_gemm_host call on pinned host buffers: the copy of
    # that step's A and B to the device, the product, and the copy of C back
    # to the host. Steps alternate over two streams (one set of library-owned
    # device buffers each), so one step's copies overlap the neighbouring
    # step's product and copies in the other direction.
    e2e = None
    if not args.no_e2e:
        hA, hB = A.pin_memory(), B.pin_memory()
        lanes = [torch.cuda.Stream(), torch.cuda.Stream()]
        hCs = [torch.empty(w.M, w.N, dtype=out_dtype).pin_memory() for _ in lanes]
        e2e_steps = max(8, min(args.steps, 48))

        def e2e_run(n):
            for lane in lanes:
                lane.wait_stream(stream)
            for i in range(n):
                j = i % 2
                sptg.gemm_host(hA, hB, C=hCs[j], stream=lanes[j], config=cfg)
            for lane in lanes:
                stream.wait_stream(lane)

        e2e_run(4)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        if sptg.device_error() != 0:
            raise RuntimeError("kernel reported a timed-out wait in the end-to-end leg")
        e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
        isz = A.element_size()
        h2d = (A.numel() + B.numel()) * isz
        d2h = hCs[0].numel() * hCs[0].element_size()
        e2e = {"value": world * w.flops / (e_ms * 1e-3) / 1e12, "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms, "api": "sptg_gemm_host, steps alternating over 2 streams"}
        link = host_link(hA, hCs[0], dev)
        # the step's copies alone, at the link's measured rates: each direction
        # on its own, and both directions sharing the link
        bound_ms = max(h2d / link["h2d_gbs"], d2h / link["d2h_gbs"],
                       (h2d + d2h) / link["both_gbs"]) / 1e6
        link["copy_bound_ms_per_step"] = bound_ms
        link["e2e_over_copy_bound"] = e_ms / bound_ms
        e2e["host_link"] = link

    # ---- the other workloads, each timed on its own (all ranks), with its
    # roofline, the oracle on a bounded sample and a parity verdict (rank 0)
    extras = {}
    if not args.no_workloads and not args.shape:
        for name in WORKLOAD_ORDER:
            if name != w.name:
                entry = run_workload(args, WORKLOADS[name], rank, world, local, sptg)
                if entry is not None:
                    extras[name] = entry

    if rank != 0:
        return None

    clocks = sampler.summary()
    roof = roofline(w, ms_per_step, ms, clocks, kernel_name, set_bytes)

    tl = None
    if args.trace:
        fields = (args.kernel, args.bn, args.stages, 0, 0, 0, args.cta_pair, int(args.no_overlap),
                  args.stream_k)
        tl = timeline(sptg, As[0], Bs[0], Cs[0], fields)
    cpu, parity = None, None
    if not args.no_cpu_baseline:
        cpu, rows, res = cpu_baseline(w, A, B)
        parity = parity_verdict(w, C_check, A, B, rows, res)
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.in_type, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype_pair": w.dtype,
                   "distribution": w.dist, "seed": w.seed, "kernel": sptg.last_config(),
                   "l2": f"{n_sets} rotating input/output sets of {set_bytes / 2**20:.0f} MiB "
                         f"(> L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof, "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
        "launch": {"mode": "cuda-graph" if graph is not None else "stream",
                   "host_us_per_step": host_us,
                   "overlap_previous": not args.no_overlap},
    }
    if tl is not None:
        line["timeline"] = tl
    if extras:
        line["workloads"] = extras
    return line


# NVIDIA's published dense (no 2:4 sparsity) FP16/BF16 tensor peaks for one
# Blackwell Ultra GPU, in TFLOP/s: the HGX B300 board lists 36 PFLOPS with
# sparsity for 8 GPUs, the GB300 NVL72 rack 360 PFLOPS with sparsity for 72;
# halving for sparsity gives 2.25 and 2.5 PFLOPS dense per GPU. The int8 path
# runs on the binary16 tensor pipe (sm_103a has no tcgen05 int8 MMA), so the
# same figures bound it.
DENSE_SPEC_TFLOPS = {"hgx_b300": 2250.0, "gb300_nvl72": 2500.0}


def roofline(w, ms_per_step, timed_ms, clocks, kernel_name, set_bytes):
    """The roofline record of one timed workload (achieved = algorithmic work
    per launch / the launch's event-timed average duration)."""
    peaks, peak_src = measured_peaks()
    bound = bound_for(w)
    # The timed region runs the kernel back to back. Once that lasts over a
    # second, or the power cap pulled the SM clock down (median under load
    # below 90 % of its maximum), the sustained figure, taken under the same
    # cap at lowered clocks, is the matching denominator; else the burst one.
    # A cap that is flagged while the clock stays at its maximum does not
    # slow the kernel, so the burst figure stays.
    sm, sm_max = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    clock_dropped = bool(sm and sm_max and sm < 0.9 * sm_max)
    sustained = timed_ms > 1000.0 or ("sw_power_cap" in clocks.get("reasons", [])
                                      and clock_dropped)
    if bound == "tensor":
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        achieved = w.flops / (ms_per_step * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "frac_burst": achieved / peaks["bf16_tflops"],
                "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peak_src} bf16 {'sustained' if sustained else 'burst'} "
                               f"(binary16 and the int8 path run at the bfloat16 rate)",
                "frac_dense_spec": achieved / DENSE_SPEC_TFLOPS["hgx_b300"],
                "frac_dense_spec_nvl72": achieved / DENSE_SPEC_TFLOPS["gb300_nvl72"],
                "dense_spec_tflops": dict(DENSE_SPEC_TFLOPS)}
    else:
        peak = peaks["hbm_gbs"]
        achieved = set_bytes / (ms_per_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} copy bandwidth"}
    roof["traffic"] = recorded_traffic(kernel_name, w.name)
    roof["algorithmic_bytes"] = set_bytes
    roof["kernel"] = kernel_name
    return roof


WORKLOAD_ORACLE_S = 4.0  # oracle seconds per additional workload
WORKLOAD_MIN_MS = 20.0   # shortest timed region of an additional workload


def run_workload(args, w, rank, world, local, sptg):
    """One additional workload: its own inputs in rotating device sets (> L2),
    W warm-up steps, then a timed region of back-to-back steps (at least
    args.steps, more for tiny products so that it lasts WORKLOAD_MIN_MS),
    CUDA events on the launching stream, max over ranks. Rank 0 adds the
    roofline, the oracle on a bounded sample of output rows and a parity
    verdict on the output of the last timed step."""
    dev = torch.device("cuda", local)
    A, B = workload_inputs(w)
    out_dtype = TORCH_DTYPE[w.out_type]
    set_bytes = algorithmic_bytes(w)
    n_sets = max(2, -(-3 * L2_BYTES // set_bytes) + 1)
    As = [A.to(dev) for _ in range(n_sets)]
    Bs = [B.to(dev) for _ in range(n_sets)]
    Cs = [torch.empty(w.M, w.N, dtype=out_dtype, device=dev) for _ in range(n_sets)]
    stream = torch.cuda.current_stream()

    def run(n):
        for i in range(n):
            j = i % n_sets
            sptg.gemm(As[j], Bs[j], C=Cs[j])

    run(args.warmup)
    torch.cuda.synchronize()
    if sptg.device_error() != 0:
        raise RuntimeError(f"{w.name}: a kernel reported a timed-out wait during warm-up")
    kernel_cfg = sptg.last_config()
    launches_per_step = int(kernel_cfg.split("launches=")[-1].split()[0])
    kernel_name = kernel_cfg.split()[0].split("=")[1]
    # size the timed region: one probe batch of args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    probe_ms = max_over_ranks(e0.elapsed_time(e1), world)
    steps = args.steps
    if probe_ms < WORKLOAD_MIN_MS:
        steps = int(min(20000, -(-args.steps * WORKLOAD_MIN_MS // max(probe_ms, 1e-3))))
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    e0.record(stream)
    run(steps)
    e1.record(stream)
    host_us = (time.perf_counter() - h0) * 1e6 / steps
    torch.cuda.synchronize()
    barrier(world)
    if rank == 0:
        sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    if sptg.device_error() != 0:
        raise RuntimeError(f"{w.name}: a kernel reported a timed-out wait in the timed region")
    launch = {"mode": "stream", "host_us_per_step": host_us, "stream_ms_per_step": ms / steps}
    # A product so small that issuing it from the host takes about as long as
    # running it measures the host: then the same steps are also captured as
    # one CUDA graph and replayed, and the graph's time is the device's.
    if host_us >= 0.8 * 1e3 * ms / steps:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            run(args.warmup)  # the library's buffers for this stream exist before capture
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            run(steps)
        torch.cuda.synchronize()
        graph.replay()  # warm
        torch.cuda.synchronize()
        barrier(world)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(e0.elapsed_time(e1), world)
        if sptg.device_error() != 0:
            raise RuntimeError(f"{w.name}: a kernel reported a timed-out wait in the graph replay")
        launch["mode"] = "cuda-graph"
        launch["why"] = "host issue time per step >= 0.8 x the stream-launched step time"
    if rank != 0:
        return None
    ms_per_step = ms / steps
    metric, unit = metric_for(w)
    C = Cs[(steps - 1) % n_sets].cpu()
    del As, Bs, Cs
    clocks = sampler.summary()
    entry = {"metric": metric, "value": job_throughput(w.flops, world, ms_per_step) * 1e3 / 1e12,
             "unit": unit, "ms_per_step": ms_per_step, "steps": steps, "warmup": args.warmup,
             "dtype": w.in_type,
             "config": {"M": w.M, "N": w.N, "K": w.K, "dtype_pair": w.dtype,
                        "distribution": w.dist, "seed": w.seed, "kernel": kernel_cfg,
                        "l2": f"{n_sets} rotating input/output sets of "
                              f"{set_bytes / 2**20:.1f} MiB (> L2)"},
             "roofline": roofline(w, ms_per_step, ms, clocks, kernel_name, set_bytes),
             "gpu_launches": launches_per_step * steps, "clocks": clocks, "launch": launch}
    if bound_for(w) == "hbm":
        entry["gbs"] = entry["roofline"]["achieved"]
    if w.M * w.N <= 256 * 256:
        entry["roofline"]["note"] = "latency-bound: the product is two output tiles"
    if not args.no_cpu_baseline:
        cpu, rows, res = cpu_baseline(w, A, B, target_s=WORKLOAD_ORACLE_S)
        entry["cpu_baseline"] = cpu
        entry["parity"] = parity_verdict(w, C, A, B, rows, res,
                                         n_random=0 if rows == w.M else 4096)
    return entry


TRACE_EVENTS = ["setup", "first_load", "first_data", "last_load", "last_mma", "epi_done",
                "exit", "fixup_done"]
TRACE_WORDS = 8 * 1024 + 2 * 64


def timeline(sptg, A, B, C, cfg_fields):
    """One traced call: per-event spread over CTAs and CTA 0's K-tile detail."""
    import numpy as np
    buf = torch.zeros(TRACE_WORDS, dtype=torch.int64, device=A.device)
    cfg = sptg.Config(*cfg_fields[:8])
    if len(cfg_fields) > 8:
        cfg.stream_k = cfg_fields[8]
    cfg.trace = buf.data_ptr()
    sptg.gemm(A, B, C=C, config=cfg)
    torch.cuda.synchronize()
    t = buf.cpu().numpy().astype(np.int64)
    grid = int(sptg.last_config().split("grid=")[1].split()[0])
    ev = t[:8 * 1024].reshape(1024, 8)[:grid]
    t0 = ev[:, 0][ev[:, 0] > 0].min()
    out = {"ctas": grid}
    for i, name in enumerate(TRACE_EVENTS):
        col = ev[:, i][ev[:, i] > 0]
        if len(col):
            us = (col - t0) / 1e3
            out[name + "_us"] = [round(float(us.min()), 2), round(float(np.median(us)), 2),
                                 round(float(us.max()), 2)]
    issue = t[8 * 1024: 8 * 1024 + 64]
    full = t[8 * 1024 + 64: 8 * 1024 + 128]
    n = int(min((issue > 0).sum(), (full > 0).sum()))
    if n:
        lat = (full[:n] - issue[:n]) / 1e3
        ahead = [int(((issue[:n] > 0) & (issue[:n] <= full[i])).sum()) - (i + 1) for i in range(n)]
        out["cta0_ktiles"] = n
        out["cta0_issue_to_full_us"] = [round(float(lat.min()), 2), round(float(np.median(lat)), 2),
                                        round(float(lat.max()), 2)]
        out["cta0_tiles_in_flight_at_consume"] = [int(min(ahead)), int(np.median(ahead)),
                                                  int(max(ahead))]
    return out


VERSUS_SHAPES = ("4096,4096,4096,f16_f16;2048,2048,2048,f16_f16;8192,8192,4096,f16_f16;"
                 "6144,6144,6144,f16_f16;8192,8192,8192,bf16_bf16;8192,8192,16384,bf16_bf16;"
                 "8192,8192,16384,bf16_f32;16384,16384,4096,bf16_bf16;4096,4096,4096,s8_s32;"
                 "64,8192,8192,bf16_bf16;128,8192,8192,bf16_bf16;64,16384,4096,bf16_bf16")


def torch_product(pair: str):
    """The PyTorch call that computes the same product, and its name.

    Same-type outputs use torch.matmul; a 16-bit product with a binary32
    output uses torch.mm's out_dtype where this PyTorch has it; int8 uses
    torch._int_mm (int32 output).  None where PyTorch has no such call.
    """
    in_t, out_t = pair.split("_")
    if in_t == "s8":
        return (lambda A, Bcm, C: torch._int_mm(A, Bcm.t(), out=C)), "torch._int_mm"
    if in_t == out_t:
        return (lambda A, Bcm, C: torch.matmul(A, Bcm.t(), out=C)), "torch.matmul"
    return (lambda A, Bcm, C: torch.mm(A, Bcm.t(), out_dtype=torch.float32, out=C)), \
        "torch.mm(out_dtype=float32)"


def run_versus_torch(args):
    """This library against PyTorch's own GEMM on the same inputs and outputs.

    Per shape: inputs drawn as the workloads draw them (uniform, seed 3; int8
    over its whole range), rotated over device sets whose total is above L2.
    Each side runs `iters` back-to-back calls between CUDA events, five
    times, medians kept; the order is ours, PyTorch, ours, PyTorch and the
    better median of each side is reported.  One JSON line per shape.
    """
    import statistics
    import software_pipelined_tiled_gb300 as sptg
    from workloads import DTYPE_PAIRS, make_inputs

    sptg.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()

    def timed(fn, iters, n_sets):
        meds = []
        for _ in range(5):
            for i in range(3):
                fn(i % n_sets)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(iters):
                fn(i % n_sets)
            e1.record(stream)
            torch.cuda.synchronize()
            meds.append(e0.elapsed_time(e1) * 1e3 / iters)
        return statistics.median(meds)

    sampler = ClockSampler(0)
    sampler.start()
    lines = []
    for spec in args.shapes.split(";"):
        m, n, k, pair = spec.split(",")
        M, N, K = int(m), int(n), int(k)
        in_t, out_t = DTYPE_PAIRS[pair]
        A, B = make_inputs(M, N, K, in_t, "int8" if in_t == "s8" else "uniform", 3)
        el_in, el_out = A.element_size(), torch.empty((), dtype=TORCH_DTYPE[out_t]).element_size()
        set_bytes = (M * K + N * K) * el_in + M * N * el_out
        n_sets = max(2, -(-3 * L2_BYTES // set_bytes) + 1)
        As = [A.to(dev) for _ in range(n_sets)]
        Bs = [B.to(dev) for _ in range(n_sets)]
        Cs = [torch.empty(M, N, dtype=TORCH_DTYPE[out_t], device=dev) for _ in range(n_sets)]
        est_s = max(2.0 * M * N * K / 1.5e15, set_bytes / 5e12)
        iters = int(min(2000, max(10, 0.03 / est_s)))
        theirs_fn, theirs_name = torch_product(pair)

        def ours(j):
            sptg.gemm(As[j], Bs[j], C=Cs[j])

        def theirs(j):
            theirs_fn(As[j], Bs[j], Cs[j])

        try:
            theirs(0)
            torch.cuda.synchronize()
        except (RuntimeError, TypeError) as e:
            theirs_fn = None
            theirs_note = f"{theirs_name} unavailable: {str(e).splitlines()[0][:120]}"
        t_ours = [timed(ours, iters, n_sets)]
        t_theirs = []
        if theirs_fn is not None:
            t_theirs.append(timed(theirs, iters, n_sets))
        t_ours.append(timed(ours, iters, n_sets))
        if theirs_fn is not None:
            t_theirs.append(timed(theirs, iters, n_sets))
        if sptg.device_error() != 0:
            raise RuntimeError("kernel reported a timed-out wait")
        us_ours = min(t_ours)
        us_theirs = min(t_theirs) if t_theirs else None
        flops = 2.0 * M * N * K
        line = {"shape": [M, N, K], "dtype": pair, "iters": iters, "sets": n_sets,
                "ours_us": round(us_ours, 3), "ours_tflops": round(flops / us_ours / 1e6, 1),
                "ours_config": sptg.last_config(),
                "torch_call": theirs_name, "torch_us": None, "torch_tflops": None,
                "torch_us_over_ours": None}
        if us_theirs is not None:
            line.update(torch_us=round(us_theirs, 3),
                        torch_tflops=round(flops / us_theirs / 1e6, 1),
                        torch_us_over_ours=round(us_theirs / us_ours, 3))
        else:
            line["torch_note"] = theirs_note
        lines.append(line)
        del As, Bs, Cs
        torch.cuda.empty_cache()
    sampler.stop()
    clocks = sampler.summary()
    for line in lines:
        line["clocks"] = clocks
        line["torch_version"] = torch.__version__
    return lines


def run_stream(args):
    """The streaming ring on its own (out = alpha * in, binary32): HBM roofline probe."""
    import software_pipelined_tiled_gb300 as sptg
    torch.cuda.set_device(0)
    n = args.stream
    nbytes = 8 * n  # read + write
    n_sets = max(2, -(-3 * L2_BYTES // nbytes) + 1)
    g = torch.Generator("cpu").manual_seed(1)
    x = torch.randn(n, generator=g)
    xs = [x.cuda() for _ in range(n_sets)]
    ys = [torch.empty_like(xs[0]) for _ in range(n_sets)]
    for i in range(args.warmup):
        sptg.stream_scale(xs[i % n_sets], 2.0, out=ys[i % n_sets])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(0)
    sampler.start()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        sptg.stream_scale(xs[i % n_sets], 2.0, out=ys[i % n_sets])
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    if sptg.device_error() != 0:
        raise RuntimeError("kernel reported a timed-out wait")
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, src = measured_peaks()
    tl = None
    if args.trace:
        buf = torch.zeros(TRACE_WORDS, dtype=torch.int64, device="cuda")
        cfg = sptg.Config()
        cfg.trace = buf.data_ptr()
        sptg.stream_scale(xs[0], 2.0, out=ys[0], config=cfg)
        torch.cuda.synchronize()
        tl = buf[:16].cpu().tolist()
    return {"metric": "stream scale GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"stream_scale_f32_n{n}", "kernel": sptg.last_config(),
                       "l2": f"{n_sets} rotating buffer pairs of {nbytes / 2**20:.0f} MiB"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{src} copy bandwidth",
                         "traffic": None, "algorithmic_bytes": nbytes},
            "clocks": sampler.summary(), "gpu_launches": args.steps}


def run_reference(args, w):
    """The CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return None
    import oracle
    metric, unit = metric_for(w)
    A, B = workload_inputs(w)
    total_budget = 150.0  # seconds for warm-up + timed steps together
    per_step = total_budget / max(1, args.steps + args.warmup)
    rows, cores = oracle_sample(w, A, B, target_s=min(12.0, per_step))
    it = {"f16": oracle.IN_F16, "bf16": oracle.IN_BF16}.get(w.in_type)

    def step():
        if w.in_type == "s8":
            oracle.gemm_s8(A[:rows], B)
        else:
            oracle.gemm_float(A[:rows], B, it)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * w.N * w.K / dt / 1e12
    sample = f"each step: output rows 0..{rows - 1} of {w.M} ({rows}x{w.N}x{w.K})"
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.in_type,
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype_pair": w.dtype,
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="M,N,K,dtype_pair: time another shape (seed 1, values per --dist)")
    ap.add_argument("--dist", default=None, choices=["uniform", "normal", "int8", "zeros"],
                    help="--shape inputs: 2 U[0,1) - 1 (default for floats), N(0,1), every "
                         "int8 value (default for int8), or all zero")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--stages", type=int, default=0, help="force the ring depth (ablation)")
    ap.add_argument("--bn", type=int, default=0, help="force the square tile width")
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3, 4, 5],
                    help="0 choose, 1 square, 2 skinny stream-K, 3 skinny cluster split, "
                         "4 skinny column strips (M <= 64), 5 skinny CTA pairs (M <= 256)")
    ap.add_argument("--cta-pair", type=int, default=0, choices=[0, 1, 2],
                    help="square kernel: 0 choose, 1 one CTA per tile, 2 CTA pair (2-SM MMA)")
    ap.add_argument("--stream-k", type=int, default=0, choices=[0, 1, 2],
                    help="square kernel: 0 stream-K for a partial last round, 1 never, 2 always")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stream", type=int, default=0,
                    help="time the streaming ring out = 2 * in over this many binary32 values")
    ap.add_argument("--graph", action="store_true",
                    help="capture the timed steps as one CUDA graph and replay it")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--trace", action="store_true",
                    help="add one traced call's in-kernel timeline to the JSON line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the chosen workload only (not the other four as well)")
    ap.add_argument("--sweep", default=None, metavar="DTYPE_PAIR",
                    help="time M = N = K over --sizes for one dtype pair (one JSON line per size; "
                         "no end-to-end or CPU legs)")
    ap.add_argument("--sizes", default="512,1024,2048,4096,8192")
    ap.add_argument("--versus-torch", action="store_true",
                    help="time this library beside PyTorch's own GEMM over --shapes "
                         "(one JSON line per shape)")
    ap.add_argument("--shapes", default=VERSUS_SHAPES, metavar="M,N,K,PAIR;...")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.shape:
        from workloads import Workload
        m, n, k, pair = args.shape.split(",")
        dist = args.dist or ("int8" if pair.startswith("s8") else "uniform")
        w = Workload(f"{pair}_{m}x{n}x{k}" + (f"_{dist}" if args.dist else ""), int(m), int(n),
                     int(k), pair, dist, 1.0, 1)
    else:
        w = WORKLOADS[args.workload]
    if args.sweep:
        from workloads import Workload
        args.no_e2e = args.no_cpu_baseline = args.no_workloads = True
        for size in (int(x) for x in args.sizes.split(",")):
            sw = Workload(f"{args.sweep}_{size}x{size}x{size}", size, size, size, args.sweep,
                          "int8" if args.sweep.startswith("s8") else "uniform", 1.0, 1)
            # about 50 ms of timed work per size at ~1.5 PFLOP/s
            args.steps = int(min(2000, max(20, 0.05 / (2.0 * size ** 3 / 1.5e15))))
            line = run_ours(args, sw)
            if line is not None:
                print(json.dumps(line), flush=True)
        return
    if args.versus_torch:
        for line in run_versus_torch(args):
            print(json.dumps(line), flush=True)
        return
    if args.stream:
        line = run_stream(args)
    else:
        line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)
    if args.impl == "ours" and int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
