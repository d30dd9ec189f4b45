"""Benchmark: Reverse All2All (combine) GB/s on the DeepSeek-V3-shaped workload.

One step = one all2all_combine through the C ABI over W=8 emulated PEs
(per PE (16384, 1, 7168) bf16 -> (2048, 8, 7168)): T = 1.879 GB read and
1.879 GB written.  GB/s = 2*T / step time.  The input (1.88 GB) is larger
than L2, so no flush is needed between steps.  After the timed steps the
other configurations' headline variants are timed in the same process and
reported under `variants`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--variant direct|pc]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Ranks: under torchrun (WORLD_SIZE set) this process is one rank.  Otherwise
`--gpus N` with N > 1 starts N processes itself, one per GPU (RANK,
LOCAL_RANK, WORLD_SIZE, MASTER_ADDR=127.0.0.1 and a free MASTER_PORT in
their environment).  Every rank runs its own replica on its own GPU (the W
PEs are emulated inside one GPU; there is no cross-GPU exchange); the
process group carries only the barrier and the max of the step times, and
the value is all ranks' bytes over that max.  `--dry-run` runs the same
orchestration without a GPU (gloo, a host-side stand-in step) so that the
launcher can be checked on CPU; it prints no benchmark figure.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "reverse-All2All combine GB/s (read+write) and % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "dsv3"
# producer/consumer tiling of the DeepSeek-V3 step: 12 x 1024 tiles, 3
# buffers (a 33 MB staging ring; measured best of 6-24 rows, 512-2048
# columns, 2-4 buffers)
PC_TILE_S, PC_BLOCK_D, PC_BUFFERS = 12, 1024, 3
# the tail shape's producer/consumer tiles are the workload's 32 rows; buffers measured best
TAIL_PC_BUFFERS = 3
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
L2_BYTES = 126 * 2**20  # smaller than the part's L2: data this size stays resident


def _hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def bench_config(world: int, variant: str) -> dict:
    """The workload as both arms report it."""
    return {"workload": "combine DeepSeek-V3-shaped: W=8 emulated PEs, per PE "
                        "(16384,1,7168) bf16 -> (2048,8,7168)",
            "W": 8, "S": 2048, "H": 1, "D": 7168, "dtype": "bf16", "variant": variant,
            "bytes_per_step": 2 * 8 * 16384 * 7168 * 2, "parallelism": f"replicas{world}",
            "l2": "no flush: 1.88 GB input and output per step, >> 126 MB L2",
            "pc_tile_s": PC_TILE_S, "pc_block_d": PC_BLOCK_D, "pc_buffer_num": PC_BUFFERS}


def _kernel_sources_hash(files) -> str:
    """Hash of the csrc files a kernel is compiled from (its translation unit
    and the headers it includes)."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "symmetric_memory_moe_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, launch_bytes: int):
    """DRAM bytes of a launch moving `launch_bytes` algorithmic bytes, from the
    committed ncu captures, while the kernel sources still hash to the
    captured ones (else None).  Two captures of different sizes give the
    DRAM bytes per algorithmic byte as their slope: a launch that leaves dirty
    lines in L2 at its end writes them back during the next one, so the
    per-launch traffic of a long run of launches is the slope times the
    launch's bytes, not one capture scaled."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t["kernels"][kernel]
        if e.get("sources_hash") != _kernel_sources_hash(e["sources"]):
            return None
        (a0, d0), (a1, d1) = [(c["algorithmic_bytes"], c["dram_bytes"]) for c in e["captures"]]
        return int(round((d1 - d0) / (a1 - a0) * launch_bytes))
    except Exception:
        return None


# --------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        inside = [s for (t, s) in self.samples if any(a - 0.05 <= t <= b + 0.05
                                                      for a, b in self.windows)]
        used = inside or [s for (_, s) in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        sm = [float(s[0]) for s in used if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in used if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in used for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower() == "active"})
        power = [float(s[2]) for s in used if s[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(used), "in_timed_region": bool(inside),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------- distributed ---
def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the process group (x itself without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch(args, argv) -> int:
    """Runs this script as args.gpus ranks (one process each, rank r on GPU r)
    and returns the first non-zero exit code, else 0.  Rank 0 prints the
    line; the ranks inherit this process's stdout and stderr."""
    port = _free_port()
    procs = []
    for r in range(args.gpus):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(args.gpus),
                   LOCAL_WORLD_SIZE=str(args.gpus), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + argv,
                                      env=env))
    codes = [p.wait() for p in procs]
    return next((c for c in codes if c), 0)


def _init_group(backend: str, device=None):
    import torch.distributed as dist

    world, _, _ = _dist_env()
    if world > 1 and not dist.is_initialized():
        if device is not None:
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)


def run_dry(args):
    """The launcher and rank plumbing without a GPU: gloo, a host-side
    stand-in step, the same barrier / max-over-ranks / rank-0 line.  Prints
    no benchmark figure."""
    import torch.distributed as dist

    world, rank, local = _dist_env()
    _init_group("gloo")
    buf = bytearray(1 << 20)
    for _ in range(args.warmup):
        bytes(buf)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        bytes(buf)
    t = max_over_ranks(time.perf_counter() - t0)
    reports = [None] * world
    if world > 1:
        dist.all_gather_object(reports, {"rank": rank, "local_rank": local})
    else:
        reports = [{"rank": rank, "local_rank": local}]
    if rank == 0:
        print(json.dumps({"dry_run": True, "metric": METRIC, "value": None, "unit": UNIT,
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ranks_reported": sorted(r["rank"] for r in reports),
                          "local_ranks": sorted(r["local_rank"] for r in reports),
                          "max_host_step_s": t / max(1, args.steps)}), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------- oracle ---
def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def _oracle_sample(wl, rows: int):
    import torch

    from symmetric_memory_moe_gb300 import inputs

    sample = inputs.Workload(wl.name, "combine", wl.W, rows, wl.H, wl.D, wl.dtype, wl.dist,
                             wl.seed)
    x = inputs.make_input(sample)
    return (x.view(torch.int16) if x.dtype == torch.bfloat16 else x).numpy()


def oracle_rate(o, xb, wl, rows: int, min_s: float, max_runs: int = 50):
    """Times the oracle `o` on a token sample `xb` of the workload (`rows` rows
    per (source, destination) block); returns (GB/s, median s per run, runs,
    bytes moved per run)."""
    moved = 2 * xb.nbytes
    times = []
    t_start = time.perf_counter()
    while len(times) < max_runs:
        t0 = time.perf_counter()
        o.combine(xb, wl.W, rows, wl.H, wl.D)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= min_s:
            break
    med = statistics.median(times)
    return moved / med / 1e9, med, len(times), moved


def cpu_baseline(wl, min_s: float = 8.0) -> dict:
    """The oracle on the machine's host cores: its OpenMP build (the combine's loops
    over the destinations and rows split across nproc threads) and the plain
    build on one thread, each on a token sample for about min_s seconds."""
    import oracle

    nproc = os.cpu_count() or 1
    threads = nproc  # the parallel loops have W x rows iterations
    rows = 512
    xb = _oracle_sample(wl, rows)
    one, sec1, runs1, moved = oracle_rate(oracle.load(), xb, wl, rows, min_s)
    line = {"value": round(one, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"oracle combine on W={wl.W} S={rows} H={wl.H} D={wl.D} bf16 ({rows}/"
                      f"{wl.S} of the tokens, {moved / 1e9:.3f} GB moved), median of {runs1} "
                      f"runs ({sec1:.2f} s each), one thread",
            "nproc": nproc, "cpu_model": _cpu_model()}
    try:
        os.environ["OMP_NUM_THREADS"] = str(threads)
        many, secn, runsn, _ = oracle_rate(oracle.load_openmp(), xb, wl, rows, min_s)
    except Exception as e:  # no OpenMP runtime on this host
        line["parallel_unavailable"] = str(e)[:200]
        return line
    line.update({"value": round(many, 4), "cores": threads,
                 "sample": f"oracle combine on W={wl.W} S={rows} H={wl.H} D={wl.D} bf16 ({rows}/"
                           f"{wl.S} of the tokens, {moved / 1e9:.3f} GB moved): its OpenMP build "
                           f"over (destination, row) on {threads} threads, median of {runsn} "
                           f"runs ({secn:.2f} s each); the plain build on one thread, median of "
                           f"{runs1} runs ({sec1:.2f} s each)",
                 "single_thread": {"value": round(one, 4), "unit": UNIT, "cores": 1}})
    return line


def run_reference(args):
    """--impl reference: the CPU oracle is the reference arm (rank 0 only)."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    import oracle
    from symmetric_memory_moe_gb300 import inputs

    wl = inputs.WORKLOADS[WORKLOAD]
    nproc = os.cpu_count() or 1
    threads = nproc
    os.environ["OMP_NUM_THREADS"] = str(threads)
    try:
        o, kind = oracle.load_openmp(), f"OpenMP build over (destination, row), " \
                                        f"{threads} threads"
    except Exception:
        o, kind, threads = oracle.load(), "plain build, one thread", 1
    # size each step so that warm-up + steps end within about two minutes
    probe = _oracle_sample(wl, 8)
    rate, _, _, _ = oracle_rate(o, probe, wl, 8, 0.0, max_runs=1)
    per_row = 2 * wl.W * wl.W * wl.H * wl.D * wl.es
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.S, budget * rate * 1e9 / per_row)))
    xb = _oracle_sample(wl, rows)
    moved = rows * per_row
    for _ in range(args.warmup):
        o.combine(xb, wl.W, rows, wl.H, wl.D)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.combine(xb, wl.W, rows, wl.H, wl.D)
    sec = (time.perf_counter() - t0) / max(1, args.steps)
    value = round(moved / sec / 1e9, 4)
    desc = (f"oracle combine on W={wl.W} S={rows} H={wl.H} D={wl.D} bf16 "
            f"({rows}/{wl.S} of the tokens), {moved / 1e9:.3f} GB moved per step; {kind}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
        "config": bench_config(world, args.variant),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc, "nproc": nproc, "cpu_model": _cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ variants ---
def _fill_random(heap, ptr, nbytes, seed):
    """Seeded random bytes in every PE's copy of an object (the path moves
    raw bits, so bytes stand in for the workload's values when timing)."""
    import torch

    g = torch.Generator(device=heap.mem.device).manual_seed(seed)
    heap.views(ptr, nbytes).copy_(torch.randint(0, 256, (heap.npes, nbytes), generator=g,
                                                dtype=torch.uint8, device=heap.mem.device))


def _time_calls(call, steps, warmup, graph):
    """GPU ms per call: `steps` launches timed with CUDA events, or, for
    calls whose data stay in L2 (launch-bound from Python), `steps` replays
    of a CUDA graph of 20 calls."""
    import torch

    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    if graph:
        per_graph = 20
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(per_graph):
                    call()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (steps * per_graph)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def _check_runs(heap, inp, out, W, S, run, inverse=False, samples=16, seed=0):
    """Sampled runs of the permutation: out_d[s, r] == in_r[d*S + s] (combine,
    dispatch with S per block), or its inverse."""
    import torch

    n = W * S * run
    outv = heap.views(out, n).view(W, S if not inverse else W, W if not inverse else S, run)
    inv = heap.views(inp, n).view(W, W if not inverse else S, S if not inverse else W, run)
    g = torch.Generator().manual_seed(seed)
    for _ in range(samples):
        d, s, r = (int(torch.randint(0, k, (1,), generator=g)) for k in (W, S, W))
        if not inverse:
            ok = torch.equal(outv[d, s, r], inv[r, d, s])   # out_d[s, r] = in_r[d*S + s]
        else:
            ok = torch.equal(outv[r, d, s], inv[d, s, r])   # out_r[d*S + s] = in_d[s, r]
        if not ok:
            raise RuntimeError("a timed variant produced a wrong output run")


def time_variants(args, peak):
    """The other configurations' headline variants (and the two-phase
    combine on the DeepSeek-V3 shape), each timed in this process."""
    from symmetric_memory_moe_gb300 import abi
    from symmetric_memory_moe_gb300.torch_heap import CombineBuffers, TorchSymmHeap

    out = {}

    def done(heap):
        rc, info = abi.symm_check_error(heap.handle)
        heap.close()
        if rc != abi.SYMM_OK:
            raise RuntimeError(f"a timed variant's device wait gave up (info {info})")

    def record(name, workload, bytes_step, ms, timing, extra=None):
        gbs = bytes_step / (ms * 1e-3) / 1e9
        e = {"workload": workload, "gbs": round(gbs, 1), "ms_per_step": round(ms, 5),
             "frac_of_peak": round(gbs / peak, 4), "bytes_per_step": bytes_step,
             "l2_resident": bytes_step <= L2_BYTES, "timing": timing}
        e.update(extra or {})
        out[name] = e

    steps = max(args.steps, 10)
    # small: W8 S128 H8 D128 bf16 (16.8 MB in, L2-resident), direct and P/C;
    # P/C with one 128-row tile per task and one buffer, measured fastest on
    # this shape (every handshake costs more than pipelining S blocks saves)
    W, S, H, D, es = 8, 128, 8, 128, 2
    for variant, tile, nbuf in (("direct", 0, 2), ("pc", 128, 1)):
        b = CombineBuffers(W, S * W, H, D, es, pc=variant == "pc", S=S, tile_s=tile or 16,
                           buffer_num=nbuf)
        _fill_random(b.heap, b.inp, b.nbytes, 1)
        kind = abi.SYMM_A2A_PC if variant == "pc" else abi.SYMM_A2A_DIRECT

        def call(b=b, kind=kind, tile=tile, nbuf=nbuf):
            abi.all2all_combine(b.heap.handle, b.inp, b.out, W, S, H, D, es, kind, tile or 16, 0,
                                nbuf, b.staging, b.signals)
        ms = _time_calls(call, steps, args.warmup, graph=True)
        _check_runs(b.heap, b.inp, b.out, W, S, H * D * es)
        record(f"small_{variant}", "combine small: W=8 S=128 H=8 D=128 bf16", 2 * W * b.nbytes,
               ms, "CUDA graph of 20 calls",
               {"tile_s": tile, "buffer_num": nbuf} if tile else None)
        done(b.heap)
    # round trip: W16 S1024 H4 D128 fp16, dispatch then its inverse
    W, S, H, D, es = 16, 1024, 4, 128, 2
    n = S * H * D * es
    heap = TorchSymmHeap(W, 3 * n + (4 << 20))
    x, y, z = heap.malloc(n), heap.malloc(n), heap.malloc(n)
    _fill_random(heap, x, n, 3)
    ms = _time_calls(lambda: abi.all2all_dispatch(heap.handle, x, y, W, S, H, D, es), steps,
                     args.warmup, graph=True)
    _check_runs(heap, x, y, W, S // W, H * D * es)
    record("roundtrip_dispatch", "dispatch: W=16 S=1024 H=4 D=128 fp16", 2 * W * n, ms,
           "CUDA graph of 20 calls")
    ms = _time_calls(lambda: abi.all2all_combine_back(heap.handle, y, z, W, S // W, H, D, es),
                     steps, args.warmup, graph=True)
    if not heap.views(z, n).equal(heap.views(x, n)):
        raise RuntimeError("dispatch then its inverse did not round-trip")
    record("roundtrip_combine_back", "combine back: W=16 S'=64 H=4 D=128 fp16", 2 * W * n, ms,
           "CUDA graph of 20 calls")
    done(heap)
    # tail: W32 S256 H2 D999 fp16 (1998-byte rows), direct and P/C with 32-row tiles
    W, S, H, D, es = 32, 256, 2, 999, 2
    for variant in ("direct", "pc"):
        b = CombineBuffers(W, S * W, H, D, es, pc=variant == "pc", S=S, tile_s=32,
                           buffer_num=TAIL_PC_BUFFERS)
        _fill_random(b.heap, b.inp, b.nbytes, 4)
        kind = abi.SYMM_A2A_PC if variant == "pc" else abi.SYMM_A2A_DIRECT

        def call(b=b, kind=kind):
            abi.all2all_combine(b.heap.handle, b.inp, b.out, W, S, H, D, es, kind, 32, 0,
                                TAIL_PC_BUFFERS, b.staging, b.signals)
        ms = _time_calls(call, steps, args.warmup, graph=False)
        _check_runs(b.heap, b.inp, b.out, W, S, H * D * es)
        record(f"tail_{variant}", "combine tail: W=32 S=256 H=2 D=999 fp16", 2 * W * b.nbytes,
               ms, "launches",
               {"tile_s": 32, "buffer_num": TAIL_PC_BUFFERS} if variant == "pc" else None)
        done(b.heap)
    # the two-phase combine on the DeepSeek-V3 shape (tiles of 64 x 1024)
    W, S, H, D, es = 8, 2048, 1, 7168, 2
    n = S * W * H * D * es
    nb, ns = abi.all2all_two_phase_workspace(W, S, H, D, es, 64, 1024, 2)
    heap = TorchSymmHeap(W, 2 * n + nb + ns + (4 << 20))
    x, y, bulk, sig = heap.malloc(n), heap.malloc(n), heap.malloc(nb), heap.malloc(ns)
    _fill_random(heap, x, n, 2)
    ms = _time_calls(lambda: abi.all2all_combine_two_phase(heap.handle, x, y, W, S, H, D, es, 64,
                                                           1024, 2, bulk, sig),
                     steps, args.warmup, graph=False)
    _check_runs(heap, x, y, W, S, H * D * es)
    record("dsv3_two_phase", "combine DeepSeek-V3-shaped, two-phase", 2 * W * n, ms, "launches",
           {"tile_s": 64, "block_d": 1024})
    done(heap)
    return out


# ------------------------------------------------------------------ ours ---
def run_ours(args):
    import torch
    import torch.distributed as dist

    from symmetric_memory_moe_gb300 import abi, inputs
    from symmetric_memory_moe_gb300.torch_heap import CombineBuffers

    world, rank, local = _dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU (or --dry-run)"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    _init_group("nccl", device)

    wl = inputs.WORKLOADS[WORKLOAD]
    W, S, H, D, es = wl.W, wl.S, wl.H, wl.D, wl.es
    T = wl.total_bytes
    step_bytes = 2 * T
    bufs = CombineBuffers(W, S * W, H, D, es, pc=True, S=S, tile_s=PC_TILE_S,
                          block_d=PC_BLOCK_D, buffer_num=PC_BUFFERS)
    heap = bufs.heap
    host_in = torch.empty((W, S * W, H, D), dtype=wl.dtype).pin_memory()
    inputs.make_input(wl, out=host_in)
    host_out = torch.empty((W, S, H * W, D), dtype=wl.dtype).pin_memory()
    heap.upload(bufs.inp, host_in.reshape(W, -1))
    torch.cuda.synchronize()

    kinds = {"direct": abi.SYMM_A2A_DIRECT, "pc": abi.SYMM_A2A_PC}
    launches_per_step = {"direct": 1, "pc": 1}  # pc: the pipeline zeroes its own slots

    def step(kind):
        abi.all2all_combine(heap.handle, bufs.inp, bufs.out, W, S, H, D, es, kind, PC_TILE_S,
                            PC_BLOCK_D, PC_BUFFERS, bufs.staging, bufs.signals)

    sampler = ClockSampler(local)
    sampler.start()
    results = {}
    order = ["direct", "pc"]
    order.sort(key=lambda v: v == args.variant)  # the headline variant runs last
    for name in order:
        kind = kinds[name]
        for _ in range(args.warmup):
            step(kind)
        torch.cuda.synchronize()
        barrier(device)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        t_wall0 = time.time()
        ev[0].record()
        for i in range(args.steps):
            step(kind)
            ev[i + 1].record()
        torch.cuda.synchronize()
        t_wall1 = time.time()
        barrier(device)
        torch.cuda.synchronize()
        sampler.mark(t_wall0, t_wall1)
        rc, info = abi.symm_check_error(heap.handle)
        if rc != abi.SYMM_OK:
            raise RuntimeError(f"{name}: device wait timed out (signal offset {info})")
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
        total_ms = ev[0].elapsed_time(ev[-1])
        total_ms = max_over_ranks(total_ms, device)
        results[name] = {"ms_per_step": total_ms / args.steps, "launch_ms_avg": statistics.mean(per),
                         "launch_ms_median": statistics.median(per),
                         "gbs": world * step_bytes * args.steps / (total_ms * 1e-3) / 1e9}
        # sampled check that the timed launches did the permutation:
        # out_d[s, r*H:(r+1)*H] must equal in_r[d*S + s]
        g = torch.Generator().manual_seed(rank)
        outv = heap.views(bufs.out, bufs.nbytes).view(W, S, W, H * D * es)
        inv = heap.views(bufs.inp, bufs.nbytes).view(W, W, S, H * D * es)
        for _ in range(32):
            d, s, r = (int(torch.randint(0, n, (1,), generator=g)) for n in (W, S, W))
            assert torch.equal(outv[d, s, r], inv[r, d, s]), f"{name}: wrong output run"
    sampler.stop()

    # end to end through the host-buffer C-ABI call: H2D inputs, combine, D2H outputs
    e2e_steps = max(3, min(args.steps, 10))
    kind = kinds[args.variant]

    def e2e_step():
        abi.all2all_combine_host(heap.handle, host_in.data_ptr(), host_out.data_ptr(), bufs.inp,
                                 bufs.out, W, S, H, D, es, kind, PC_TILE_S, PC_BLOCK_D,
                                 PC_BUFFERS, bufs.staging, bufs.signals)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    torch.cuda.synchronize()
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), device) / e2e_steps
    assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    heap.close()
    del host_in, host_out

    # plain cudaMemcpyAsync device-to-device of the same T bytes, for context
    src = torch.empty(T, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    for _ in range(3):
        dst.copy_(src)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(10):
        dst.copy_(src)
    c1.record()
    torch.cuda.synchronize()
    d2d_gbs = 2 * T * 10 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    del src, dst
    torch.cuda.empty_cache()

    peak, peak_src = _hbm_peak()
    variants = {k: {"workload": "combine DeepSeek-V3-shaped", "gbs": round(v["gbs"], 1),
                    "ms_per_step": round(v["ms_per_step"], 4),
                    "frac_of_peak": round(v["gbs"] / world / peak, 4),
                    "bytes_per_step": step_bytes, "l2_resident": False, "timing": "launches"}
                for k, v in results.items()}
    if not args.no_variants:
        variants.update(time_variants(args, peak))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    head = results[args.variant]
    kernel_name = "a2a_pc_rel_kernel" if args.variant == "pc" else "a2a_runs_kernel"
    achieved = step_bytes / (head["launch_ms_avg"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(head["gbs"], 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(head["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, moved as raw bits)",
        "config": bench_config(world, args.variant),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "kernel": kernel_name,
                     "traffic": _traffic(kernel_name, step_bytes),
                     "traffic_method": "ncu DRAM bytes of two captures (S=256, S=512): their "
                                       "slope per algorithmic byte times this launch's bytes"},
        "variants": variants,
        "d2d_memcpy_gbs": round(d2d_gbs, 1),
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": T, "d2h_bytes_per_step": T, "steps": e2e_steps,
                "ms_per_step": round(e2e_ms, 3),
                "call": "all2all_combine_host (pinned host buffers: the direct combine reads and writes them in place over the host link)"},
        "gpu_launches": args.steps * launches_per_step[args.variant],
        "clocks": sampler.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="direct", choices=["direct", "pc"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="time only the DeepSeek-V3-shaped combine")
    ap.add_argument("--dry-run", action="store_true",
                    help="the launcher and rank plumbing on CPU (gloo); no benchmark figure")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch(args, argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.dry_run:
        run_dry(args)
    else:
        run_ours(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
