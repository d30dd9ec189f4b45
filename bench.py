"""Benchmark: Reverse All2All (combine) GB/s on the DeepSeek-V3-shaped workload.

One step = one all2all_combine through the C ABI over W=8 emulated PEs
(per PE (16384, 1, 7168) bf16 -> (2048, 8, 7168)): T = 1.879 GB read and
1.879 GB written.  GB/s = 2*T / step time.  The input (1.88 GB) is larger
than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--variant pc|direct]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

For N > 1 (torchrun), every rank runs its own replica on its own GPU (the
W PEs are emulated inside one GPU; there is no cross-GPU exchange), the step
time is the max over ranks and the value the sum of all ranks' bytes over it.
"""
from __future__ import annotations

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

METRIC = "reverse-All2All combine GB/s (read+write) and % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "dsv3"
PC_TILE_S, PC_BLOCK_D, PC_BUFFERS = 16, 1024, 2
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def _hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


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
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was taken (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t["kernels"][kernel]
        if e.get("sources_hash") != _kernel_sources_hash(e["sources"]):
            return None
        # scaled from the captured launch by the bytes one launch moves
        return int(round(e["dram_bytes"] * launch_bytes / e["algorithmic_bytes"]))
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


# --------------------------------------------------------------- oracle ---
def oracle_rate(wl, rows: int, repeats_min_s: float, max_runs: int = 50):
    """The CPU oracle (as it stands, one thread) on the workload's shape with
    `rows` rows per (source, destination) block; returns (GB/s, seconds per
    run, runs, sample bytes moved per run)."""
    import torch

    import oracle
    from symmetric_memory_moe_gb300 import inputs

    o = oracle.load()
    sample = inputs.Workload(wl.name, "combine", wl.W, rows, wl.H, wl.D, wl.dtype, wl.dist,
                             wl.seed)
    x = inputs.make_input(sample)
    xb = (x.view(torch.int16) if x.dtype == torch.bfloat16 else x).numpy()
    moved = 2 * xb.nbytes
    times = []
    t_start = time.perf_counter()
    while len(times) < max_runs:
        t0 = time.perf_counter()
        o.combine(xb, wl.W, rows, wl.H, wl.D)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= repeats_min_s and len(times) >= 1:
            break
    med = statistics.median(times)
    return moved / med / 1e9, med, len(times), moved


def run_reference(args):
    """--impl reference: the CPU oracle is the reference arm (rank 0 only)."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    from symmetric_memory_moe_gb300 import inputs

    wl = inputs.WORKLOADS[WORKLOAD]
    # size each step so warm-up + steps end within ~2 minutes
    rate, _, _, _ = oracle_rate(wl, 8, 0.0, max_runs=1)
    per_row = 2 * wl.W * wl.W * wl.H * wl.D * wl.es
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.S, budget * rate * 1e9 / per_row)))
    sample_rate, sec, _, moved = 0.0, 0.0, 0, rows * per_row
    import oracle
    import torch

    o = oracle.load()
    sample = inputs.Workload(wl.name, "combine", wl.W, rows, wl.H, wl.D, wl.dtype, wl.dist,
                             wl.seed)
    xb = inputs.make_input(sample).view(torch.int16).numpy()
    for _ in range(args.warmup):
        o.combine(xb, wl.W, rows, wl.H, wl.D)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.combine(xb, wl.W, rows, wl.H, wl.D)
    sec = (time.perf_counter() - t0) / max(1, args.steps)
    sample_rate = moved / sec / 1e9
    desc = (f"oracle combine on W={wl.W} S={rows} H={wl.H} D={wl.D} bf16 "
            f"({rows}/{wl.S} of the tokens), {moved / 1e9:.3f} GB moved per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(sample_rate, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": "combine DeepSeek-V3-shaped (W=8 S=2048 H=1 D=7168 bf16), "
                               "CPU oracle on a token sample", "W": wl.W, "S_sample": rows,
                   "H": wl.H, "D": wl.D},
        "cpu_baseline": {"value": round(sample_rate, 4), "unit": UNIT, "cores": 1,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(sample_rate, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours ---
def run_ours(args):
    import torch
    import torch.distributed as dist

    from symmetric_memory_moe_gb300 import abi, inputs
    from symmetric_memory_moe_gb300.torch_heap import CombineBuffers

    world, rank, local = _dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=device)

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
    launches_per_step = {"direct": 1, "pc": 2}  # pc: signal reset + pipeline

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

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = 512
        rate, sec, runs, moved = oracle_rate(wl, rows, 10.0)
        cpu = {"value": round(rate, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"oracle combine on W={W} S={rows} H={H} D={D} bf16 ({rows}/{S} of "
                         f"the tokens, {moved / 1e9:.3f} GB moved), median of {runs} runs "
                         f"({sec:.2f} s each), one host thread"}

    head = results[args.variant]
    peak, peak_src = _hbm_peak()
    kernel_name = "a2a_pc_kernel" if args.variant == "pc" else "a2a_runs_kernel"
    achieved = step_bytes / (head["launch_ms_avg"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(head["gbs"], 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(head["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, moved as raw bits)",
        "config": {"workload": "combine DeepSeek-V3-shaped: W=8 emulated PEs, per PE "
                               "(16384,1,7168) bf16 -> (2048,8,7168)",
                   "W": W, "S": S, "H": H, "D": D, "variant": args.variant,
                   "bytes_per_step": step_bytes, "parallelism": f"replicas{world}",
                   "l2": "no flush: 1.88 GB input and output per step, >> 126 MB L2",
                   "pc_tile_s": PC_TILE_S, "pc_block_d": PC_BLOCK_D,
                   "pc_buffer_num": PC_BUFFERS},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "kernel": kernel_name,
                     "traffic": _traffic(kernel_name, step_bytes)},
        "variants": {k: {"gbs": round(v["gbs"], 1), "ms_per_step": round(v["ms_per_step"], 4),
                         "frac_of_peak": round(v["gbs"] / world / peak, 4)}
                     for k, v in results.items()},
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
    heap.close()
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="direct", choices=["direct", "pc"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
