"""Runs one all-to-all variant on one shape for a few steps (for profilers
such as ncu, or quick timing), through the C ABI.

  python -m symmetric_memory_moe_gb300.profile_case --variant pc --S 256 --steps 4

Each step is the whole call (for pc: the signal reset and the pipeline; for
the collectives: metadata, push and wait).  Prints one JSON line with per-step
CUDA-event times and GB/s (bytes read + bytes written / time).

  python -m symmetric_memory_moe_gb300.profile_case --variant alltoall --tokens 4096
  python -m symmetric_memory_moe_gb300.profile_case --variant allgather --bytes 33554432
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import abi, inputs
from .torch_heap import CombineBuffers, TorchSymmHeap

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "int32": torch.int32,
          "uint8": torch.uint8}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--variant", default="pc",
                    choices=["direct", "pc", "noalloc", "dispatch", "combine_back", "two_phase",
                             "alltoall", "allgather", "ag_matmul"])
    ap.add_argument("--W", type=int, default=8)
    ap.add_argument("--S", type=int, default=256)
    ap.add_argument("--H", type=int, default=1)
    ap.add_argument("--D", type=int, default=7168)
    ap.add_argument("--dtype", default="bf16", choices=sorted(DTYPES))
    ap.add_argument("--tile-s", type=int, default=16)
    ap.add_argument("--block-d", type=int, default=1024)
    ap.add_argument("--buffers", type=int, default=2)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--vector", action="store_true",
                    help="pc: 16-byte vector copies only (no bulk prefetch)")
    ap.add_argument("--bulk", action="store_true",
                    help="direct and pc: bulk (TMA) copies through shared memory")
    ap.add_argument("--tokens", type=int, default=4096, help="alltoall: tokens per PE")
    ap.add_argument("--experts", type=int, default=256, help="alltoall: routed experts")
    ap.add_argument("--topk", type=int, default=8, help="alltoall: experts per token")
    ap.add_argument("--skew", type=float, default=1.0, help="alltoall: Zipf exponent")
    ap.add_argument("--bytes", type=int, default=32 << 20, help="allgather: bytes per PE")
    ap.add_argument("--m-local", type=int, default=512, help="ag_matmul: rows per PE")
    ap.add_argument("--k", type=int, default=1024, help="ag_matmul: inner dimension")
    ap.add_argument("--n", type=int, default=2048, help="ag_matmul: columns of b")
    ap.add_argument("--cublas", action="store_true",
                    help="ag_matmul: also time torch.bmm on the gathered rows (context)")
    args = ap.parse_args(argv)
    if args.variant in ("alltoall", "allgather"):
        return collective(args)
    if args.variant == "two_phase":
        return two_phase(args)
    if args.variant == "ag_matmul":
        return ag_matmul(args)

    dt = DTYPES[args.dtype]
    es = torch.empty((), dtype=dt).element_size()
    W, S, H, D = args.W, args.S, args.H, args.D
    rows_in = S * W if args.variant in ("direct", "pc", "noalloc") else S
    if args.variant == "combine_back":
        rows_in = S  # per PE (S/W, H*W, D): same bytes as (S, H, D)
    bufs = CombineBuffers(W, rows_in, H, D, es, pc=args.variant == "pc", S=S,
                          tile_s=args.tile_s, block_d=args.block_d, buffer_num=args.buffers)
    heap = bufs.heap
    # the path moves raw bits, so seeded random bytes drawn on the device
    # stand in for the workload's values here
    g = torch.Generator(device=heap.mem.device).manual_seed(7)
    heap.views(bufs.inp, bufs.nbytes).copy_(
        torch.randint(0, 256, (W, bufs.nbytes), generator=g, dtype=torch.uint8,
                      device=heap.mem.device))

    def step():
        if args.variant in ("direct", "pc"):
            kind = abi.SYMM_A2A_PC if args.variant == "pc" else abi.SYMM_A2A_DIRECT
            if args.vector:
                kind |= abi.SYMM_A2A_FLAG_VECTOR
            if args.bulk:
                kind |= abi.SYMM_A2A_FLAG_BULK
            abi.all2all_combine(heap.handle, bufs.inp, bufs.out, W, S, H, D, es, kind,
                                args.tile_s, args.block_d, args.buffers, bufs.staging,
                                bufs.signals)
        elif args.variant == "noalloc":
            abi.all2all_combine_pc_noalloc(heap.handle, bufs.inp, bufs.out, W, S, H, D, es,
                                           args.tile_s, args.block_d, args.buffers)
        elif args.variant == "dispatch":
            abi.all2all_dispatch(heap.handle, bufs.inp, bufs.out, W, S, H, D, es)
        else:
            abi.all2all_combine_back(heap.handle, bufs.inp, bufs.out, W, S // W, H, D, es)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record()
    for i in range(args.steps):
        step()
        ev[i + 1].record()
    torch.cuda.synchronize()
    rc, info = abi.symm_check_error(heap.handle)
    if rc != abi.SYMM_OK:
        raise SystemExit(f"device wait timed out at signal offset {info}")
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    moved = 2 * W * bufs.nbytes
    checked = 0
    if args.variant in ("direct", "pc", "noalloc"):
        # sampled runs of the combine: out_d[s, r*H + h] == in_r[d*S + s, h]
        run = H * D * es
        outv = heap.views(bufs.out, bufs.nbytes).view(W, S, W, run)
        inv = heap.views(bufs.inp, bufs.nbytes).view(W, W, S, run)
        gc = torch.Generator().manual_seed(11)
        for _ in range(64):
            d, s, r = (int(torch.randint(0, n, (1,), generator=gc)) for n in (W, S, W))
            if not torch.equal(outv[d, s, r], inv[r, d, s]):
                raise SystemExit(f"wrong output run (d={d}, s={s}, r={r})")
            checked += 1
    print(json.dumps({"variant": args.variant, "W": W, "S": S, "H": H, "D": D, "es": es,
                      "bytes_per_step": moved, "ms": [round(m, 4) for m in ms],
                      "gbs_median": round(moved / (statistics.median(ms) * 1e-3) / 1e9, 1),
                      "runs_checked": checked}))
    heap.close()


def _time(step, steps):
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        step()
        ev[i + 1].record()
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def two_phase(args):
    W, S, H, D = args.W, args.S, args.H, args.D
    es = torch.empty((), dtype=DTYPES[args.dtype]).element_size()
    n = S * W * H * D * es
    nb, ns = abi.all2all_two_phase_workspace(W, S, H, D, es, args.tile_s, args.block_d,
                                             args.buffers)
    heap = TorchSymmHeap(W, 2 * n + nb + ns + (4 << 20))
    inp, out, bulk, sig = heap.malloc(n), heap.malloc(n), heap.malloc(nb), heap.malloc(ns)
    g = torch.Generator(device="cuda").manual_seed(7)
    heap.views(inp, n).copy_(torch.randint(0, 256, (W, n), generator=g, dtype=torch.uint8,
                                           device="cuda"))

    def step():
        abi.all2all_combine_two_phase(heap.handle, inp, out, W, S, H, D, es, args.tile_s,
                                      args.block_d, args.buffers, bulk, sig)
    _time(step, 3)
    ms = _time(step, args.steps)
    rc, info = abi.symm_check_error(heap.handle)
    if rc != abi.SYMM_OK:
        raise SystemExit(f"two-phase combine failed on the device: code {rc}, info {info}")
    moved = 2 * W * n
    print(json.dumps({"variant": "two_phase", "W": W, "S": S, "H": H, "D": D, "es": es,
                      "tile_s": args.tile_s, "block_d": args.block_d, "buffers": args.buffers,
                      "bytes_per_step": moved, "ms": [round(m, 4) for m in ms],
                      "gbs_median": round(moved / (statistics.median(ms) * 1e-3) / 1e9, 1)}))
    heap.close()


def ag_matmul(args):
    W, m, k, n = args.W, args.m_local, args.k, args.n
    dtype = {"bf16": torch.bfloat16, "fp16": torch.float16}[args.dtype]
    code = abi.SYMM_DTYPE_BF16 if dtype == torch.bfloat16 else abi.SYMM_DTYPE_F16
    sig_bytes = abi.shmem_fused_ag_matmul_workspace(W, m, k, n)
    sizes = [m * k * 2, k * n * 2, W * m * n * 2, W * m * k * 2, sig_bytes]
    heap = TorchSymmHeap(W, sum(sizes) + 256 * len(sizes) + (4 << 20))
    pa, pb, pc, pg, ps = [heap.malloc(s) for s in sizes]
    g = torch.Generator(device="cuda").manual_seed(7)
    for p, nb in ((pa, sizes[0]), (pb, sizes[1])):
        heap.views(p, nb).view(dtype).copy_(
            torch.randn(W, nb // 2, generator=g, device="cuda").to(dtype))

    def step():
        abi.shmem_fused_all_gather_matmul(heap.handle, pa, pb, pc, pg, W, m, k, n, code, 128, ps)
    _time(step, 3)
    ms = _time(step, args.steps)
    rc, info = abi.symm_check_error(heap.handle)
    if rc != abi.SYMM_OK:
        raise SystemExit(f"fused AllGather + MatMul failed on the device: code {rc}, info {info}")
    flops = 2.0 * W * (W * m) * k * n
    out = {"variant": "ag_matmul", "W": W, "m_local": m, "k": k, "n": n, "dtype": args.dtype,
           "flops_per_step": flops, "ms": [round(x, 4) for x in ms],
           "tflops_median": round(flops / (statistics.median(ms) * 1e-3) / 1e12, 1)}
    if args.cublas:  # the same matmuls on already-gathered rows, by the library
        A = torch.randn(W, W * m, k, generator=g, device="cuda").to(dtype)
        B = torch.randn(W, k, n, generator=g, device="cuda").to(dtype)
        _time(lambda: torch.bmm(A, B), 3)
        cms = _time(lambda: torch.bmm(A, B), args.steps)
        out["cublas_bmm_tflops_median"] = round(flops / (statistics.median(cms) * 1e-3) / 1e12, 1)
    print(json.dumps(out))
    heap.close()


def collective(args):
    W = args.W
    ws = torch.empty(abi.shmem_collective_workspace(W) // 8, dtype=torch.int64, device="cuda")
    if args.variant == "alltoall":
        row = args.H * args.D * torch.empty((), dtype=DTYPES[args.dtype]).element_size()
        counts = inputs.moe_counts(W, args.tokens, args.experts, args.topk, seed=5,
                                   skew=args.skew)
        in_rows, out_rows = int(counts.sum(1).max()), int(counts.sum(0).max())
        heap = TorchSymmHeap(W, (in_rows + out_rows) * row + (4 << 20))
        inp, out, sig = heap.malloc(in_rows * row), heap.malloc(out_rows * row), heap.malloc(64)
        nin, moved = in_rows * row, 2 * int(counts.sum()) * row
        dcounts = counts.cuda()

        def step():
            abi.shmem_alltoall(heap.handle, inp, out, dcounts.data_ptr(), W, row, in_rows,
                               out_rows, ws.data_ptr(), sig)
        shape = {"tokens": args.tokens, "experts": args.experts, "topk": args.topk,
                 "skew": args.skew, "row_bytes": row, "rows": int(counts.sum())}
    else:
        n = args.bytes
        heap = TorchSymmHeap(W, (W + 1) * n + (4 << 20))
        inp, out, sig = heap.malloc(n), heap.malloc(W * n), heap.malloc(64)
        nin, moved = n, W * n + W * W * n   # every input read once, W copies written

        def step():
            abi.shmem_allgather(heap.handle, inp, out, W, n, ws.data_ptr(), sig)
        shape = {"bytes": n}
    g = torch.Generator(device="cuda").manual_seed(7)
    heap.views(inp, nin).copy_(torch.randint(0, 256, (W, nin), generator=g, dtype=torch.uint8,
                                             device="cuda"))
    _time(step, 3)
    ms = _time(step, args.steps)
    rc, info = abi.symm_check_error(heap.handle)
    if rc != abi.SYMM_OK:
        raise SystemExit(f"collective failed on the device: code {rc}, info {info}")
    print(json.dumps({"variant": args.variant, "W": W, **shape, "bytes_per_step": moved,
                      "ms": [round(m, 4) for m in ms],
                      "gbs_median": round(moved / (statistics.median(ms) * 1e-3) / 1e9, 1)}))
    heap.close()


if __name__ == "__main__":
    main()
