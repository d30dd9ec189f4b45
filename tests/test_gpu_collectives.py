"""GPU parity of the push-mode collectives (HyperParallel RFC "Symmetric
Memory", section 10) against the oracle, byte for byte: AllToAll with uneven
per-pair row counts (MoE routing, random, empty, single PE, unaligned rows and
pointers) and AllGather (sizes around the 16 KB piece, empty, unaligned).
Output rows a PE does not receive must keep their old bytes; every PE's
signal ends at W; device-detected size errors come back as SYMM_ERANGE with
nothing copied, and the heap stays usable."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

POISON = 0xA5


def _heap(W, nbytes):
    slab = nbytes + (4 << 20)
    h = TorchSymmHeap(W, slab)
    h.mem.zero_()
    return h


def _workspace(W):
    n = abi.shmem_collective_workspace(W)
    return torch.empty(n // 8, dtype=torch.int64, device="cuda")


def _signals(heap, sig):
    torch.cuda.synchronize()
    return heap.views(sig, 8).view(torch.int64)[:, 0].cpu()


def _run_alltoall(W, row_bytes, counts, in_rows, out_rows, *, in_shift=0, out_shift=0, seed=0,
                  repeat=1):
    """Fills every PE's input with random rows, poisons the outputs, runs
    shmem_alltoall `repeat` times and compares with the oracle."""
    o = oracle.load()
    heap = _heap(W, (in_rows + out_rows) * row_bytes + 4096)
    try:
        in_p = heap.malloc(in_rows * row_bytes + 16) + in_shift
        out_p = heap.malloc(out_rows * row_bytes + 16) + out_shift
        sig = heap.malloc(64)
        x = inputs.random_bytes(W * in_rows * row_bytes, seed).view(W, in_rows * row_bytes)
        heap.views(in_p, in_rows * row_bytes).copy_(x.cuda())
        heap.views(out_p, out_rows * row_bytes).fill_(POISON)
        dcounts = counts.to(torch.int64).cuda()
        ws = _workspace(W)
        for _ in range(repeat):
            abi.shmem_alltoall(heap.handle, in_p, out_p, dcounts.data_ptr(), W, row_bytes, in_rows,
                               out_rows, ws.data_ptr(), sig)
        rc, _ = abi.symm_check_error(heap.handle)
        assert rc == abi.SYMM_OK
        got = heap.views(out_p, out_rows * row_bytes).cpu().numpy()
        want = np.full((W, out_rows, row_bytes), POISON, np.uint8)
        want = o.alltoallv(x.numpy().reshape(W, in_rows, row_bytes), counts.numpy(), out_rows,
                           out=want)
        assert np.array_equal(got, want.reshape(W, out_rows * row_bytes))
        assert torch.equal(_signals(heap, sig), torch.full((W,), W, dtype=torch.int64))
    finally:
        heap.close()


@pytest.mark.parametrize("W,tokens,row_bytes,seed", [
    (8, 512, 7168 * 2, 5),     # DeepSeek-V3 hidden rows, bf16
    (16, 256, 4096 * 2, 6),
    (4, 300, 999 * 2, 7),      # rows that are not a multiple of 16 bytes
])
def test_alltoall_moe_routing(W, tokens, row_bytes, seed):
    counts = inputs.moe_counts(W, tokens, 32 * W, 8, seed)
    in_rows = int(counts.sum(1).max())
    out_rows = int(counts.sum(0).max()) + 3   # the last rows of every PE stay untouched
    _run_alltoall(W, row_bytes, counts, in_rows, out_rows, seed=seed)


@pytest.mark.parametrize("W,high,zero_frac,row_bytes,in_shift,out_shift", [
    (2, 5, 0.0, 8, 0, 0),
    (3, 40, 0.3, 1, 0, 0),          # one-byte rows
    (5, 17, 0.5, 4, 1, 3),          # byte-shifted pointers
    (7, 64, 0.2, 1998, 5, 11),
    (8, 33, 0.0, 16384, 0, 0),
    (32, 9, 0.6, 240, 0, 8),        # many PEs, mostly empty segments
])
def test_alltoall_random_counts(W, high, zero_frac, row_bytes, in_shift, out_shift):
    counts = inputs.random_counts(W, high, seed=W, zero_frac=zero_frac)
    in_rows = int(counts.sum(1).max()) + 1
    out_rows = int(counts.sum(0).max()) + 2
    _run_alltoall(W, row_bytes, counts, in_rows, out_rows, in_shift=in_shift,
                  out_shift=out_shift, seed=W + 100)


def test_alltoall_golden_counts_exact_capacity():
    counts = torch.tensor([[1, 2], [3, 0]])
    _run_alltoall(2, 8, counts, 3, 4, seed=1)   # PE 0 receives exactly out_rows rows


@pytest.mark.parametrize("W", [1, 4])
def test_alltoall_degenerate(W):
    _run_alltoall(W, 64, torch.zeros(W, W, dtype=torch.int64), 4, 4)          # nothing moves
    _run_alltoall(W, 0, torch.full((W, W), 3, dtype=torch.int64), 3 * W, 3 * W)  # empty rows
    _run_alltoall(W, 100, torch.full((W, W), 2, dtype=torch.int64), 2 * W, 2 * W, repeat=3)


def test_alltoall_size_errors_found_on_device():
    W, row_bytes, in_rows, out_rows = 4, 32, 10, 10
    heap = _heap(W, 4096)
    try:
        in_p, out_p, sig = heap.malloc(in_rows * row_bytes), heap.malloc(out_rows * row_bytes), \
            heap.malloc(64)
        heap.views(out_p, out_rows * row_bytes).fill_(POISON)
        ws = _workspace(W)
        ok = torch.full((W, W), 2, dtype=torch.int64)
        for bad in (ok.clone().index_put_((torch.tensor(1), torch.tensor(2)), torch.tensor(-1)),
                    ok.clone().index_put_((torch.tensor(0), torch.tensor(3)), torch.tensor(5)),
                    ok.clone().index_put_((torch.tensor(2), torch.tensor(1)), torch.tensor(1 << 62))):
            d = bad.cuda()
            abi.shmem_alltoall(heap.handle, in_p, out_p, d.data_ptr(), W, row_bytes, in_rows,
                               out_rows, ws.data_ptr(), sig)
            rc, _ = abi.symm_check_error(heap.handle)
            assert rc == abi.SYMM_ERANGE, bad
            assert bool((heap.views(out_p, out_rows * row_bytes) == POISON).all())
        d = ok.cuda()   # the heap and the context stay usable
        abi.shmem_alltoall(heap.handle, in_p, out_p, d.data_ptr(), W, row_bytes, in_rows,
                           out_rows, ws.data_ptr(), sig)
        assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
        assert torch.equal(_signals(heap, sig), torch.full((W,), W, dtype=torch.int64))
    finally:
        heap.close()


@pytest.mark.parametrize("W,nbytes,in_shift,out_shift", [
    (1, 1000, 0, 0), (3, 0, 0, 0), (3, 1, 0, 0), (4, 17, 1, 2), (8, 16384, 0, 0),
    (8, 16385, 0, 0), (5, 100_003, 3, 7), (8, 1 << 20, 0, 0), (16, 300_000, 0, 4),
])
def test_allgather(W, nbytes, in_shift, out_shift):
    o = oracle.load()
    heap = _heap(W, (W + 1) * nbytes + 4096)
    try:
        in_p = heap.malloc(nbytes + 16) + in_shift
        out_p = heap.malloc(W * nbytes + 16) + out_shift
        sig = heap.malloc(64)
        x = inputs.random_bytes(W * nbytes, seed=W * 7 + nbytes % 97).view(W, nbytes)
        if nbytes:
            heap.views(in_p, nbytes).copy_(x.cuda())
            heap.views(out_p, W * nbytes).fill_(POISON)
        ws = _workspace(W)
        for _ in range(2):
            abi.shmem_allgather(heap.handle, in_p, out_p, W, nbytes, ws.data_ptr(), sig)
        assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
        if nbytes:
            got = heap.views(out_p, W * nbytes).cpu().numpy()
            assert np.array_equal(got, o.allgather(x.numpy()))
        assert torch.equal(_signals(heap, sig), torch.full((W,), W, dtype=torch.int64))
    finally:
        heap.close()
