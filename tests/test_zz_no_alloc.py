"""all2all_combine_pc_noalloc: the producer/consumer combine for callers that
cannot allocate device memory (their device memory is all handed out by
another allocator, or their hot path must not pay for cudaMalloc/cudaFree).
Its staging ring and signal slots live in the library's own static device
array; the caller passes only the input and output.

Checked through the C ABI, on two calls in a row with different shapes (the
second call must not be disturbed by what the first left in the shared
array), against both the CPU oracle and the regular all2all_combine; the
path moves bits, so both comparisons are exact.  A repeated call must leave
the device's free memory and torch's reserved memory unchanged.  This file
runs last so that a failure here leaves every other test already run; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

W = 8
POISON = 0xA5


def _expect(x, S, H, D, es):
    """The oracle's combine of raw es-byte elements."""
    xv = np.ascontiguousarray(x.numpy()).view(np.dtype((np.void, es))).reshape(W, S * W, H, D)
    return oracle.load().combine(xv, W, S, H, D).view(np.uint8).reshape(W, -1)


def _case(heap, inp, out_a, out_b, S, H, D, dtype, tile_s, block_d, seed):
    es = torch.empty((), dtype=dtype).element_size()
    n = S * W * H * D * es
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(0, 256, (W, n), generator=g, dtype=torch.uint8)
    heap.upload(inp, x)
    heap.views(out_a, n).fill_(POISON)
    heap.views(out_b, n).fill_(POISON)
    # the existing entry point, with its staging and signals in the heap
    st, sg = abi.all2all_pc_workspace(W, S, H, D, es, tile_s, block_d, 2)
    staging = heap.malloc(st)
    signals = heap.malloc(sg)
    abi.all2all_combine(heap.handle, inp, out_a, W, S, H, D, es, abi.SYMM_A2A_PC, tile_s, block_d,
                        2, staging, signals)
    # the allocation-free entry point
    abi.all2all_combine_pc_noalloc(heap.handle, inp, out_b, W, S, H, D, es, tile_s, block_d, 2)
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)
    a = heap.download(out_a, n)
    b = heap.download(out_b, n)
    want = _expect(x, S, H, D, es)
    assert np.array_equal(b.numpy(), want), "allocation-free combine differs from the oracle"
    assert np.array_equal(a.numpy(), want), "heap-workspace combine differs from the oracle"
    assert torch.equal(a, b)


def test_noalloc_matches_oracle_and_combine_two_calls_in_a_row():
    assert torch.cuda.is_available()
    cap = 16 << 20
    heap = TorchSymmHeap(W, 4 * cap)
    inp, out_a, out_b = heap.malloc(cap), heap.malloc(cap), heap.malloc(cap)
    # call 1: bf16, aligned 400-byte rows in 4 D blocks
    _case(heap, inp, out_a, out_b, 48, 2, 200, torch.bfloat16, 16, 64, seed=1)
    # call 2: fp16 unaligned 1998-byte rows, one D block, taller tiles
    _case(heap, inp, out_a, out_b, 70, 1, 999, torch.float16, 32, 0, seed=2)
    heap.close()


def test_noalloc_call_allocates_nothing():
    """After a first call, further calls change neither the device's free
    memory nor the bytes torch's caching allocator holds."""
    assert torch.cuda.is_available()
    S, H, D, es = 64, 1, 2048, 2
    n = S * W * H * D * es
    heap = TorchSymmHeap(W, 2 * n + (1 << 20))
    inp, out = heap.malloc(n), heap.malloc(n)
    heap.views(inp, n).copy_(torch.randint(0, 256, (W, n), dtype=torch.uint8))
    abi.all2all_combine_pc_noalloc(heap.handle, inp, out, W, S, H, D, es, 16, 1024, 2)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        abi.all2all_combine_pc_noalloc(heap.handle, inp, out, W, S, H, D, es, 16, 1024, 2)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert torch.cuda.memory_reserved() == reserved0
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)
    heap.close()


def test_noalloc_rejects_more_than_its_static_scratch():
    assert torch.cuda.is_available()
    heap = TorchSymmHeap(W, 8 << 20)
    inp, out = heap.malloc(1 << 20), heap.malloc(1 << 20)
    # DeepSeek-V3 rows with 64-row tiles need W*2*64*8*7168*2 = 117 MB > 32 MiB
    with pytest.raises(abi.SymmError) as e:
        abi.all2all_combine_pc_noalloc(heap.handle, inp, out, W, 8, 1, 7168, 2, 64, 0, 2)
    assert e.value.code in (abi.SYMM_EINVAL,)
    heap.close()
