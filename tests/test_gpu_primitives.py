"""GPU parity of the one-sided primitives against the oracle's host-memory
heap model, and the bounded waits: a wait that nothing satisfies gives up
with SYMM_ETIMEDOUT after its budget and leaves the context usable."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import CombineBuffers, TorchSymmHeap

pytestmark = pytest.mark.gpu

W = 4
SLAB = 2 << 20
HDR = abi.SYMM_HEAP_HEADER_BYTES


@pytest.fixture()
def heap():
    assert torch.cuda.is_available()
    h = TorchSymmHeap(W, SLAB)
    h.mem.zero_()
    yield h
    h.close()


def _device_heap(h: TorchSymmHeap) -> np.ndarray:
    torch.cuda.synchronize()
    a = h.mem.cpu().numpy().copy()
    for pe in range(W):  # the header is the library's own
        a[pe * h.slab: pe * h.slab + HDR] = 0
    return a


def test_put_get_match_oracle(heap):
    o = oracle.load()
    model = np.zeros(W * heap.slab, np.uint8)
    obj = heap.malloc(600_000)
    src_dev = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    src_host = inputs.random_bytes(1 << 20, seed=11)
    src_dev.copy_(src_host)
    rng = np.random.default_rng(0)
    # sizes and offsets covering every phase mod 16 on both sides, and long runs
    cases = [(0, 0, 1), (3, 5, 15), (17, 1, 16), (1, 2, 33), (5, 12, 4099), (8, 24, 65536),
             (7, 3, 300_001), (0, 0, 524_288)]
    cases += [(int(rng.integers(0, 4000)), int(rng.integers(0, 4000)),
               int(rng.integers(1, 50000))) for _ in range(12)]
    for i, (toff, soff, n) in enumerate(cases):
        pe = i % W
        abi.shmem_put(heap.handle, obj, toff, src_dev.data_ptr(), soff, n, pe)
        assert o.put(model, heap.slab, W, heap.offset(obj) + toff,
                     src_host[soff:soff + n].numpy(), pe) == 0
    assert np.array_equal(_device_heap(heap), model)
    # get back from every PE, at shifted offsets
    dst = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for i, (off, doff, n) in enumerate([(0, 0, 70000), (5, 3, 4097), (13, 0, 31), (2, 9, 600)]):
        pe = (i + 1) % W
        abi.shmem_get(heap.handle, dst.data_ptr(), doff, obj, off, n, pe)
        want = np.zeros(n, np.uint8)
        assert o.get(model, heap.slab, W, want, heap.offset(obj) + off, pe) == 0
        torch.cuda.synchronize()
        assert np.array_equal(dst[doff:doff + n].cpu().numpy(), want)


def test_signal_ops_and_put_with_signal(heap):
    o = oracle.load()
    model = np.zeros(W * heap.slab, np.uint8)
    data = heap.malloc(1 << 16)
    sig = heap.malloc(64 * 8)
    src_host = inputs.random_bytes(1 << 16, seed=12)
    src = src_host.cuda()
    sig_off = heap.offset(sig)
    # RFC example 1: rank 0 puts 4096 elements to rank 1 and SETs signal 1
    abi.shmem_put_with_signal(heap.handle, data, 0, src.data_ptr(), 0, 8192, sig, 0, 1,
                              abi.SYMM_SIGNAL_SET, 1)
    o.put_with_signal(model, heap.slab, W, heap.offset(data), src_host[:8192].numpy(), sig_off,
                      1, 0, 1)
    # push mode: every rank puts a segment to PE 0 and ADDs 1 to its counter
    seg = 1000
    for r in range(W):
        abi.shmem_put_with_signal(heap.handle, data, 9000 + r * seg, src.data_ptr(), r * seg, seg,
                                  sig, 8, 1, abi.SYMM_SIGNAL_ADD, 0)
        o.put_with_signal(model, heap.slab, W, heap.offset(data) + 9000 + r * seg,
                          src_host[r * seg:(r + 1) * seg].numpy(), sig_off + 64, 1, 1, 0)
    # plain signal ops, including negative values and wrap-around
    for (v, op, pe, el) in [(-7, 0, 2, 16), (5, 1, 2, 16), (2**62, 1, 3, 24), (2**62, 1, 3, 24),
                            (0, 1, 3, 24)]:
        abi.shmem_signal_op(heap.handle, sig, el, v, op, pe)
        o.signal_op(model, heap.slab, W, sig_off + 8 * el, v, op, pe)
    assert np.array_equal(_device_heap(heap), model)
    # waits that hold already return without error: EQ W on PE 0, GT/LT
    abi.shmem_wait_for_signal(heap.handle, sig, 8, W, abi.SYMM_CMP_EQ, 0, 10**9)
    abi.shmem_wait_for_signal(heap.handle, sig, 0, 0, abi.SYMM_CMP_GT, 1, 10**9)
    abi.shmem_wait_for_signal(heap.handle, sig, 16, -1, abi.SYMM_CMP_LT, 2, 10**9)
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)


def test_put_with_signal_zero_bytes_only_signals(heap):
    sig = heap.malloc(64)
    abi.shmem_put_with_signal(heap.handle, sig, 0, 0, 0, 0, sig, 0, 3, abi.SYMM_SIGNAL_SET, 2)
    torch.cuda.synchronize()
    assert heap.views(sig, 8)[2].view(torch.int64).item() == 3


@pytest.mark.parametrize("cmp,value", [(abi.SYMM_CMP_EQ, 1), (abi.SYMM_CMP_GT, 0),
                                       (abi.SYMM_CMP_LT, 0)])
def test_wait_on_unset_signal_times_out(heap, cmp, value):
    """A flag that nothing sets: the wait gives up after ~20 ms and reports
    which signal it was; the stream and context keep working afterwards."""
    sig = heap.malloc(64 * 4)
    abi.shmem_wait_for_signal(heap.handle, sig, 2, value, cmp, 3, 20_000_000)
    rc, info = abi.symm_check_error(heap.handle)
    assert rc == abi.SYMM_ETIMEDOUT
    assert info == 3 * heap.slab + heap.offset(sig) + 16
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)  # cleared
    abi.shmem_signal_op(heap.handle, sig, 2, 1, abi.SYMM_SIGNAL_SET, 3)
    abi.shmem_wait_for_signal(heap.handle, sig, 2, 1, abi.SYMM_CMP_EQ, 3, 10**9)
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)


@pytest.mark.parametrize("H,D", [
    (2, 64),      # 128-byte rows: whole-tile group copies, no prefetch
    (1, 1024),    # 2 KB rows: the prefetching kernel with release threads
    (2, 999),     # 1998-byte rows: shift-merged group copies
])
def test_pc_stale_signal_times_out_then_recovers(H, D):
    """A producer/consumer slot left at a value nobody expects (2): with the
    launch's slot reset skipped, its producer (waits for 0) and consumer
    (waits for 1) give up after the budget and every other group and release
    thread aborts; the next call with the reset runs clean and bit-exact."""
    Wp, S = 4, 32
    bufs = CombineBuffers(Wp, S * Wp, H, D, 2, pc=True, S=S, tile_s=8)
    heap = bufs.heap
    g = torch.Generator().manual_seed(3)
    x = torch.randint(-30000, 30000, (Wp, S * Wp, H, D), generator=g, dtype=torch.int16)
    heap.upload(bufs.inp, x.reshape(Wp, -1))
    heap.views(bufs.signals, bufs.signal_bytes).zero_()
    abi.symm_set_spin_budget(heap.handle, 50_000_000)
    slot = 2 * H + H - 1  # ((buf*W + r)*nbd + bd)*H + h with buf 0, source r 2, block 0, h H-1; on PE 2
    abi.shmem_signal_op(heap.handle, bufs.signals, slot * 8, 2, abi.SYMM_SIGNAL_SET, 2)
    abi.all2all_combine(heap.handle, bufs.inp, bufs.out, Wp, S, H, D, 2,
                        abi.SYMM_A2A_PC | abi.SYMM_A2A_FLAG_NO_RESET, 8, 0, 2, bufs.staging,
                        bufs.signals)
    rc, info = abi.symm_check_error(heap.handle)
    assert rc == abi.SYMM_ETIMEDOUT
    assert info == 2 * heap.slab + heap.offset(bufs.signals) + slot * 64
    abi.symm_set_spin_budget(heap.handle, 2_000_000_000)
    abi.all2all_combine(heap.handle, bufs.inp, bufs.out, Wp, S, H, D, 2, abi.SYMM_A2A_PC, 8, 0, 2,
                        bufs.staging, bufs.signals)
    assert abi.symm_check_error(heap.handle) == (abi.SYMM_OK, 0)
    got = heap.download(bufs.out, bufs.nbytes).numpy()
    want = oracle.load().combine(x.numpy(), Wp, S, H, D).view(np.uint8).reshape(Wp, -1)
    assert np.array_equal(got, want)
    heap.close()


def test_put_based_combine(heap):
    """The combine composed from the primitives, in the RFC's push mode: PE r
    puts every run it owes PE d (its rows d*S + s) into out_d's column r*H
    with put_with_signal ADD 1 on d's counter; each PE then waits for its
    counter to reach W*S.  The result equals the oracle's combine."""
    o = oracle.load()
    S, H, D, es = 6, 2, 12, 2
    R = H * D * es
    x = inputs.random_bytes(W * S * W * R, seed=21).view(W, S * W * R)
    inp = heap.malloc(S * W * R)
    out = heap.malloc(S * W * R)
    sig = heap.malloc(64)
    heap.upload(inp, x)
    heap.views(out, S * W * R).fill_(0xA5)
    heap.views(sig, 64).zero_()
    for r in range(W):
        src = abi.symm_at(heap.handle, inp, r)  # PE r's own input
        for d in range(W):
            for s in range(S):
                abi.shmem_put_with_signal(heap.handle, out, (s * W + r) * R, src,
                                          (d * S + s) * R, R, sig, 0, 1, abi.SYMM_SIGNAL_ADD, d)
    for d in range(W):
        abi.shmem_wait_for_signal(heap.handle, sig, 0, W * S, abi.SYMM_CMP_EQ, d)
    torch.cuda.synchronize()
    assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    want = o.combine(x.numpy().reshape(W, S * W, H, D * es), W, S, H, D * es)
    assert np.array_equal(heap.download(out, S * W * R).numpy(),
                          want.view(np.uint8).reshape(W, -1))
