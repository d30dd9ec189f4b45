"""Every entry point on objects placed past 4.5 GiB inside each PE's slab:
the heap's address arithmetic (PE index times slab, plus the object offset)
must be 64-bit all the way through.  Results are checked against the oracle
as in the other GPU tests (bit for bit; the fused matmul within its fp32
accumulation bound)."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

W = 2
FILLER = (9 << 29)  # 4.5 GiB of every slab before the objects under test


@pytest.fixture(scope="module")
def heap():
    h = TorchSymmHeap(W, FILLER + (64 << 20))
    h.malloc(FILLER)
    yield h
    h.close()


@pytest.fixture(autouse=True)
def _fresh(heap):
    abi.symm_heap_reset(heap.handle)
    heap.malloc(FILLER)
    yield


def _check_ok(heap):
    rc, info = abi.symm_check_error(heap.handle)
    assert rc == abi.SYMM_OK, (rc, info)


def test_objects_are_past_4_gib(heap):
    p = heap.malloc(64)
    assert heap.offset(p) >= FILLER > (1 << 32)


@pytest.mark.parametrize("kind", ["direct", "pc", "two_phase"])
def test_combine(heap, kind):
    o = oracle.load()
    S, H, D = 24, 2, 40
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-2**15, 2**15, (W, S * W, H, D), generator=g, dtype=torch.int16)
    n = x[0].numel() * 2
    pin, pout = heap.malloc(n), heap.malloc(n)
    heap.upload(pin, x.reshape(W, -1))
    heap.views(pout, n).fill_(0xA5)
    if kind == "two_phase":
        nb, ns = abi.all2all_two_phase_workspace(W, S, H, D, 2, 8, 16, 2)
        bulk, sig = heap.malloc(nb), heap.malloc(ns)
        abi.all2all_combine_two_phase(heap.handle, pin, pout, W, S, H, D, 2, 8, 16, 2, bulk, sig)
    else:
        variant = abi.SYMM_A2A_PC if kind == "pc" else abi.SYMM_A2A_DIRECT
        st, sg = abi.all2all_pc_workspace(W, S, H, D, 2, 8, 16, 2)
        staging, sig = heap.malloc(st), heap.malloc(sg)
        abi.all2all_combine(heap.handle, pin, pout, W, S, H, D, 2, variant, 8, 16, 2, staging, sig)
    _check_ok(heap)
    want = o.combine(x.numpy(), W, S, H, D).view(np.uint8).reshape(W, -1)
    assert np.array_equal(heap.download(pout, n).numpy(), want)


def test_put_get_and_collectives(heap):
    o = oracle.load()
    g = torch.Generator().manual_seed(6)
    # put to PE 1, get back from it
    obj = heap.malloc(5000)
    src = torch.randint(0, 256, (5000,), generator=g, dtype=torch.uint8).cuda()
    dst = torch.zeros(5000, dtype=torch.uint8, device="cuda")
    abi.shmem_put(heap.handle, obj, 0, src.data_ptr(), 0, 5000, 1)
    abi.shmem_get(heap.handle, dst.data_ptr(), 0, obj, 0, 5000, 1)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
    # AllToAll with uneven counts, then AllGather
    counts = torch.tensor([[2, 3], [1, 0]])
    rb, in_rows, out_rows = 24, 5, 4
    x = torch.randint(0, 256, (W, in_rows * rb), generator=g, dtype=torch.uint8)
    ws = torch.empty(abi.shmem_collective_workspace(W) // 8, dtype=torch.int64, device="cuda")
    pin, pout, sig = heap.malloc(in_rows * rb), heap.malloc(out_rows * rb), heap.malloc(64)
    heap.upload(pin, x)
    heap.views(pout, out_rows * rb).fill_(0xA5)
    dc = counts.cuda()
    abi.shmem_alltoall(heap.handle, pin, pout, dc.data_ptr(), W, rb, in_rows, out_rows,
                       ws.data_ptr(), sig)
    _check_ok(heap)
    want = o.alltoallv(x.numpy().reshape(W, in_rows, rb), counts.numpy(), out_rows,
                       out=np.full((W, out_rows, rb), 0xA5, np.uint8))
    assert np.array_equal(heap.download(pout, out_rows * rb).numpy(), want.reshape(W, -1))
    abi.shmem_allgather(heap.handle, pin, pout, W, 2 * rb, ws.data_ptr(), sig)
    _check_ok(heap)
    got = heap.download(pout, W * 2 * rb).numpy()
    assert np.array_equal(got, o.allgather(x[:, :2 * rb].numpy()))


def test_fused_all_gather_matmul(heap):
    o = oracle.load()
    m, k, n = 128, 64, 256
    g = torch.Generator().manual_seed(7)
    a = torch.randn(W, m, k, generator=g).to(torch.bfloat16)
    b = torch.randn(W, k, n, generator=g).to(torch.bfloat16)
    sizes = [m * k * 2, k * n * 2, W * m * n * 2, W * m * k * 2,
             abi.shmem_fused_ag_matmul_workspace(W, m, k, n)]
    pa, pb, pc, pg, ps = [heap.malloc(z) for z in sizes]
    heap.upload(pa, a.reshape(W, -1))
    heap.upload(pb, b.reshape(W, -1))
    abi.shmem_fused_all_gather_matmul(heap.handle, pa, pb, pc, pg, W, m, k, n,
                                      abi.SYMM_DTYPE_BF16, 128, ps)
    _check_ok(heap)
    a64, b64 = a.double().numpy(), b.double().numpy()
    gather, ref = o.ag_matmul(a64, b64)
    _, mag = o.ag_matmul(np.abs(a64), np.abs(b64))
    gg = heap.download(pg, sizes[3]).view(torch.bfloat16).double().numpy().reshape(gather.shape)
    cc = heap.download(pc, sizes[2]).view(torch.bfloat16).double().numpy().reshape(ref.shape)
    assert np.array_equal(gg, gather)
    # bf16 output rounding plus k fp32 additions of at most 2^-23 each
    assert (np.abs(cc - ref) <= 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * k * 2.0 ** -23 * mag).all()
