"""GPU parity of the fused AllGather + MatMul (RFC "Symmetric Memory",
section 10, example 2) against the oracle.

gather_out must equal the stacked inputs bit for bit.  c is a floating-point
contraction: the kernel multiplies fp16/bf16 inputs exactly (a product of
two 11-bit significands fits fp32's 24), adds the k products in fp32 on the
tensor cores and rounds the sum to the input type.  Error model: each of the
k - 1 fp32 additions errs by at most one unit in the last place of its
result, 2^-23 relative -- what a truncating adder can do; round-to-nearest
gives half of it -- so the accumulated sum c^ satisfies

    |c^ - c| <= (k - 1) 2^-23 (1 + O(k 2^-23)) sum_x |a_ix| |b_xj|
             <= k 2^-23 sum_x |a_ix| |b_xj|        (k 2^-23 <= 2^-9 here),

and the final rounding adds u_out |c^| <= u_out (|c| + |c^ - c|).  Each
element must therefore lie within

    u_out |c| + (1 + u_out) k 2^-23 sum_x |a_ix| |b_xj|

of the oracle's fp64 value (u_out = 2^-11 for fp16, 2^-8 for bf16).  Small
shapes are checked on every element; the RFC example's size and the large
shapes whose throughput is reported are checked on sampled elements."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

POISON = 0xA5
DT = {"f16": (torch.float16, abi.SYMM_DTYPE_F16, 2.0 ** -11),
      "bf16": (torch.bfloat16, abi.SYMM_DTYPE_BF16, 2.0 ** -8)}


def tolerance(dt, k, ref, mag):
    """The bound above for reference values `ref` and sum |a| |b| values `mag`."""
    u_out = DT[dt][2]
    return u_out * np.abs(ref) + (1.0 + u_out) * k * 2.0 ** -23 * mag


def run(W, m_local, k, n, dt, seed=0, repeat=1):
    """Returns (a, b, gather [W, m_total, k] torch, c [W, m_total, n] float64 numpy,
    signals [W, slots])."""
    dtype, code, _ = DT[dt]
    a, b = inputs.ag_matmul_inputs(W, m_local, k, n, dtype, seed)
    m_total = W * m_local
    sig_bytes = abi.shmem_fused_ag_matmul_workspace(W, m_local, k, n)
    sizes = [a[0].numel() * 2, b[0].numel() * 2, m_total * n * 2, m_total * k * 2, sig_bytes]
    heap = TorchSymmHeap(W, sum(sizes) + 256 * len(sizes) + (4 << 20))
    try:
        pa, pb, pc, pg, ps = [heap.malloc(s) for s in sizes]
        heap.upload(pa, a.reshape(W, -1))
        heap.upload(pb, b.reshape(W, -1))
        heap.views(pc, sizes[2]).fill_(POISON)
        heap.views(pg, sizes[3]).fill_(POISON)
        for _ in range(repeat):
            abi.shmem_fused_all_gather_matmul(heap.handle, pa, pb, pc, pg, W, m_local, k, n, code,
                                              128, ps)
        torch.cuda.synchronize()
        rc, info = abi.symm_check_error(heap.handle)
        assert rc == abi.SYMM_OK, (rc, info)
        gather = heap.download(pg, sizes[3]).view(dtype).reshape(W, m_total, k)
        c = heap.download(pc, sizes[2]).view(dtype).reshape(W, m_total, n).double().numpy()
        sig = heap.download(ps, sig_bytes).view(torch.int64).reshape(W, -1)
        return a, b, gather, c, sig[:, :W * (m_local // 128) * 8:8]
    finally:
        heap.close()


def check_gather(a, gather):
    W = a.shape[0]
    stacked = a.reshape(W * a.shape[1], a.shape[2])
    for d in range(W):
        assert torch.equal(gather[d].view(torch.int16), stacked.view(torch.int16)), d


@pytest.mark.parametrize("W,m_local,k,n,dt", [
    (1, 128, 64, 256, "bf16"),     # one tile, one K slice
    (1, 128, 256, 256, "f16"),
    (2, 256, 320, 512, "bf16"),
    (3, 128, 200, 264, "f16"),     # k and n not multiples of the tile
    (4, 256, 72, 1000, "bf16"),
    (2, 128, 8, 64, "f16"),        # the smallest k and n: zero-filled K slice, N boxes past n
    (16, 128, 64, 256, "bf16"),    # 16 PEs
    (2, 256, 128, 256, "f16"),     # two row blocks per PE, one column tile
    (3, 384, 64, 512, "bf16"),     # odd row blocks per PE
])
def test_small_shapes_every_element(W, m_local, k, n, dt):
    o = oracle.load()
    a, b, gather, c, sig = run(W, m_local, k, n, dt, seed=W * 10 + k)
    check_gather(a, gather)
    assert torch.equal(sig, torch.ones_like(sig))
    a64, b64 = a.double().numpy(), b.double().numpy()
    _, ref = o.ag_matmul(a64, b64)
    _, mag = o.ag_matmul(np.abs(a64), np.abs(b64))
    tol = tolerance(dt, k, ref, mag)
    err = np.abs(c - ref)
    assert (err <= tol).all(), f"max err {err.max()}, worst ratio {(err / tol).max()}"


@pytest.mark.parametrize("dt,W,m_local,k,n", [
    ("bf16", 8, 512, 1024, 2048), ("f16", 8, 512, 1024, 2048),
    ("bf16", 4, 256, 2048, 4096),   # 64 MB of b in all: the PE-major tile order
    ("bf16", 8, 1024, 4096, 4096),  # the large shapes whose TFLOP/s are reported
    ("bf16", 8, 2048, 7168, 2048),
    ("bf16", 4, 1024, 8192, 8192),
])
def test_example_size_sampled(dt, W, m_local, k, n):
    """The RFC example's shapes with 8 PEs (m_local 512, k 1024, n 2048,
    blocks of 128 rows), cases whose b matrices do not fit in L2 together,
    and the large shapes up to k = 8192; 3000 sampled elements plus strided
    elements of the first and last rows."""
    o = oracle.load()
    a, b, gather, c, sig = run(W, m_local, k, n, dt, seed=7, repeat=2)
    check_gather(a, gather)
    assert torch.equal(sig, torch.ones_like(sig))
    a64 = np.ascontiguousarray(a.double().numpy())
    b64 = np.ascontiguousarray(b.double().numpy())
    aa, ab = np.abs(a64), np.abs(b64)
    rng = np.random.default_rng(3)
    picks = [(int(rng.integers(W)), int(rng.integers(W * m_local)), int(rng.integers(n)))
             for _ in range(3000)]
    picks += [(d, i, j) for d in (0, W - 1) for i in (0, W * m_local - 1) for j in range(0, n, 97)]
    for d, i, j in picks:
        ref = o.ag_matmul_at(a64, b64, d, i, j)
        tol = tolerance(dt, k, ref, o.ag_matmul_at(aa, ab, d, i, j))
        assert abs(c[d, i, j] - ref) <= tol, (d, i, j, c[d, i, j], ref)


def test_empty_rows_launch_nothing():
    heap = TorchSymmHeap(2, 4 << 20)
    try:
        p = [heap.malloc(4096) for _ in range(5)]
        abi.shmem_fused_all_gather_matmul(heap.handle, p[0], p[1], p[2], p[3], 2, 0, 64, 64,
                                          abi.SYMM_DTYPE_F16, 128, p[4])
        torch.cuda.synchronize()
        assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    finally:
        heap.close()
