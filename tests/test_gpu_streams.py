"""Every entry point on a stream of the caller's (not the default stream):
the work is enqueued on that stream, so after the stream is synchronised --
and only the stream -- the results match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

W = 4


def test_all_entry_points_on_a_side_stream():
    o = oracle.load()
    st = torch.cuda.Stream()
    heap = TorchSymmHeap(W, 16 << 20)
    try:
        g = torch.Generator().manual_seed(31)
        # combine: direct, producer/consumer, two-phase; dispatch and its inverse
        S, H, D = 32, 2, 64
        x = torch.randint(-2**15, 2**15, (W, S * W, H, D), generator=g, dtype=torch.int16)
        n = x[0].numel() * 2
        pin, pout, back = heap.malloc(n), heap.malloc(n), heap.malloc(n)
        stg_b, sig_b = abi.all2all_pc_workspace(W, S, H, D, 2, 8, 32, 2)
        staging, sig = heap.malloc(stg_b), heap.malloc(sig_b)
        nb, ns = abi.all2all_two_phase_workspace(W, S, H, D, 2, 8, 32, 2)
        bulk, tsig = heap.malloc(nb), heap.malloc(ns)
        heap.upload(pin, x.reshape(W, -1))
        torch.cuda.synchronize()
        want = o.combine(x.numpy(), W, S, H, D).view(np.uint8).reshape(W, -1)
        calls = [
            lambda: abi.all2all_combine(heap.handle, pin, pout, W, S, H, D, 2,
                                        abi.SYMM_A2A_DIRECT, stream=st),
            lambda: abi.all2all_combine(heap.handle, pin, pout, W, S, H, D, 2, abi.SYMM_A2A_PC,
                                        8, 32, 2, staging, sig, stream=st),
            lambda: abi.all2all_combine_two_phase(heap.handle, pin, pout, W, S, H, D, 2, 8, 32, 2,
                                                  bulk, tsig, stream=st),
        ]
        for call in calls:
            with torch.cuda.stream(st):
                heap.views(pout, n).fill_(0xA5)
            call()
            st.synchronize()
            assert abi.symm_check_error(heap.handle, st)[0] == abi.SYMM_OK
            assert np.array_equal(heap.download(pout, n).numpy(), want)
        abi.all2all_dispatch(heap.handle, pin, pout, W, S * W, H, D, 2, stream=st)
        abi.all2all_combine_back(heap.handle, pout, back, W, S, H, D, 2, stream=st)
        st.synchronize()
        assert np.array_equal(heap.download(back, n).numpy(),
                              x.numpy().view(np.uint8).reshape(W, -1))
        abi.symm_heap_reset(heap.handle)
        # AllToAll and AllGather
        counts = torch.tensor([[2, 0, 1, 3], [1, 1, 1, 1], [0, 3, 2, 0], [4, 0, 0, 1]])
        rb, in_rows, out_rows = 36, 6, 8
        xa = torch.randint(0, 256, (W, in_rows * rb), generator=g, dtype=torch.uint8)
        ws = torch.empty(abi.shmem_collective_workspace(W) // 8, dtype=torch.int64, device="cuda")
        pa_in, pa_out = heap.malloc(in_rows * rb), heap.malloc(out_rows * rb)
        psig = heap.malloc(64)
        heap.upload(pa_in, xa)
        heap.views(pa_out, out_rows * rb).fill_(0xA5)
        dc = counts.cuda()
        torch.cuda.synchronize()
        abi.shmem_alltoall(heap.handle, pa_in, pa_out, dc.data_ptr(), W, rb, in_rows, out_rows,
                           ws.data_ptr(), psig, stream=st)
        st.synchronize()
        want = o.alltoallv(xa.numpy().reshape(W, in_rows, rb), counts.numpy(), out_rows,
                           out=np.full((W, out_rows, rb), 0xA5, np.uint8))
        assert np.array_equal(heap.download(pa_out, out_rows * rb).numpy(), want.reshape(W, -1))
        abi.shmem_allgather(heap.handle, pa_in, pa_out, W, 2 * rb, ws.data_ptr(), psig, stream=st)
        st.synchronize()
        assert np.array_equal(heap.download(pa_out, W * 2 * rb).numpy(),
                              o.allgather(xa[:, :2 * rb].numpy()))
        abi.symm_heap_reset(heap.handle)
        # fused AllGather + MatMul
        m, k, nn = 128, 64, 256
        a, b = inputs.ag_matmul_inputs(W, m, k, nn, torch.float16, seed=8)
        sizes = [m * k * 2, k * nn * 2, W * m * nn * 2, W * m * k * 2,
                 abi.shmem_fused_ag_matmul_workspace(W, m, k, nn)]
        pa, pb, pc, pg, ps = [heap.malloc(z) for z in sizes]
        heap.upload(pa, a.reshape(W, -1))
        heap.upload(pb, b.reshape(W, -1))
        torch.cuda.synchronize()
        abi.shmem_fused_all_gather_matmul(heap.handle, pa, pb, pc, pg, W, m, k, nn,
                                          abi.SYMM_DTYPE_F16, 128, ps, stream=st)
        st.synchronize()
        a64, b64 = a.double().numpy(), b.double().numpy()
        _, ref = o.ag_matmul(a64, b64)
        _, mag = o.ag_matmul(np.abs(a64), np.abs(b64))
        cc = heap.download(pc, sizes[2]).view(torch.float16).double().numpy().reshape(ref.shape)
        # fp16 output rounding plus k fp32 additions of at most 2^-23 each
        tol = 2.0 ** -11 * np.abs(ref) + (1 + 2.0 ** -11) * k * 2.0 ** -23 * mag
        assert (np.abs(cc - ref) <= tol).all()
        assert abi.symm_check_error(heap.handle, st)[0] == abi.SYMM_OK
    finally:
        torch.cuda.synchronize()
        heap.close()
