"""GPU parity of the two-phase combine ("UDMA Optimized Implementation" with
its wait/notify signal regions) against the oracle, bit for bit: the output
equals the combine's definition on the combine workloads and on ragged,
odd-sized and shifted layouts (all three copy instances: bulk sends with
group-wide tile copies, bulk sends with per-row copies, vector copies
everywhere); on small shapes the bulk rank slots and both signal regions
also equal the sequential replay of the page's algorithm after the call."""
import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import TorchSymmHeap

pytestmark = pytest.mark.gpu

POISON = 0xA5


def _np_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy()


def run_two_phase(x, W, S, H, D, tile_s, block_d=0, buffer_num=2, in_shift=0, out_shift=0,
                  repeat=1):
    """x: CPU [W][S*W][H][D].  Returns (out bytes [W, n], bulk bytes [W, n],
    signals [W, slots, 8] int64) after `repeat` calls."""
    es = x.element_size()
    n = S * W * H * D * es
    bulk_bytes, sig_bytes = abi.all2all_two_phase_workspace(W, S, H, D, es, tile_s, block_d,
                                                            buffer_num)
    assert bulk_bytes == n
    heap = TorchSymmHeap(W, 3 * n + sig_bytes + (4 << 20))
    try:
        inp = heap.malloc(n + 64) + in_shift
        out = heap.malloc(n + 64) + out_shift
        bulk = heap.malloc(bulk_bytes)
        sig = heap.malloc(sig_bytes)
        heap.upload(inp, x.reshape(W, -1))
        heap.views(out, n).fill_(POISON)
        heap.views(bulk, bulk_bytes).fill_(POISON)
        heap.views(sig, sig_bytes).fill_(0x7F)   # the call resets its signals itself
        for _ in range(repeat):
            abi.all2all_combine_two_phase(heap.handle, inp, out, W, S, H, D, es, tile_s, block_d,
                                          buffer_num, bulk, sig)
        torch.cuda.synchronize()
        rc, info = abi.symm_check_error(heap.handle)
        assert rc == abi.SYMM_OK, (rc, info)
        return (heap.download(out, n).numpy(), heap.download(bulk, bulk_bytes).numpy(),
                heap.download(sig, sig_bytes).view(torch.int64).numpy().reshape(W, -1, 8))
    finally:
        heap.close()


def _check(x, W, S, H, D, tile_s, block_d=0, buffer_num=2, replay=True, **kw):
    got, bulk, sig = run_two_phase(x, W, S, H, D, tile_s, block_d, buffer_num, **kw)
    o = oracle.load()
    xb = _np_bits(x)
    want = o.combine(xb, W, S, H, D).view(np.uint8).reshape(W, -1)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} output bytes differ"
    nbs = -(-S // tile_s)
    # region A: 1 for every (block, sender r != d), 0 for r == d; region B: 0
    region_a = sig[:, :nbs * W, 0].reshape(W, nbs, W)
    want_a = np.ones((W, nbs, W), np.int64)
    for d in range(W):
        want_a[d, :, d] = 0
    assert np.array_equal(region_a, want_a)
    assert not sig[:, nbs * W:, 0].any()
    if replay:  # the rank slots r != d hold what the page's phase 1 leaves there
        _, peer, rsig = o.two_phase_replay(xb, W, S, H, D, tile_s, block_d or D, buffer_num)
        peer = peer.view(np.uint8).reshape(W, W, -1)
        bulk = bulk.reshape(W, W, -1)
        for d in range(W):
            for r in range(W):
                if r != d:
                    assert np.array_equal(bulk[d, r], peer[d, r]), (d, r)
        assert np.array_equal(sig[:, :, 0], rsig[:, :, 0])


@pytest.mark.parametrize("name,tile_s,block_d", [
    ("tiny", 2, 0), ("small", 16, 64), ("dsv3", 16, 0), ("dsv3", 64, 1024), ("tail", 32, 0)])
def test_workload_shapes(name, tile_s, block_d):
    wl = inputs.WORKLOADS[name]
    x = inputs.make_input(wl)
    _check(x, wl.W, wl.S, wl.H, wl.D, tile_s, block_d, replay=wl.total_bytes < (64 << 20))


@pytest.mark.parametrize("W,S,H,D,dtype,tile_s,block_d,nbuf", [
    (3, 7, 1, 5, torch.int16, 2, 3, 3),       # ragged S and D blocks, 10-byte rows
    (5, 9, 2, 6, torch.int32, 4, 4, 1),       # one buffer
    (1, 6, 3, 4, torch.int16, 2, 2, 2),       # one PE: the self loop only
    (2, 3, 1, 7, torch.uint8, 8, 16, 2),      # tile taller than S
    (4, 40, 2, 999, torch.float16, 8, 256, 2),
    (8, 64, 4, 64, torch.bfloat16, 16, 0, 3),  # 16-byte rows: bulk sends, group tile copies
    (6, 33, 1, 520, torch.float32, 5, 100, 2),  # bulk sends, unaligned D blocks
])
def test_shapes_and_replay(W, S, H, D, dtype, tile_s, block_d, nbuf):
    g = torch.Generator().manual_seed(W * 100 + S)
    x = torch.randint(-30000, 30000, (W, S * W, H, D), generator=g, dtype=torch.int32).to(dtype)
    _check(x, W, S, H, D, tile_s, block_d, nbuf)


@pytest.mark.parametrize("in_shift,out_shift", [(2, 0), (0, 6), (10, 14)])
def test_shifted_pointers(in_shift, out_shift):
    W, S, H, D = 4, 24, 2, 64
    g = torch.Generator().manual_seed(in_shift + out_shift)
    x = torch.randint(-30000, 30000, (W, S * W, H, D), generator=g).to(torch.int16)
    _check(x, W, S, H, D, 8, 32, in_shift=in_shift, out_shift=out_shift)


def test_repeated_calls_reuse_the_workspace():
    W, S, H, D = 8, 96, 1, 512
    g = torch.Generator().manual_seed(3)
    x = torch.randint(-30000, 30000, (W, S * W, H, D), generator=g).to(torch.bfloat16)
    _check(x, W, S, H, D, 16, 0, 2, repeat=4)


def test_empty_extents_launch_nothing():
    heap = TorchSymmHeap(2, 4 << 20)
    try:
        p = heap.malloc(4096)
        q = heap.malloc(4096)
        b = heap.malloc(4096)
        s = heap.malloc(4096)
        for S, H, D in [(0, 2, 8), (4, 0, 8), (4, 2, 0)]:
            abi.all2all_combine_two_phase(heap.handle, p, q, 2, S, H, D, 2, 2, 0, 2, b, s)
        torch.cuda.synchronize()
        assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    finally:
        heap.close()
