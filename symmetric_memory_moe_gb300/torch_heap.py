"""A symmetric heap whose memory is one PyTorch CUDA tensor.

PyTorch only provides the device allocation and host<->device copies for
setting up inputs and reading results; every step of the all-to-all runs in
libsymm_a2a.so through :mod:`abi`.
"""
from __future__ import annotations

import torch

from . import abi

SLAB_ALIGN = 2 << 20  # slabs are rounded up to 2 MiB


def _up(n: int, a: int) -> int:
    return (n + a - 1) // a * a


class TorchSymmHeap:
    """W slabs of ``slab`` bytes in one uint8 CUDA tensor, registered with
    ``symm_heap_init``."""

    def __init__(self, npes: int, slab_bytes: int, device=None):
        self.npes = npes
        self.slab = _up(max(slab_bytes, abi.SYMM_HEAP_HEADER_BYTES + 256), SLAB_ALIGN)
        dev = torch.device(device) if device is not None else torch.device("cuda",
                                                                           torch.cuda.current_device())
        self.mem = torch.empty(npes * self.slab, dtype=torch.uint8, device=dev)
        self.base = self.mem.data_ptr()
        self.handle = abi.symm_heap_init(self.base, self.slab, npes)

    def malloc(self, nbytes: int, align: int = 0) -> int:
        return abi.symm_malloc(self.handle, nbytes, align)

    def offset(self, ptr: int) -> int:
        return (ptr - self.base) % self.slab

    def views(self, ptr: int, nbytes: int) -> torch.Tensor:
        """[W, nbytes] uint8 view: row k is PE k's copy of the object at ptr."""
        return self.mem.as_strided((self.npes, nbytes), (self.slab, 1), self.offset(ptr))

    def upload(self, ptr: int, host: torch.Tensor) -> None:
        """Copies host [W, ...] (any dtype) into every PE's copy of ptr's object."""
        flat = host.contiguous().view(torch.uint8).reshape(self.npes, -1)
        self.views(ptr, flat.shape[1]).copy_(flat, non_blocking=flat.is_pinned())

    def download(self, ptr: int, nbytes: int) -> torch.Tensor:
        """[W, nbytes] uint8 host copy of every PE's object at ptr."""
        return self.views(ptr, nbytes).cpu()

    def close(self) -> None:
        if self.handle:
            abi.symm_heap_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CombineBuffers:
    """Heap + symmetric in/out (+ producer/consumer staging and signals) for
    one all-to-all shape: per-PE input rows_in x H x D, output the same bytes."""

    def __init__(self, W: int, rows_in: int, H: int, D: int, elem_bytes: int, *, pc: bool = False,
                 S: int | None = None, tile_s: int = 16, block_d: int = 0, buffer_num: int = 2,
                 extra: int = 0, device=None):
        self.W, self.H, self.D, self.es = W, H, D, elem_bytes
        self.nbytes = rows_in * H * D * elem_bytes
        self.tile_s, self.block_d, self.buffer_num = tile_s, block_d, buffer_num
        st = sg = 0
        if pc:
            st, sg = abi.all2all_pc_workspace(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num)
        slab = abi.SYMM_HEAP_HEADER_BYTES + 2 * _up(self.nbytes, 256) + _up(st, 256) + \
            _up(sg, 256) + extra + 4 * 256
        self.heap = TorchSymmHeap(W, slab, device)
        self.inp = self.heap.malloc(self.nbytes)
        self.out = self.heap.malloc(self.nbytes)
        self.staging = self.heap.malloc(st) if pc else None
        self.signals = self.heap.malloc(sg) if pc else None
        self.staging_bytes, self.signal_bytes = st, sg
