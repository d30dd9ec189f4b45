"""Thin ctypes binding of libsymm_a2a.so (include/symm_a2a.h).

Functions carry the C names and argument order; this module only marshals
arguments (ints for device pointers, an int or an object with ``.cuda_stream``
for the stream) and turns negative return codes into ``SymmError``.  All
work runs in the library's CUDA kernels; there is no other code path.  If the
library cannot be loaded (or built with nvcc) every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SYMM_OK = 0
SYMM_EINVAL = -1
SYMM_ENOMEM = -2
SYMM_ETIMEDOUT = -3
SYMM_ECUDA = -4
SYMM_ERANGE = -5
SYMM_SIGNAL_SET = 0
SYMM_SIGNAL_ADD = 1
SYMM_CMP_EQ = 0
SYMM_CMP_GT = 1
SYMM_CMP_LT = 2
SYMM_A2A_DIRECT = 0
SYMM_A2A_PC = 1
SYMM_A2A_FLAG_NO_RESET = 0x100
SYMM_A2A_FLAG_VECTOR = 0x200
SYMM_A2A_FLAG_BULK = 0x400
SYMM_A2A_FLAG_PHASED = 0x800
SYMM_HEAP_HEADER_BYTES = 4096
SYMM_SIGNAL_STRIDE_BYTES = 64
SYMM_NOALLOC_SCRATCH_BYTES = 32 << 20

_NAMES = {SYMM_EINVAL: "SYMM_EINVAL", SYMM_ENOMEM: "SYMM_ENOMEM",
          SYMM_ETIMEDOUT: "SYMM_ETIMEDOUT", SYMM_ECUDA: "SYMM_ECUDA", SYMM_ERANGE: "SYMM_ERANGE"}


class SymmError(RuntimeError):
    def __init__(self, code: int, func: str, msg: str):
        super().__init__(f"{func}: {_NAMES.get(code, code)}: {msg}")
        self.code = code


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64

_SIGS = {
    "symm_heap_init": [_P, _SZ, _I, ctypes.POINTER(_P)],
    "symm_heap_destroy": [_P],
    "symm_malloc": [_P, _SZ, _SZ, ctypes.POINTER(_P)],
    "symm_heap_reset": [_P],
    "symm_at": [_P, _P, _I],
    "symm_set_spin_budget": [_P, _U64],
    "symm_check_error": [_P, _P, ctypes.POINTER(_I64)],
    "symm_last_error": [],
    "shmem_put": [_P, _P, _SZ, _P, _SZ, _SZ, _I, _P],
    "shmem_get": [_P, _P, _SZ, _P, _SZ, _SZ, _I, _P],
    "shmem_signal_op": [_P, _P, _SZ, _I64, _I, _I, _P],
    "shmem_wait_for_signal": [_P, _P, _SZ, _I64, _I, _I, _U64, _P],
    "shmem_put_with_signal": [_P, _P, _SZ, _P, _SZ, _SZ, _P, _SZ, _I64, _I, _I, _P],
    "all2all_pc_workspace": [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ),
                             ctypes.POINTER(_SZ)],
    "all2all_combine": [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P],
    "all2all_dispatch": [_P, _P, _P, _I, _I, _I, _I, _I, _P],
    "all2all_combine_back": [_P, _P, _P, _I, _I, _I, _I, _I, _P],
    "all2all_combine_host": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P],
    "all2all_combine_pc_noalloc": [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P],
    "shmem_collective_workspace": [_I, ctypes.POINTER(_SZ)],
    "all2all_two_phase_workspace": [_I] * 8 + [ctypes.POINTER(_SZ)] * 2,
    "shmem_fused_ag_matmul_workspace": [_I] * 5 + [ctypes.POINTER(_SZ)],
    "shmem_fused_all_gather_matmul": [_P] * 5 + [_I] * 6 + [_P, _P],
    "all2all_combine_two_phase": [_P, _P, _P] + [_I] * 8 + [_P, _P, _P],
    "shmem_alltoall": [_P, _P, _P, _P, _I, _SZ, _SZ, _SZ, _P, _P, _P],
    "shmem_allgather": [_P, _P, _P, _I, _SZ, _P, _P, _P],
}

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return os.environ.get("SYMM_A2A_LIB") or _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library: $SYMM_A2A_LIB if set (a prebuilt libsymm_a2a.so),
    else the in-tree build (compiled with nvcc first if missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("SYMM_A2A_LIB") or _build.build()
            if not os.path.exists(path):
                raise ImportError(f"libsymm_a2a.so missing at {path}")
            cdll = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(cdll, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name == "symm_last_error" else (
                    _P if name == "symm_at" else _I)
            _lib = cdll
        return _lib


def symm_last_error() -> str:
    return lib().symm_last_error().decode()


def _check(rc: int, func: str) -> int:
    if rc < 0:
        raise SymmError(rc, func, symm_last_error())
    return rc


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# ------------------------------------------------------------------ heap --
def symm_heap_init(base: int, slab_stride: int, npes: int) -> int:
    h = _P()
    _check(lib().symm_heap_init(base, slab_stride, npes, ctypes.byref(h)), "symm_heap_init")
    return h.value


def symm_heap_destroy(heap: int) -> None:
    _check(lib().symm_heap_destroy(heap), "symm_heap_destroy")


def symm_malloc(heap: int, nbytes: int, align: int = 0) -> int:
    p = _P()
    _check(lib().symm_malloc(heap, nbytes, align, ctypes.byref(p)), "symm_malloc")
    return p.value


def symm_heap_reset(heap: int) -> None:
    _check(lib().symm_heap_reset(heap), "symm_heap_reset")


def symm_at(heap: int, ptr: int, pe: int):
    """PE pe's address of ptr's object, or None."""
    return lib().symm_at(heap, ptr, pe)


def symm_set_spin_budget(heap: int, budget_ns: int) -> None:
    _check(lib().symm_set_spin_budget(heap, budget_ns), "symm_set_spin_budget")


def symm_check_error(heap: int, stream=None):
    """(code, info): SYMM_OK, SYMM_ETIMEDOUT (info: the timed-out signal's byte
    offset), or SYMM_ERANGE; raises SymmError only for a failure of the check
    itself."""
    info = _I64(0)
    rc = lib().symm_check_error(heap, _stream(stream), ctypes.byref(info))
    if rc not in (SYMM_OK, SYMM_ETIMEDOUT, SYMM_ERANGE):
        _check(rc, "symm_check_error")
    return rc, info.value


# ------------------------------------------------------------ primitives --
def shmem_put(heap, target, target_off, src, src_off, nbytes, target_pe, stream=None):
    _check(lib().shmem_put(heap, target, target_off, src, src_off, nbytes, target_pe,
                           _stream(stream)), "shmem_put")


def shmem_get(heap, dst, dst_off, src, src_off, nbytes, src_pe, stream=None):
    _check(lib().shmem_get(heap, dst, dst_off, src, src_off, nbytes, src_pe, _stream(stream)),
           "shmem_get")


def shmem_signal_op(heap, signal, signal_off, value, op, target_pe, stream=None):
    _check(lib().shmem_signal_op(heap, signal, signal_off, value, op, target_pe,
                                 _stream(stream)), "shmem_signal_op")


def shmem_wait_for_signal(heap, signal, signal_off, cmp_value, cmp, pe, budget_ns=0,
                          stream=None):
    _check(lib().shmem_wait_for_signal(heap, signal, signal_off, cmp_value, cmp, pe, budget_ns,
                                       _stream(stream)), "shmem_wait_for_signal")


def shmem_put_with_signal(heap, target, target_off, src, src_off, nbytes, signal, signal_off,
                          value, op, target_pe, stream=None):
    _check(lib().shmem_put_with_signal(heap, target, target_off, src, src_off, nbytes, signal,
                                       signal_off, value, op, target_pe, _stream(stream)),
           "shmem_put_with_signal")


# -------------------------------------------------------------- all2all --
def all2all_pc_workspace(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num):
    """(staging_bytes, signal_bytes) per PE."""
    st, sg = _SZ(0), _SZ(0)
    _check(lib().all2all_pc_workspace(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num,
                                      ctypes.byref(st), ctypes.byref(sg)), "all2all_pc_workspace")
    return st.value, sg.value


def all2all_combine(heap, inp, out, W, S, H, D, elem_bytes, variant=SYMM_A2A_DIRECT, tile_s=16,
                    block_d=0, buffer_num=2, staging=None, signals=None, stream=None):
    _check(lib().all2all_combine(heap, inp, out, W, S, H, D, elem_bytes, variant, tile_s, block_d,
                                 buffer_num, staging, signals, _stream(stream)),
           "all2all_combine")


def all2all_dispatch(heap, inp, out, W, S, H, D, elem_bytes, stream=None):
    _check(lib().all2all_dispatch(heap, inp, out, W, S, H, D, elem_bytes, _stream(stream)),
           "all2all_dispatch")


def all2all_combine_back(heap, inp, out, W, Sp, H, D, elem_bytes, stream=None):
    _check(lib().all2all_combine_back(heap, inp, out, W, Sp, H, D, elem_bytes, _stream(stream)),
           "all2all_combine_back")


def all2all_combine_host(heap, host_in, host_out, inp, out, W, S, H, D, elem_bytes,
                         variant=SYMM_A2A_DIRECT, tile_s=16, block_d=0, buffer_num=2,
                         staging=None, signals=None, stream=None):
    _check(lib().all2all_combine_host(heap, host_in, host_out, inp, out, W, S, H, D, elem_bytes,
                                      variant, tile_s, block_d, buffer_num, staging, signals,
                                      _stream(stream)), "all2all_combine_host")


def all2all_combine_pc_noalloc(heap, inp, out, W, S, H, D, elem_bytes, tile_s=16, block_d=0,
                               buffer_num=2, stream=None):
    """The producer/consumer combine with its staging and signals in the
    library's static scratch array, for callers that cannot allocate device
    memory; see include/symm_a2a.h."""
    _check(lib().all2all_combine_pc_noalloc(heap, inp, out, W, S, H, D, elem_bytes, tile_s,
                                            block_d, buffer_num, _stream(stream)),
           "all2all_combine_pc_noalloc")


# ------------------------------------------------------ two-phase combine --
def all2all_two_phase_workspace(W, S, H, D, elem_bytes, tile_s=16, block_d=0, buffer_num=2):
    """(bulk_bytes, signal_bytes) per PE."""
    b, g = _SZ(0), _SZ(0)
    _check(lib().all2all_two_phase_workspace(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num,
                                             ctypes.byref(b), ctypes.byref(g)),
           "all2all_two_phase_workspace")
    return b.value, g.value


def all2all_combine_two_phase(heap, inp, out, W, S, H, D, elem_bytes, tile_s, block_d,
                              buffer_num, bulk, signals, stream=None):
    _check(lib().all2all_combine_two_phase(heap, inp, out, W, S, H, D, elem_bytes, tile_s,
                                           block_d, buffer_num, bulk, signals, _stream(stream)),
           "all2all_combine_two_phase")


# ---------------------------------------------- fused AllGather + MatMul --
SYMM_DTYPE_F16 = 0
SYMM_DTYPE_BF16 = 1


def shmem_fused_ag_matmul_workspace(W, m_local, k, n, block_size=128):
    """signal_bytes per PE."""
    g = _SZ(0)
    _check(lib().shmem_fused_ag_matmul_workspace(W, m_local, k, n, block_size, ctypes.byref(g)),
           "shmem_fused_ag_matmul_workspace")
    return g.value


def shmem_fused_all_gather_matmul(heap, a, b, c, gather_out, W, m_local, k, n, dtype,
                                  block_size, signals, stream=None):
    _check(lib().shmem_fused_all_gather_matmul(heap, a, b, c, gather_out, W, m_local, k, n, dtype,
                                               block_size, signals, _stream(stream)),
           "shmem_fused_all_gather_matmul")


# ------------------------------------------------------------ collectives --
def shmem_collective_workspace(W: int) -> int:
    n = _SZ(0)
    _check(lib().shmem_collective_workspace(W, ctypes.byref(n)), "shmem_collective_workspace")
    return n.value


def shmem_alltoall(heap, inp, out, counts, W, row_bytes, in_rows, out_rows, workspace, signals,
                   stream=None):
    _check(lib().shmem_alltoall(heap, inp, out, counts, W, row_bytes, in_rows, out_rows, workspace,
                                signals, _stream(stream)), "shmem_alltoall")


def shmem_allgather(heap, inp, out, W, nbytes, workspace, signals, stream=None):
    _check(lib().shmem_allgather(heap, inp, out, W, nbytes, workspace, signals, _stream(stream)),
           "shmem_allgather")
