"""ctypes wrapper of the plain-C oracle (``a2a_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
smoke check and the benchmark's CPU-baseline leg may import this module.  It
shares nothing with the CUDA path: it compiles its own C file with gcc and
works on host numpy arrays.

Every function takes and returns contiguous numpy arrays of any dtype; values
are moved as raw ``itemsize``-byte elements, never converted.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "a2a_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liba2a_oracle.so")
# the same source built with -fopenmp: oracle_combine splits its loops over the
# destination rank d and the row s across threads.  Only the timed CPU
# baseline uses it.
OMP_LIB_PATH = os.path.join(BUILD_DIR, "liba2a_oracle_omp.so")


def build(src: str = SOURCE, out: str = LIB_PATH, force: bool = False,
          werror: bool = True, openmp: bool = False) -> str:
    """Compile the oracle with gcc -O2 (and -fopenmp if asked) into a shared
    library; return its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall"] + (["-Werror"] if werror else [])
    cmd += (["-fopenmp"] if openmp else []) + ["-shared", "-fPIC", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_I64 = ctypes.c_int64
_P = ctypes.c_void_p


class Oracle:
    """Loaded oracle library with numpy-level entry points."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_combine", "oracle_dispatch", "oracle_combine_back"):
            fn = getattr(lib, name)
            fn.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I64]
            fn.restype = ctypes.c_int
        lib.oracle_pc_replay.argtypes = [_P, _P] + [_I64] * 8 + [_P, _P]
        lib.oracle_pc_replay.restype = ctypes.c_int
        lib.oracle_put.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64]
        lib.oracle_get.argtypes = [_P, _I64, _I64, _P, _I64, _I64, _I64]
        lib.oracle_signal_op.argtypes = [_P, _I64, _I64, _I64, _I64, _I64, _I64]
        lib.oracle_wait_satisfied.argtypes = [_I64, _I64, _I64]
        lib.oracle_put_with_signal.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64,
                                               _I64, _I64]
        for name in ("oracle_put", "oracle_get", "oracle_signal_op", "oracle_wait_satisfied",
                     "oracle_put_with_signal"):
            getattr(lib, name).restype = ctypes.c_int
        lib.oracle_two_phase_replay.argtypes = [_P, _P] + [_I64] * 8 + [_P, _P]
        lib.oracle_two_phase_replay.restype = ctypes.c_int
        lib.oracle_alltoallv.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64]
        lib.oracle_alltoallv.restype = ctypes.c_int
        lib.oracle_allgather.argtypes = [_P, _P, _I64, _I64]
        lib.oracle_allgather.restype = ctypes.c_int
        lib.oracle_ag_matmul.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64]
        lib.oracle_ag_matmul.restype = ctypes.c_int
        lib.oracle_ag_matmul_at.argtypes = [_P, _P] + [_I64] * 7
        lib.oracle_ag_matmul_at.restype = ctypes.c_double
        self.lib = lib

    # -- permutations ------------------------------------------------------
    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data

    def combine(self, x: np.ndarray, W: int, S: int, H: int, D: int) -> np.ndarray:
        """x: [W, S*W, H, D] -> [W, S, H*W, D]."""
        x = np.ascontiguousarray(x)
        assert x.size == W * S * W * H * D, (x.shape, W, S, H, D)
        out = np.empty((W, S, H * W, D), dtype=x.dtype)
        rc = self.lib.oracle_combine(self._ptr(x), self._ptr(out), W, S, H, D, x.itemsize)
        if rc:
            raise ValueError(f"oracle_combine rc={rc}")
        return out

    def dispatch(self, x: np.ndarray, W: int, S: int, H: int, D: int) -> np.ndarray:
        """x: [W, S, H, D] -> [W, S/W, H*W, D]."""
        x = np.ascontiguousarray(x)
        assert x.size == W * S * H * D
        if S % W:
            raise ValueError("dispatch needs S % W == 0")
        out = np.empty((W, S // W, H * W, D), dtype=x.dtype)
        rc = self.lib.oracle_dispatch(self._ptr(x), self._ptr(out), W, S, H, D, x.itemsize)
        if rc:
            raise ValueError(f"oracle_dispatch rc={rc}")
        return out

    def combine_back(self, y: np.ndarray, W: int, Sp: int, H: int, D: int) -> np.ndarray:
        """y: [W, Sp, H*W, D] -> [W, Sp*W, H, D]."""
        y = np.ascontiguousarray(y)
        assert y.size == W * Sp * H * W * D
        out = np.empty((W, Sp * W, H, D), dtype=y.dtype)
        rc = self.lib.oracle_combine_back(self._ptr(y), self._ptr(out), W, Sp, H, D, y.itemsize)
        if rc:
            raise ValueError(f"oracle_combine_back rc={rc}")
        return out

    def pc_replay(self, x: np.ndarray, W: int, S: int, H: int, D: int, block_s: int,
                  block_d: int, buffer_num: int = 2):
        """Sequential replay of the page's MTE producer/consumer kernel.

        Returns (out, signals_after) where out is [W, S, H*W, D]."""
        x = np.ascontiguousarray(x)
        nbd = -(-D // block_d)
        out = np.empty((W, S, H * W, D), dtype=x.dtype)
        staging = np.zeros(W * buffer_num * block_s * H * W * D * x.itemsize + 1, np.uint8)
        signals = np.zeros(W * buffer_num * nbd * H * W * 8, np.int64)
        rc = self.lib.oracle_pc_replay(self._ptr(x), self._ptr(out), W, S, H, D, x.itemsize,
                                       block_s, block_d, buffer_num, self._ptr(staging),
                                       self._ptr(signals))
        if rc:
            raise ValueError(f"oracle_pc_replay rc={rc}")
        return out, signals

    def two_phase_replay(self, x: np.ndarray, W: int, S: int, H: int, D: int, block_s: int,
                         block_d: int, buffer_num: int = 2):
        """Sequential replay of the page's two-phase (bulk + self-loop) kernel.

        Returns (out, peer_mem, signals_after): out is [W, S, H*W, D]; peer_mem
        [W, W, S, H, D] (rank slots; slot d of PE d holds only the self-loop
        double buffer at its start); signals [W, nbs*W + buffer_num*nbd*H, 8]."""
        x = np.ascontiguousarray(x)
        nbs, nbd = -(-S // block_s), -(-D // block_d)
        out = np.empty((W, S, H * W, D), dtype=x.dtype)
        peer = np.zeros((W, W, S, H, D), dtype=x.dtype)
        signals = np.zeros((W, nbs * W + buffer_num * nbd * H, 8), np.int64)
        rc = self.lib.oracle_two_phase_replay(self._ptr(x), self._ptr(out), W, S, H, D,
                                              x.itemsize, block_s, block_d, buffer_num,
                                              self._ptr(peer), self._ptr(signals))
        if rc:
            raise ValueError(f"oracle_two_phase_replay rc={rc}")
        return out, peer, signals

    def alltoallv(self, x: np.ndarray, counts: np.ndarray, out_rows: int,
                  out: np.ndarray | None = None) -> np.ndarray:
        """x: [W, in_rows, ...] rows; counts: [W, W] int64, counts[r, d] rows
        from r to d -> out [W, out_rows, ...] (rows not received keep `out`'s
        values, zeros when out is None)."""
        x = np.ascontiguousarray(x)
        W, in_rows = x.shape[0], x.shape[1]
        row_bytes = x[0, 0].nbytes if in_rows else int(np.prod(x.shape[2:])) * x.itemsize
        c = np.ascontiguousarray(counts, dtype=np.int64)
        assert c.shape == (W, W)
        if out is None:
            out = np.zeros((W, out_rows) + x.shape[2:], dtype=x.dtype)
        out = np.ascontiguousarray(out)
        rc = self.lib.oracle_alltoallv(self._ptr(x), self._ptr(out), self._ptr(c), W, row_bytes,
                                       in_rows, out_rows)
        if rc:
            raise ValueError(f"oracle_alltoallv rc={rc}")
        return out

    def allgather(self, x: np.ndarray) -> np.ndarray:
        """x: [W, n] -> [W, W*n]."""
        x = np.ascontiguousarray(x)
        W = x.shape[0]
        out = np.empty((W, W * x[0].size), dtype=x.dtype)
        rc = self.lib.oracle_allgather(self._ptr(x), self._ptr(out), W, x[0].nbytes)
        if rc:
            raise ValueError(f"oracle_allgather rc={rc}")
        return out

    def ag_matmul(self, a: np.ndarray, b: np.ndarray):
        """a: [W, m_local, k], b: [W, k, n] (any real dtype; widened to float64
        exactly for fp16) -> (gather [W, W*m_local, k], c [W, W*m_local, n]),
        float64."""
        a = np.ascontiguousarray(a, dtype=np.float64)
        b = np.ascontiguousarray(b, dtype=np.float64)
        W, m_local, k = a.shape
        n = b.shape[2]
        assert b.shape == (W, k, n)
        gather = np.empty((W, W * m_local, k), np.float64)
        c = np.empty((W, W * m_local, n), np.float64)
        rc = self.lib.oracle_ag_matmul(self._ptr(a), self._ptr(b), self._ptr(gather),
                                       self._ptr(c), W, m_local, k, n)
        if rc:
            raise ValueError(f"oracle_ag_matmul rc={rc}")
        return gather, c

    def ag_matmul_at(self, a: np.ndarray, b: np.ndarray, d: int, i: int, j: int) -> float:
        """c_d[i, j] alone (for sampled checks at full size); a, b float64."""
        assert a.dtype == np.float64 and b.dtype == np.float64
        assert a.flags["C_CONTIGUOUS"] and b.flags["C_CONTIGUOUS"]
        W, m_local, k = a.shape
        return self.lib.oracle_ag_matmul_at(self._ptr(a), self._ptr(b), W, m_local, k,
                                            b.shape[2], d, i, j)

    # -- primitives on a host-memory heap -----------------------------------
    def put(self, heap: np.ndarray, slab: int, npes: int, target_off: int, src: np.ndarray,
            pe: int) -> int:
        src = np.ascontiguousarray(src)
        return self.lib.oracle_put(self._ptr(heap), slab, npes, target_off, self._ptr(src),
                                   src.nbytes, pe)

    def get(self, heap: np.ndarray, slab: int, npes: int, dst: np.ndarray, src_off: int,
            pe: int) -> int:
        return self.lib.oracle_get(self._ptr(heap), slab, npes, self._ptr(dst), src_off,
                                   dst.nbytes, pe)

    def signal_op(self, heap: np.ndarray, slab: int, npes: int, sig_off: int, value: int,
                  op: int, pe: int) -> int:
        return self.lib.oracle_signal_op(self._ptr(heap), slab, npes, sig_off, value, op, pe)

    def wait_satisfied(self, current: int, value: int, cmp: int) -> int:
        return self.lib.oracle_wait_satisfied(current, value, cmp)

    def put_with_signal(self, heap: np.ndarray, slab: int, npes: int, target_off: int,
                        src: np.ndarray, sig_off: int, value: int, op: int, pe: int) -> int:
        src = np.ascontiguousarray(src)
        return self.lib.oracle_put_with_signal(self._ptr(heap), slab, npes, target_off,
                                               self._ptr(src), src.nbytes, sig_off, value, op,
                                               pe)


_DEFAULT: Oracle | None = None


def load(path: str | None = None) -> Oracle:
    """Return the oracle loaded from ``path`` (default: build and cache)."""
    global _DEFAULT
    if path is not None:
        return Oracle(path)
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def load_openmp() -> Oracle:
    """The oracle built with -fopenmp (its combine runs over (d, s) in
    parallel, OMP_NUM_THREADS threads), for the timed CPU baseline."""
    return Oracle(build(out=OMP_LIB_PATH, openmp=True))


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))
