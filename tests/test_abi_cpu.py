"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports
every symbol include/symm_a2a.h declares, and its host-side logic (heap
arithmetic, argument validation) behaves; no call here launches a kernel."""
import os
import re
import subprocess

import pytest

from symmetric_memory_moe_gb300 import abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "symm_a2a.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^(?:const\s+)?(?:int|void|char)\s*\**\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("symm_heap_init", "symm_malloc", "symm_at", "shmem_put", "shmem_get",
                 "shmem_signal_op", "shmem_wait_for_signal", "shmem_put_with_signal",
                 "all2all_dispatch", "all2all_combine", "all2all_combine_back"):
        assert must in names


def test_binding_constants_match_the_header():
    """Every integer SYMM_* constant the binding defines has the header's
    value (codes, enums, flags, sizes)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    defines = {}
    for name, value in re.findall(r"^#define\s+(SYMM_\w+)\s+(.+?)\s*$", text, flags=re.M):
        try:
            # drop C integer suffixes (32u, 1ll) before evaluating the expression
            expr = re.sub(r"\b(\d+)(?:[uU]?[lL]{0,2}|[lL]{1,2}[uU])\b", r"\1", value)
            defines[name] = int(eval(expr, {}))
        except Exception:
            continue
    shared = [n for n in dir(abi) if n.startswith("SYMM_") and isinstance(getattr(abi, n), int)]
    assert len(shared) > 10
    for name in shared:
        assert name in defines, f"{name} is not #defined in the header"
        assert getattr(abi, name) == defines[name], name


def test_library_exports_every_declared_symbol():
    path = build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = abi.lib()
    for n in declared_functions():
        assert hasattr(lib, n)
    assert set(declared_functions()) == set(abi._SIGS), "binding and header disagree"


FAKE_BASE = 0x7F0000000000  # never dereferenced: host-only calls below


def test_heap_arithmetic():
    slab = 4 << 20
    h = abi.symm_heap_init(FAKE_BASE, slab, 8)
    try:
        p = abi.symm_malloc(h, 1000)
        assert p == FAKE_BASE + abi.SYMM_HEAP_HEADER_BYTES  # first allocation after the header
        q = abi.symm_malloc(h, 10, 4096)
        assert q % 4096 == 0 and q >= p + 1024  # previous one padded to 256
        r = abi.symm_malloc(h, 1)
        assert r % 256 == 0 and r == q + 256
        # symm_at(p, pe) = base + pe*slab + (p - base) mod slab, from any slab
        for pe in range(8):
            assert abi.symm_at(h, p, pe) == FAKE_BASE + pe * slab + (p - FAKE_BASE)
            assert abi.symm_at(h, abi.symm_at(h, q, 5), pe) == abi.symm_at(h, q, pe)
        assert abi.symm_at(h, p, 8) is None and abi.symm_at(h, p, -1) is None
        assert abi.symm_at(h, FAKE_BASE - 1, 0) is None
        assert abi.symm_at(h, FAKE_BASE + 8 * slab, 0) is None
        with pytest.raises(abi.SymmError) as e:
            abi.symm_malloc(h, slab)
        assert e.value.code == abi.SYMM_ENOMEM
        with pytest.raises(abi.SymmError) as e:
            abi.symm_malloc(h, 16, 3)
        assert e.value.code == abi.SYMM_EINVAL
        abi.symm_heap_reset(h)
        assert abi.symm_malloc(h, 5) == p
    finally:
        abi.symm_heap_destroy(h)


@pytest.mark.parametrize("base,slab,npes", [(FAKE_BASE + 16, 4 << 20, 2), (FAKE_BASE, 4096, 2),
                                            (FAKE_BASE, (4 << 20) + 8, 2), (FAKE_BASE, 4 << 20, 0),
                                            (0, 4 << 20, 2)])
def test_heap_init_rejects(base, slab, npes):
    with pytest.raises(abi.SymmError) as e:
        abi.symm_heap_init(base, slab, npes)
    assert e.value.code == abi.SYMM_EINVAL


def test_pc_workspace_sizes():
    # staging [buffer][tile_s][H*W][D], signals buffer*nbd*H*W slots of 64 B
    st, sg = abi.all2all_pc_workspace(8, 2048, 1, 7168, 2, 16, 1792, 2)
    assert st == 2 * 16 * 8 * 7168 * 2 and sg == 2 * 4 * 1 * 8 * 64
    st, sg = abi.all2all_pc_workspace(32, 256, 2, 999, 2, 32, 0, 2)
    assert st == 2 * 32 * 64 * 999 * 2 and sg == 2 * 1 * 2 * 32 * 64
    with pytest.raises(abi.SymmError):
        abi.all2all_pc_workspace(8, 16, 1, 8, 2, 0, 0, 2)


def test_two_phase_workspace_sizes():
    # bulk: W rank slots of [S][H][D]; signals: region A nbs*W + region B buffer_num*nbd*H slots
    b, g = abi.all2all_two_phase_workspace(8, 2048, 1, 7168, 2, 16, 1024, 2)
    assert b == 8 * 2048 * 7168 * 2 and g == (128 * 8 + 2 * 7 * 1) * 64
    b, g = abi.all2all_two_phase_workspace(3, 7, 2, 5, 4, 2, 0, 3)   # block_d 0 = D
    assert b == 3 * 7 * 2 * 5 * 4 and g == (4 * 3 + 3 * 1 * 2) * 64
    for bad in [(0, 4, 1, 8, 2, 2, 0, 2), (2, 4, 1, 8, 0, 2, 0, 2), (2, 4, 1, 8, 2, 0, 0, 2),
                (2, 4, 1, 8, 2, 2, -1, 2), (2, 4, 1, 8, 2, 2, 0, 0)]:
        with pytest.raises(abi.SymmError) as e:
            abi.all2all_two_phase_workspace(*bad)
        assert e.value.code == abi.SYMM_EINVAL


def test_fused_ag_matmul_workspace_sizes():
    # signals: W*m_local/128 slots of 64 B plus 8-byte counters
    assert abi.shmem_fused_ag_matmul_workspace(8, 512, 1024, 2048) == 8 * 4 * (64 + 8)
    for bad in [(0, 128, 64, 64), (2, 100, 64, 64), (2, 128, 60, 64), (2, 128, 64, 12),
                (2, 128, 0, 64)]:
        with pytest.raises(abi.SymmError) as e:
            abi.shmem_fused_ag_matmul_workspace(*bad)
        assert e.value.code == abi.SYMM_EINVAL
    with pytest.raises(abi.SymmError):
        abi.shmem_fused_ag_matmul_workspace(2, 128, 64, 64, 64)   # block_size != 128


def test_collective_workspace_sizes():
    # send/recv offsets and done counters (W*W each), receive totals (W), a flag
    for W in (1, 2, 8, 100):
        words = 3 * W * W + W + 1
        assert abi.shmem_collective_workspace(W) == (words * 8 + 255) // 256 * 256
    for W in (0, -1, 4097):
        with pytest.raises(abi.SymmError) as e:
            abi.shmem_collective_workspace(W)
        assert e.value.code == abi.SYMM_EINVAL


def test_validation_happens_before_any_launch():
    W, slab = 4, 8 << 20
    h = abi.symm_heap_init(FAKE_BASE, slab, W)
    try:
        n = 16 * W * 2 * 8 * 2
        a = abi.symm_malloc(h, n)
        b = abi.symm_malloc(h, n)

        def code(fn, *args):
            with pytest.raises(abi.SymmError) as e:
                fn(h, *args, stream=0)
            return e.value.code

        E = abi.SYMM_EINVAL
        assert code(abi.all2all_combine, a, b, W + 1, 16, 2, 8, 2) == E       # W != npes
        assert code(abi.all2all_combine, a, a, W, 16, 2, 8, 2) == E           # in == out
        assert code(abi.all2all_combine, a, a + 64, W, 16, 2, 8, 2) == E      # overlap
        assert code(abi.all2all_combine, a, b, W, 16, 2, 8, 0) == E           # elem_bytes 0
        assert code(abi.all2all_combine, a, b, W, 16 << 10, 2, 8, 2) == E     # past the slab
        assert code(abi.all2all_combine, FAKE_BASE, b, W, 16, 2, 8, 2) == E   # header
        assert code(abi.all2all_combine, 0x1000, b, W, 16, 2, 8, 2) == E      # not in the heap
        assert code(abi.all2all_combine, a, b, W, 16, 2, 8, 2, 7) == E        # bad variant
        assert code(abi.all2all_dispatch, a, b, W, 18, 2, 8, 2) == E          # S % W
        assert code(abi.all2all_combine_back, a, b, W, -1, 2, 8, 2) == E
        # PC without (or with too small) workspace
        assert code(abi.all2all_combine, a, b, W, 16, 2, 8, 2, abi.SYMM_A2A_PC, 4, 0, 2,
                    None, None) == E
        assert code(abi.all2all_combine, a, b, W, 16, 2, 8, 2, abi.SYMM_A2A_PC, 4, 0, 2,
                    a, b) == E                                                  # overlaps in/out
        # primitives
        assert code(abi.shmem_put, a, 0, 0x1000, 0, 64, W) == E               # bad PE
        assert code(abi.shmem_put, a, n, 0x1000, 0, slab, 0) == E             # past the slab
        assert code(abi.shmem_get, 0x1000, 0, a, 0, 64, -1) == E
        assert code(abi.shmem_signal_op, a, 0, 1, 2, 0) == E                  # op 2
        assert code(abi.shmem_signal_op, a + 4, 0, 1, 0, 0) == E              # misaligned
        assert code(abi.shmem_wait_for_signal, a, 0, 1, 3, 0) == E            # cmp 3
        assert code(abi.shmem_put_with_signal, a, 0, 0x1000, 0, 64, b, 0, 1, 5, 0) == E
        # collectives: every check is on the host, before the metadata kernel
        sig = abi.symm_malloc(h, 64)
        ws, cnt = 0x10000, 0x20000   # plain device words, never touched here
        assert code(abi.shmem_alltoall, a, b, None, W, 64, 8, 8, ws, sig) == E     # no counts
        assert code(abi.shmem_alltoall, a, b, cnt, W - 1, 64, 8, 8, ws, sig) == E  # W != npes
        assert code(abi.shmem_alltoall, a, b, cnt, W, 64, 8, 8, ws + 4, sig) == E  # workspace
        assert code(abi.shmem_alltoall, a, b, cnt, W, 64, 8, 8, None, sig) == E
        assert code(abi.shmem_alltoall, a, a + 8, cnt, W, 64, 8, 8, ws, sig) == E  # overlap
        assert code(abi.shmem_alltoall, a, b, cnt, W, 64, 8, 8, ws, a) == E        # sig in `in`
        assert code(abi.shmem_alltoall, a, b, cnt, W, 64, 8, 8, ws, sig + 4) == E  # misaligned
        assert code(abi.shmem_alltoall, a, b, cnt, W, 1 << 20, 8, 8, ws, sig) == E  # past slab
        assert code(abi.shmem_alltoall, a, b, cnt, W, 1 << 62, 8, 8, ws, sig) == E  # overflow
        assert code(abi.shmem_allgather, a, b, W, 64, ws, None) == E
        assert code(abi.shmem_allgather, a, b, W, n, ws, sig) == E                # out too small
        assert code(abi.shmem_allgather, a, b, W, 1 << 62, ws, sig) == E
        assert code(abi.shmem_allgather, a, b, W + 2, 64, ws, sig) == E
        # two-phase combine: workspace ranges, overlaps, W, tiles
        blk = abi.symm_malloc(h, n)
        tsig = abi.symm_malloc(h, 4096)
        tp = abi.all2all_combine_two_phase
        assert code(tp, a, b, W + 1, 16, 2, 8, 2, 4, 0, 2, blk, tsig) == E   # W != npes
        assert code(tp, a, b, W, 16, 2, 8, 2, 0, 0, 2, blk, tsig) == E       # tile_s 0
        assert code(tp, a, b, W, 16, 2, 8, 2, 4, 0, 0, blk, tsig) == E       # no buffers
        assert code(tp, a, b, W, 16, 2, 8, 2, 4, 0, 2, a, tsig) == E         # bulk is in
        assert code(tp, a, b, W, 16, 2, 8, 2, 4, 0, 2, blk, blk) == E        # signals in bulk
        assert code(tp, a, b, W, 16, 2, 8, 2, 4, 0, 2, blk, tsig + 4) == E   # misaligned
        assert code(tp, a, b, W, 16, 2, 8, 2, 4, 0, 2, 0x1000, tsig) == E    # not in the heap
        assert code(tp, a, a, W, 16, 2, 8, 2, 4, 0, 2, blk, tsig) == E       # in == out
        # fused AllGather + MatMul: W = 4, m_local 128, k 8, n 8 (2 KB a, 8 KB gather)
        fa, fb, fc, fg, fs = [abi.symm_malloc(h, 16384) for _ in range(5)]
        fm = abi.shmem_fused_all_gather_matmul
        F16 = abi.SYMM_DTYPE_F16
        assert code(fm, fa, fb, fc, fg, W, 128, 8, 8, 7, 128, fs) == E          # dtype
        assert code(fm, fa, fb, fc, fg, W + 1, 128, 8, 8, F16, 128, fs) == E    # W
        assert code(fm, fa, fb, fc, fg, W, 100, 8, 8, F16, 128, fs) == E        # m_local
        assert code(fm, fa, fb, fc, fg, W, 128, 8, 8, F16, 64, fs) == E         # block
        assert code(fm, fa, fb, fc, fa, W, 128, 8, 8, F16, 128, fs) == E        # overlap
        assert code(fm, fa + 8, fb, fc, fg, W, 128, 8, 8, F16, 128, fs) == E    # alignment
        assert code(fm, fa, fb, fc, 0x1000, W, 128, 8, 8, F16, 128, fs) == E   # not heap
        assert code(fm, fa, fb, fc, fg, W, 128 * 16, 8, 8, F16, 128, fs) == E   # too big
    finally:
        abi.symm_heap_destroy(h)


def test_header_is_plain_c(tmp_path):
    """The boundary header compiles as strict C99 (no C++ in the interface)."""
    src = tmp_path / "use.c"
    src.write_text('#include "symm_a2a.h"\n'
                   "int main(void) { size_t b = 0; return shmem_collective_workspace(8, &b); }\n")
    res = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                          "-fsyntax-only", "-I", os.path.join(ROOT, "include"), str(src)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_readme_example_uses_the_binding():
    """The README's usage example parses, and every `abi.` name and heap
    method it calls exists in the binding."""
    import ast

    from symmetric_memory_moe_gb300 import torch_heap

    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README has no python example"
    for code in blocks:
        tree = ast.parse(code)
        for node in ast.walk(tree):
            if isinstance(node, ast.Attribute) and isinstance(node.value, ast.Name):
                if node.value.id == "abi":
                    assert hasattr(abi, node.attr), f"abi.{node.attr}"
                if node.value.id == "heap":
                    assert hasattr(torch_heap.TorchSymmHeap, node.attr) or node.attr == "handle", \
                        f"heap.{node.attr}"
