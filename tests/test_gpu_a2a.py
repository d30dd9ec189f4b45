"""GPU parity: the CUDA all-to-all through the C ABI against the CPU oracle.

Results must be bit-exact (the path moves bits, it does no arithmetic).
Outputs are poisoned (0xA5) before every call so an unwritten byte shows.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from symmetric_memory_moe_gb300 import abi, inputs
from symmetric_memory_moe_gb300.torch_heap import CombineBuffers, TorchSymmHeap

pytestmark = pytest.mark.gpu

POISON = 0xA5
# producer/consumer D-block per workload: several blocks where D allows
BLOCK_D = {"tiny": 0, "small": 64, "dsv3": 1792, "tail": 0}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()


@functools.lru_cache(maxsize=2)
def _workload_data(name):
    wl = inputs.WORKLOADS[name]
    x = inputs.make_input(wl)
    return wl, x


def _np_view(t: torch.Tensor) -> np.ndarray:
    """Raw-bit numpy view of a CPU tensor (bf16 viewed as int16)."""
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy()


# variant name -> all2all_combine variant bits: "direct" copies 16-byte
# vectors, "direct_bulk" bulk (TMA) copies where rows are 16-byte aligned;
# "pc" prefetches the producer's input by bulk copies where rows are 16-byte
# aligned, "pc_vec" uses 16-byte vectors only
KINDS = {"direct": abi.SYMM_A2A_DIRECT, "pc": abi.SYMM_A2A_PC,
         "direct_bulk": abi.SYMM_A2A_DIRECT | abi.SYMM_A2A_FLAG_BULK,
         "pc_vec": abi.SYMM_A2A_PC | abi.SYMM_A2A_FLAG_VECTOR}


def run_combine(x: torch.Tensor, W, S, H, D, variant, tile_s=16, block_d=0, buffer_num=2,
                in_shift=0, out_shift=0, repeat=1):
    """Runs all2all_combine on x ([W][S*W][H][D], CPU); returns [W, bytes] uint8."""
    es = x.element_size()
    pc = variant.startswith("pc")
    extra = 2048
    bufs = CombineBuffers(W, S * W, H, D, es, pc=pc, S=S, tile_s=tile_s, block_d=block_d,
                          buffer_num=buffer_num, extra=extra)
    heap, n = bufs.heap, bufs.nbytes
    inp, out = bufs.inp + in_shift, bufs.out + out_shift
    heap.upload(inp, x.reshape(W, -1))
    heap.views(out, n).fill_(POISON)
    kind = KINDS[variant]
    for _ in range(repeat):
        abi.all2all_combine(heap.handle, inp, out, W, S, H, D, es, kind, tile_s, block_d,
                            buffer_num, bufs.staging, bufs.signals)
    torch.cuda.synchronize()
    rc, info = abi.symm_check_error(heap.handle)
    assert rc == abi.SYMM_OK, (rc, info)
    res = heap.download(out, n)
    if pc:  # every slot (first int64 of each 64-byte line) returned to 0 by its consumer
        sig = heap.download(bufs.signals, bufs.signal_bytes).view(torch.int64)[:, ::8]
        assert not sig.any()
    heap.close()
    return res


def expect_combine(x, W, S, H, D):
    y = oracle.load().combine(_np_view(x), W, S, H, D)
    return y.view(np.uint8).reshape(W, -1)


def assert_bits_equal(got: torch.Tensor, want: np.ndarray):
    g = got.numpy()
    if not np.array_equal(g, want):
        bad = np.argwhere(g != want)
        raise AssertionError(f"{len(bad)} bytes differ; first at (pe, byte) {bad[:5].tolist()}, "
                             f"got {g[tuple(bad[0])]} want {want[tuple(bad[0])]}")


# ------------------------------------------------ the five workloads ------
@pytest.mark.parametrize("name,variant", [
    ("tiny", "direct"), ("tiny", "pc"), ("small", "direct"), ("small", "pc"),
    ("small", "direct_bulk"), ("small", "pc_vec"), ("tail", "direct"), ("tail", "pc"),
    ("dsv3", "direct"), ("dsv3", "pc"), ("dsv3", "direct_bulk"), ("dsv3", "pc_vec")])
def test_workload_combine_bit_exact(name, variant):
    wl, x = _workload_data(name)
    got = run_combine(x, wl.W, wl.S, wl.H, wl.D, variant, tile_s=wl.tile_s,
                      block_d=BLOCK_D[name])
    assert_bits_equal(got, expect_combine(x, wl.W, wl.S, wl.H, wl.D))


def test_tiny_golden_values():
    """Hand-worked entries of the W=2 iota case, read off the GPU output."""
    wl, x = _workload_data("tiny")
    for variant in ("direct", "pc"):
        got = run_combine(x, wl.W, wl.S, wl.H, wl.D, variant, tile_s=2).view(torch.int32)
        got = got.reshape(wl.W, wl.S, wl.H * wl.W, wl.D)
        assert got[0, 0, 2, 0] == 1000000 and got[0, 3, 1, 7] == 63
        assert got[1, 0, 0, 0] == 64 and got[1, 3, 3, 7] == 1000127


def test_roundtrip_dispatch_then_inverse():
    """W=16 fp16 dispatch (1024,4,128) -> (64,64,128) matches the oracle, and
    the inverse brings back the input bit for bit."""
    wl, x = _workload_data("roundtrip")
    W, S, H, D, es = wl.W, wl.S, wl.H, wl.D, wl.es
    bufs = CombineBuffers(W, S, H, D, es, extra=S * H * D * es + 256)
    heap, n = bufs.heap, bufs.nbytes
    back = heap.malloc(n)
    heap.upload(bufs.inp, x.reshape(W, -1))
    heap.views(bufs.out, n).fill_(POISON)
    heap.views(back, n).fill_(POISON)
    abi.all2all_dispatch(heap.handle, bufs.inp, bufs.out, W, S, H, D, es)
    abi.all2all_combine_back(heap.handle, bufs.out, back, W, S // W, H, D, es)
    torch.cuda.synchronize()
    want = oracle.load().dispatch(_np_view(x), W, S, H, D).view(np.uint8).reshape(W, -1)
    assert_bits_equal(heap.download(bufs.out, n), want)
    assert_bits_equal(heap.download(back, n), _np_view(x).view(np.uint8).reshape(W, -1))
    heap.close()


# ------------------------------------------------------------ edge cases --
def _rand_bytes(W, rows, H, D, es, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (W, rows, H, D * es), generator=g, dtype=torch.uint8)


@pytest.mark.parametrize("op,W,S,H,D", [
    ("combine", 3, 5, 1, 8),         # 16-byte runs: one batch holds a whole period (3 runs)
    ("combine", 5, 3, 1, 2048),      # 4 KB runs: batches of 2, the last of a period holds 1
    ("combine", 7, 4, 1, 520),       # 1040-byte runs: batches of 7
    ("combine", 1, 6, 2, 64),        # one PE: a period of 1 run, the per-run kernel
    ("combine", 4, 3, 1, 2056),      # 4112-byte runs: past the batches, the per-run kernel
    ("dispatch", 6, 12, 3, 16),      # 96-byte runs, S' = 2
    ("combine_back", 4, 9, 1, 1024), # inverse, period S' = 9 in batches of 4, 4, 1
    ("combine_back", 3, 1, 2, 32),   # inverse with S' = 1: the per-run kernel
])
def test_short_run_batches(op, W, S, H, D):
    """Aligned runs of at most 4 KB are copied in batches of consecutive runs
    per warp (a period: the W source PEs of one output row for the combine
    and dispatch, the S' rows of one (PE, PE) pair for the inverse); batches
    end with the period.  S is the combine's S, dispatch's S or the inverse's
    S'.  Bit-exact against the oracle, on bf16-sized elements."""
    es = 2
    rows_in = {"combine": S * W, "dispatch": S, "combine_back": S * W}[op]
    xe = _rand_bytes(W, rows_in, H, D, es, seed=W * 100 + S + D)
    n = rows_in * H * D * es
    bufs = CombineBuffers(W, rows_in, H, D, es, extra=256)
    heap = bufs.heap
    heap.upload(bufs.inp, xe.reshape(W, -1))
    heap.views(bufs.out, n).fill_(POISON)
    xv = np.ascontiguousarray(xe.numpy()).view(np.dtype((np.void, es)))
    o = oracle.load()
    if op == "combine":
        abi.all2all_combine(heap.handle, bufs.inp, bufs.out, W, S, H, D, es, abi.SYMM_A2A_DIRECT,
                            16, 0, 2, 0, 0)
        want = o.combine(xv.reshape(W, S * W, H, D), W, S, H, D)
    elif op == "dispatch":
        abi.all2all_dispatch(heap.handle, bufs.inp, bufs.out, W, S, H, D, es)
        want = o.dispatch(xv.reshape(W, S, H, D), W, S, H, D)
    else:
        abi.all2all_combine_back(heap.handle, bufs.inp, bufs.out, W, S, H, D, es)
        want = o.combine_back(xv.reshape(W, S, H * W, D), W, S, H, D)
    torch.cuda.synchronize()
    assert_bits_equal(heap.download(bufs.out, n), want.view(np.uint8).reshape(W, -1))
    heap.close()


@pytest.mark.parametrize("op,W,S,H,D,es,in_shift,out_shift", [
    ("combine", 3, 5, 1, 3, 2, 0, 0),         # 6-byte runs: one batch holds a period
    ("combine", 5, 7, 1, 17, 2, 0, 0),        # 34-byte runs, period of 35 in one batch
    ("combine", 7, 40, 1, 130, 2, 0, 0),      # 260-byte runs: batches of 23, the last of 4
    ("combine", 4, 64, 1, 250, 2, 0, 0),      # 500-byte runs: batches of 16, none ragged
    ("combine", 3, 20, 1, 511, 2, 0, 0),      # 1022-byte runs: batches of 7, the last of 4
    ("combine", 3, 9, 2, 256, 2, 3, 0),       # 1024-byte runs made unaligned: batches of 7
    ("combine", 3, 9, 2, 384, 2, 3, 0),       # 1536-byte runs made unaligned: one run per slot
    ("combine", 7, 40, 1, 130, 2, 5, 11),     # shifted bases on both sides
    ("combine", 1, 50, 1, 13, 1, 1, 2),       # one PE: a period of S runs
    ("combine", 16, 512, 1, 250, 2, 0, 0),    # 8192 batches: warps stride over several
    ("dispatch", 6, 12, 3, 15, 2, 0, 0),      # 90-byte runs, S' = 2
    ("dispatch", 4, 8, 1, 301, 2, 7, 3),      # 602-byte runs, shifted
    ("combine_back", 4, 9, 1, 333, 2, 0, 0),  # inverse: 666-byte runs, batches of 12
    ("combine_back", 5, 3, 1, 7, 1, 0, 9),    # inverse: 7-byte runs
    ("combine", 1, 1, 1, 5, 2, 3, 0),         # a single 10-byte run
    ("combine_back", 1, 4, 1, 300, 2, 0, 5),  # inverse on one PE: 600-byte runs
    ("dispatch", 3, 3, 1, 700, 2, 1, 0),      # 1400-byte runs, S' = 1: whole-warp batches of 3
    ("combine_back", 4, 9, 1, 100, 2, 6, 2),  # inverse, 200-byte runs: groups of 8 lanes, shifted
])
def test_unaligned_run_rings(op, W, S, H, D, es, in_shift, out_shift):
    """Runs that are not 16-byte aligned stream through per-warp shared-memory
    rings: one run per slot from 1536 bytes, batches of runs consecutive in
    the input below (2, 6 or 8 KB by run length; a batch ends with its input
    PE's runs), written by groups of 8, 16 or 32 lanes.  S is the combine's S, dispatch's S or the inverse's
    S'.  Bit-exact against the oracle, bytes around the output untouched."""
    rows_in = {"combine": S * W, "dispatch": S, "combine_back": S * W}[op]
    xe = _rand_bytes(W, rows_in, H, D, es, seed=W * 7 + S * 3 + D + in_shift)
    n = rows_in * H * D * es
    heap = TorchSymmHeap(W, abi.SYMM_HEAP_HEADER_BYTES + 2 * n + 4096)
    pin, pout = heap.malloc(n + 64), heap.malloc(n + 64)  # room for the shifts
    inp, out = pin + in_shift, pout + out_shift
    heap.upload(inp, xe.reshape(W, -1))
    heap.views(pout, n + 64).fill_(POISON)
    xv = np.ascontiguousarray(xe.numpy()).view(np.dtype((np.void, es)))
    o = oracle.load()
    if op == "combine":
        abi.all2all_combine(heap.handle, inp, out, W, S, H, D, es, abi.SYMM_A2A_DIRECT,
                            16, 0, 2, 0, 0)
        want = o.combine(xv.reshape(W, S * W, H, D), W, S, H, D)
    elif op == "dispatch":
        abi.all2all_dispatch(heap.handle, inp, out, W, S, H, D, es)
        want = o.dispatch(xv.reshape(W, S, H, D), W, S, H, D)
    else:
        abi.all2all_combine_back(heap.handle, inp, out, W, S, H, D, es)
        want = o.combine_back(xv.reshape(W, S, H * W, D), W, S, H, D)
    torch.cuda.synchronize()
    assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    got = heap.download(pout, n + 64)
    assert_bits_equal(got[:, out_shift:out_shift + n].contiguous(),
                      want.view(np.uint8).reshape(W, -1))
    assert (got[:, :out_shift] == POISON).all() and (got[:, out_shift + n:] == POISON).all()
    heap.close()


@pytest.mark.parametrize("W,S,H,D,es,tile_s,block_d,buf", [
    (1, 7, 3, 5, 2, 4, 0, 2),        # one PE: identity
    (3, 37, 2, 999, 2, 16, 256, 2),   # odd W, ragged S and D blocks
    (5, 9, 1, 33, 1, 4, 8, 3),        # bytes, 3 buffers
    (4, 16, 2, 7, 3, 1, 0, 1),        # 3-byte elements, one row per tile, one buffer
    (2, 5, 4, 16, 8, 2, 5, 2),        # 8-byte elements
    (8, 12, 1, 1, 16, 5, 0, 2),       # 16-byte elements, one element per run
    (6, 3, 3, 100, 4, 64, 17, 2),     # tile taller than S
    (4, 21, 2, 24, 2, 8, 16, 2),      # 16-byte rows: bulk path, ragged S and D blocks
    (3, 10, 1, 40000, 2, 2, 0, 2),    # 80 kB runs: several bulk chunks per run
    (2, 33, 4, 8, 4, 4, 4, 3),        # 16-byte rows of 4-byte elements, 3 buffers
    (2, 9, 1, 16, 2, 2, 8, 1),        # aligned, one buffer: each slot reused by the next task
])
@pytest.mark.parametrize("variant", ["direct", "pc", "direct_bulk", "pc_vec"])
def test_shapes(W, S, H, D, es, tile_s, block_d, buf, variant):
    xe = _rand_bytes(W, S * W, H, D, es, seed=W * 1000 + S).reshape(W, S * W, H, D, es)
    got = _run_es(xe, W, S, H, D, es, variant, tile_s, block_d, buf)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


def _expect_es(xe, W, S, H, D, es):
    """Oracle combine of raw es-byte elements (numpy void dtype)."""
    xv = np.ascontiguousarray(xe.numpy()).view(np.dtype((np.void, es))).reshape(W, S * W, H, D)
    return oracle.load().combine(xv, W, S, H, D).view(np.uint8).reshape(W, -1)


def _run_es(xe, W, S, H, D, es, variant, tile_s, block_d, buf, in_shift=0, out_shift=0):
    pc = variant.startswith("pc")
    bufs = CombineBuffers(W, S * W, H, D, es, pc=pc, S=S, tile_s=tile_s, block_d=block_d,
                          buffer_num=buf, extra=2048)
    heap, n = bufs.heap, bufs.nbytes
    inp, out = bufs.inp + in_shift, bufs.out + out_shift
    heap.upload(inp, xe.reshape(W, -1))
    heap.views(out, n).fill_(POISON)
    abi.all2all_combine(heap.handle, inp, out, W, S, H, D, es, KINDS[variant], tile_s, block_d,
                        buf, bufs.staging, bufs.signals)
    torch.cuda.synchronize()
    assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    res = heap.download(out, n)
    heap.close()
    return res


@pytest.mark.parametrize("in_shift,out_shift", [(2, 0), (0, 6), (3, 9), (14, 1), (16, 32)])
@pytest.mark.parametrize("variant", ["direct", "pc"])
def test_unaligned_base_pointers(in_shift, out_shift, variant):
    """Input and output at arbitrary byte offsets: every src/dst phase mod 16."""
    W, S, H, D, es = 4, 10, 2, 45, 2
    xe = _rand_bytes(W, S * W, H, D, es, seed=in_shift * 31 + out_shift).reshape(W, S * W, H, D,
                                                                                  es)
    got = _run_es(xe, W, S, H, D, es, variant, 4, 16, 2, in_shift, out_shift)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("in_shift,out_shift,tile_s", [
    (0, 0, 8),      # 16-byte-aligned 16 KB tiles: bulk prefetch, whole-tile group copies
    (0, 8, 8),      # output off 16 bytes: group copies with shifted vectors, byte edges
    (4, 0, 8),      # input off 16 bytes: the same, the source phase off instead
    (5, 11, 8),     # both off, by different amounts
    (0, 0, 40),     # a tile too big for the prefetch ring: whole-tile group copies
    (16, 48, 40),
    (3, 0, 40),     # unaligned, tiles taller than the last S block
])
def test_pc_copy_instances(in_shift, out_shift, tile_s):
    """The producer/consumer kernel's copy instances, chosen by alignment and
    tile size, on 2064-byte rows (wide enough for the bulk prefetch) and a
    ragged last S block (40-row tiles are 81 KB, more than the prefetch ring
    takes).  Each object leaves 128 bytes of its 256-byte allocation granule
    free for the shifts."""
    W, S, H, D, es = 4, 45, 2, 1032, 2
    xe = _rand_bytes(W, S * W, H, D, es, seed=tile_s + in_shift).reshape(W, S * W, H, D, es)
    got = _run_es(xe, W, S, H, D, es, "pc", tile_s, 0, 2, in_shift, out_shift)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("W,S,H,D,es,shift", [
    (4, 19, 2, 999, 2, 0),    # 1998-byte rows: source phase changes from row to row
    (4, 19, 2, 999, 2, 6),
    (8, 9, 1, 15, 2, 0),      # rows shorter than 16 bytes: head and tail bytes only
    (16, 9, 1, 17, 1, 9),     # 17-byte rows: one vector at most
    (2, 33, 8, 7, 3, 1),      # 3-byte elements, 21-byte rows
])
def test_pc_any_alignment_tiles(W, S, H, D, es, shift):
    """Tiles whose staging and output rows share one 16-byte phase (H*W*D*es a
    multiple of 16) but whose rows are not 16-byte aligned: every group
    copies whole tiles with shifted vectors, on several row lengths and
    source phases, with tiles of 4 and 32 rows."""
    xe = _rand_bytes(W, S * W, H, D, es, seed=D * 7 + shift).reshape(W, S * W, H, D, es)
    for tile_s in (4, 32):
        got = _run_es(xe, W, S, H, D, es, "pc", tile_s, 0, 2, shift, 0)
        assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("W,S,H,D,es,tile_s,block_d,buf,shift", [
    (4, 19, 2, 999, 2, 32, 600, 2, 6),    # D blocks of 1200 and 798 bytes; chunks of 16 + 3 rows
    (4, 37, 4, 1501, 1, 40, 0, 1, 3),     # odd 1501-byte rows, one buffer; chunks of 21 + 16 rows
    (2, 50, 8, 1099, 2, 16, 0, 3, 13),    # 2198-byte rows, 3 buffers; chunks of 14 + 2 rows
    (16, 5, 1, 601, 2, 3, 0, 2, 1),       # 1202-byte rows
    (32, 9, 2, 999, 2, 2, 0, 1, 5),       # 2048 tasks per S block: several per CTA, one buffer
    (32, 9, 2, 999, 2, 2, 0, 3, 5),       # the same with 3 buffers (slots fresh for 3 S blocks)
    (32, 9, 3, 1101, 2, 2, 550, 2, 3),    # 9216 tasks: more per CTA than the task table holds
])
def test_pc_any_prefetch(W, S, H, D, es, tile_s, block_d, buf, shift):
    """Rows of 1 KB and more that are not 16-byte aligned, with staging and
    output rows in one 16-byte phase: the producer's input arrives by bulk
    copies of each row's aligned covering range, in chunks of rows (a tile
    taller than a ring entry takes several), and is shift-merged from shared
    memory.  Ragged S and D blocks, one to three buffers, input shifted so
    that the rows' source phases differ from the destination's (each input
    object ends at least 13 bytes before its 256-byte granule does).  With
    W = 32 each CTA owns several tasks and walks them one after another:
    the producer is paced on its own consumer across task boundaries, and a
    slot's staging lines are dropped from L2 after its last use."""
    xe = _rand_bytes(W, S * W, H, D, es, seed=D * 3 + shift).reshape(W, S * W, H, D, es)
    got = _run_es(xe, W, S, H, D, es, "pc", tile_s, block_d, buf, shift, 0)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("W,S,H,D,es,tile_s,block_d,buf,shift", [
    (4, 19, 2, 999, 2, 32, 600, 2, 6),   # unaligned rows, ragged S and D blocks
    (8, 40, 1, 1024, 2, 12, 0, 3, 0),    # 2 KB rows, 3 buffers
    (3, 10, 2, 7, 3, 4, 0, 1, 0),        # 3-byte elements, one buffer
])
def test_pc_phased_mode(W, S, H, D, es, tile_s, block_d, buf, shift):
    """SYMM_A2A_FLAG_PHASED, the debugging mode in which each S block's
    producers and then its consumers run as separate launches (a barrier
    between the roles): the oracle's result, every slot back at 0, also when
    the slots held stale values before the call (the mode zeroes them)."""
    xe = _rand_bytes(W, S * W, H, D, es, seed=D + tile_s + buf).reshape(W, S * W, H, D, es)
    bufs = CombineBuffers(W, S * W, H, D, es, pc=True, S=S, tile_s=tile_s, block_d=block_d,
                          buffer_num=buf, extra=2048)
    heap, n = bufs.heap, bufs.nbytes
    inp = bufs.inp + shift
    heap.upload(inp, xe.reshape(W, -1))
    heap.views(bufs.out, n).fill_(POISON)
    heap.views(bufs.signals, bufs.signal_bytes).fill_(0x7F)
    abi.all2all_combine(heap.handle, inp, bufs.out, W, S, H, D, es,
                        abi.SYMM_A2A_PC | abi.SYMM_A2A_FLAG_PHASED, tile_s, block_d, buf,
                        bufs.staging, bufs.signals)
    torch.cuda.synchronize()
    assert abi.symm_check_error(heap.handle)[0] == abi.SYMM_OK
    assert_bits_equal(heap.download(bufs.out, n), _expect_es(xe, W, S, H, D, es))
    sig = heap.download(bufs.signals, bufs.signal_bytes).view(torch.int64)[:, ::8]
    assert not sig.any()
    heap.close()


@pytest.mark.parametrize("W,S,H,buf,tile_s", [
    (2, 24, 1, 1, 4),    # one slot per CTA, one buffer: reused by the very next tile
    (2, 24, 1, 2, 4),    # two slots in rotation
    (2, 24, 1, 3, 4),    # three
    (2, 22, 1, 2, 4),    # ragged last S block
    (16, 8, 2, 1, 4),    # 512 tasks per S block: CTAs own two or more tasks each
    (16, 9, 2, 2, 2),
])
def test_pc_slot_rotations(W, S, H, buf, tile_s):
    """2 KB rows (the prefetching instance) with one to three buffers and one
    or several tasks per CTA: each slot is reused every tasks x buffers tiles
    of its CTA, from one to several times per S block."""
    D, es = 1024, 2
    xe = _rand_bytes(W, S * W, H, D, es, seed=W * 100 + S + buf).reshape(W, S * W, H, D, es)
    got = _run_es(xe, W, S, H, D, es, "pc", tile_s, 0, buf)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("D,tile_s,block_d", [
    (16000, 4, 0),      # 32000-byte rows, 125 KB tiles: no prefetch
    (7168, 64, 1024),   # tiles of 64 2 KB rows: no prefetch
    (7168, 2, 0),       # 14 KB rows, 28 KB tiles: prefetched
    (3000, 8, 1032),    # ragged D blocks (2064 + 2064 + 1872 bytes): prefetched
])
def test_pc_wide_rows_and_tall_tiles(D, tile_s, block_d):
    """Aligned rows of 2 KB to 32 KB: tiles that the input prefetch ring takes
    (up to 32 KB) and tiles taller than it (copied without the prefetch),
    with ragged D blocks and S blocks."""
    W, S, H, es = 4, 37, 1, 2
    xe = _rand_bytes(W, S * W, H, D, es, seed=D + tile_s).reshape(W, S * W, H, D, es)
    got = _run_es(xe, W, S, H, D, es, "pc", tile_s, block_d, 2)
    assert_bits_equal(got, _expect_es(xe, W, S, H, D, es))


@pytest.mark.parametrize("S,H,D", [(0, 2, 8), (4, 0, 8), (4, 2, 0)])
def test_empty_extents_are_noops(S, H, D):
    W = 2
    bufs = CombineBuffers(W, 8, 2, 8, 2, pc=True, S=4, tile_s=2)
    heap = bufs.heap
    heap.views(bufs.out, 64).fill_(POISON)
    for kind in (abi.SYMM_A2A_DIRECT, abi.SYMM_A2A_PC):
        abi.all2all_combine(heap.handle, bufs.inp, bufs.out, W, S, H, D, 2, kind, 2, 0, 2,
                            bufs.staging, bufs.signals)
    abi.all2all_dispatch(heap.handle, bufs.inp, bufs.out, W, S, H, D, 2)
    torch.cuda.synchronize()
    assert (heap.download(bufs.out, 64) == POISON).all()
    heap.close()


@pytest.mark.parametrize("variant", ["pc", "pc_vec"])
def test_repeated_pc_calls_reuse_signals(variant):
    """Back-to-back PC launches on one workspace (reset in-stream each time)."""
    W, S, H, D = 4, 24, 2, 40
    x = _rand_bytes(W, S * W, H, D, 2, seed=5).view(torch.int16).reshape(W, S * W, H, D)
    got = run_combine(x, W, S, H, D, variant, tile_s=4, block_d=16, repeat=3)
    assert_bits_equal(got, expect_combine(x, W, S, H, D))


@pytest.mark.parametrize("S", [10, 16, 37])
def test_host_buffer_entry_point(S):
    """all2all_combine_host: host in -> device -> combine -> host out.  S 10
    takes the single-chunk path; S 16 and 37 the 8-chunk pipeline (37: a
    ragged last chunk).  Two calls in a row with different inputs on the
    same objects, pinned and (once) pageable host buffers."""
    W, H, D = 4, 2, 24
    for variant, kind in (("direct", abi.SYMM_A2A_DIRECT), ("pc", abi.SYMM_A2A_PC)):
        bufs = CombineBuffers(W, S * W, H, D, 2, pc=variant == "pc", S=S, tile_s=4)
        for call in range(2):
            x = _rand_bytes(W, S * W, H, D, 2, seed=9 + call + S).view(torch.int16)
            x = x.reshape(W, S * W, H, D).contiguous()
            pinned = not (variant == "direct" and call == 1)
            host_in = x.pin_memory() if pinned else x.clone()
            host_out = torch.full((W, S, H * W, D), -1, dtype=torch.int16)
            if pinned:
                host_out = host_out.pin_memory()
            abi.all2all_combine_host(bufs.heap.handle, host_in.data_ptr(), host_out.data_ptr(),
                                     bufs.inp, bufs.out, W, S, H, D, 2, kind, 4, 0, 2,
                                     bufs.staging, bufs.signals)
            torch.cuda.synchronize()
            want = expect_combine(x, W, S, H, D)
            assert np.array_equal(host_out.view(torch.uint8).reshape(W, -1).numpy(), want), \
                (variant, call)
        bufs.heap.close()
