"""Pins of the CPU oracle against facts the pages and mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle given to it is
wrong.  They are collected by ``test_oracle_pins.py`` and re-run against
deliberately broken copies of the oracle by ``test_oracle_mutants.py`` (each
broken copy must fail at least one pin), so a plausible slip anywhere in the
oracle -- a dropped term, a swapped index, a transposed operand -- is caught.

The pins never retype the oracle's formula: they use hand-worked values
(``golden/combine_tiny_w2.txt``), closed forms (W=1 is the identity), invariants
(a permutation: every iota value appears exactly once), a library routine
(numpy's transpose of the 5-d view), round trips (dispatch followed by its
inverse is the identity) and an independent replay of the page's own tile
loop.
"""
from __future__ import annotations

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "combine_tiny_w2.txt")


def _iota(W, rows, H, D, base=1_000_000, dtype=np.int32):
    per = rows * H * D
    x = np.arange(per, dtype=np.int64)[None, :] + base * np.arange(W, dtype=np.int64)[:, None]
    return x.astype(dtype).reshape(W, rows, H, D)


def _rand(shape, seed, dtype):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 2**15, size=shape, dtype=np.int64).astype(dtype)


# -- hand-worked values ----------------------------------------------------
def pin_golden_tiny(o):
    """Hand-worked W=2 entries of the combine and the dispatch."""
    W, S, H, D = 2, 4, 2, 8
    comb = o.combine(_iota(W, S * W, H, D), W, S, H, D)
    disp = o.dispatch(_iota(W, S, H, D), W, S, H, D)
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            op, d, row, col, x, value = line[0], *map(int, line[1:])
            got = (comb if op == "combine" else disp)[d, row, col, x]
            assert got == value, (op, d, row, col, x, got, value)
            n += 1
    assert n >= 12


# -- closed forms ----------------------------------------------------------
def pin_w1_identity(o):
    """One rank: combine, dispatch and its inverse leave the tensor unchanged."""
    for (S, H, D, dt) in [(5, 3, 7, np.int16), (4, 1, 33, np.int32), (3, 2, 5, np.uint8)]:
        x = _rand((1, S, H, D), 1, dt)
        np.testing.assert_array_equal(o.combine(x, 1, S, H, D).reshape(x.shape), x)
        np.testing.assert_array_equal(o.dispatch(x, 1, S, H, D).reshape(x.shape), x)
        np.testing.assert_array_equal(o.combine_back(x, 1, S, H, D).reshape(x.shape), x)


def pin_self_block(o):
    """Block d of rank d stays on rank d, at column group d*H (its own experts):
    with H=1, D=1 the combine of rank d's block d is the diagonal of the grid."""
    W, S = 3, 2
    x = _iota(W, S * W, 1, 1, base=100)
    y = o.combine(x, W, S, 1, 1)
    for d in range(W):
        for s in range(S):
            assert y[d, s, d, 0] == 100 * d + d * S + s


# -- invariants ------------------------------------------------------------
SHAPES = [  # (W, S, H, D): tiny, small, DeepSeek-V3 hidden size, tail (D=999)
    (2, 4, 2, 8), (8, 16, 8, 128), (8, 4, 1, 7168), (4, 10, 2, 999), (3, 5, 3, 1),
]


def pin_bijection(o):
    """Every input element appears exactly once in the output (iota input)."""
    for (W, S, H, D) in SHAPES:
        x = _iota(W, S * W, H, D, base=1 << 32, dtype=np.int64)
        y = o.combine(x, W, S, H, D)
        assert np.array_equal(np.sort(y, axis=None), np.sort(x, axis=None))
        if W > 1:
            assert not np.array_equal(y.reshape(-1), x.reshape(-1))
        xd = _iota(W, S * W, H, D, base=1 << 32, dtype=np.int64)
        yd = o.dispatch(xd, W, S * W, H, D)
        assert np.array_equal(np.sort(yd, axis=None), np.sort(xd, axis=None))


# -- library routine -------------------------------------------------------
def pin_numpy_transpose(o):
    """The combine is the (1, 2, 0, 3, 4) transpose of the [r][d][s][h][x] view;
    dispatch is the same with S/W rows per block; the inverse swaps back."""
    for (W, S, H, D) in SHAPES:
        x = _rand((W, S * W, H, D), 7, np.int16)
        ref = x.reshape(W, W, S, H, D).transpose(1, 2, 0, 3, 4).reshape(W, S, W * H, D)
        np.testing.assert_array_equal(o.combine(x, W, S, H, D), ref)
        xd = _rand((W, S * W, H, D), 8, np.int32)
        refd = xd.reshape(W, W, S, H, D).transpose(1, 2, 0, 3, 4).reshape(W, S, W * H, D)
        np.testing.assert_array_equal(o.dispatch(xd, W, S * W, H, D), refd)
        y = _rand((W, S, W * H, D), 9, np.uint8)
        refb = y.reshape(W, S, W, H, D).transpose(2, 0, 1, 3, 4).reshape(W, S * W, H, D)
        np.testing.assert_array_equal(o.combine_back(y, W, S, H, D), refb)


# -- round trips -----------------------------------------------------------
def pin_round_trip(o):
    """dispatch then its inverse, and the inverse then dispatch, are identities."""
    for (W, S, H, D) in [(16, 64, 4, 8), (4, 12, 2, 999), (2, 8, 3, 5)]:
        x = _rand((W, S, H, D), 3, np.float16)
        y = o.dispatch(x, W, S, H, D)
        assert y.shape == (W, S // W, H * W, D)
        np.testing.assert_array_equal(o.combine_back(y, W, S // W, H, D), x)
        z = _rand((W, S // W, H * W, D), 4, np.int16)
        np.testing.assert_array_equal(o.dispatch(o.combine_back(z, W, S // W, H, D), W, S, H, D),
                                      z)


# -- the page's own tile loop ----------------------------------------------
def pin_page_tile_loop(o):
    """The sequential replay of the page's producer/consumer kernel (staging
    layout, signal slots, masks for ragged S and D) gives the combine, and
    leaves every signal slot back at 0."""
    cases = [((2, 4, 2, 8), 2, 8), ((8, 16, 8, 128), 16, 64), ((4, 40, 2, 999), 32, 256),
             ((3, 7, 1, 5), 4, 3)]
    for (W, S, H, D), bs, bd in cases:
        x = _rand((W, S * W, H, D), 5, np.int16)
        y, sig = o.pc_replay(x, W, S, H, D, bs, bd, 2)
        np.testing.assert_array_equal(y, o.combine(x, W, S, H, D))
        assert not sig.any()


def pin_page_two_phase_loop(o):
    """The sequential replay of the page's two-phase kernel (bulk rank slots,
    self-loop double buffer, region A / region B signals) gives the (1, 2, 0,
    3, 4) transpose; afterwards slot r of PE d holds PE r's rows d*S.. for
    every r != d (the bulk arrives whole), every region-A slot of a sender
    r != d reads 1 and its own slot 0, and every region-B slot is back at 0."""
    cases = [((2, 4, 2, 8), 2, 8, 2), ((8, 16, 8, 128), 4, 64, 2), ((4, 40, 2, 999), 8, 256, 2),
             ((3, 7, 1, 5), 2, 3, 3), ((5, 9, 2, 6), 4, 4, 1), ((1, 6, 3, 4), 2, 2, 2),
             ((2, 3, 1, 7), 8, 16, 2)]
    for (W, S, H, D), bs, bd, nbuf in cases:
        x = _rand((W, S * W, H, D), 6, np.int16)
        y, peer, sig = o.two_phase_replay(x, W, S, H, D, bs, bd, nbuf)
        ref = x.reshape(W, W, S, H, D).transpose(1, 2, 0, 3, 4).reshape(W, S, W * H, D)
        np.testing.assert_array_equal(y, ref)
        nbs = -(-S // bs)
        for d in range(W):
            for r in range(W):
                if r != d:
                    np.testing.assert_array_equal(peer[d, r], x[r, d * S:(d + 1) * S])
            region_a = sig[d, :nbs * W, 0].reshape(nbs, W)
            want = np.ones((nbs, W), np.int64)
            want[:, d] = 0
            np.testing.assert_array_equal(region_a, want)
            assert not sig[d, nbs * W:].any() and not sig[d, :, 1:].any()


# -- bit patterns ----------------------------------------------------------
def pin_bit_patterns(o):
    """Values move as raw bits: NaN payloads, -0 and infinities survive."""
    W, S, H, D = 2, 2, 1, 4
    pats = np.array([0x7E01, 0xFE77, 0x8000, 0x7C00, 0xFC00, 0x0001, 0x7BFF, 0x3C00],
                    dtype=np.uint16)
    x = np.resize(pats, W * S * W * H * D).reshape(W, S * W, H, D).view(np.float16)
    y = o.combine(x, W, S, H, D)
    ref = x.view(np.uint16).reshape(W, W, S, H, D).transpose(1, 2, 0, 3, 4)
    np.testing.assert_array_equal(y.view(np.uint16).reshape(-1), ref.reshape(-1))


# -- edge cases ------------------------------------------------------------
def pin_edges(o):
    """Empty extents give empty outputs; dispatch rejects S not divisible by W."""
    x = np.zeros((4, 0, 2, 3), np.int16)
    assert o.combine(x, 4, 0, 2, 3).shape == (4, 0, 8, 3)
    x = np.zeros((2, 6, 2, 0), np.int16)
    assert o.combine(x, 2, 3, 2, 0).size == 0
    try:
        o.dispatch(np.zeros((3, 4, 1, 1), np.int8), 3, 4, 1, 1)
    except ValueError:
        pass
    else:
        raise AssertionError("dispatch accepted S % W != 0")


# -- one-sided primitives --------------------------------------------------
def pin_primitives(o):
    """put/get address PE k at k*slab + offset; SET overwrites, ADD accumulates;
    the RFC's producer/consumer example (SET 1, wait EQ 1) and its push-mode
    AllToAll (each of W ranks ADDs 1, the receiver waits for EQ W) hold."""
    W, slab = 4, 256
    heap = np.zeros(W * slab, np.uint8)
    src = (np.arange(40) * 7 % 251).astype(np.uint8)
    assert o.put(heap, slab, W, 16, src, 2) == 0
    np.testing.assert_array_equal(heap[2 * slab + 16: 2 * slab + 56], src)
    assert heap[:2 * slab + 16].sum() == 0 and heap[2 * slab + 56:].sum() == 0
    dst = np.zeros(40, np.uint8)
    assert o.get(heap, slab, W, dst, 16, 2) == 0
    np.testing.assert_array_equal(dst, src)
    assert o.put(heap, slab, W, 0, src, W) != 0          # no PE W
    assert o.put(heap, slab, W, slab - 8, src, 0) != 0   # past the slab
    # RFC example 1: the producer SETs 1, the consumer waits for EQ 1
    sig_off = 128
    assert o.wait_satisfied(int(heap[3 * slab + sig_off:3 * slab + sig_off + 8].view(np.int64)[0]),
                            1, 0) == 0
    assert o.put_with_signal(heap, slab, W, 32, src[:8], sig_off, 1, 0, 3) == 0
    np.testing.assert_array_equal(heap[3 * slab + 32:3 * slab + 40], src[:8])
    cur = int(heap[3 * slab + sig_off:3 * slab + sig_off + 8].view(np.int64)[0])
    assert cur == 1 and o.wait_satisfied(cur, 1, 0) == 1
    # push mode: every rank ADDs 1 on PE 0; the receiver waits for EQ world_size
    for _ in range(W):
        assert o.signal_op(heap, slab, W, 192, 1, 1, 0) == 0
    cur = int(heap[192:200].view(np.int64)[0])
    assert cur == W
    assert o.wait_satisfied(cur, W, 0) == 1 and o.wait_satisfied(cur, W - 1, 1) == 1
    assert o.wait_satisfied(cur, W, 1) == 0 and o.wait_satisfied(cur, W + 1, 2) == 1
    assert o.wait_satisfied(cur, W, 2) == 0
    assert o.signal_op(heap, slab, W, 192, -5, 0, 0) == 0   # SET overwrites
    assert int(heap[192:200].view(np.int64)[0]) == -5
    assert o.signal_op(heap, slab, W, 192, 1, 2, 0) != 0    # no op 2


# -- collectives: AllToAll with uneven counts, AllGather ---------------------
GOLDEN_A2AV = os.path.join(HERE, "golden", "alltoallv_w2.txt")


def _random_counts(W, seed, hi=5, zero_frac=0.3):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, hi, size=(W, W)).astype(np.int64)
    c[rng.random((W, W)) < zero_frac] = 0
    return c


def pin_alltoallv_golden(o):
    """Hand-worked W=2 uneven exchange (rows are one int32)."""
    vals = {}
    with open(GOLDEN_A2AV) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                vals.setdefault(line[0], []).append([int(v) for v in line[1:]])
    counts = np.array(vals["counts"][0], np.int64).reshape(2, 2)
    x = np.array([row[1:] for row in sorted(vals["in"])], np.int32).reshape(2, 3, 1)
    want = np.array([row[1:] for row in sorted(vals["out"])], np.int32).reshape(2, 4, 1)
    got = o.alltoallv(x, counts, 4, out=np.full((2, 4, 1), -1, np.int32))
    np.testing.assert_array_equal(got, want)


def pin_alltoallv_w1_and_equal_split(o):
    """One PE keeps its first n rows; equal counts S are the block transpose
    of the [r][d][S] view (numpy)."""
    x = _rand((1, 9, 5), 21, np.int16)
    np.testing.assert_array_equal(o.alltoallv(x, np.array([[6]]), 9)[0, :6], x[0, :6])
    for W, S, rb in [(2, 3, 4), (4, 5, 7), (8, 2, 16)]:
        x = _rand((W, W * S, rb), 22, np.uint8)
        y = o.alltoallv(x, np.full((W, W), S, np.int64), W * S)
        ref = x.reshape(W, W, S, rb).transpose(1, 0, 2, 3).reshape(W, W * S, rb)
        np.testing.assert_array_equal(y, ref)


def pin_alltoallv_round_trip_and_bijection(o):
    """Counts C then C^T bring every sent row home; with iota rows the rows
    received are exactly the rows sent."""
    for W, seed in [(2, 1), (5, 2), (8, 3), (3, 4)]:
        c = _random_counts(W, seed)
        in_rows = int(c.sum(1).max()) + 2
        mid_rows = int(c.sum(0).max()) + 1
        x = np.arange(W * in_rows * 3, dtype=np.int64).reshape(W, in_rows, 3) + 10**6
        y = o.alltoallv(x, c, mid_rows)
        back = o.alltoallv(y, c.T.copy(), in_rows)
        for r in range(W):
            n = int(c[r].sum())
            np.testing.assert_array_equal(back[r, :n], x[r, :n])
        sent = np.concatenate([x[r, :int(c[r].sum())] for r in range(W)]).reshape(-1, 3)
        got = np.concatenate([y[d, :int(c[:, d].sum())] for d in range(W)]).reshape(-1, 3)
        assert np.array_equal(np.sort(sent[:, 0]), np.sort(got[:, 0]))


def pin_alltoallv_rejects(o):
    """Negative counts and rows that do not fit are refused."""
    x = np.zeros((2, 3, 1), np.int32)
    for c, out_rows in [(np.array([[1, -1], [0, 0]]), 4), (np.array([[2, 2], [0, 0]]), 4),
                        (np.array([[2, 0], [3, 0]]), 4)]:
        try:
            o.alltoallv(x, c, out_rows)
        except ValueError:
            continue
        raise AssertionError(f"accepted counts {c.tolist()}")


def pin_allgather(o):
    """Every PE's output is the concatenation of all inputs in rank order;
    one PE is the identity."""
    x = _rand((1, 11), 31, np.uint8)
    np.testing.assert_array_equal(o.allgather(x), x)
    for W, n in [(2, 3), (4, 17), (8, 64)]:
        x = _rand((W, n), 32, np.int16)
        y = o.allgather(x)
        for d in range(W):
            np.testing.assert_array_equal(y[d], x.reshape(-1))
    x = np.array([[7, 8], [9, 10], [11, 12]], np.int32)
    assert o.allgather(x)[1].tolist() == [7, 8, 9, 10, 11, 12]


def pin_ag_matmul_golden(o):
    """Hand-worked W=2 values (golden/ag_matmul_w2.txt)."""
    rows = {}
    with open(os.path.join(HERE, "golden", "ag_matmul_w2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *vals = line.split()
                rows.setdefault(key, []).append([float(v) for v in vals])
    a = np.array([r[1:] for r in rows["a"]]).reshape(2, 1, 2)
    b = np.array([r[1:] for r in rows["b"]]).reshape(2, 2, 2)
    gather, c = o.ag_matmul(a, b)
    for d in range(2):
        np.testing.assert_array_equal(gather[d].reshape(-1), rows["gather"][0])
    for d, *vals in rows["c"]:
        np.testing.assert_array_equal(c[int(d)].reshape(-1), vals)
        for i in range(2):
            for j in range(2):
                assert o.ag_matmul_at(a, b, int(d), i, j) == vals[i * 2 + j]


def pin_ag_matmul_library(o):
    """Small integer inputs (exact in float64): the gather is numpy's
    concatenation of the ranks' rows, the result numpy's matmul of it with each
    rank's b; one rank reduces to a plain matmul; the result is linear in b;
    sampled single elements agree with the full result."""
    rng = np.random.default_rng(41)
    for W, m, k, n in [(1, 3, 4, 5), (2, 4, 3, 2), (3, 2, 5, 7), (4, 3, 8, 3)]:
        a = rng.integers(-9, 10, (W, m, k)).astype(np.float64)
        b1 = rng.integers(-9, 10, (W, k, n)).astype(np.float64)
        b2 = rng.integers(-9, 10, (W, k, n)).astype(np.float64)
        gather, c = o.ag_matmul(a, b1)
        stacked = np.concatenate(list(a), axis=0)
        for d in range(W):
            np.testing.assert_array_equal(gather[d], stacked)
            np.testing.assert_array_equal(c[d], np.matmul(stacked, b1[d]))
        _, c2 = o.ag_matmul(a, b2)
        _, c12 = o.ag_matmul(a, b1 + b2)
        np.testing.assert_array_equal(c12, c + c2)
        for _ in range(10):
            d, i, j = rng.integers(0, W), rng.integers(0, W * m), rng.integers(0, n)
            assert o.ag_matmul_at(a, b1, int(d), int(i), int(j)) == c[d, i, j]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(o) -> None:
    for pin in ALL_PINS:
        pin(o)
