/*
 * a2a_oracle.c -- plain CPU oracle for the EP-MoE all-to-all permutations.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may build, load or call
 * this file.  It shares no code, header, table or helper with the CUDA path:
 * every function here is the plain definition written out as nested loops,
 * copying `es` bytes per element with memcpy (no arithmetic on the values, so
 * any dtype -- including NaN payloads and -0 -- passes through bit for bit).
 *
 * Layouts (all contiguous, rank-major, row-major inside a rank):
 *   combine      in  [W][S*W][H][D]   out [W][S][H*W][D]
 *   dispatch     in  [W][S][H][D]     out [W][S/W][H*W][D]
 *   combine_back in  [W][Sp][H*W][D]  out [W][Sp*W][H][D]     (Sp = S/W)
 *
 * Return value: 0 on success, -1 on an invalid shape.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Reverse All2All (combine).
 * Source: "Reverse All2All (EP MoE Distributed Kernel)", section "Reverse
 * All2All Operator Semantics": per rank the input (S*world_size, H, D) becomes
 * the output (S, H*world_size, D).  Which input row lands in which output
 * column follows the same page's "MTE Implementation": the producer of rank
 * r reads row target*S + s, expert column h, and writes the target's column
 * r*H + h; the consumer of rank d keeps row s and column r*H + h.  Hence
 *     out_d[s, r*H + h, x] = in_r[d*S + s, h, x].                            */
int oracle_combine(const void *in, void *out, int64_t W, int64_t S, int64_t H,
                   int64_t D, int64_t es)
{
    if (W < 1 || S < 0 || H < 0 || D < 0 || es < 1) return -1;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    /* Each (d, s) writes only row s of out_d: the OpenMP build (timed CPU
     * baseline only) splits the loops over d and s across threads; the plain
     * build ignores this. */
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static)
#endif
    for (int64_t d = 0; d < W; d++)
        for (int64_t s = 0; s < S; s++)
            for (int64_t r = 0; r < W; r++)
                for (int64_t h = 0; h < H; h++)
                    for (int64_t x = 0; x < D; x++) {
                        /* in_r has S*W rows of H*D elements */
                        int64_t i_in = ((r * (S * W) + (d * S + s)) * H + h) * D + x;
                        /* out_d has S rows of (H*W)*D elements */
                        int64_t i_out = ((d * S + s) * (H * W) + (r * H + h)) * D + x;
                        memcpy(dst + i_out * es, src + i_in * es, (size_t)es);
                    }
    return 0;
}

/* Forward All2All (dispatch).
 * Source: same page, "Reverse All2All Operator Semantics" and "EP MoE
 * Scenario": per rank (S, H, D) becomes (S/world_size, H*world_size, D).  The
 * page gives shapes only; the row/column placement is the combine's with the
 * block length S' = S/W:
 *     out_d[s', r*H + h, x] = in_r[d*S' + s', h, x].
 * S must be a multiple of W.                                                 */
int oracle_dispatch(const void *in, void *out, int64_t W, int64_t S, int64_t H,
                    int64_t D, int64_t es)
{
    if (W < 1 || S < 0 || H < 0 || D < 0 || es < 1 || S % W != 0) return -1;
    const int64_t Sp = S / W;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t d = 0; d < W; d++)
        for (int64_t sp = 0; sp < Sp; sp++)
            for (int64_t r = 0; r < W; r++)
                for (int64_t h = 0; h < H; h++)
                    for (int64_t x = 0; x < D; x++) {
                        /* in_r has S rows of H*D elements */
                        int64_t i_in = ((r * S + (d * Sp + sp)) * H + h) * D + x;
                        /* out_d has Sp rows of (H*W)*D elements */
                        int64_t i_out = ((d * Sp + sp) * (H * W) + (r * H + h)) * D + x;
                        memcpy(dst + i_out * es, src + i_in * es, (size_t)es);
                    }
    return 0;
}

/* Inverse of dispatch ("results must be sent back ... to the token's original
 * rank", same page, introduction).  Per rank (Sp, H*W, D) becomes (Sp*W, H, D):
 *     out_r[d*Sp + s', h, x] = in_d[s', r*H + h, x].                         */
int oracle_combine_back(const void *in, void *out, int64_t W, int64_t Sp,
                        int64_t H, int64_t D, int64_t es)
{
    if (W < 1 || Sp < 0 || H < 0 || D < 0 || es < 1) return -1;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t r = 0; r < W; r++)
        for (int64_t d = 0; d < W; d++)
            for (int64_t sp = 0; sp < Sp; sp++)
                for (int64_t h = 0; h < H; h++)
                    for (int64_t x = 0; x < D; x++) {
                        /* in_d has Sp rows of (H*W)*D elements */
                        int64_t i_in = ((d * Sp + sp) * (H * W) + (r * H + h)) * D + x;
                        /* out_r has Sp*W rows of H*D elements */
                        int64_t i_out = ((r * (Sp * W) + (d * Sp + sp)) * H + h) * D + x;
                        memcpy(dst + i_out * es, src + i_in * es, (size_t)es);
                    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sequential replay of the tile-level producer/consumer algorithm of the    */
/* page's "MTE Implementation" (sections "Producer-Consumer Pipeline",       */
/* "Signal Memory Layout", "Symmetric Memory Layout").  It exists to pin the  */
/* definition above against the page's own index arithmetic: the staging     */
/* ("peer memory") layout [buffer][block_s rows][H*W][D] per rank, the        */
/* per-task int64 signal slots spaced 8 elements apart, the wait-for-0 /      */
/* notify-1 / wait-for-1 / reset-to-0 handshake, and the boundary masks.      */
/*                                                                            */
/* Every "core" of the page runs one after another: within one S block all    */
/* producer tasks of every rank, then all consumer tasks of every rank.  That */
/* is one legal interleaving of the concurrent pipeline.  A wait whose        */
/* condition does not hold in this order is a protocol error (returns -2).    */
/*                                                                            */
/* staging: W * buffer_num * block_s * (H*W) * D * es bytes (rank-major)      */
/* signals: W * buffer_num * nbd * H * W * 8 int64 (rank-major), zeroed by    */
/*          the caller first, as the page's host side does before launch.     */
/* ------------------------------------------------------------------------ */
int oracle_pc_replay(const void *in, void *out, int64_t W, int64_t S, int64_t H,
                     int64_t D, int64_t es, int64_t block_s, int64_t block_d,
                     int64_t buffer_num, void *staging, int64_t *signals)
{
    if (W < 1 || S < 0 || H < 0 || D < 0 || es < 1 || block_s < 1 || block_d < 1 ||
        buffer_num < 1)
        return -1;
    const unsigned char *a = (const unsigned char *)in;
    unsigned char *c = (unsigned char *)out;
    unsigned char *peer = (unsigned char *)staging;
    const int64_t nbs = (S + block_s - 1) / block_s;
    const int64_t nbd = (D + block_d - 1) / block_d;
    const int64_t tasks = nbd * H * W;                 /* per buffer, per rank */
    const int64_t chunk = H * W * D;                   /* one staging row      */
    const int64_t peer_rank_elems = buffer_num * block_s * chunk;
    const int64_t sig_rank_elems = buffer_num * tasks * 8;
    const int64_t a_rank_rows = S * W;                 /* input rows per rank  */

    for (int64_t bs = 0; bs < nbs; bs++) {
        const int64_t buf = bs % buffer_num;

        /* producers: every source rank, every task (rank_loop, h, d block) */
        for (int64_t rank = 0; rank < W; rank++) {
            for (int64_t task = 0; task < tasks; task++) {
                const int64_t rank_loop = task % W;
                const int64_t hd = task / W;           /* = block_d*H + h */
                const int64_t h = hd % H;
                const int64_t bd = hd / H;
                const int64_t target = (rank + rank_loop) % W;
                int64_t *slot = signals + target * sig_rank_elems +
                                (buf * tasks + rank * nbd * H + hd) * 8;
                if (*slot != 0) return -2;             /* wait(slot == 0) */
                for (int64_t i = 0; i < block_s; i++) {
                    const int64_t s = bs * block_s + i;
                    if (s >= S) continue;              /* row mask */
                    for (int64_t j = 0; j < block_d; j++) {
                        const int64_t x = bd * block_d + j;
                        if (x >= D) continue;          /* column mask */
                        const int64_t i_a = ((rank * a_rank_rows + target * S + s) * H + h) * D + x;
                        const int64_t i_p = target * peer_rank_elems +
                                            (buf * block_s + i) * chunk +
                                            (rank * H + h) * D + x;
                        memcpy(peer + i_p * es, a + i_a * es, (size_t)es);
                    }
                }
            }
            /* after its fence, the producer notifies every task's slot */
            for (int64_t task = 0; task < tasks; task++) {
                const int64_t hd = task / W;
                const int64_t target = (rank + task % W) % W;
                signals[target * sig_rank_elems + (buf * tasks + rank * nbd * H + hd) * 8] = 1;
            }
        }

        /* consumers: every destination rank, every task (r, h, d block) */
        for (int64_t rank = 0; rank < W; rank++) {
            for (int64_t task = 0; task < tasks; task++) {
                const int64_t r = task % W;
                const int64_t hd = task / W;
                const int64_t h = hd % H;
                const int64_t bd = hd / H;
                const int64_t *slot = signals + rank * sig_rank_elems +
                                      (buf * tasks + r * nbd * H + hd) * 8;
                if (*slot != 1) return -2;             /* wait(slot == 1) */
                for (int64_t i = 0; i < block_s; i++) {
                    const int64_t s = bs * block_s + i;
                    if (s >= S) continue;
                    for (int64_t j = 0; j < block_d; j++) {
                        const int64_t x = bd * block_d + j;
                        if (x >= D) continue;
                        const int64_t i_p = rank * peer_rank_elems +
                                            (buf * block_s + i) * chunk +
                                            (r * H + h) * D + x;
                        const int64_t i_c = ((rank * S + s) * (H * W) + (r * H + h)) * D + x;
                        memcpy(c + i_c * es, peer + i_p * es, (size_t)es);
                    }
                }
            }
            /* after its fence, the consumer returns every slot to 0 */
            for (int64_t task = 0; task < tasks; task++) {
                const int64_t r = task % W;
                const int64_t hd = task / W;
                signals[rank * sig_rank_elems + (buf * tasks + r * nbd * H + hd) * 8] = 0;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sequential replay of the page's two-phase combine ("UDMA Optimized         */
/* Implementation" with its "Wait/Notify Optimization": sections "Two-Phase   */
/* Data Copy", "Symmetric Memory Layout" and "Dual Signal Memory Region       */
/* Design").  Like the replay above it pins the combine's definition against */
/* the page's own index arithmetic, here for the other staging layout:        */
/*   peer memory per rank: W rank slots of [S][H][D]; slot r != rank receives */
/*   rank r's whole segment for this rank (bulk, no buffering); slot rank     */
/*   holds only the self-loop double buffer [buffer][block_s][H][D] at its    */
/*   start.                                                                   */
/*   signals per rank: region A [nbs][W] ("sender r has sent S block b",      */
/*   written once, never reset), then region B [buffer][nbd*H] (self-loop     */
/*   handshake: wait 0, write, notify 1; the consumer returns the credit by   */
/*   setting 0), slots 8 int64 apart.                                        */
/* Order per S block: every rank's bulk sends of that block, then every       */
/* rank's self-loop tiles, then every rank's consumer tasks -- one legal      */
/* interleaving of the concurrent kernel.  The bulk phase is replayed block   */
/* by block, as the wait/notify version sends it (one send per S block and   */
/* target, each followed by its region-A notify).  A wait whose condition     */
/* does not hold in this order, or a region-A slot written twice, is a        */
/* protocol error (returns -2).                                               */
/*                                                                            */
/* peer:    W * W*S*H*D * es bytes (rank-major)                               */
/* signals: W * (nbs*W + buffer_num*nbd*H) * 8 int64 (rank-major), zeroed by  */
/*          the caller first.                                                 */
/* ------------------------------------------------------------------------ */
int oracle_two_phase_replay(const void *in, void *out, int64_t W, int64_t S, int64_t H,
                            int64_t D, int64_t es, int64_t block_s, int64_t block_d,
                            int64_t buffer_num, void *peer_mem, int64_t *signals)
{
    /* The double buffer always fits slot rank: buffer buf holds S block buf
     * (rows < S) while nbs <= buffer_num, and S > buffer_num*block_s after. */
    if (W < 1 || S < 0 || H < 0 || D < 0 || es < 1 || block_s < 1 || block_d < 1 ||
        buffer_num < 1)
        return -1;
    const unsigned char *a = (const unsigned char *)in;
    unsigned char *c = (unsigned char *)out;
    unsigned char *peer = (unsigned char *)peer_mem;
    const int64_t nbs = (S + block_s - 1) / block_s;
    const int64_t nbd = (D + block_d - 1) / block_d;
    const int64_t row = H * D;                         /* one [H][D] row, elements */
    const int64_t peer_rank_elems = W * S * row;
    const int64_t tasks = nbd * H;                     /* self-loop tasks per block */
    const int64_t region_b = nbs * W * 8;
    const int64_t sig_rank_elems = region_b + buffer_num * tasks * 8;

    for (int64_t bs = 0; bs < nbs; bs++) {
        const int64_t buf = bs % buffer_num;
        const int64_t s0 = bs * block_s;
        const int64_t rows = (S - s0 < block_s) ? S - s0 : block_s;

        /* phase 1: rank sends its rows target*S + s0 .. to the target's slot rank */
        for (int64_t rank = 0; rank < W; rank++)
            for (int64_t target = 0; target < W; target++) {
                if (target == rank) continue;
                const int64_t i_a = (rank * (S * W) + target * S + s0) * row;
                const int64_t i_p = target * peer_rank_elems + (rank * S + s0) * row;
                memcpy(peer + i_p * es, a + i_a * es, (size_t)(rows * row * es));
                int64_t *slot = signals + target * sig_rank_elems + (bs * W + rank) * 8;
                if (*slot != 0) return -2;             /* written once */
                *slot = 1;
            }

        /* phase 2: self-loop tiles into the double buffer of slot rank */
        for (int64_t rank = 0; rank < W; rank++)
            for (int64_t task = 0; task < tasks; task++) {
                const int64_t h = task % H;
                const int64_t bd = task / H;
                int64_t *slot = signals + rank * sig_rank_elems + region_b +
                                (buf * tasks + task) * 8;
                if (*slot != 0) return -2;             /* wait(slot == 0) */
                for (int64_t i = 0; i < rows; i++)
                    for (int64_t j = 0; j < block_d; j++) {
                        const int64_t x = bd * block_d + j;
                        if (x >= D) continue;          /* column mask */
                        const int64_t i_a = ((rank * (S * W) + rank * S + s0 + i) * H + h) * D + x;
                        const int64_t i_p = rank * peer_rank_elems + rank * S * row +
                                            (buf * block_s + i) * row + h * D + x;
                        memcpy(peer + i_p * es, a + i_a * es, (size_t)es);
                    }
                *slot = 1;                             /* notify after the fence */
            }

        /* consumers: every destination rank, every task (r, h, d block) */
        for (int64_t rank = 0; rank < W; rank++)
            for (int64_t task = 0; task < tasks * W; task++) {
                const int64_t r = task % W;
                const int64_t hd = task / W;           /* = block_d*H + h */
                const int64_t h = hd % H;
                const int64_t bd = hd / H;
                int64_t *slot;
                int64_t first_row;                     /* row of s0 inside slot r */
                if (r == rank) {
                    slot = signals + rank * sig_rank_elems + region_b + (buf * tasks + hd) * 8;
                    first_row = buf * block_s;
                } else {
                    slot = signals + rank * sig_rank_elems + (bs * W + r) * 8;
                    first_row = s0;
                }
                if (*slot != 1) return -2;             /* wait(slot == 1) */
                for (int64_t i = 0; i < rows; i++)
                    for (int64_t j = 0; j < block_d; j++) {
                        const int64_t x = bd * block_d + j;
                        if (x >= D) continue;
                        const int64_t i_p = rank * peer_rank_elems + r * S * row +
                                            (first_row + i) * row + h * D + x;
                        const int64_t i_c = ((rank * S + s0 + i) * (H * W) + (r * H + h)) * D + x;
                        memcpy(c + i_c * es, peer + i_p * es, (size_t)es);
                    }
                if (r == rank) *slot = 0;              /* credit return */
            }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One-sided primitives on a symmetric heap held in host memory.              */
/* Source: "Distributed Architecture Design" section 5.3 (remote address =    */
/* target PE's heap base + the pointer's offset from the local heap base),    */
/* and the HyperParallel "Symmetric Memory" RFC, section 4 (Python API) and   */
/* section 6 (primitive semantics): put copies size bytes to the target PE,   */
/* get copies from the source PE, signal_op is SET (0) or ADD (1), wait       */
/* compares with EQ (0), GT (1) or LT (2).                                    */
/* The heap here is npes slabs of slab_stride bytes, slab k = PE k.           */
/* ------------------------------------------------------------------------ */

/* Address of `offset` (bytes from the start of a slab) on PE `pe`. */
static unsigned char *oracle_heap_at(unsigned char *heap, int64_t slab_stride,
                                     int64_t pe, int64_t offset)
{
    return heap + pe * slab_stride + offset;
}

/* put: target slab `pe`, byte offset target_off, receives `bytes` from src. */
int oracle_put(void *heap, int64_t slab_stride, int64_t npes, int64_t target_off,
               const void *src, int64_t bytes, int64_t pe)
{
    if (pe < 0 || pe >= npes || target_off < 0 || bytes < 0 ||
        target_off + bytes > slab_stride)
        return -1;
    memcpy(oracle_heap_at((unsigned char *)heap, slab_stride, pe, target_off), src,
           (size_t)bytes);
    return 0;
}

/* get: dst receives `bytes` from slab `pe` at byte offset src_off. */
int oracle_get(const void *heap, int64_t slab_stride, int64_t npes, void *dst,
               int64_t src_off, int64_t bytes, int64_t pe)
{
    if (pe < 0 || pe >= npes || src_off < 0 || bytes < 0 || src_off + bytes > slab_stride)
        return -1;
    memcpy(dst, oracle_heap_at((unsigned char *)heap, slab_stride, pe, src_off),
           (size_t)bytes);
    return 0;
}

/* signal_op on the int64 signal at byte offset sig_off of slab `pe`. */
int oracle_signal_op(void *heap, int64_t slab_stride, int64_t npes, int64_t sig_off,
                     int64_t value, int64_t op, int64_t pe)
{
    if (pe < 0 || pe >= npes || sig_off < 0 || sig_off + 8 > slab_stride) return -1;
    int64_t cur;
    unsigned char *p = oracle_heap_at((unsigned char *)heap, slab_stride, pe, sig_off);
    memcpy(&cur, p, 8);
    if (op == 0)
        cur = value;                                  /* SET */
    else if (op == 1)
        cur = (int64_t)((uint64_t)cur + (uint64_t)value); /* ADD, wrapping */
    else
        return -1;
    memcpy(p, &cur, 8);
    return 0;
}

/* wait predicate: 1 if `current` satisfies (cmp, value), 0 if not, -1 bad cmp */
int oracle_wait_satisfied(int64_t current, int64_t value, int64_t cmp)
{
    if (cmp == 0) return current == value;            /* EQ */
    if (cmp == 1) return current > value;             /* GT */
    if (cmp == 2) return current < value;             /* LT */
    return -1;
}

/* put_with_signal: the data lands before the signal changes (the RFC's     */
/* "fence before signal" rule); sequentially that is put, then signal_op.   */
int oracle_put_with_signal(void *heap, int64_t slab_stride, int64_t npes,
                           int64_t target_off, const void *src, int64_t bytes,
                           int64_t sig_off, int64_t value, int64_t op, int64_t pe)
{
    int rc = oracle_put(heap, slab_stride, npes, target_off, src, bytes, pe);
    if (rc) return rc;
    return oracle_signal_op(heap, slab_stride, npes, sig_off, value, op, pe);
}

/* ------------------------------------------------------------------------ */
/* Collectives built on the one-sided primitives: HyperParallel RFC          */
/* "Symmetric Memory", section 10 (advanced algorithms, push mode).          */
/* ------------------------------------------------------------------------ */

/* AllToAll with per-pair row counts (push mode).  counts[r*W + d] rows of   */
/* row_bytes go from PE r to PE d.  PE r's input holds its rows for d = 0,   */
/* 1, ... back to back; PE d's output holds the rows it receives from r = 0, */
/* 1, ... back to back (the receive offsets the RFC exchanges first).        */
/*   in  [W][in_rows][row_bytes]    out [W][out_rows][row_bytes]            */
/* Output rows past what PE d receives are left untouched.  Returns -1 when  */
/* a count is negative or a PE would send or receive more rows than fit.     */
int oracle_alltoallv(const void *in, void *out, const int64_t *counts, int64_t W,
                     int64_t row_bytes, int64_t in_rows, int64_t out_rows)
{
    if (W < 1 || row_bytes < 0 || in_rows < 0 || out_rows < 0) return -1;
    for (int64_t r = 0; r < W; r++) {
        int64_t sent = 0;
        for (int64_t d = 0; d < W; d++) {
            if (counts[r * W + d] < 0) return -1;
            sent += counts[r * W + d];
        }
        if (sent > in_rows) return -1;
    }
    for (int64_t d = 0; d < W; d++) {
        int64_t got = 0;
        for (int64_t r = 0; r < W; r++) got += counts[r * W + d];
        if (got > out_rows) return -1;
    }
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t d = 0; d < W; d++) {
        int64_t pos = 0;                               /* next receive row of d */
        for (int64_t r = 0; r < W; r++) {
            int64_t first = 0;                         /* r's first row for d */
            for (int64_t e = 0; e < d; e++) first += counts[r * W + e];
            for (int64_t i = 0; i < counts[r * W + d]; i++) {
                memcpy(dst + (d * out_rows + pos) * row_bytes,
                       src + (r * in_rows + first + i) * row_bytes, (size_t)row_bytes);
                pos++;
            }
        }
    }
    return 0;
}

/* AllGather (push mode): every PE r places its `bytes` at byte r*bytes of  */
/* every PE's output.   in [W][bytes]   out [W][W*bytes]                     */
int oracle_allgather(const void *in, void *out, int64_t W, int64_t bytes)
{
    if (W < 1 || bytes < 0) return -1;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t d = 0; d < W; d++)
        for (int64_t r = 0; r < W; r++)
            memcpy(dst + (d * W + r) * bytes, src + r * bytes, (size_t)bytes);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fused AllGather + MatMul.                                                  */
/* Source: HyperParallel RFC "Symmetric Memory", section 10                   */
/* (fused_all_gather_matmul) and its example 2 (fused AllGather + MatMul):    */
/* every rank r holds a_r (m_local x k) and its own b (k x n); the gathered   */
/* gather_out (m_total x k, m_total = W * m_local) stacks a_0, a_1, ... in    */
/* rank order, and the result on rank d is gather_out @ b_d (m_total x n).    */
/* The section's formula also names a ReduceScatter, but the example's        */
/* result is (m_total, n) on every rank: the plain reading, taken here, is    */
/* the matmul of the gathered rows with no reduction.                         */
/* Values are doubles (the caller widens fp16 / bf16 exactly); the sum runs   */
/* over the k index in increasing order.                                      */
/*   a [W][m_local][k], b [W][k][n] -> gather [W][m_total][k],                */
/*   c [W][m_total][n]                                                        */
/* ------------------------------------------------------------------------ */
int oracle_ag_matmul(const double *a, const double *b, double *gather, double *c, int64_t W,
                     int64_t m_local, int64_t k, int64_t n)
{
    if (W < 1 || m_local < 0 || k < 0 || n < 0)
        return -1;
    const int64_t m_total = W * m_local;
    for (int64_t d = 0; d < W; d++)
        for (int64_t r = 0; r < W; r++)
            for (int64_t i = 0; i < m_local; i++)
                for (int64_t x = 0; x < k; x++)
                    gather[(d * m_total + r * m_local + i) * k + x] = a[(r * m_local + i) * k + x];
    for (int64_t d = 0; d < W; d++)
        for (int64_t i = 0; i < m_total; i++)
            for (int64_t j = 0; j < n; j++) {
                double acc = 0.0;
                for (int64_t x = 0; x < k; x++)
                    acc += gather[(d * m_total + i) * k + x] * b[(d * k + x) * n + j];
                c[(d * m_total + i) * n + j] = acc;
            }
    return 0;
}

/* One output element c_d[i, j] of the same operation, straight from the     */
/* inputs: row i of gather_out is row i % m_local of a_(i / m_local).         */
double oracle_ag_matmul_at(const double *a, const double *b, int64_t W, int64_t m_local,
                           int64_t k, int64_t n, int64_t d, int64_t i, int64_t j)
{
    const int64_t r = i / m_local, row = i % m_local;
    double acc = 0.0;
    for (int64_t x = 0; x < k; x++)
        acc += a[(r * m_local + row) * k + x] * b[(d * k + x) * n + j];
    (void)W;
    return acc;
}
