/*
 * symm_a2a.h -- C ABI of the GB300 symmetric-heap all-to-all library
 * (libsymm_a2a.so, sm_103a).
 *
 * W processing elements (PEs, "ranks") are emulated on one GPU as W equal
 * slabs of one device allocation that the caller owns.  Every call takes
 * plain pointers and sizes; device pointers are marked "device", the CUDA
 * stream is passed as `void *stream` (a cudaStream_t; NULL = legacy default
 * stream).  Calls that launch work are asynchronous on that stream: a zero
 * return means "validated and enqueued".  A wait that gives up on the device
 * is reported later by symm_check_error().
 *
 * Return codes: SYMM_OK, or a negative SYMM_E* code; symm_last_error() then
 * holds a one-line message (per calling thread).  No call allocates device
 * memory; none frees memory it did not allocate; none ever traps the GPU.
 *
 * Sources (page, section) of the operations:
 *  [RA2A]  "Reverse All2All (EP MoE Distributed Kernel)": sections "Reverse
 *          All2All Operator Semantics", "EP MoE Scenario", "MTE
 *          Implementation" (Producer-Consumer Pipeline, Signal Memory Layout,
 *          Symmetric Memory Layout, Performance Considerations).
 *  [RFC]   HyperParallel RFC "Symmetric Memory (one-sided communication)":
 *          section 2 (symmetric memory), 4 (Python API), 5 (push/pull
 *          modes), 6 (primitive semantics), 8 (kernel notes).
 *  [ARCH]  "Distributed Architecture Design": section 5 (symmetric heap
 *          runtime, 5.3 symm_at address resolution), section 6 (signal,
 *          wait, fence mechanisms).
 */
#ifndef SYMM_A2A_H
#define SYMM_A2A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes -- */
#define SYMM_OK 0
#define SYMM_EINVAL (-1)    /* bad argument: shape, PE, pointer, range, alignment */
#define SYMM_ENOMEM (-2)    /* the heap's slab has no room for the request */
#define SYMM_ETIMEDOUT (-3) /* a device-side wait ran past its budget */
#define SYMM_ECUDA (-4)     /* a CUDA runtime call failed (message in symm_last_error) */
#define SYMM_ERANGE (-5)    /* device-side sizes (counts) exceed a buffer; reported by symm_check_error */

/* signal operations and comparisons, numbered as the [RFC] Python API numbers
 * them (section 4: signal_op 0=SET, 1=ADD; compare_op 0=EQ, 1=GT, 2=LT) */
#define SYMM_SIGNAL_SET 0
#define SYMM_SIGNAL_ADD 1
#define SYMM_CMP_EQ 0
#define SYMM_CMP_GT 1
#define SYMM_CMP_LT 2

/* all2all_combine variants */
#define SYMM_A2A_DIRECT 0 /* one pass over every (source, destination, row) run */
#define SYMM_A2A_PC 1     /* persistent producer/consumer through staging slots */
/* OR-ed into the variant: skip the signal reset that precedes a PC launch
 * (the caller has zeroed the signal slots itself) */
#define SYMM_A2A_FLAG_NO_RESET 0x100
/* Copy paths.  By default each variant uses the path measured fastest on
 * GB300: DIRECT moves 16-byte vectors through registers where every run is
 * 16-byte aligned, and otherwise (in device memory) bulk-loads each run's, or
 * each batch of short runs', 16-byte-aligned covering range into shared
 * memory and stores aligned 16-byte vectors from there; PC prefetches the
 * producer's input tiles with bulk (TMA) copies into shared memory when its
 * rows are long enough to pay (2 KB aligned, 1 KB at any alignment), and
 * uses 16-byte vectors otherwise.
 * OR-ed into the variant: SYMM_A2A_FLAG_VECTOR makes PC use 16-byte vectors
 * only; SYMM_A2A_FLAG_BULK makes DIRECT use bulk (TMA) copies through
 * shared memory both ways where every run is 16-byte aligned. */
#define SYMM_A2A_FLAG_VECTOR 0x200
#define SYMM_A2A_FLAG_BULK 0x400
/* OR-ed into SYMM_A2A_PC, for debugging: a barrier between producers and
 * consumers.  Each S block runs as two launches -- every producer stages its
 * tile and releases its slot, then every consumer acquires, copies out and
 * returns its slot -- so no consumer overlaps any producer ([RA2A] "MTE
 * Implementation" with a global barrier per S block in place of the
 * pipelining).  Same staging, slots and results, far slower: a result that
 * is right with this flag and wrong without it points at the
 * synchronisation rather than at the index arithmetic.  Slots are always
 * zeroed first (SYMM_A2A_FLAG_NO_RESET is ignored). */
#define SYMM_A2A_FLAG_PHASED 0x800

/* bytes at the start of every slab that the heap keeps for itself */
#define SYMM_HEAP_HEADER_BYTES 4096
/* distance between two producer/consumer signal slots (one 64-byte line) */
#define SYMM_SIGNAL_STRIDE_BYTES 64

typedef struct symm_heap symm_heap_t;

/* ------------------------------------------------------- symmetric heap -- */

/* [ARCH] 5, [RFC] 2: a symmetric heap is memory of the same size and layout
 * on every PE, so an offset means the same object on every PE.
 * base        device; caller-owned; >= npes * slab_stride bytes; 256-byte
 *             aligned.  The heap never frees it.  The first
 *             SYMM_HEAP_HEADER_BYTES of every slab are reserved.
 * slab_stride bytes per PE; a multiple of 256 (2 MiB recommended) and
 *             > SYMM_HEAP_HEADER_BYTES.  PE k's slab starts at base + k*slab_stride.
 * npes        number of PEs (W), >= 1.
 * heap        out: host handle.  Writes no device memory (the header is
 *             zeroed on the stream of the first call that launches work).
 *             With a current CUDA device, it looks up the address of
 *             all2all_combine_pc_noalloc's static array on that device (see
 *             there), which makes CUDA load and reserve that array; a
 *             failure there is not reported here (the entry point reports it).
 * Errors: SYMM_EINVAL. */
int symm_heap_init(void *base, size_t slab_stride, int npes, symm_heap_t **heap);

/* Releases the host handle only. */
int symm_heap_destroy(symm_heap_t *heap);

/* [ARCH] 5.2 (symmetric allocation: same size on every PE).  Bump-allocates
 * `bytes` at one offset, reserved in every slab; returns PE 0's address.
 * align: power of two (0 = 256); the result is always 256-byte aligned and
 * every allocation is padded to a multiple of 256 bytes.
 * Errors: SYMM_EINVAL (bad align), SYMM_ENOMEM (slab full). */
int symm_malloc(symm_heap_t *heap, size_t bytes, size_t align, void **ptr);

/* Frees every symm_malloc allocation at once (offsets restart after the header). */
int symm_heap_reset(symm_heap_t *heap);

/* [ARCH] 5.3: the address of `ptr`'s object on PE `pe`:
 *   base + pe*slab_stride + ((ptr - base) mod slab_stride).
 * ptr may point into any slab.  Returns NULL when pe is out of range or ptr
 * is outside the heap.  Host-only arithmetic. */
void *symm_at(symm_heap_t *heap, const void *ptr, int pe);

/* Default spin budget of producer/consumer waits, in ns (initially 2 s). */
int symm_set_spin_budget(symm_heap_t *heap, uint64_t budget_ns);

/* Marks, in the *info of symm_check_error, a timed-out signal slot of
 * all2all_combine_pc_noalloc: *info = SYMM_INFO_NOALLOC_SIGNAL + the slot's
 * byte offset in the signal area of that call's static array. */
#define SYMM_INFO_NOALLOC_SIGNAL (1ll << 62)

/* Synchronises `stream`, then returns the first device-side error recorded in
 * the heap header since the last check (SYMM_OK; SYMM_ETIMEDOUT; SYMM_ERANGE
 * from shmem_alltoall) and clears it.  Until it is cleared, every later
 * device wait on this heap gives up at once (the abort flag stays raised),
 * so check after any launch that may have timed out.  *info (optional)
 * receives, for a wait that gave up, the byte offset from base of its
 * signal, or SYMM_INFO_NOALLOC_SIGNAL + an offset for a signal of
 * all2all_combine_pc_noalloc (see there).  Errors: SYMM_ECUDA. */
int symm_check_error(symm_heap_t *heap, void *stream, int64_t *info);

/* Message of the last failed call on this thread ("" if none). */
const char *symm_last_error(void);

/* ------------------------------------------------- one-sided primitives -- */

/* [RFC] 4, 6 (shmem_put; push): copy `bytes` from device src + src_off to
 * PE target_pe's copy of the symmetric object `target`, at byte target_off.
 * The destination range must lie in one slab past the header; src is any
 * device memory inside a 16-byte-aligned allocation (cudaMalloc, torch).
 * Any alignment of either side.  Errors: SYMM_EINVAL. */
int shmem_put(symm_heap_t *heap, void *target, size_t target_off, const void *src,
              size_t src_off, size_t bytes, int target_pe, void *stream);

/* [RFC] 4, 6 (shmem_get; pull): copy `bytes` from PE src_pe's copy of the
 * symmetric object `src`, at byte src_off, to device dst + dst_off. */
int shmem_get(symm_heap_t *heap, void *dst, size_t dst_off, const void *src, size_t src_off,
              size_t bytes, int src_pe, void *stream);

/* [RFC] 4, 6; [ARCH] 6.2: apply SET or ADD of `value` to the int64 at
 * element `signal_off` of PE target_pe's copy of the symmetric array
 * `signal` (8-byte aligned), with release semantics at GPU scope: writes
 * ordered before this call on the stream are visible to whoever observes
 * the new value.  op: SYMM_SIGNAL_SET or SYMM_SIGNAL_ADD (wrapping). */
int shmem_signal_op(symm_heap_t *heap, int64_t *signal, size_t signal_off, int64_t value, int op,
                    int target_pe, void *stream);

/* [RFC] 4, 6; [ARCH] 6.3: block the stream until the int64 at element
 * signal_off of PE pe's copy of `signal` compares (cmp: EQ/GT/LT) true
 * against cmp_value, with acquire semantics; work later on the stream sees
 * what the signaller wrote before its signal.  The wait does not consume the
 * signal (several waiters may wait on one slot).  It gives up after
 * budget_ns (0 = the heap's spin budget) and then records SYMM_ETIMEDOUT for
 * symm_check_error(); it never hangs the GPU.  Another kernel that must run
 * concurrently to satisfy it is not guaranteed to: signal first in stream
 * order, or expect the timeout. */
int shmem_wait_for_signal(symm_heap_t *heap, const int64_t *signal, size_t signal_off,
                          int64_t cmp_value, int cmp, int pe, uint64_t budget_ns, void *stream);

/* [RFC] 4, 6, 8 (put_mem_signal): shmem_put, then -- after every byte of it
 * is visible at GPU scope -- shmem_signal_op on PE target_pe, in one launch.
 * Calls of it that overlap on the device share one arrival counter in the
 * heap header and race; issue them in stream order. */
int shmem_put_with_signal(symm_heap_t *heap, void *target, size_t target_off, const void *src,
                          size_t src_off, size_t bytes, int64_t *signal, size_t signal_off,
                          int64_t value, int op, int target_pe, void *stream);

/* ------------------------------------------------------------ all-to-all -- */

/* Sizes of the producer/consumer workspace, per PE ([RA2A] "Signal Memory
 * Layout", "Symmetric Memory Layout"):
 *   staging : buffer_num * tile_s * (H*W) * D * elem_bytes bytes
 *             (layout [buffer][tile_s rows][H*W][D])
 *   signals : buffer_num * nbd * H * W slots of SYMM_SIGNAL_STRIDE_BYTES
 *             (int64 each; slot (buf, r, bd, h) at
 *              ((buf*W + r)*nbd + bd)*H + h), nbd = ceil(D / block_d).
 * block_d = 0 means D.  Errors: SYMM_EINVAL. */
int all2all_pc_workspace(int W, int S, int H, int D, int elem_bytes, int tile_s, int block_d,
                         int buffer_num, size_t *staging_bytes, size_t *signal_bytes);

/* [RA2A] "Reverse All2All Operator Semantics" / "MTE Implementation":
 * Reverse All2All (combine).  Per PE the input (S*W, H, D) becomes the
 * output (S, H*W, D):
 *     out_d[s, r*H + h, x] = in_r[d*S + s, h, x]
 * for every destination PE d, source PE r, row s < S, h < H, x < D.
 * in, out     symmetric (heap) pointers; PE k's tensors are symm_at(in|out, k),
 *             contiguous row-major, elem_bytes per element, any alignment.
 *             The input and output ranges must not overlap.
 * variant     SYMM_A2A_DIRECT, or SYMM_A2A_PC [| SYMM_A2A_FLAG_NO_RESET]:
 *             producers copy tile_s x block_d tiles of every source PE into
 *             the destination PE's staging slot and release its signal; the
 *             destination's consumers acquire it, copy the tile into the
 *             output and return the slot (signal 0).  The launch zeroes the
 *             W signal arrays first (unless NO_RESET).  Its grid never
 *             exceeds the CTAs that fit on the GPU at once.
 * tile_s, block_d, buffer_num, staging, signals: PC only (see
 *             all2all_pc_workspace; staging and signals are symmetric
 *             pointers of at least those sizes); ignored by DIRECT.
 * elem_bytes  any size >= 1; values move as raw bits.
 * S, H or D = 0 is a no-op.  Errors: SYMM_EINVAL, SYMM_ECUDA; a PC wait that
 * gives up shows in symm_check_error(). */
int all2all_combine(symm_heap_t *heap, const void *in, void *out, int W, int S, int H, int D,
                    int elem_bytes, int variant, int tile_s, int block_d, int buffer_num,
                    void *staging, int64_t *signals, void *stream);

/* [RA2A] "Reverse All2All Operator Semantics" / "EP MoE Scenario": Forward
 * All2All (dispatch).  Per PE (S, H, D) becomes (S/W, H*W, D):
 *     out_d[s', r*H + h, x] = in_r[d*S' + s', h, x],   S' = S/W.
 * S % W != 0 is SYMM_EINVAL.  Same pointer rules as all2all_combine. */
int all2all_dispatch(symm_heap_t *heap, const void *in, void *out, int W, int S, int H, int D,
                     int elem_bytes, void *stream);

/* Inverse of all2all_dispatch (results returned to the tokens' ranks,
 * [RA2A] introduction).  Per PE (Sp, H*W, D) becomes (Sp*W, H, D):
 *     out_r[d*Sp + s', h, x] = in_d[s', r*H + h, x]. */
int all2all_combine_back(symm_heap_t *heap, const void *in, void *out, int W, int Sp, int H,
                         int D, int elem_bytes, void *stream);

/* all2all_combine on host buffers: host_in ([W][S*W][H][D], contiguous) in,
 * host_out ([W][S][H*W][D]) out.  For the direct variant with both buffers
 * page-locked and mapped (cudaHostAlloc / torch pin_memory), each lying in
 * one allocation, the combine kernel reads and writes them in place over
 * the host link; `in`, `out`, staging and signals are then not used.
 * Otherwise `in` and `out` (symmetric, S*W rows per PE each) are device
 * space, and for S >= 16 the work is pipelined in 8
 * chunks of S rows: each chunk's input rows are gathered into a compact
 * buffer at the start of `in` (one 2-D copy per PE), combined into a buffer
 * at the start of `out`, and copied out (one copy per PE), with two buffers
 * alternating and the copies on two streams of the library's own, so that
 * copies in, the combine and copies out of neighbouring chunks overlap.
 * The caller's `stream` runs the combines and waits for the last copies, so
 * work enqueued on it afterwards sees host_out complete.  After the call
 * the device objects hold chunk buffers, not the whole input and output.
 * Smaller S: one copy per slab and direction on `stream`.  Page-locked host
 * buffers make the copies asynchronous.  Calls from several host threads
 * are serialised while they enqueue.  Returns once enqueued. */
int all2all_combine_host(symm_heap_t *heap, const void *host_in, void *host_out, const void *in,
                         void *out, int W, int S, int H, int D, int elem_bytes, int variant,
                         int tile_s, int block_d, int buffer_num, void *staging, int64_t *signals,
                         void *stream);

/* ------------------------------------------------- two-phase combine -- */

/* Workspace of all2all_combine_two_phase, per PE (allocate each with
 * symm_malloc):
 *   bulk    W rank slots of [S][H][D] (= the input's bytes);
 *   signals region A, nbs*W slots (nbs = ceil(S / tile_s)), then region B,
 *           buffer_num * nbd * H slots (nbd = ceil(D / block_d)), each slot
 *           SYMM_SIGNAL_STRIDE_BYTES apart.
 * block_d = 0 means D.  Errors: SYMM_EINVAL. */
int all2all_two_phase_workspace(int W, int S, int H, int D, int elem_bytes, int tile_s,
                                int block_d, int buffer_num, size_t *bulk_bytes,
                                size_t *signal_bytes);

/* [Reverse All2All (EP MoE Distributed Kernel), "UDMA Optimized
 * Implementation" with its "Wait/Notify Optimization"]  The same combine as
 * all2all_combine (out_d[s, r*H + h, x] = in_r[d*S + s, h, x]), in two phases:
 *   phase 1  for every r != d, PE r's rows d*S .. d*S + S - 1 are sent in bulk
 *            (S block by S block) to rank slot r of PE d's `bulk`, and each
 *            arrived S block sets its region-A slot (b, r) of PE d to 1 once;
 *   phase 2  PE d's own rows d*S .. go tile by tile (tile_s rows, block_d
 *            elements) through the double buffer at the start of rank slot d
 *            (buffer_num buffers), handshaking on region B (wait 0, write,
 *            set 1; the consumer resets 0 after reading);
 *   consumer PE d copies every tile from rank slot r (r != d) or from the
 *            double buffer (r == d) into out_d.
 * All W PEs run in one cooperative launch (preceded by an in-stream reset of
 * the signals).  On return (in stream order), region A of every PE holds 1
 * for each (block, r != d) and 0 for r == d, region B is all 0, and the bulk
 * slots r != d hold the senders' segments.
 * in, out: as for all2all_combine.  bulk, signals: from
 * all2all_two_phase_workspace; no two of in/out/bulk/signals may overlap.
 * Bulk (TMA) copies are used when H*D*elem_bytes and the in and bulk offsets
 * are multiples of 16 bytes, 16-byte vector copies otherwise.
 * Errors: SYMM_EINVAL (shapes, ranges, W != npes), SYMM_ECUDA (launch,
 * including a grid the device cannot keep resident); a wait that gives up
 * is reported by symm_check_error() as SYMM_ETIMEDOUT. */
int all2all_combine_two_phase(symm_heap_t *heap, const void *in, void *out, int W, int S, int H,
                              int D, int elem_bytes, int tile_s, int block_d, int buffer_num,
                              void *bulk, int64_t *signals, void *stream);

/* --------------------------------------------------------- collectives -- */

/* Bytes of device workspace (plain device memory, 8-byte aligned; no need to
 * be symmetric) that shmem_alltoall and shmem_allgather need for W PEs:
 * offsets, per-segment completion counters and a validity word.
 * Errors: SYMM_EINVAL (W outside [1, 4096]). */
int shmem_collective_workspace(int W, size_t *bytes);

/* [RFC] 10 (AllToAll, push mode): every PE r sends counts[r*W + d] rows of
 * row_bytes to every PE d.  PE r's input (symmetric, in_rows rows) holds its
 * rows for d = 0, 1, ... back to back; PE d's output (symmetric, out_rows
 * rows) receives the rows of r = 0, 1, ... back to back; output rows past
 * what PE d receives are not written.
 * counts      device; W*W int64, read by the kernels (the host never
 *             synchronises to learn them).  A negative count, a PE sending
 *             more than in_rows or receiving more than out_rows rows is
 *             found on the device: nothing is copied and symm_check_error()
 *             reports SYMM_ERANGE.
 * workspace   device; shmem_collective_workspace(W) bytes.
 * signals     symmetric int64 (one per PE): zeroed, then ADDed to (release)
 *             once per completed (r, d) segment; the call ends with every
 *             PE's wait for the value W, so on return (in stream order) the
 *             output is complete.
 * Errors: SYMM_EINVAL, SYMM_ECUDA; later SYMM_ERANGE/SYMM_ETIMEDOUT via
 * symm_check_error(). */
int shmem_alltoall(symm_heap_t *heap, const void *in, void *out, const int64_t *counts, int W,
                   size_t row_bytes, size_t in_rows, size_t out_rows, void *workspace,
                   int64_t *signals, void *stream);

/* [RFC] 10 (AllGather, push mode): every PE r pushes its `bytes` (symmetric
 * `in`) to byte r*bytes of every PE's symmetric `out` (W*bytes per PE) and
 * ADDs 1 to that PE's signal; the call ends with every PE waiting for W.
 * workspace and signals as for shmem_alltoall.  Any alignment.
 * Errors: SYMM_EINVAL, SYMM_ECUDA; later SYMM_ETIMEDOUT via symm_check_error(). */
int shmem_allgather(symm_heap_t *heap, const void *in, void *out, int W, size_t bytes,
                    void *workspace, int64_t *signals, void *stream);

/* ------------------------------------------ fused AllGather + MatMul -- */

#define SYMM_DTYPE_F16 0
#define SYMM_DTYPE_BF16 1

/* Signal object of shmem_fused_all_gather_matmul, per PE (allocate with
 * symm_malloc): W * m_local / block_size slots SYMM_SIGNAL_STRIDE_BYTES
 * apart, followed by as many 8-byte counters (used on PE 0).  Errors:
 * SYMM_EINVAL (shapes as for the call). */
int shmem_fused_ag_matmul_workspace(int W, int m_local, int k, int n, int block_size,
                                    size_t *signal_bytes);

/* [RFC] 10 (fused_all_gather_matmul) and its example 2: every PE r holds a_r
 * (m_local x k) and b_r (k x n), row-major, elements of `dtype`
 * (SYMM_DTYPE_F16 or SYMM_DTYPE_BF16).  Computes, on every PE d,
 *   gather_out_d = [a_0; a_1; ...; a_(W-1)]     (m_total x k, m_total = W*m_local)
 *   c_d          = gather_out_d @ b_d           (m_total x n)
 * with fp32 accumulation on the tensor cores and c rounded to `dtype`.  The
 * rows are pushed in blocks of block_size rows; each block's signal slot
 * (source r, block j) on PE d is set to 1 when it has arrived, and the
 * matmul of the rows of that block starts as soon as its slot is set.  All W
 * PEs run in one cooperative launch, preceded by an in-stream reset of the
 * signals.
 * Shapes: block_size must be 128 and m_local a multiple of it; k and n
 * multiples of 8, at least 8.  a, b, c, gather_out, signals: symmetric
 * objects, 16-byte aligned, pairwise disjoint; signals sized by
 * shmem_fused_ag_matmul_workspace.
 * Errors: SYMM_EINVAL (shapes, ranges, W != npes), SYMM_ECUDA (launch or
 * tensor-map set-up); a wait that gives up is reported by symm_check_error()
 * as SYMM_ETIMEDOUT. */
int shmem_fused_all_gather_matmul(symm_heap_t *heap, const void *a, const void *b, void *c,
                                  void *gather_out, int W, int m_local, int k, int n, int dtype,
                                  int block_size, int64_t *signals, void *stream);

/* ------------------------------------------- allocation-free variant -- */

/* Size of the library's own static device array used by
 * all2all_combine_pc_noalloc (32 MiB, held on every GPU that loads the
 * library until the process exits). */
#define SYMM_NOALLOC_SCRATCH_BYTES (32u << 20)

/* No counterpart on the pages: an addition for callers that cannot allocate
 * device memory -- code whose device memory is all handed out beforehand by
 * another allocator, or a hot path that must not pay the device-wide
 * synchronisation of cudaMalloc/cudaFree -- but still want the staged,
 * signalled combine.  Same operation and arguments as
 * all2all_combine(SYMM_A2A_PC) except that the staging ring and the signal
 * slots live in the library's static SYMM_NOALLOC_SCRATCH_BYTES array
 * instead of the caller's heap; the caller passes only the symmetric input
 * and output.  It runs the same kernels as all2all_combine(SYMM_A2A_PC) and
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Needs W * (roundup256(buffer_num*tile_s*H*W*D*elem_bytes) +
 *    roundup256(buffer_num*W*nbd*H*64)) bytes of scratch; larger requests
 *    return SYMM_EINVAL before launching anything.
 *  - Each call zeroes its signal slots in the array first (the array keeps
 *    the last call's contents).  All calls share the one array per device:
 *    calls that overlap on the GPU (other streams, other threads, other
 *    heaps) race and give undefined output; order them on one stream.
 *  - The array's device address is looked up (cudaGetSymbolAddress, with the
 *    device current) and cached once per device.  symm_heap_init does this
 *    for the device current at init, which also loads the part of the
 *    library that holds the array: that is when CUDA reserves the array's
 *    memory, so a device without 32 MiB free fails there, not here.  On any
 *    other device the first call does the look-up itself; make that call
 *    before any stream capture.
 * Errors: SYMM_EINVAL, SYMM_ECUDA; a wait that gives up shows in
 * symm_check_error(), with *info = SYMM_INFO_NOALLOC_SIGNAL + the offset of
 * the slot in the array's signal area. */
int all2all_combine_pc_noalloc(symm_heap_t *heap, const void *in, void *out, int W, int S, int H,
                               int D, int elem_bytes, int tile_s, int block_d, int buffer_num,
                               void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SYMM_A2A_H */
