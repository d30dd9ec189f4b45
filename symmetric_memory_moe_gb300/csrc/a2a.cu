// a2a.cu -- the EP-MoE all-to-all permutations on the emulated symmetric heap.
//
// Source: "Reverse All2All (EP MoE Distributed Kernel)".
//  * "Reverse All2All Operator Semantics": combine turns each PE's
//    (S*W, H, D) into (S, H*W, D); dispatch turns (S, H, D) into
//    (S/W, H*W, D).  Element placement (section "MTE Implementation"):
//        out_d[s, r*H + h, x] = in_r[d*S + s, h, x].
//  * "MTE Implementation": the producer/consumer pipeline -- producers of
//    source PE r copy a tile (COMM_BLOCK_S rows x COMM_BLOCK_D columns of one
//    expert column h) of the rows bound for destination t into t's staging
//    slot [buffer][row][r*H + h][d-block] after waiting for the slot's signal
//    to read 0, fence, and set it to 1; consumers of t wait for 1, copy the
//    staged tile into output column r*H + h, fence, and set it back to 0.
//    Double buffering over S blocks (buffer_num = 2), per-task signal slots
//    spaced 8 int64 apart, masks for ragged S and D.
//
// GB300 design (what differs from the page, and why):
//  * All W PEs run in ONE launch (one GPU holds every slab).  Each CTA is
//    warp-specialised: warps 0-3 are a producer group, warps 4-7 a consumer
//    group, each synchronised by its own named barrier.  The grid is capped at
//    the CTAs that are resident at once, so every spin can be satisfied.
//  * A task (destination d, source r, expert h, D block) is one signal slot;
//    like the page's cores, each CTA owns a fixed set of tasks and walks each
//    task's S blocks in order (task by task, where the page's cores go S
//    block by S block), its consumer group consuming exactly the tiles its
//    own producer group staged.  Every wait is thus satisfied by the same
//    CTA, and successive producers of a slot are ordered.  The page's target
//    rotation (rank + i) % W staggers one PE's producers across
//    destinations; here every (r, d) pair is in flight at once, so it has
//    nothing left to stagger.
//  * Copies move 16-byte vectors per lane (funnel-shifted when source and
//    destination disagree mod 16) instead of masked 2-D tile loads; ragged
//    S and D blocks are bounds in the row loop and the byte count.
//  * The direct variant is one pass with no staging: every contiguous run of
//    H*D elements (fixed r, d, s) is copied once, the minimum traffic.
#include <stdio.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

namespace {

// Tuning knobs (compile-time): 16-byte vectors in flight per lane, and the
// minimum resident CTAs per SM that register allocation must allow.
// Run copies: layouts whose runs are all 16-byte aligned use the aligned
// copy with SYMM_RUNS_UNROLL vectors in flight per lane; any other layout
// uses the general copy (head/tail bytes, shift-merge) with fewer vectors in
// flight and more resident warps, which measured faster there.
#ifndef SYMM_RUNS_UNROLL
#define SYMM_RUNS_UNROLL 16
#endif
#ifndef SYMM_RUNS_MIN_BLOCKS
#define SYMM_RUNS_MIN_BLOCKS 2
#endif
#ifndef SYMM_RUNS_GENERAL_UNROLL
#define SYMM_RUNS_GENERAL_UNROLL 3
#endif
#ifndef SYMM_RUNS_GENERAL_MIN_BLOCKS
#define SYMM_RUNS_GENERAL_MIN_BLOCKS 6
#endif
// 16-byte vectors in flight per lane in the row-by-row producer/consumer
// copies (rows whose staging stride is not a multiple of 16 bytes); 2 fits
// the register budget of 3 CTAs per SM without spills
#ifndef SYMM_PC_UNROLL
#define SYMM_PC_UNROLL 2
#endif
// 16-byte vectors in flight per thread in the producer/consumer tile copies
// that spread a whole tile over the group (tiles with 16-byte-aligned rows)
#ifndef SYMM_PC_FLAT_UNROLL
#define SYMM_PC_FLAT_UNROLL 4
#endif
// 16-byte vectors in flight per thread in the tile copies for rows of any
// alignment (two aligned source blocks per output vector)
#ifndef SYMM_PC_ANY_UNROLL
#define SYMM_PC_ANY_UNROLL 4
#endif
#ifndef SYMM_PC_MIN_BLOCKS
#define SYMM_PC_MIN_BLOCKS 3
#endif

constexpr int kRunThreads = 256;
constexpr int kPcThreads = 256;  // 4 producer warps + 4 consumer warps
constexpr int kPcGroup = 128;
constexpr int kPcMinBlocks = SYMM_PC_MIN_BLOCKS;
// a2a_pc_kernel's residency for its kCopyRows and kCopyAligned instances
// (kCopyAny keeps kPcMinBlocks: its shift-merge spills at 64 registers).
// Four CTAs per SM give a CTA to each of the small shape's 512 tasks.
#ifndef SYMM_PC_KERNEL_MIN_BLOCKS
#define SYMM_PC_KERNEL_MIN_BLOCKS 4
#endif

// --------------------------------------------------------------- direct ---
// One warp per run of R = H*D*elem_bytes contiguous bytes, destination-major.
// INVERSE = false (combine, dispatch with Sb = S/W):
//   run k = (d*Sb + s)*W + r : in slab r row d*Sb + s  ->  out slab d row s*W + r
// INVERSE = true (combine_back):
//   run k = (r*W + d)*Sb + s : in slab d row s*W + r   ->  out slab r row d*Sb + s
// (a "row" here is one run of R bytes).
template <bool INVERSE, bool ALIGNED>
__global__ void __launch_bounds__(kRunThreads,
                                  ALIGNED ? SYMM_RUNS_MIN_BLOCKS : SYMM_RUNS_GENERAL_MIN_BLOCKS)
    a2a_runs_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, size_t in_pe,
                    size_t out_pe, uint32_t W, uint32_t Sb, size_t R, uint32_t nruns) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * kRunThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kRunThreads) >> 5;
  for (uint32_t k = warp; k < nruns; k += nwarps) {
    const uint8_t* src;
    uint8_t* dst;
    if (!INVERSE) {
      const uint32_t r = k % W, t = k / W, s = t % Sb, d = t / Sb;
      src = in + r * in_pe + (size_t)(d * Sb + s) * R;
      dst = out + d * out_pe + (size_t)(s * W + r) * R;
    } else {
      const uint32_t s = k % Sb, t = k / Sb, d = t % W, r = t / W;
      src = in + d * in_pe + (size_t)(s * W + r) * R;
      dst = out + r * out_pe + (size_t)(d * Sb + s) * R;
    }
    if (ALIGNED)
      symm::warp_copy_aligned<SYMM_RUNS_UNROLL, symm::kRO, symm::kCS>(dst, src, R >> 4, lane);
    else
      symm::warp_copy<SYMM_RUNS_GENERAL_UNROLL, symm::kRO, symm::kCS, SYMM_RUNS_GENERAL_UNROLL>(
          dst, src, R, lane);
  }
}

// --------------------------------------------------- direct, short runs ---
// The same permutation for runs of at most kBatchMaxVec 16-byte vectors
// (16-byte aligned): one warp per run would keep only a few vectors in
// flight per lane and pay a whole memory round trip per run.  Consecutive
// runs of a period are linear in one index -- the source PE r for the
// combine and dispatch (period W: run k = (d*Sb + s)*W + r, sources in_pe
// apart, destinations R apart), the row s for the inverse (period Sb: run
// k = (r*W + d)*Sb + s, sources W*R apart, destinations R apart) -- so a
// warp copies a batch of m of them as one tile of m rows, kBatchUnroll
// vectors in flight per lane.  Batches never cross a period.
#ifndef SYMM_RUNS_BATCH_UNROLL
#define SYMM_RUNS_BATCH_UNROLL 8
#endif
#ifndef SYMM_RUNS_BATCH_MIN_BLOCKS
#define SYMM_RUNS_BATCH_MIN_BLOCKS 4
#endif
constexpr int kBatchUnroll = SYMM_RUNS_BATCH_UNROLL;
constexpr uint32_t kBatchMaxVec = 256;  // runs of at most 4 KB take the batches
template <bool INVERSE>
__global__ void __launch_bounds__(kRunThreads, SYMM_RUNS_BATCH_MIN_BLOCKS)
    a2a_runs_batch_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, size_t in_pe,
                          size_t out_pe, uint32_t W, uint32_t Sb, uint32_t R, uint32_t nruns,
                          uint32_t m) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * kRunThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kRunThreads) >> 5;
  const uint32_t P = INVERSE ? Sb : W;  // runs per period
  const uint32_t nbp = (P + m - 1) / m;  // batches per period
  const uint32_t nbatch = nruns / P * nbp;
  const uint32_t nvec = R >> 4;
  const symm::TileStep step = symm::tile_step(32, nvec);
  const uint32_t i0 = (uint32_t)lane / nvec, c0 = (uint32_t)lane - i0 * nvec;
  for (uint32_t bi = warp; bi < nbatch; bi += nwarps) {
    const uint32_t pi = bi / nbp, j0 = (bi - pi * nbp) * m;  // period, its first run
    const uint32_t rows = min(m, P - j0);
    const uint8_t* src;
    uint8_t* dst;
    size_t sstride;
    if (!INVERSE) {
      const uint32_t s = pi % Sb, d = pi / Sb;
      src = in + j0 * in_pe + (size_t)(d * Sb + s) * R;
      dst = out + d * out_pe + (size_t)(s * W + j0) * R;
      sstride = in_pe;
    } else {
      const uint32_t d = pi % W, r = pi / W;
      src = in + d * in_pe + (size_t)(j0 * W + r) * R;
      dst = out + r * out_pe + (size_t)(d * Sb + j0) * R;
      sstride = (size_t)W * R;
    }
    const uint32_t nv = rows * nvec;
    uint32_t i = i0, c = c0;
    for (uint32_t v0 = 0; v0 < nv; v0 += 32 * kBatchUnroll) {
      uint4 x[kBatchUnroll];
      uint32_t doff[kBatchUnroll];
#pragma unroll
      for (int u = 0; u < kBatchUnroll; ++u) {
        doff[u] = i * R + 16 * c;
        if (v0 + 32 * u + lane < nv) x[u] = symm::ld16_ro(src + i * sstride + 16 * c);
        step.advance(i, c, nvec);
      }
#pragma unroll
      for (int u = 0; u < kBatchUnroll; ++u)
        if (v0 + 32 * u + lane < nv) symm::st16_cs(dst + doff[u], x[u]);
    }
  }
}

// ----------------------------------------------- direct, unaligned runs ---
// Runs that are not 16-byte aligned, up to a slot: the general instance
// above keeps only a few vectors in flight in registers and is bound by
// memory latency.  Here each warp streams its runs (or batches of short
// runs, below) through its own ring of kRingSlots shared-memory slots: lane
// 0 loads the 16-byte-aligned block range covering a unit with one bulk (TMA)
// copy (at most 15 bytes on either side, inside the granules of the unit's
// first and last bytes), completing on the slot's mbarrier; the warp
// then funnel-shifts the slot into aligned 16-byte stores (byte heads and
// tails) and lane 0 reloads the slot with the unit kRingSlots ahead.  Device
// memory only.  Shared memory bounds the residency, so CTAs are small (4
// warps of 2 slots: 28 warps on an SM for the tail shape's 4 KB runs).
#ifndef SYMM_RUNS_RING
#define SYMM_RUNS_RING 1
#endif
#ifndef SYMM_RING_WARPS
#define SYMM_RING_WARPS 4
#endif
#ifndef SYMM_RING_SLOTS
#define SYMM_RING_SLOTS 2
#endif
#ifndef SYMM_RING_UNROLL
#define SYMM_RING_UNROLL 2
#endif
#ifndef SYMM_RING_ORDER  // 0: consecutive warps write consecutive runs; 1: read them
#define SYMM_RING_ORDER 0
#endif
constexpr int kRingWarps = SYMM_RING_WARPS;
constexpr int kRingSlots = SYMM_RING_SLOTS;
constexpr int kRingUnroll = SYMM_RING_UNROLL;
#ifndef SYMM_RING_MIN_RUN
#define SYMM_RING_MIN_RUN 1536
#endif
constexpr uint32_t kRingMinRun = SYMM_RING_MIN_RUN;
// kRingWarps x kRingSlots mbarriers, rounded up to 128 bytes
constexpr uint32_t kRingHeader = (8u * kRingWarps * kRingSlots + 127u) & ~127u;
// the largest slot: 8 KB, or what fits 227 KB of shared memory
constexpr uint32_t kRingMaxSlot =
    ((232448u - kRingHeader) / (kRingWarps * kRingSlots) & ~15u) < 8192u
        ? ((232448u - kRingHeader) / (kRingWarps * kRingSlots) & ~15u)
        : 8192u;
// Bytes of a batch of short runs, at most, by run length: large runs gain
// from large bulk copies, short ones (more byte edges and index work per
// byte in the copy-out) from the residency of smaller slots.
#ifndef SYMM_RING_BATCH_BYTES
#define SYMM_RING_BATCH_BYTES 8160
#endif
constexpr uint32_t kRingBatchBytes = SYMM_RING_BATCH_BYTES;  // runs of 384 bytes and up
constexpr uint32_t kRingMidBatchBytes = 6144;                // 32 to 383 bytes
constexpr uint32_t kRingTinyBatchBytes = 2048;               // under 32 bytes
static_assert(kRingBatchBytes + 30 <= kRingMaxSlot, "a batch's covering range fits a slot");
// MODE kRingPerRun: a unit is one run, in a2a_runs_kernel's order.  Runs
// shorter than kRingMinRun travel in batches of up to `mb` runs that are
// consecutive in the input (one input PE's rows: the combine's source r, the
// inverse's destination d; a batch ends with that PE's runs), one bulk copy
// per batch.  kRingBatchWarp: the whole warp writes the batch's runs one
// after another (runs of 512 bytes and up); kRingBatchGroups: groups of
// `glanes` lanes (8 or 16) write one run each.
// (One instance per way of writing: sharing one, each slowed the other.)
enum { kRingPerRun = 0, kRingBatchWarp = 1, kRingBatchGroups = 2 };
template <bool INVERSE, int MODE>
__global__ void __launch_bounds__(32 * kRingWarps)
    a2a_runs_ring_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, size_t in_pe,
                         size_t out_pe, uint32_t W, uint32_t Sb, uint32_t R, uint32_t nunits,
                         uint32_t mb, uint32_t nbp, uint32_t glanes, uint32_t slot_bytes,
                         uint64_t budget_ns, Control* ctl) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem) + wib * kRingSlots;
  uint8_t* ring = smem + kRingHeader + (size_t)wib * kRingSlots * slot_bytes;
  const uint32_t warp = blockIdx.x * kRingWarps + wib;
  const uint32_t nwarps = gridDim.x * kRingWarps;
  const uint32_t period = W * Sb;  // runs of one input PE
  // run (r, s, d) -> its source and destination
  auto ends = [&](uint32_t r, uint32_t s, uint32_t d, const uint8_t** src, uint8_t** dst) {
    if (!INVERSE) {
      *src = in + r * in_pe + (size_t)(d * Sb + s) * R;
      *dst = out + d * out_pe + (size_t)(s * W + r) * R;
    } else {
      *src = in + d * in_pe + (size_t)(s * W + r) * R;
      *dst = out + r * out_pe + (size_t)(d * Sb + s) * R;
    }
  };
  // unit u -> source of its first run and its run count
  auto unit_at = [&](uint32_t u, const uint8_t** src, uint8_t** dst, uint32_t* cnt) {
    if (MODE != kRingPerRun) {
      // run t of input PE p (its runs in input order: the combine's
      // t = d*Sb + s of source p, the inverse's t = s*W + r of destination p)
      // starts at in + p*in_pe + t*R
      // whole-warp batches: unit u is batch u / W of PE u % W, so output runs
      // that share a boundary sector (same d and s, next r) are written by
      // warps at work at the same time; lane-group batches: batch u % nbp of
      // PE u / nbp, consecutive warps reading consecutive input
      const uint32_t p = MODE == kRingBatchWarp ? u % W : u / nbp;
      const uint32_t t0 = (MODE == kRingBatchWarp ? u / W : u % nbp) * mb;
      *cnt = min(mb, period - t0);
      *src = in + p * in_pe + (size_t)t0 * R;
      *dst = nullptr;  // each run's own, in the copy-out
    } else {
      const bool r_fastest = (SYMM_RING_ORDER == 0) != INVERSE;
      uint32_t r, s, d;
      if (r_fastest) {
        r = u % W;
        const uint32_t t = u / W;
        s = t % Sb;
        d = t / Sb;
      } else {
        s = u % Sb;
        const uint32_t t = u / Sb;
        d = t % W;
        r = t / W;
      }
      ends(r, s, d, src, dst);
      *cnt = 1;
    }
  };
  auto load = [&](uint32_t u, int slot) {  // lane 0: unit u's covering range into `slot`
    const uint8_t* src;
    uint8_t* dst;
    uint32_t cnt;
    unit_at(u, &src, &dst, &cnt);
    const uintptr_t lo = (uintptr_t)src & ~(uintptr_t)15;
    const uint32_t n =
        (uint32_t)((((uintptr_t)src + (size_t)cnt * R + 15) & ~(uintptr_t)15) - lo);
    symm::mbar_arrive_expect_tx(&full[slot], n);
    symm::bulk_load(ring + (size_t)slot * slot_bytes, reinterpret_cast<const void*>(lo), n,
                    &full[slot]);
  };
  // one run: slot bytes [q0, q0 + R) to dst, by the G lanes gl = 0..G-1
  // (whole: G = 32, more lanes than head or tail bytes)
  auto copy_run = [&](const uint8_t* sl, uint32_t q0, uint8_t* dst, uint32_t gl, uint32_t G,
                      bool whole) {
    uint32_t head = (uint32_t)((16 - ((uintptr_t)dst & 15)) & 15);
    if (head > R) head = R;
    const uint32_t nvec = (R - head) >> 4, tail = R - head - (nvec << 4);
#pragma unroll kRingUnroll
    for (uint32_t c = gl; c < nvec; c += G) {
      const uint32_t q = q0 + head + 16 * c;
      const uint8_t* p = sl + (q & ~15u);
      uint4 x = *reinterpret_cast<const uint4*>(p);
      if (q & 15) x = symm::funnel16(x, *reinterpret_cast<const uint4*>(p + 16), q & 15);
      symm::st16_cs(dst + head + 16 * c, x);
    }
    if (whole) {  // G = 32 > 15 >= head, tail
      if (gl < head) symm::st1(dst + gl, sl[q0 + gl]);
      if (gl < tail) symm::st1(dst + head + (nvec << 4) + gl, sl[q0 + head + (nvec << 4) + gl]);
    } else {
      for (uint32_t b = gl; b < head; b += G) symm::st1(dst + b, sl[q0 + b]);
      for (uint32_t b = gl; b < tail; b += G) {
        const uint32_t x = head + (nvec << 4) + b;
        symm::st1(dst + x, sl[q0 + x]);
      }
    }
  };
  if (lane == 0) {
    for (int i = 0; i < kRingSlots; ++i) symm::mbar_init(&full[i], 1);
    symm::fence_mbar_init();
    for (int i = 0; i < kRingSlots; ++i)
      if (warp + (uint64_t)i * nwarps < nunits) load(warp + i * nwarps, i);
  }
  __syncwarp();
  uint32_t it = 0;
  for (uint32_t u = warp; u < nunits; u += nwarps, ++it) {
    const int slot = (int)(it % kRingSlots);
    int ok = 1;
    if (lane == 0) ok = symm::mbar_wait(&full[slot], (it / kRingSlots) & 1u, budget_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // lane 0 saw the slot land; the others read it after this
    if (!ok) {
      if (lane == 0) {
        symm::record_error(ctl, symm::kErrTimedOut, -1);
        // let this warp's loads still in flight land before it leaves (bounded)
        for (uint32_t j = 0; j < (uint32_t)kRingSlots && u + (uint64_t)j * nwarps < nunits; ++j)
          symm::mbar_wait(&full[(it + j) % kRingSlots], ((it + j) / kRingSlots) & 1u, budget_ns);
      }
      return;  // uniform across the warp
    }
    symm::mbar_try_wait(&full[slot], (it / kRingSlots) & 1u);  // every lane observes the phase
    const uint8_t* src;
    uint8_t* dst;
    uint32_t cnt;
    unit_at(u, &src, &dst, &cnt);
    const uint8_t* sl = ring + (size_t)slot * slot_bytes;
    const uint32_t m0 = (uint32_t)((uintptr_t)src & 15);  // the unit's first byte in the slot
    if (MODE == kRingPerRun) {
      copy_run(sl, m0, dst, (uint32_t)lane, 32, true);
    } else {
      const uint32_t p = MODE == kRingBatchWarp ? u % W : u / nbp;
      const uint32_t t0 = (MODE == kRingBatchWarp ? u / W : u % nbp) * mb;
      const uint32_t gl = (uint32_t)lane % glanes, groups = 32 / glanes;
      uint32_t j = (uint32_t)lane / glanes;
      if (MODE == kRingBatchWarp) {
        for (; j < cnt; j += groups) {
          const uint8_t* sj;
          uint8_t* dj;
          const uint32_t t = t0 + j;
          if (!INVERSE)
            ends(p, t % Sb, t / Sb, &sj, &dj);  // p = r, t = d*Sb + s
          else
            ends(t % W, t / W, p, &sj, &dj);  // p = d, t = s*W + r
          copy_run(sl, m0 + j * R, dj, gl, glanes, false);
        }
      } else {
        // run t = hi * L + lo: the combine's (d, s), the inverse's (s, r); a
        // cursor per lane group steps `groups` runs without dividing
        const uint32_t L = INVERSE ? W : Sb;
        uint32_t hi = (t0 + j) / L, lo = (t0 + j) - hi * L;
        for (; j < cnt; j += groups) {
          uint8_t* dj = INVERSE ? out + lo * out_pe + (size_t)(p * Sb + hi) * R
                                : out + hi * out_pe + (size_t)(lo * W + p) * R;
          copy_run(sl, m0 + j * R, dj, gl, glanes, false);
          lo += groups;
          while (lo >= L) {
            lo -= L;
            ++hi;
          }
        }
      }
    }
    __syncwarp();  // every lane has read the slot
    if (lane == 0 && u + (uint64_t)kRingSlots * nwarps < nunits) {
      symm::fence_proxy_async_shared();  // those reads precede the reload
      load(u + kRingSlots * nwarps, slot);
    }
  }
}

// ------------------------------------------------------ direct, bulk ---
// The same run permutation moved by the Tensor Memory Accelerator: one thread
// per CTA streams units (runs cut into <= kBulkChunk-byte pieces) through a
// ring of kBulkStages shared-memory buffers -- a bulk load global->shared
// completing on the stage's mbarrier, then a bulk store shared->global --
// keeping kBulkStages loads in flight without holding data in registers.
// Needs 16-byte-aligned runs (R % 16 == 0, 16-byte-aligned bases).
#ifndef SYMM_BULK_STAGES
#define SYMM_BULK_STAGES 4
#endif
#ifndef SYMM_BULK_CHUNK
#define SYMM_BULK_CHUNK 16384
#endif
constexpr int kBulkStages = SYMM_BULK_STAGES;
constexpr uint32_t kBulkChunk = SYMM_BULK_CHUNK;
constexpr size_t kBulkSmem = 128 + (size_t)kBulkStages * kBulkChunk;

template <bool INVERSE>
__device__ __forceinline__ void run_unit(const uint8_t* in, uint8_t* out, size_t slab, uint32_t W,
                                         uint32_t Sb, size_t R, uint32_t nchunks, uint64_t u,
                                         const uint8_t** src, uint8_t** dst, uint32_t* len) {
  const uint32_t k = (uint32_t)(u / nchunks), c = (uint32_t)(u % nchunks);
  const size_t off = (size_t)c * kBulkChunk;
  if (!INVERSE) {
    const uint32_t r = k % W, t = k / W, s = t % Sb, d = t / Sb;
    *src = in + r * slab + (size_t)(d * Sb + s) * R + off;
    *dst = out + d * slab + (size_t)(s * W + r) * R + off;
  } else {
    const uint32_t s = k % Sb, t = k / Sb, d = t % W, r = t / W;
    *src = in + d * slab + (size_t)(s * W + r) * R + off;
    *dst = out + r * slab + (size_t)(d * Sb + s) * R + off;
  }
  *len = (uint32_t)(R - off < kBulkChunk ? R - off : kBulkChunk);
}

template <bool INVERSE>
__global__ void __launch_bounds__(32)
    a2a_runs_bulk_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, size_t slab,
                         uint32_t W, uint32_t Sb, size_t R, uint32_t nruns, uint32_t nchunks,
                         uint64_t budget_ns, Control* ctl) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint8_t* buf = smem + 128;
  if (threadIdx.x != 0) return;
  for (int st = 0; st < kBulkStages; ++st) symm::mbar_init(&bar[st], 1);
  symm::fence_mbar_init();
  const uint64_t units = (uint64_t)nruns * nchunks;
  const uint64_t mine = units > blockIdx.x ? (units - blockIdx.x - 1) / gridDim.x + 1 : 0;
  const uint8_t* src;
  uint8_t* dst;
  uint32_t len;
  uint64_t issued = 0;
  for (; issued < mine && issued < (uint64_t)kBulkStages; ++issued) {
    run_unit<INVERSE>(in, out, slab, W, Sb, R, nchunks, blockIdx.x + issued * gridDim.x, &src,
                      &dst, &len);
    symm::mbar_arrive_expect_tx(&bar[issued], len);
    symm::bulk_load(buf + issued * kBulkChunk, src, len, &bar[issued]);
  }
  uint64_t i = 0;
  for (; i < mine; ++i) {
    const int st = (int)(i % kBulkStages);
    if (!symm::mbar_wait(&bar[st], (uint32_t)(i / kBulkStages) & 1u, budget_ns)) {
      symm::record_error(ctl, symm::kErrTimedOut, -1);
      break;
    }
    run_unit<INVERSE>(in, out, slab, W, Sb, R, nchunks, blockIdx.x + i * gridDim.x, &src, &dst,
                      &len);
    symm::bulk_store(dst, buf + (size_t)st * kBulkChunk, len);
    symm::bulk_commit();
    if (issued < mine) {  // refill this stage once the store has read it
      symm::bulk_wait_read<0>();
      run_unit<INVERSE>(in, out, slab, W, Sb, R, nchunks, blockIdx.x + issued * gridDim.x, &src,
                        &dst, &len);
      symm::mbar_arrive_expect_tx(&bar[st], len);
      symm::bulk_load(buf + (size_t)st * kBulkChunk, src, len, &bar[st]);
      ++issued;
    }
  }
  // after a give-up, let the loads still in flight land (again bounded)
  for (; i < issued; ++i)
    symm::mbar_wait(&bar[i % kBulkStages], (uint32_t)(i / kBulkStages) & 1u, budget_ns);
  symm::bulk_wait<0>();
}

// ------------------------------------------------ producer / consumer ---
// The staging ring and the signal slots of PE k sit at staging + k*stage_pe
// and signals + k*sig_pe: in the destination slab of the symmetric heap
// (stride = the slab), or in any other device array laid out per PE.
struct PcArgs {
  const uint8_t* in;  // PE 0's input and output; PE k's at +k*slab
  uint8_t* out;
  size_t slab;
  uint8_t* staging;  // PE 0's staging ring [buffer][tile_s rows][H*W][D]
  uint8_t* signals;  // PE 0's signal slots, SYMM_SIGNAL_STRIDE_BYTES apart
  size_t stage_pe, sig_pe;
  uint32_t W, H, S, D, es;
  uint32_t tile_s, block_d, nbd, nbs, buffer_num;
  size_t tile_src;   // input bytes from one S block to the next (tile_s rows)
  size_t tile_dst;   // output bytes from one S block to the next
  size_t stage_buf;  // staging bytes from one buffer to the next
  size_t slot_buf;   // signal bytes from one buffer to the next
  uint32_t reset;    // zero this launch's signal slots first (each CTA its own)
  uint32_t discard;  // drop a slot's staging lines from L2 after its last use
  uint64_t budget_ns;
  Control* ctl;
  const uint8_t* err_base;  // a slot that times out is reported as its offset
  int64_t err_bias;         // from err_base, plus err_bias
};

// One task of one S block: the tile of source PE r bound for destination d,
// expert column h, D block bd.  q = ((d*W + r)*H + h)*nbd + bd.
struct PcTask {
  int64_t* slot;       // the signal slot (buffer b % buffer_num) on PE d
  const uint8_t* src;  // input row d*S + s0 of PE r, at column x0
  uint8_t* stage;      // staging row 0 of the slot, column r*H + h, x0
  uint8_t* dst;        // output row s0 of PE d, column r*H + h, x0
  uint32_t rows;       // rows of the tile (the last S block may be short)
  uint32_t len;        // bytes per tile row (the last D block may be short)
};

// Task q at S block 0, buffer 0; the other S blocks and buffers are fixed
// strides from it (PcArgs::tile_src, tile_dst, slot_buf, stage_buf).
struct PcBase {
  int64_t* slot;
  const uint8_t* src;
  uint8_t* stage;
  uint8_t* dst;
  uint32_t len;
};

__device__ __forceinline__ PcBase pc_base(const PcArgs& a, size_t q) {
  const uint32_t bd = (uint32_t)(q % a.nbd);
  q /= a.nbd;
  const uint32_t h = (uint32_t)(q % a.H);
  q /= a.H;
  const uint32_t r = (uint32_t)(q % a.W);
  const uint32_t d = (uint32_t)(q / a.W);
  const uint32_t x0 = bd * a.block_d;
  const size_t col = ((size_t)(r * a.H + h) * a.D + x0) * a.es;
  PcBase k;
  // slot (0, r, bd, h) of destination d, one 64-byte line each
  k.slot = reinterpret_cast<int64_t*>(
      a.signals + d * a.sig_pe + (((size_t)r * a.nbd + bd) * a.H + h) * SYMM_SIGNAL_STRIDE_BYTES);
  k.src = a.in + r * a.slab + (((size_t)d * a.S * a.H + h) * a.D + x0) * a.es;
  k.stage = a.staging + d * a.stage_pe + col;
  k.dst = a.out + d * a.slab + col;
  k.len = min(a.block_d, a.D - x0) * a.es;
  return k;
}

__device__ __forceinline__ PcTask pc_task_of(const PcArgs& a, const PcBase& k0, uint32_t b,
                                             uint32_t buf) {
  PcTask k;
  k.slot = reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(k0.slot) + buf * a.slot_buf);
  k.src = k0.src + b * a.tile_src;
  k.stage = k0.stage + buf * a.stage_buf;
  k.dst = k0.dst + b * a.tile_dst;
  k.rows = min(a.tile_s, a.S - b * a.tile_s);
  k.len = k0.len;
  return k;
}

// CTA c owns the tasks q = c + j*gridDim.x (j < nq) of every S block (the
// page's fixed core-to-task mapping), and walks them task by task: its tile
// number t = j*nbs + b is S block b of task j, in buffer b % buffer_num.  A
// slot's successive producers are then one CTA, in S-block order, as on the
// page, whose cores walk S block by S block instead; with several tasks per
// CTA that order keeps every task's slots in use at once (the whole staging
// ring), this one only each CTA's current task's buffer_num slots, which
// L2 can hold.  SYMM_PC_TASK_MAJOR = 0 selects the page's order
// (t = b*nq + j).
#ifndef SYMM_PC_TASK_MAJOR
#define SYMM_PC_TASK_MAJOR 1
#endif
__device__ __forceinline__ uint32_t pc_tasks_per_cta(const PcArgs& a) {
  const size_t per_block = (size_t)a.W * a.W * a.H * a.nbd;
  return (uint32_t)((per_block - blockIdx.x - 1) / gridDim.x + 1);
}

// The CTA's tasks decoded once: up to kPcOwned of them in shared memory
// (the loops then take a task with a few adds and no divisions); more are
// decoded again at each use.
constexpr uint32_t kPcOwned = 16;
struct PcTable {
  PcBase base[kPcOwned];
};
__device__ __forceinline__ void pc_table_fill(const PcArgs& a, uint32_t nq, PcTable& tab) {
  for (uint32_t j = threadIdx.x; j < nq && j < kPcOwned; j += blockDim.x)
    tab.base[j] = pc_base(a, blockIdx.x + (size_t)j * gridDim.x);
}
__device__ __forceinline__ PcBase pc_table_get(const PcArgs& a, const PcTable& tab, uint32_t j) {
  return j < kPcOwned ? tab.base[j] : pc_base(a, blockIdx.x + (size_t)j * gridDim.x);
}

// Zeroes the signal slots of the CTA's tasks, every buffer (the page's reset
// before each launch, done by each slot's owner: a slot belongs to exactly
// one task and a task to one CTA, so no other CTA touches it).  gpu-scope
// stores, then a CTA barrier (the caller's) before any acquire.
__device__ __forceinline__ void pc_zero_own_slots(const PcArgs& a, uint32_t nq,
                                                  const PcTable& tab) {
  for (uint32_t i = threadIdx.x; i < nq * a.buffer_num; i += blockDim.x) {
    const uint32_t j = i / a.buffer_num, buf = i - j * a.buffer_num;
    int64_t* slot = reinterpret_cast<int64_t*>(
        reinterpret_cast<uint8_t*>(pc_table_get(a, tab, j).slot) + buf * a.slot_buf);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(slot), "l"((int64_t)0) : "memory");
  }
}

// Position (S block, task, buffer) in a CTA's task sequence, advanced
// without divisions.
struct PcCursor {
  uint32_t b = 0, j = 0, buf = 0;
  __device__ __forceinline__ void next(uint32_t nq, uint32_t nbs, uint32_t buffer_num) {
    if (SYMM_PC_TASK_MAJOR) {
      if (++b == nbs) {
        b = 0;
        buf = 0;
        ++j;
      } else if (++buf == buffer_num) {
        buf = 0;
      }
    } else if (++j == nq) {
      j = 0;
      ++b;
      if (++buf == buffer_num) buf = 0;
    }
  }
};
// Fewest tiles between two uses of one slot in a CTA's sequence.
__device__ __forceinline__ uint64_t pc_slot_reuse(uint32_t nq, uint32_t buffer_num) {
  return SYMM_PC_TASK_MAJOR ? (uint64_t)buffer_num : (uint64_t)nq * buffer_num;
}
__device__ __forceinline__ PcTask pc_task_at(const PcArgs& a, const PcTable& tab,
                                             const PcCursor& c) {
  return pc_task_of(a, pc_table_get(a, tab, c.j), c.b, c.buf);
}

// L2 policies of the producer/consumer copies: SYMM_PC_L2HINT marks the
// prefetched input reads evict-first and the staging writes evict-last, so
// streamed input and output lines leave L2 before staged tiles do (measured
// on GB300, DeepSeek-V3 rows: 5078 against 4986 GB/s, and 476 against 504 MB
// of DRAM writes at S = 512, fewer staging lines written back).
#ifndef SYMM_PC_L2HINT
#define SYMM_PC_L2HINT 1
#endif

// Issues the bulk loads of a tile's input rows into `tile` (one mbarrier phase).
__device__ __forceinline__ void pc_prefetch(const PcArgs& a, const PcTask& k, uint8_t* tile,
                                            uint64_t* bar) {
  const size_t src_row = (size_t)a.H * a.D * a.es;
  symm::mbar_arrive_expect_tx(bar, k.rows * k.len);
  if (SYMM_PC_L2HINT) {
    const uint64_t pol = symm::policy_evict_first();
    for (uint32_t i = 0; i < k.rows; ++i)
      symm::bulk_load_hint(tile + i * k.len, k.src + i * src_row, k.len, bar, pol);
  } else {
    for (uint32_t i = 0; i < k.rows; ++i)
      symm::bulk_load(tile + i * k.len, k.src + i * src_row, k.len, bar);
  }
}


// PREFETCH: the producer group's thread 0 keeps the input tiles of the next
// kPcPrefetch tasks in flight with bulk (TMA) loads into a shared-memory
// ring, so producer warps only copy shared memory -> staging (16-byte
// vectors); needs 16-byte-aligned tile rows.  Without it, producer warps
// load the input with 16-byte vectors themselves.
#ifndef SYMM_PC_PREFETCH
#define SYMM_PC_PREFETCH 2
#endif
constexpr int kPcPrefetch = SYMM_PC_PREFETCH;
// The prefetching instance with release warps (a2a_pc_rel_kernel, below).
#ifndef SYMM_PC_RELEASE_WARPS
#define SYMM_PC_RELEASE_WARPS 1
#endif

constexpr uint32_t kPcMaxPrefetchTile = 32 * 1024;
// Narrowest tile row worth a bulk copy: measured on GB300, rows of 256 B to
// 1 KB went faster without the prefetch (e.g. 1425 against 936 GB/s on 256 B
// rows), rows of 2 KB faster with it (4742 against 4302 GB/s).
constexpr size_t kPcMinPrefetchRow = 2048;
// The same for rows of any alignment, whose copies without the prefetch
// shift-merge two loaded blocks per vector (a2a_pc_rel_kernel<true>).
#ifndef SYMM_PC_ANY_PREFETCH
#define SYMM_PC_ANY_PREFETCH 1
#endif
constexpr size_t kPcMinPrefetchRowAny = 1024;
// Bytes of input rows per ring entry of the unaligned instance (at most
// kPcMaxPrefetchTile; a row wider than this takes an entry of its own).
#ifndef SYMM_PC_ANY_CHUNK
#define SYMM_PC_ANY_CHUNK 32768
#endif
constexpr uint32_t kPcAnyChunk = SYMM_PC_ANY_CHUNK;

// How a group copies its tile (a tile always spans less than 4 GiB here):
//   kCopyAligned  every tile row, base and row stride is 16-byte aligned:
//                 symm::group_copy_tile, the tile flattened to 16-byte vectors;
//   kCopyAny      the staging and output rows share one 16-byte phase (their
//                 stride H*W*D*elem_bytes is a multiple of 16), any other
//                 alignment: symm::group_copy_tile_any, flattened too, with
//                 funnel-shifted vectors and byte heads and tails;
//   kCopyRows     anything else: one warp per row with symm::warp_copy.
enum { kCopyRows = 0, kCopyAligned = 1, kCopyAny = 2 };

template <bool PREFETCH, int MODE>
__global__ void __launch_bounds__(kPcThreads,
                                  MODE == kCopyAny ? kPcMinBlocks : SYMM_PC_KERNEL_MIN_BLOCKS)
    a2a_pc_kernel(const PcArgs a, uint32_t tile_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int status[2];
  __shared__ PcTable tab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int role = warp >> 2;          // 0 = producer group, 1 = consumer group
  const int gwarp = warp & 3;          // warp inside its group
  const int gtid = threadIdx.x & (kPcGroup - 1);
  const int bar_id = 1 + role;         // named barrier of the group
  const size_t stage_row = (size_t)a.H * a.W * a.D * a.es;  // one staging row, bytes
  const size_t src_row = (size_t)a.H * a.D * a.es;
  const uint32_t nq = pc_tasks_per_cta(a);
  const uint64_t ntasks = (uint64_t)a.nbs * nq;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + 128;
  pc_table_fill(a, nq, tab);
  __syncthreads();
  if (a.reset) {
    pc_zero_own_slots(a, nq, tab);
    __syncthreads();
  }
  uint64_t issued = 0;
  PcCursor pre;  // the next task whose input the producer prefetches
  if (PREFETCH && role == 0) {
    if (gtid == 0) {
      for (int i = 0; i < kPcPrefetch; ++i) symm::mbar_init(&bars[i], 1);
      symm::fence_mbar_init();
      for (; issued < ntasks && issued < (uint64_t)kPcPrefetch; ++issued, pre.next(nq, a.nbs, a.buffer_num))
        pc_prefetch(a, pc_task_at(a, tab, pre), ring + issued * tile_bytes, &bars[issued]);
    }
    symm::group_sync(bar_id, kPcGroup);
  }

  // The producer of S block b and the consumer of S block b - buffer_num on
  // the same slot are this CTA's own two groups, so no wait depends on
  // another CTA.
  PcCursor cur;
  for (uint64_t t = 0; t < ntasks; ++t, cur.next(nq, a.nbs, a.buffer_num)) {
    const PcTask k = pc_task_at(a, tab, cur);
    const int st = (int)(t % kPcPrefetch);
    if (gtid == 0) {
      int rc = symm::kSpinOk;
      if (PREFETCH && role == 0 &&
          !symm::mbar_wait(&bars[st], (uint32_t)(t / kPcPrefetch) & 1u, a.budget_ns)) {
        symm::record_error(a.ctl, symm::kErrTimedOut, -1);
        rc = symm::kSpinTimeout;
      }
      if (rc == symm::kSpinOk)
        rc = symm::spin_wait(k.slot, symm::kCmpEq, role == 0 ? 0 : 1, a.budget_ns, a.ctl,
                             a.err_base, a.err_bias);
      status[role] = rc;
    }
    symm::group_sync(bar_id, kPcGroup);
    if (status[role] != symm::kSpinOk) {
      // let this group's prefetches still in flight land (bounded), then leave
      if (PREFETCH && role == 0 && gtid == 0)
        for (uint64_t i = t; i < issued; ++i)
          symm::mbar_wait(&bars[i % kPcPrefetch], (uint32_t)(i / kPcPrefetch) & 1u, a.budget_ns);
      return;  // uniform across the group
    }

    if (role == 0) {
      if (PREFETCH) {
        // shared-memory tile -> destination d's slot, 16 bytes per thread-step
        const uint8_t* tile = ring + (size_t)st * tile_bytes;
        const uint32_t vrow = k.len >> 4, nv = k.rows * vrow;
        const uint64_t pol = SYMM_PC_L2HINT ? symm::policy_evict_last() : 0;
        const symm::TileStep step = symm::tile_step(kPcGroup, vrow);
        uint32_t i = (uint32_t)gtid / vrow, c = (uint32_t)gtid - i * vrow;
        for (uint32_t v = gtid; v < nv; v += kPcGroup, step.advance(i, c, vrow)) {
          const uint4 x = *reinterpret_cast<const uint4*>(tile + i * k.len + 16 * c);
          if (SYMM_PC_L2HINT)
            symm::st16_hint(k.stage + i * stage_row + 16 * c, x, pol);
          else
            symm::st16(k.stage + i * stage_row + 16 * c, x);
        }
      } else if (MODE == kCopyAligned) {
        // input rows d*S + s0 + i of source r -> destination d's slot
        symm::group_copy_tile<kPcGroup, SYMM_PC_FLAT_UNROLL, symm::kRO, symm::kST>(
            k.stage, (uint32_t)stage_row, k.src, (uint32_t)src_row, k.rows, k.len >> 4, gtid);
      } else if (MODE == kCopyAny) {
        symm::group_copy_tile_any<kPcGroup, SYMM_PC_ANY_UNROLL, symm::kRO, symm::kST>(
            k.stage, (uint32_t)stage_row, k.src, (uint32_t)src_row, k.rows, k.len, gtid);
      } else {
        for (uint32_t i = gwarp; i < k.rows; i += 4)
          symm::warp_copy<SYMM_PC_UNROLL, symm::kRO, symm::kST>(k.stage + i * stage_row,
                                                                 k.src + i * src_row, k.len, lane);
      }
    } else {
      // staged tile -> output rows s0 + i, column r*H + h
      if (MODE == kCopyAligned)
        symm::group_copy_tile<kPcGroup, SYMM_PC_FLAT_UNROLL, symm::kCG, symm::kCS>(
            k.dst, (uint32_t)stage_row, k.stage, (uint32_t)stage_row, k.rows, k.len >> 4, gtid);
      else if (MODE == kCopyAny)
        symm::group_copy_tile_any<kPcGroup, SYMM_PC_ANY_UNROLL, symm::kCG, symm::kCS>(
            k.dst, (uint32_t)stage_row, k.stage, (uint32_t)stage_row, k.rows, k.len, gtid);
      else
        for (uint32_t i = gwarp; i < k.rows; i += 4)
          symm::warp_copy<SYMM_PC_UNROLL, symm::kCG, symm::kCS>(k.dst + i * stage_row,
                                                                 k.stage + i * stage_row, k.len,
                                                                 lane);
    }
    symm::group_sync(bar_id, kPcGroup);  // the group's copies precede the release
    if (gtid == 0) {
      symm::st_release(k.slot, role == 0 ? 1 : 0);
      if (PREFETCH && role == 0 && issued < ntasks) {
        // every producer thread has read this ring slot: refill it
        symm::fence_proxy_async_shared();
        pc_prefetch(a, pc_task_at(a, tab, pre), ring + (size_t)st * tile_bytes, &bars[st]);
        pre.next(nq, a.nbs, a.buffer_num);
        ++issued;
      }
    }
  }
}

// ------------------------------- producer / consumer, release warps ---
// a2a_pc_kernel's prefetching instance with the releases taken off the copy
// groups.  A gpu-scope release waits for the memory system -- about 2 µs
// while the GPU streams at HBM rate, measured -- and in a2a_pc_kernel the
// whole group waits behind it.  Here:
//   warps 0-3  producer group: thread 0 acquires the slot (== 0); for each
//              input chunk of the tile (below) thread 0 waits for the chunk
//              in the prefetch ring, the group copies it into the staging
//              slot and arrives on the chunk's done barrier (one of
//              kPcRelLag that alternate);
//   warps 4-7  consumer group: thread 0 acquires (== 1), the group copies the
//              staged tile out and arrives on the tile's done barrier;
//   (a slot's last holder is always this CTA's other group, so thread 0
//   first waits for that group's release count in shared memory -- the
//   release is then performed in L2 -- and acquires with a single load
//   instead of polling L2; the producer group also starts tile t only once
//   the consumer group has released tile t - R, R as below, when tile t's
//   slot is fresh (a task's first S blocks): a CTA's staged tiles not yet
//   consumed then never exceed R, which bounds what L2 must hold);
//   warp 8     producer release thread: per chunk, waits for its done
//              barrier and refills its ring entry with the next input chunk;
//              after a tile's last chunk, releases the slot (1), counts it in
//              released[0], and only then refills that chunk's entry;
//   warp 9     consumer release warp: per tile, waits for done[1], drops the
//              staging lines of a slot's last use from L2 when
//              PcArgs::discard is set (below), releases (0) and counts it
//              in released[1].
// A group may acquire tile t only once tile t - min(R, kPcRelLag) is
// released (R = the fewest tiles between two uses of a slot in the CTA's
// sequence: buffer_num when it walks task by task, tasks x buffers when S
// block by S block): the slot of tile t - R then no longer holds the value
// the group waits for from its last use, and the done barrier of tile
// t - kPcRelLag (the same one of the kPcRelLag that alternate) has been
// consumed.  The producer group arrives on a done barrier per chunk; it is
// never more than a ring's worth of chunks ahead of its release thread (a
// chunk's ring entry is refilled only after the chunk one ring earlier is
// done), so kPcRelLag >= the ring's entries keeps those phases apart too.
// The release is an atomic exchange whose
// result the count depends on, so the count moves only once the release is
// performed in L2, where the group's acquire reads.  Waits on another role's
// progress (a release thread on its group, a group on its release thread)
// have twice the spin budget, so that a stuck slot is what a give-up
// reports, not a wait that depends on it.
//
// Input chunks: a tile's input rows arrive in chunks of up to
// PcRing::chunk_rows rows, one ring entry each, so a tile taller than a ring
// entry still streams through the ring.
//   ANY = false  16-byte-aligned rows, loaded as they are and packed in the
//                entry (row pitch = the row's bytes); both groups copy
//                aligned 16-byte vectors.
//   ANY = true   rows of any alignment whose staging and output rows share
//                one 16-byte phase.  Bulk copies need 16-byte-aligned
//                addresses and sizes, so each row's aligned covering block
//                range is loaded, PcRing::pitch bytes apart; the producer
//                funnel-shifts it into aligned 16-byte stores
//                (symm::group_copy_ring_any) and the consumer copies head
//                bytes, aligned vectors and tail bytes
//                (symm::group_copy_tile_phase).  The covering range reads at
//                most 15 bytes on either side of a row, inside the 16-byte
//                granules of its first and last bytes.
//
// Discards: a slot is used for S blocks b, b + buffer_num, ... of its task;
// after its last use its staging lines stay dirty in L2 (marked evict-last)
// until they are written back, which costs DRAM bandwidth and, while they
// wait, crowds the slots still in use out of L2.  With PcArgs::discard the
// consumer release warp drops, after a slot's last use in the launch, every
// 128-byte line that lies wholly inside the tile's rows (discard.global.L2),
// before the release; lines shared with a neighbouring task's bytes are left
// alone.  The CTA's last task is left out: nothing of this launch follows it
// that its lines could crowd out, and discards there only delay the end of
// the launch.  Discarding after every use instead measured slower (the
// release waits for the discards, and the slot is rewritten while still in
// L2).
constexpr int kPcRelThreads = 320;
#ifndef SYMM_PC_REL_LAG
#define SYMM_PC_REL_LAG 4
#endif
constexpr int kPcRelLag = SYMM_PC_REL_LAG;  // done barriers per group (a power of two)
static_assert((kPcRelLag & (kPcRelLag - 1)) == 0 && kPcRelLag >= 1, "lag: a power of two");
// Ring entries of the release-warp kernel's instance for aligned rows.
#ifndef SYMM_PC_REL_PREFETCH
#define SYMM_PC_REL_PREFETCH 2
#endif
constexpr int kPcRelPrefetch = SYMM_PC_REL_PREFETCH;
// The instance for rows of any alignment (ANY = true) has its own ring depth,
// consumer vectors in flight and residency: its producer shift-merges from
// shared memory and its consumer copies byte edges, which need more
// registers than 3 CTAs per SM leave.
#ifndef SYMM_PC_ANY_RING
#define SYMM_PC_ANY_RING 2
#endif
#ifndef SYMM_PC_ANY_CONSUMER_UNROLL
#define SYMM_PC_ANY_CONSUMER_UNROLL 8
#endif
// 16-byte vectors in flight per lane in the producer's shift-merge copy
// out of the ring (symm::group_copy_ring_any).
#ifndef SYMM_PC_RING_UNROLL
#define SYMM_PC_RING_UNROLL 1
#endif
#ifndef SYMM_PC_ANY_MIN_BLOCKS
#define SYMM_PC_ANY_MIN_BLOCKS 2
#endif
template <bool ANY>
struct PcRelConf {
  static constexpr int ring = ANY ? SYMM_PC_ANY_RING : kPcRelPrefetch;
  static constexpr int min_blocks = ANY ? SYMM_PC_ANY_MIN_BLOCKS : kPcMinBlocks;
  static constexpr int consumer_unroll = ANY ? SYMM_PC_ANY_CONSUMER_UNROLL : SYMM_PC_FLAT_UNROLL;
  static_assert(kPcRelLag >= ring, "done barriers must outnumber ring entries");
  static_assert((ring + 2 * kPcRelLag) * 8 <= 128, "barriers fit the ring's header");
};
// Drop a slot's staging lines from L2 after its last use (PcArgs::discard).
#ifndef SYMM_PC_DISCARD
#define SYMM_PC_DISCARD 1
#endif

// The input ring of a2a_pc_rel_kernel.
struct PcRing {
  uint32_t stage;       // bytes per ring entry
  uint32_t chunk_rows;  // tile rows per entry
  uint32_t pitch;       // ANY: ring bytes per row (a multiple of 16)
};

__device__ __forceinline__ uint32_t pc_chunks(uint32_t rows, uint32_t chunk_rows) {
  return (rows + chunk_rows - 1) / chunk_rows;
}

// Issues the bulk loads of rows r0 .. r0 + n - 1 of task k's input tile into
// ring entry `buf` (one mbarrier phase): ANY, each row's 16-byte-aligned
// covering block range, `pitch` bytes apart; otherwise the rows, packed.
template <bool ANY>
__device__ __forceinline__ void pc_prefetch_chunk(const PcArgs& a, const PcTask& k, uint32_t r0,
                                                  uint32_t n, uint32_t pitch, uint8_t* buf,
                                                  uint64_t* bar) {
  const size_t src_row = (size_t)a.H * a.D * a.es;
  const uint8_t* s0 = k.src + (size_t)r0 * src_row;
  const uint64_t pol = symm::policy_evict_first();
  if (!ANY) {
    symm::mbar_arrive_expect_tx(bar, n * k.len);
    for (uint32_t i = 0; i < n; ++i)
      symm::bulk_load_hint(buf + i * k.len, s0 + i * src_row, k.len, bar, pol);
    return;
  }
  const uintptr_t m16 = ~(uintptr_t)15;
  uint32_t total = 0;
  for (uint32_t i = 0; i < n; ++i) {
    const uintptr_t s = (uintptr_t)(s0 + i * src_row);
    total += (uint32_t)(((s + k.len + 15) & m16) - (s & m16));
  }
  symm::mbar_arrive_expect_tx(bar, total);
  for (uint32_t i = 0; i < n; ++i) {
    const uintptr_t s = (uintptr_t)(s0 + i * src_row);
    const uintptr_t lo = s & m16;
    symm::bulk_load_hint(buf + i * pitch, reinterpret_cast<const void*>(lo),
                         (uint32_t)(((s + k.len + 15) & m16) - lo), bar, pol);
  }
}

__device__ __forceinline__ uint64_t atom_exch_release(int64_t* p, int64_t v) {
  uint64_t old;
  asm volatile("atom.release.gpu.global.exch.b64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}
// 0, computed from x so that what uses it waits for x
__device__ __forceinline__ uint32_t zero_after(uint64_t x) {
  uint32_t z;
  asm volatile("{\n\t.reg .b64 t;\n\tand.b64 t, %1, 0;\n\tcvt.u32.u64 %0, t;\n\t}"
               : "=r"(z)
               : "l"(x));
  return z;
}
// Bounded wait on an mbarrier phase that also gives up once the heap's abort
// flag is raised.
__device__ __forceinline__ bool pc_mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns,
                                             Control* ctl) {
  if (symm::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = symm::globaltimer_ns();
  const uint64_t max_iters = budget_ns / 32 + (1u << 20);
  for (uint64_t it = 0;; ++it) {
    if (symm::mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63 && (symm::ld_relaxed_u32(&ctl->abort) ||
                            symm::globaltimer_ns() - t0 > budget_ns || it > max_iters))
      return false;
  }
}
// Bounded wait until a shared-memory count reaches `want`.
__device__ __forceinline__ bool pc_count_wait(volatile uint32_t* count, uint32_t want,
                                              uint64_t budget_ns, Control* ctl) {
  if (*count >= want) return true;
  const uint64_t t0 = symm::globaltimer_ns();
  const uint64_t max_iters = budget_ns / 64 + 4096;
  for (uint64_t it = 0;; ++it) {
    if (*count >= want) return true;
    if (symm::ld_relaxed_u32(&ctl->abort)) return false;
    if (symm::globaltimer_ns() - t0 > budget_ns || it > max_iters) {
      symm::record_error(ctl, symm::kErrTimedOut, -1);
      return false;
    }
    __nanosleep(32);
  }
}
__device__ __forceinline__ void pc_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(symm::smem_addr(bar)) : "memory");
}

// Warps of the producer group (the rest of warps 0-7 form the consumer group).
#ifndef SYMM_PC_REL_PRODUCER_WARPS
#define SYMM_PC_REL_PRODUCER_WARPS 4
#endif
constexpr int kPcRelPW = SYMM_PC_REL_PRODUCER_WARPS;
constexpr int kPcRelPG = 32 * kPcRelPW;        // producer group threads
constexpr int kPcRelCG = 32 * (8 - kPcRelPW);  // consumer group threads

template <bool ANY>
__global__ void __launch_bounds__(kPcRelThreads, PcRelConf<ANY>::min_blocks)
    a2a_pc_rel_kernel(const PcArgs a, const PcRing rg) {
  constexpr int kRing = PcRelConf<ANY>::ring;
  extern __shared__ __align__(128) uint8_t smem[];
  // [role][parity of the group's barrier count]: thread 0 writes entry p
  // again only after the group's next barrier, which every reader of the
  // previous value has passed
  __shared__ int status[2][2];
  __shared__ PcTable tab;
  __shared__ volatile uint32_t released[2];
  uint64_t* in_full = reinterpret_cast<uint64_t*>(smem);  // kRing ring barriers
  uint64_t* done = in_full + kRing;                        // [role][i % kPcRelLag]
  uint8_t* ring = smem + 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 0 producer group, 1 consumer group, 2 release threads
  const int role = warp < kPcRelPW ? 0 : (warp < 8 ? 1 : 2);
  const int gtid = role == 0 ? (int)threadIdx.x : (int)threadIdx.x - kPcRelPG;
  const int gsize = role == 0 ? kPcRelPG : kPcRelCG;
  const int bar_id = 1 + role;
  const size_t stage_row = (size_t)a.H * a.W * a.D * a.es;
  const size_t src_row = (size_t)a.H * a.D * a.es;
  const uint32_t nq = pc_tasks_per_cta(a);
  const uint64_t ntasks = (uint64_t)a.nbs * nq;
  const uint64_t reuse = pc_slot_reuse(nq, a.buffer_num);
  const uint64_t lag = reuse < (uint64_t)kPcRelLag ? reuse : (uint64_t)kPcRelLag;
  pc_table_fill(a, nq, tab);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) symm::mbar_init(&in_full[i], 1);
    for (int i = 0; i < kPcRelLag; ++i) {
      symm::mbar_init(&done[i], kPcRelPG);
      symm::mbar_init(&done[kPcRelLag + i], kPcRelCG);
    }
    released[0] = 0;
    released[1] = 0;
    symm::fence_mbar_init();
  }
  __syncthreads();
  if (a.reset) {
    pc_zero_own_slots(a, nq, tab);
    __syncthreads();
  }

  if (role < 2) {  // ------------------------------------ copy groups
    const uint64_t pol = symm::policy_evict_last();
    const uint32_t msrc = (uint32_t)(src_row & 15);
    PcCursor cur;
    uint64_t g = 0;  // barriers passed: chunks (producer) or tiles (consumer)
    for (uint64_t t = 0; t < ntasks; ++t, cur.next(nq, a.nbs, a.buffer_num)) {
      const PcTask k = pc_task_at(a, tab, cur);
      const uint32_t nch = role == 0 ? pc_chunks(k.rows, rg.chunk_rows) : 1;
      for (uint32_t c = 0; c < nch; ++c, ++g) {
        const int par = (int)(g & 1);
        if (gtid == 0) {
          int rc = symm::kSpinOk;
          if (c == 0 && t + 1 > lag &&
              !pc_count_wait(&released[role], (uint32_t)(t + 1 - lag), 2 * a.budget_ns, a.ctl))
            rc = symm::kSpinTimeout;
          if (rc == symm::kSpinOk && role == 0 &&
              !pc_mbar_wait(&in_full[g % kRing], (uint32_t)(g / kRing) & 1u,
                            a.budget_ns, a.ctl)) {
            symm::record_error(a.ctl, symm::kErrTimedOut, -1);
            rc = symm::kSpinTimeout;
          }
          if (rc == symm::kSpinOk && c == 0) {
            // The slot's last holder is this CTA's other group: wait until
            // its release is performed (the other role's count), so that the
            // acquire finds the value at once instead of polling L2.
            if (role == 1 &&
                !pc_count_wait(&released[0], (uint32_t)(t + 1), 2 * a.budget_ns, a.ctl))
              rc = symm::kSpinTimeout;
            // (pacing: also when tile t's slot is fresh, see above)
            if (role == 0 && t >= reuse &&
                !pc_count_wait(&released[1], (uint32_t)(t + 1 - reuse), 2 * a.budget_ns, a.ctl))
              rc = symm::kSpinTimeout;
            if (rc == symm::kSpinOk)
              rc = symm::spin_wait(k.slot, symm::kCmpEq, role == 0 ? 0 : 1, a.budget_ns, a.ctl,
                                   a.err_base, a.err_bias);
          }
          status[role][par] = rc;
        }
        symm::group_sync(bar_id, gsize);
        if (status[role][par] != symm::kSpinOk) return;  // uniform across the group
        if (role == 0) {
          // ring entry -> rows r0 .. r0 + n - 1 of destination d's slot
          const uint8_t* src = ring + (size_t)(g % kRing) * rg.stage;
          const uint32_t r0 = c * rg.chunk_rows;
          const uint32_t n = min(rg.chunk_rows, k.rows - r0);
          uint8_t* dst = k.stage + (size_t)r0 * stage_row;
          if (ANY) {
            const uint32_t m0 = (uint32_t)((uintptr_t)(k.src + (size_t)r0 * src_row) & 15);
            symm::group_copy_ring_any<kPcRelPG, SYMM_PC_RING_UNROLL>(
                dst, (uint32_t)stage_row, src, rg.pitch, m0, msrc, n, k.len, gtid, pol);
          } else {
            const uint32_t vrow = k.len >> 4, nv = n * vrow;
            const symm::TileStep step = symm::tile_step(kPcRelPG, vrow);
            uint32_t i = (uint32_t)gtid / vrow, cc = (uint32_t)gtid - i * vrow;
            for (uint32_t v = gtid; v < nv; v += kPcRelPG, step.advance(i, cc, vrow))
              symm::st16_hint(dst + i * stage_row + 16 * cc,
                              *reinterpret_cast<const uint4*>(src + i * k.len + 16 * cc), pol);
          }
        } else if (ANY) {
          symm::group_copy_tile_phase<kPcRelCG, PcRelConf<ANY>::consumer_unroll, symm::kCG, symm::kCS>(
              k.dst, (uint32_t)stage_row, k.stage, (uint32_t)stage_row, k.rows, k.len, gtid);
        } else {
          symm::group_copy_tile<kPcRelCG, SYMM_PC_FLAT_UNROLL, symm::kCG, symm::kCS>(
              k.dst, (uint32_t)stage_row, k.stage, (uint32_t)stage_row, k.rows, k.len >> 4, gtid);
        }
        // this thread's copies precede the arrival
        pc_mbar_arrive(&done[role * kPcRelLag + (g % kPcRelLag)]);
      }
    }
  } else if (threadIdx.x == 256) {  // ---------------- producer release thread
    PcCursor pre;         // task of the next chunk to load
    uint64_t pre_t = 0;   // its tile number
    uint32_t pre_c = 0;   // the chunk within it
    uint64_t issued = 0;  // chunks loaded, into ring entry issued % kRing
    auto issue_next = [&]() {
      if (pre_t >= ntasks) return;
      const PcTask kp = pc_task_at(a, tab, pre);
      const uint32_t r0 = pre_c * rg.chunk_rows;
      const int e = (int)(issued % kRing);
      symm::fence_proxy_async_shared();  // the group's reads of the entry precede the load
      pc_prefetch_chunk<ANY>(a, kp, r0, min(rg.chunk_rows, kp.rows - r0), rg.pitch,
                             ring + (size_t)e * rg.stage, &in_full[e]);
      ++issued;
      if (++pre_c == pc_chunks(kp.rows, rg.chunk_rows)) {
        pre_c = 0;
        ++pre_t;
        pre.next(nq, a.nbs, a.buffer_num);
      }
    };
    while (issued < (uint64_t)kRing && pre_t < ntasks) issue_next();
    PcCursor cur;
    uint64_t g = 0;  // chunks done
    bool ok = true;
    for (uint64_t t = 0; ok && t < ntasks; ++t, cur.next(nq, a.nbs, a.buffer_num)) {
      const PcTask k = pc_task_at(a, tab, cur);
      const uint32_t nch = pc_chunks(k.rows, rg.chunk_rows);
      for (uint32_t c = 0; c < nch; ++c, ++g) {
        if (!pc_mbar_wait(&done[g % kPcRelLag], (uint32_t)(g / kPcRelLag) & 1u, 2 * a.budget_ns,
                          a.ctl)) {
          symm::record_error(a.ctl, symm::kErrTimedOut, -1);
          ok = false;
          break;
        }
        // chunk g's entry is free: load the chunk kRing ahead into it, after
        // the release and its count when this is the tile's last chunk (both
        // are on the slot's cycle; measured faster than refilling first, or
        // refilling while the release is in flight)
        if (c + 1 < nch) issue_next();
      }
      if (!ok) break;
      const uint64_t old = atom_exch_release(k.slot, 1);
      released[0] = (uint32_t)(t + 1) + zero_after(old);
      issue_next();
    }
    // let the loads still in flight land before the CTA may leave (bounded)
    for (uint64_t i = g; i < issued; ++i)
      symm::mbar_wait(&in_full[i % kRing], (uint32_t)(i / kRing) & 1u,
                      a.budget_ns);
  } else if (warp == 9) {  // ------------------------ consumer release warp
    PcCursor cur;
    for (uint64_t t = 0; t < ntasks; ++t, cur.next(nq, a.nbs, a.buffer_num)) {
      int ok = 1;
      if (lane == 0)
        ok = pc_mbar_wait(&done[kPcRelLag + (t % kPcRelLag)], (uint32_t)(t / kPcRelLag) & 1u,
                          2 * a.budget_ns, a.ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();  // lane 0's acquire of the group's copies precedes every lane's discards
      if (!ok) {
        if (lane == 0) symm::record_error(a.ctl, symm::kErrTimedOut, -1);
        break;
      }
      const PcTask k = pc_task_at(a, tab, cur);
      if (a.discard && cur.b + a.buffer_num >= a.nbs && (!SYMM_PC_TASK_MAJOR || cur.j + 1 < nq)) {
        // the slot's last use, with more of the CTA's tasks to come: every
        // 128-byte line wholly inside one of the tile's staging rows
        for (uint32_t i = 0; i < k.rows; ++i) {
          const uintptr_t row = (uintptr_t)(k.stage + (size_t)i * stage_row);
          const uintptr_t hi = (row + k.len) & ~(uintptr_t)127;
          for (uintptr_t x = ((row + 127) & ~(uintptr_t)127) + 128 * (uintptr_t)lane; x < hi;
               x += 128 * 32)
            symm::discard_l2(reinterpret_cast<const void*>(x));
        }
        __syncwarp();  // every lane's discards precede the release
      }
      if (lane == 0) {
        const uint64_t old = atom_exch_release(k.slot, 0);
        released[1] = (uint32_t)(t + 1) + zero_after(old);
      }
    }
  }
}

// ------------------------------------- producer / consumer, phased ---
// SYMM_A2A_FLAG_PHASED (a debugging aid): the producers of one S block, or
// its consumers, as one launch of one CTA per task whose warps take the
// tile's rows.  Kernel boundaries stand in for a barrier between the two
// roles; the slot protocol is the pipelined kernels' (producer: wait 0,
// copy, release 1; consumer: wait 1, copy, release 0), so a slot's waits
// are satisfied as soon as they start.
constexpr int kPcPhaseThreads = 256;
template <int ROLE>  // 0: producers, 1: consumers
__global__ void __launch_bounds__(kPcPhaseThreads) a2a_pc_phase_kernel(const PcArgs a, uint32_t b) {
  __shared__ int status;
  const PcTask k = pc_task_of(a, pc_base(a, blockIdx.x), b, b % a.buffer_num);
  if (threadIdx.x == 0)
    status = symm::spin_wait(k.slot, symm::kCmpEq, ROLE == 0 ? 0 : 1, a.budget_ns, a.ctl,
                             a.err_base, a.err_bias);
  __syncthreads();
  if (status != symm::kSpinOk) return;  // uniform across the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t stage_row = (size_t)a.H * a.W * a.D * a.es;
  const size_t src_row = (size_t)a.H * a.D * a.es;
  for (uint32_t i = warp; i < k.rows; i += kPcPhaseThreads / 32) {
    if (ROLE == 0)
      symm::warp_copy<4, symm::kRO, symm::kST>(k.stage + i * stage_row, k.src + i * src_row,
                                               k.len, lane);
    else
      symm::warp_copy<4, symm::kCG, symm::kCS>(k.dst + i * stage_row, k.stage + i * stage_row,
                                               k.len, lane);
  }
  __syncthreads();  // the CTA's copies precede the release
  if (threadIdx.x == 0) symm::st_release(k.slot, ROLE == 0 ? 1 : 0);
}
// Every signal slot of every PE to 0 (before a phased call).
__global__ void pc_phase_zero_kernel(const PcArgs a) {
  const size_t per_pe = (size_t)a.buffer_num * a.W * a.nbd * a.H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < per_pe * a.W;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t d = i / per_pe, j = i - d * per_pe;
    *reinterpret_cast<int64_t*>(a.signals + d * a.sig_pe + j * SYMM_SIGNAL_STRIDE_BYTES) = 0;
  }
}

// ------------------------------------------------------------ launching ---
// CTAs of `kernel` (launched with `threads` threads and `smem` bytes of
// dynamic shared memory) that are resident on the current device at once;
// cached.  Raises the kernel's dynamic shared memory limit first if needed.
int resident_ctas(const void* kernel, int threads, size_t smem = 0, size_t smem_limit = 0) {
  static std::mutex mu;
  static std::map<std::pair<std::pair<int, const void*>, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({{dev, kernel}, smem});
  if (it != cache.end()) return it->second;
  if (smem_limit < smem) smem_limit = smem;
  if (smem_limit > 48 * 1024) {
    // at most what the device lets a CTA opt in to, less the kernel's static part
    cudaFuncAttributes fa;
    int optin = 0;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return 0;
    const size_t most = optin > (int)fa.sharedSizeBytes ? optin - fa.sharedSizeBytes : 0;
    if (smem > most) return 0;
    if (smem_limit > most) smem_limit = most;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_limit) != cudaSuccess)
      return 0;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
    return 0;
  const int n = per_sm * sm_count();
  cache[{{dev, kernel}, smem}] = n;
  return n;
}

bool mul_ok(size_t a, size_t b, size_t* out) {
  if (a && b > SIZE_MAX / a) return false;
  *out = a * b;
  return true;
}

// Validates a permutation call; fills the slab offsets and per-PE byte sizes.
int check_perm(symm_heap* h, const void* in, const void* out, int W, size_t rows_in, int H, int D,
               int es, const char* what, size_t* in_off, size_t* out_off, size_t* bytes) {
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  if (W != h->npes)
    return fail(SYMM_EINVAL, std::string(what) + ": W=" + std::to_string(W) +
                                 " differs from the heap's " + std::to_string(h->npes) + " PEs");
  if (H < 0 || D < 0 || es < 1)
    return fail(SYMM_EINVAL, std::string(what) + ": negative extent or elem_bytes < 1");
  if (rows_in > 0x7fffffffull || (size_t)H * W > 0x7fffffffull)
    return fail(SYMM_EINVAL, std::string(what) + ": more than 2^31 rows or columns per PE");
  size_t n;
  if (!mul_ok(rows_in, (size_t)H, &n) || !mul_ok(n, (size_t)D, &n) || !mul_ok(n, (size_t)es, &n))
    return fail(SYMM_EINVAL, std::string(what) + ": size overflow");
  *bytes = n;
  int rc = check_range(h, in, n, (std::string(what) + ": in").c_str(), in_off);
  if (rc) return rc;
  rc = check_range(h, out, n, (std::string(what) + ": out").c_str(), out_off);
  if (rc) return rc;
  if (n && *in_off < *out_off + n && *out_off < *in_off + n)
    return fail(SYMM_EINVAL, std::string(what) + ": input and output ranges overlap");
  return SYMM_OK;
}

// Launches the run permutation with 16-byte vector loads/stores (measured
// fastest), or bulk (TMA) copies when `bulk` is asked and every run is
// 16-byte aligned.
int launch_runs(symm_heap* h, size_t in_off, size_t out_off, uint32_t W, uint32_t Sb, size_t R,
                bool inverse, bool bulk_asked, cudaStream_t s, const char* what) {
  const size_t nruns = (size_t)W * W * Sb;
  if (nruns == 0 || R == 0) return SYMM_OK;
  if (nruns > 0x7fffffffull)
    return fail(SYMM_EINVAL, std::string(what) + ": more than 2^31 runs");
  const uint8_t* in = h->base + in_off;
  uint8_t* out = h->base + out_off;
  const bool bulk = bulk_asked && R % 16 == 0 && in_off % 16 == 0 && out_off % 16 == 0;
  if (bulk) {
    int rc = ensure_ctrl(h, s);
    if (rc) return rc;
    const void* kfn = inverse ? (const void*)a2a_runs_bulk_kernel<true>
                              : (const void*)a2a_runs_bulk_kernel<false>;
    const int cap = resident_ctas(kfn, 32, kBulkSmem);
    if (cap <= 0) return fail(SYMM_ECUDA, std::string(what) + ": bulk kernel set-up failed");
    const uint32_t nchunks = (uint32_t)((R + kBulkChunk - 1) / kBulkChunk);
    const uint64_t units = (uint64_t)nruns * nchunks;
    const int grid = (int)(units < (uint64_t)cap ? units : (uint64_t)cap);
    Control* ctl = reinterpret_cast<Control*>(h->base);
    if (inverse)
      a2a_runs_bulk_kernel<true><<<grid, 32, kBulkSmem, s>>>(in, out, h->slab, W, Sb, R,
                                                             (uint32_t)nruns, nchunks,
                                                             h->spin_budget, ctl);
    else
      a2a_runs_bulk_kernel<false><<<grid, 32, kBulkSmem, s>>>(in, out, h->slab, W, Sb, R,
                                                              (uint32_t)nruns, nchunks,
                                                              h->spin_budget, ctl);
    return cuda_check(cudaGetLastError(), what);
  }
  int rc = ensure_ctrl(h, s);  // the heap header records a wait that gives up
  if (rc) return rc;
  return symm_host::launch_runs_raw(in, out, h->slab, h->slab, W, Sb, R, inverse, s, what,
                                    /*device_mem=*/true, h->base, h->spin_budget);
}

}  // namespace

// The run permutation between any two device-accessible buffers: PE k's
// input at in + k*in_pe, its output at out + k*out_pe (symmetric slabs, or
// page-locked host memory reached over the host link).
int symm_host::launch_runs_raw(const uint8_t* in, uint8_t* out, size_t in_pe, size_t out_pe,
                               uint32_t W, uint32_t Sb, size_t R, bool inverse, cudaStream_t s,
                               const char* what, bool device_mem, void* ctl,
                               uint64_t budget_ns) {
  const size_t nruns = (size_t)W * W * Sb;
  if (nruns == 0 || R == 0) return SYMM_OK;
  if (nruns > 0x7fffffffull) return fail(SYMM_EINVAL, std::string(what) + ": more than 2^31 runs");
  const bool aligned = R % 16 == 0 && (uintptr_t)in % 16 == 0 && (uintptr_t)out % 16 == 0 &&
                       in_pe % 16 == 0 && out_pe % 16 == 0;
  const uint32_t period = inverse ? Sb : W;
  if (aligned && R <= 16 * kBatchMaxVec && period >= 2) {
    // short runs: batches of m runs per warp, about two rounds of vectors each
    const uint32_t nvec = (uint32_t)(R >> 4);
    const uint32_t m = std::min(period, std::max(2u, (uint32_t)(64 * kBatchUnroll) / nvec));
    const void* bfn = inverse ? (const void*)a2a_runs_batch_kernel<true>
                              : (const void*)a2a_runs_batch_kernel<false>;
    int bcap = resident_ctas(bfn, kRunThreads);
    if (bcap <= 0) bcap = 4 * (sm_count() > 0 ? sm_count() : 1);
    const size_t nbatch = nruns / period * ((period + m - 1) / m);
    const size_t bneed = (nbatch + kRunThreads / 32 - 1) / (kRunThreads / 32);
    const int bgrid = (int)(bneed < (size_t)bcap ? bneed : (size_t)bcap);
    if (inverse)
      a2a_runs_batch_kernel<true><<<bgrid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb,
                                                                (uint32_t)R, (uint32_t)nruns, m);
    else
      a2a_runs_batch_kernel<false><<<bgrid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb,
                                                                 (uint32_t)R, (uint32_t)nruns, m);
    return cuda_check(cudaGetLastError(), what);
  }
  // unaligned runs in device memory: bulk loads through per-warp rings, one
  // run per slot from 1 KB up to a slot, batches of shorter runs below
  if (SYMM_RUNS_RING && !aligned && device_mem && ctl) {
    const bool batch = R < kRingMinRun;
    const size_t period = (size_t)W * Sb;  // runs of one input PE
    size_t mb = 1, units = nruns;
    uint32_t glanes = 32;
    if (batch) {
      const size_t bytes = R < 32 ? kRingTinyBatchBytes
                           : R < 384 ? kRingMidBatchBytes
                                     : kRingBatchBytes;
      mb = std::max((size_t)1, std::min(period, bytes / R));
      const size_t nbp = (period + mb - 1) / mb;
      units = (size_t)W * nbp;
      while (glanes > 8 && R < 16u * glanes) glanes >>= 1;
    }
    const size_t slot = (mb * R + 30) & ~(size_t)15;
    if (slot <= kRingMaxSlot) {
      const int mode = !batch ? kRingPerRun : glanes == 32 ? kRingBatchWarp : kRingBatchGroups;
      const void* const fns[2][3] = {
          {(const void*)a2a_runs_ring_kernel<false, kRingPerRun>,
           (const void*)a2a_runs_ring_kernel<false, kRingBatchWarp>,
           (const void*)a2a_runs_ring_kernel<false, kRingBatchGroups>},
          {(const void*)a2a_runs_ring_kernel<true, kRingPerRun>,
           (const void*)a2a_runs_ring_kernel<true, kRingBatchWarp>,
           (const void*)a2a_runs_ring_kernel<true, kRingBatchGroups>}};
      const void* rfn = fns[inverse ? 1 : 0][mode];
      const size_t smem = kRingHeader + (size_t)kRingWarps * kRingSlots * slot;
      const int rcap = resident_ctas(rfn, 32 * kRingWarps, smem,
                                     kRingHeader + (size_t)kRingWarps * kRingSlots * kRingMaxSlot);
      if (rcap > 0) {
        const size_t rneed = (units + kRingWarps - 1) / kRingWarps;
        const int rgrid = (int)(rneed < (size_t)rcap ? rneed : (size_t)rcap);
        const uint32_t nbp = (uint32_t)((period + mb - 1) / mb);
        Control* c = static_cast<Control*>(ctl);
        auto go = [&](auto kern) {
          kern<<<rgrid, 32 * kRingWarps, smem, s>>>(in, out, in_pe, out_pe, W, Sb, (uint32_t)R,
                                                   (uint32_t)units, (uint32_t)mb, nbp, glanes,
                                                   (uint32_t)slot, budget_ns, c);
        };
        if (inverse)
          mode == kRingPerRun      ? go(a2a_runs_ring_kernel<true, kRingPerRun>)
          : mode == kRingBatchWarp ? go(a2a_runs_ring_kernel<true, kRingBatchWarp>)
                                   : go(a2a_runs_ring_kernel<true, kRingBatchGroups>);
        else
          mode == kRingPerRun      ? go(a2a_runs_ring_kernel<false, kRingPerRun>)
          : mode == kRingBatchWarp ? go(a2a_runs_ring_kernel<false, kRingBatchWarp>)
                                   : go(a2a_runs_ring_kernel<false, kRingBatchGroups>);
        return cuda_check(cudaGetLastError(), what);
      }
    }
  }
  const void* kfn = inverse ? (aligned ? (const void*)a2a_runs_kernel<true, true>
                                       : (const void*)a2a_runs_kernel<true, false>)
                            : (aligned ? (const void*)a2a_runs_kernel<false, true>
                                       : (const void*)a2a_runs_kernel<false, false>);
  int cap = resident_ctas(kfn, kRunThreads);
  if (cap <= 0) cap = 4 * (sm_count() > 0 ? sm_count() : 1);
  const size_t need = (nruns + kRunThreads / 32 - 1) / (kRunThreads / 32);
  const int grid = (int)(need < (size_t)cap ? need : (size_t)cap);
  const uint32_t n32 = (uint32_t)nruns;
  if (inverse && aligned)
    a2a_runs_kernel<true, true><<<grid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb, R, n32);
  else if (inverse)
    a2a_runs_kernel<true, false><<<grid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb, R,
                                                             n32);
  else if (aligned)
    a2a_runs_kernel<false, true><<<grid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb, R,
                                                             n32);
  else
    a2a_runs_kernel<false, false><<<grid, kRunThreads, 0, s>>>(in, out, in_pe, out_pe, W, Sb, R,
                                                              n32);
  return cuda_check(cudaGetLastError(), what);
}

// -------------------------------------------------------------- C ABI ---
extern "C" int all2all_pc_workspace(int W, int S, int H, int D, int elem_bytes, int tile_s,
                                    int block_d, int buffer_num, size_t* staging_bytes,
                                    size_t* signal_bytes) {
  if (W < 1 || S < 0 || H < 0 || D < 0 || elem_bytes < 1 || tile_s < 1 || block_d < 0 ||
      buffer_num < 1)
    return fail(SYMM_EINVAL, "all2all_pc_workspace: bad arguments");
  const size_t bd = block_d ? (size_t)block_d : (size_t)D;
  const size_t nbd = bd ? ((size_t)D + bd - 1) / bd : 0;
  size_t st, sg;
  if (!mul_ok((size_t)buffer_num, (size_t)tile_s, &st) || !mul_ok(st, (size_t)H * W, &st) ||
      !mul_ok(st, (size_t)D, &st) || !mul_ok(st, (size_t)elem_bytes, &st))
    return fail(SYMM_EINVAL, "all2all_pc_workspace: size overflow");
  if (!mul_ok((size_t)buffer_num * W, nbd * H, &sg) || !mul_ok(sg, SYMM_SIGNAL_STRIDE_BYTES, &sg))
    return fail(SYMM_EINVAL, "all2all_pc_workspace: size overflow");
  if (staging_bytes) *staging_bytes = st;
  if (signal_bytes) *signal_bytes = sg;
  return SYMM_OK;
}

// Zeroes, picks the instance for and launches one producer/consumer combine.
namespace {
// The kernels' arguments for a plan; false when a tile row exceeds 4 GiB.
bool make_pc_args(const PcPlan& p, PcArgs* out) {
  const uint32_t bd = p.block_d ? (uint32_t)p.block_d : (uint32_t)p.D;
  const uint32_t nbd = (p.D + bd - 1) / bd;
  if ((uint64_t)std::min(bd, (uint32_t)p.D) * p.es > 0xffffffffull) return false;
  PcArgs a;
  a.in = p.in;
  a.out = p.out;
  a.slab = p.slab;
  a.staging = p.staging;
  a.signals = p.signals;
  a.stage_pe = p.stage_pe;
  a.sig_pe = p.sig_pe;
  a.W = p.W;
  a.H = p.H;
  a.S = p.S;
  a.D = p.D;
  a.es = p.es;
  a.tile_s = p.tile_s;
  a.block_d = bd;
  a.nbd = nbd;
  a.nbs = (p.S + p.tile_s - 1) / p.tile_s;
  a.buffer_num = p.buffer_num;
  a.reset = p.reset ? 1u : 0u;
  a.discard = SYMM_PC_DISCARD ? 1u : 0u;
  a.tile_src = (size_t)p.tile_s * p.H * p.D * p.es;
  a.tile_dst = (size_t)p.tile_s * p.H * p.W * p.D * p.es;
  a.stage_buf = a.tile_dst;
  a.slot_buf = (size_t)p.W * nbd * p.H * SYMM_SIGNAL_STRIDE_BYTES;
  a.budget_ns = p.budget_ns;
  a.ctl = static_cast<Control*>(p.ctl);
  a.err_base = p.err_base;
  a.err_bias = p.err_bias;
  *out = a;
  return true;
}

// SYMM_A2A_FLAG_PHASED: zero every slot, then per S block one launch of all
// producers and one of all consumers (see a2a_pc_phase_kernel).
int launch_pc_phased(const PcPlan& p, cudaStream_t s, const char* what) {
  PcArgs a;
  if (!make_pc_args(p, &a))
    return fail(SYMM_EINVAL, std::string(what) + ": a tile row (block_d * elem_bytes) exceeds 4 GiB");
  const size_t tasks = (size_t)a.W * a.W * a.H * a.nbd;
  if (tasks > 0x7fffffffull) return fail(SYMM_EINVAL, std::string(what) + ": too many tasks");
  const size_t slots = tasks * a.buffer_num;
  pc_phase_zero_kernel<<<(unsigned)std::min<size_t>((slots + 255) / 256, 1024), 256, 0, s>>>(a);
  int rc = cuda_check(cudaGetLastError(), what);
  for (uint32_t b = 0; rc == SYMM_OK && b < a.nbs; ++b) {
    a2a_pc_phase_kernel<0><<<(unsigned)tasks, kPcPhaseThreads, 0, s>>>(a, b);
    a2a_pc_phase_kernel<1><<<(unsigned)tasks, kPcPhaseThreads, 0, s>>>(a, b);
    rc = cuda_check(cudaGetLastError(), what);
  }
  return rc;
}
}  // namespace

int symm_host::launch_pc(const PcPlan& p, cudaStream_t s, const char* what) {
  PcArgs a;
  if (!make_pc_args(p, &a))
    return fail(SYMM_EINVAL, std::string(what) + ": a tile row (block_d * elem_bytes) exceeds 4 GiB");
  const uint32_t bd = a.block_d;
  const uint32_t nbd = a.nbd;
  // every tile row, base and row stride 16-byte aligned
  const bool aligned = ((size_t)p.D * p.es) % 16 == 0 && ((size_t)bd * p.es) % 16 == 0 &&
                       (uintptr_t)p.in % 16 == 0 && (uintptr_t)p.out % 16 == 0 &&
                       (uintptr_t)p.staging % 16 == 0 && p.slab % 16 == 0 &&
                       p.stage_pe % 16 == 0;
  // a tile's offsets fit 32 bits (stage_row = H*W*D*es is its widest row stride)
  const size_t stage_row = (size_t)p.H * p.W * p.D * p.es;
  const bool small_tile = (uint64_t)p.tile_s * stage_row < (1ull << 32);
  // the tile copies a group does (see kCopyAligned, kCopyAny, kCopyRows)
  const int mode = !small_tile ? kCopyRows
                   : aligned   ? kCopyAligned
                   : stage_row % 16 == 0 ? kCopyAny
                                         : kCopyRows;
  const size_t tile_bytes = (size_t)p.tile_s * bd * p.es;
  const size_t tasks = (size_t)p.W * p.W * p.H * nbd;
  const size_t row_max = (size_t)std::min(bd, (uint32_t)p.D) * p.es;  // bytes of a full D block
  const void* kfn;
  int threads;
  size_t smem, smem_limit;
  PcRing rg{0, 0, 0};
  bool rel = false;
  {
    // input prefetch by bulk copies (one per tile row) when every tile row is
    // 16-byte aligned and at least kPcMinPrefetchRow bytes, and a tile fits
    // the shared-memory ring; narrower rows are copied faster by the group
    const bool prefetch = !p.vector_only && mode == kCopyAligned &&
                          row_max >= kPcMinPrefetchRow && tile_bytes <= kPcMaxPrefetchTile;
    // rows of any alignment: prefetch of their covering block ranges, in
    // chunks of rows, when staging and output rows share one 16-byte phase
    const size_t any_pitch = (row_max + 30) & ~(size_t)15;
    const bool prefetch_any = SYMM_PC_ANY_PREFETCH && SYMM_PC_RELEASE_WARPS && !p.vector_only &&
                              mode == kCopyAny && row_max >= kPcMinPrefetchRowAny &&
                              any_pitch <= kPcMaxPrefetchTile &&
                              (uintptr_t)p.out % 16 == (uintptr_t)p.staging % 16 &&
                              p.slab % 16 == 0 && p.stage_pe % 16 == 0;
    kfn = prefetch                  ? (const void*)a2a_pc_kernel<true, kCopyAligned>
          : mode == kCopyAligned    ? (const void*)a2a_pc_kernel<false, kCopyAligned>
          : mode == kCopyAny        ? (const void*)a2a_pc_kernel<false, kCopyAny>
                                    : (const void*)a2a_pc_kernel<false, kCopyRows>;
    threads = kPcThreads;
    smem = prefetch ? 128 + (size_t)kPcPrefetch * tile_bytes : 0;
    smem_limit = prefetch ? 128 + (size_t)kPcPrefetch * kPcMaxPrefetchTile : 0;
    if (prefetch && SYMM_PC_RELEASE_WARPS) {
      rg.chunk_rows = (uint32_t)p.tile_s;  // a whole tile per ring entry
      rg.pitch = (uint32_t)row_max;
      rg.stage = (uint32_t)tile_bytes;
      kfn = (const void*)a2a_pc_rel_kernel<false>;
      rel = true;
    } else if (prefetch_any) {
      rg.pitch = (uint32_t)any_pitch;
      rg.chunk_rows = (uint32_t)std::min(
          (size_t)p.tile_s, std::max((size_t)1, (size_t)kPcAnyChunk / any_pitch));
      rg.stage = rg.chunk_rows * rg.pitch;
      kfn = (const void*)a2a_pc_rel_kernel<true>;
      rel = true;
    }
    if (rel) {
      const size_t ring = prefetch ? PcRelConf<false>::ring : PcRelConf<true>::ring;
      threads = kPcRelThreads;
      smem = 128 + ring * rg.stage;
      smem_limit = 128 + ring * kPcMaxPrefetchTile;
    }
  }
  // tasks of one S block, dealt evenly: k per CTA, ceil(tasks / k) CTAs,
  // never more CTAs than are resident at once (each instance measured on its
  // own), so every wait is on a CTA that is running
  const int cap = resident_ctas(kfn, threads, smem, smem_limit);
  if (cap <= 0) return fail(SYMM_ECUDA, std::string(what) + ": occupancy query failed");
  const size_t per_cta = (tasks + cap - 1) / cap;
  const int grid = (int)((tasks + per_cta - 1) / per_cta);
  uint32_t tb = (uint32_t)tile_bytes;
  void* args_pc[] = {&a, &tb};
  void* args_rel[] = {&a, &rg};
  return cuda_check(cudaLaunchKernel(kfn, dim3((unsigned)grid), dim3(threads),
                                     rel ? args_rel : args_pc, smem, s),
                    (std::string(what) + ": PC launch").c_str());
}

static int combine_pc(symm_heap* h, size_t in_off, size_t out_off, size_t nbytes, int W, int S,
                      int H, int D, int es, int flags, int tile_s, int block_d, int buffer_num,
                      void* staging, int64_t* signals, cudaStream_t s) {
  size_t st_bytes, sg_bytes;
  int rc = all2all_pc_workspace(W, S, H, D, es, tile_s, block_d, buffer_num, &st_bytes, &sg_bytes);
  if (rc) return rc;
  size_t st_off, sg_off;
  rc = check_range(h, staging, st_bytes, "all2all_combine: staging", &st_off);
  if (rc) return rc;
  rc = check_range(h, signals, sg_bytes, "all2all_combine: signals", &sg_off);
  if (rc) return rc;
  if (sg_off & 63) return fail(SYMM_EINVAL, "all2all_combine: signals not 64-byte aligned");
  const size_t offs[4] = {in_off, out_off, st_off, sg_off};
  const size_t lens[4] = {nbytes, nbytes, st_bytes, sg_bytes};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (lens[i] && lens[j] && offs[i] < offs[j] + lens[j] && offs[j] < offs[i] + lens[i])
        return fail(SYMM_EINVAL, "all2all_combine: in/out/staging/signals ranges overlap");
  if (nbytes == 0) return SYMM_OK;
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  PcPlan p;
  p.in = h->base + in_off;
  p.out = h->base + out_off;
  p.slab = h->slab;
  p.staging = h->base + st_off;
  p.stage_pe = h->slab;
  p.signals = h->base + sg_off;
  p.sig_pe = h->slab;
  p.W = W;
  p.S = S;
  p.H = H;
  p.D = D;
  p.es = es;
  p.tile_s = tile_s;
  p.block_d = block_d;
  p.buffer_num = buffer_num;
  p.reset = !(flags & SYMM_A2A_FLAG_NO_RESET);
  p.vector_only = (flags & SYMM_A2A_FLAG_VECTOR) != 0;
  p.budget_ns = h->spin_budget;
  p.ctl = h->base;
  p.err_base = h->base;
  p.err_bias = 0;
  if (flags & SYMM_A2A_FLAG_PHASED) return launch_pc_phased(p, s, "all2all_combine");
  return launch_pc(p, s, "all2all_combine");
}

extern "C" int all2all_combine(symm_heap_t* h, const void* in, void* out, int W, int S, int H,
                               int D, int elem_bytes, int variant, int tile_s, int block_d,
                               int buffer_num, void* staging, int64_t* signals, void* stream) {
  if (S < 0 || W < 1) return fail(SYMM_EINVAL, "all2all_combine: S < 0 or W < 1");
  size_t in_off, out_off, nbytes;
  int rc = check_perm(h, in, out, W, (size_t)S * W, H, D, elem_bytes, "all2all_combine", &in_off,
                      &out_off, &nbytes);
  if (rc) return rc;
  const int kind = variant & 0xff, flags = variant & ~0xff;
  if (flags &
      ~(SYMM_A2A_FLAG_NO_RESET | SYMM_A2A_FLAG_VECTOR | SYMM_A2A_FLAG_BULK | SYMM_A2A_FLAG_PHASED))
    return fail(SYMM_EINVAL, "all2all_combine: unknown flag");
  cudaStream_t s = as_stream(stream);
  if (kind == SYMM_A2A_DIRECT)
    return launch_runs(h, in_off, out_off, W, S, (size_t)H * D * elem_bytes, false,
                       (flags & SYMM_A2A_FLAG_BULK) != 0, s, "all2all_combine");
  if (kind == SYMM_A2A_PC)
    return combine_pc(h, in_off, out_off, nbytes, W, S, H, D, elem_bytes, flags, tile_s, block_d,
                      buffer_num, staging, signals, s);
  return fail(SYMM_EINVAL, "all2all_combine: unknown variant " + std::to_string(kind));
}

extern "C" int all2all_dispatch(symm_heap_t* h, const void* in, void* out, int W, int S, int H,
                                int D, int elem_bytes, void* stream) {
  if (S < 0 || W < 1) return fail(SYMM_EINVAL, "all2all_dispatch: S < 0 or W < 1");
  if (S % W) return fail(SYMM_EINVAL, "all2all_dispatch: S must be a multiple of W");
  size_t in_off, out_off, nbytes;
  int rc = check_perm(h, in, out, W, (size_t)S, H, D, elem_bytes, "all2all_dispatch", &in_off,
                      &out_off, &nbytes);
  if (rc) return rc;
  return launch_runs(h, in_off, out_off, W, S / W, (size_t)H * D * elem_bytes, false, false,
                     as_stream(stream), "all2all_dispatch");
}

extern "C" int all2all_combine_back(symm_heap_t* h, const void* in, void* out, int W, int Sp,
                                    int H, int D, int elem_bytes, void* stream) {
  if (Sp < 0 || W < 1) return fail(SYMM_EINVAL, "all2all_combine_back: Sp < 0 or W < 1");
  size_t in_off, out_off, nbytes;
  int rc = check_perm(h, in, out, W, (size_t)Sp * W, H, D, elem_bytes, "all2all_combine_back",
                      &in_off, &out_off, &nbytes);
  if (rc) return rc;
  return launch_runs(h, in_off, out_off, W, Sp, (size_t)H * D * elem_bytes, true, false,
                     as_stream(stream), "all2all_combine_back");
}

