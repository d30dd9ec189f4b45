// two_phase.cu -- the two-phase combine: bulk sends of every cross-PE
// segment into the receiver's rank slot, a double-buffered self loop for the
// segment a PE keeps, and a consumer that permutes both into the output.
//
// Source: "Reverse All2All (EP MoE Distributed Kernel)", section "UDMA
// Optimized Implementation": "Two-Phase Data Copy" (phase 1 moves each
// sender's whole segment for a target in bulk; phase 2 copies the self
// segment tile by tile through a double buffer; the consumer reads rank
// slot r for r != rank, the double buffer for r == rank), "Symmetric Memory
// Layout" (per PE: W rank slots of [S][H][D]; the self slot's first
// buffer_num * block_s rows are the double buffer), and "Wait/Notify
// Optimization" / "Dual Signal Memory Region Design" (region A: one
// write-once slot per (S block, sender), set when that block of the bulk
// send has arrived; region B: one slot per (buffer, self task) with the
// wait-0 / write / notify-1 / consume / credit-0 handshake).
//
// GB300 design: one persistent cooperative launch runs every PE's roles at
// once, each in its own warps of every CTA:
//   sender       streams its (S block, sender, target) chunks with bulk
//                (TMA) copies global -> shared -> global through a 4-stage
//                ring (the GPU's counterpart of the page's bulk engine),
//                waits for the chunk's stores to land, then does a release
//                store of 1 to the chunk's region-A slot: one thread of warp
//                0; layouts that are not 16-byte aligned use 16-byte vector
//                copies by warps 0-1 instead;
//   producer     the self-loop group (region B): warps 1-3 (vector: 2-3);
//   consumer     the consumer group: the remaining 8 warps.
// A CTA keeps the same self tiles for every S block and walks the blocks in
// order (the page's task-to-core mapping), so a self slot's successive
// producers, and its successive consumers, are one group in order.  Remote
// tiles need no credit and are dealt round robin over all CTAs.  Consumers
// wait on senders and producers of other CTAs; the cooperative launch
// guarantees that all CTAs are resident, and every wait is bounded.
#include <algorithm>
#include <map>
#include <mutex>
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

namespace {

constexpr int kTpWarps = 12;  // per CTA: sender, self-loop producer and consumer warps
constexpr int kTpThreads = 32 * kTpWarps;
// Warps per role: bulk sends need one issuing thread; vector sends carry the
// (W-1)/W cross-PE share of the bytes on SM copies and get more warps (two
// sender and two self-loop warps measured best on 1998-byte rows).
#ifndef SYMM_TP_VEC_SENDERS
#define SYMM_TP_VEC_SENDERS 2
#endif
#ifndef SYMM_TP_VEC_PRODUCERS
#define SYMM_TP_VEC_PRODUCERS 2
#endif
#ifndef SYMM_TP_ROW_UNROLL
#define SYMM_TP_ROW_UNROLL 4
#endif
template <bool BULK>
struct TpRoles {
  static constexpr int kSender = BULK ? 1 : SYMM_TP_VEC_SENDERS;
  static constexpr int kProducer = BULK ? 3 : SYMM_TP_VEC_PRODUCERS;
  static constexpr int kConsumer = kTpWarps - kSender - kProducer;
};
constexpr uint32_t kTpPiece = 16384;  // bytes of one bulk copy
constexpr int kTpStages = 4;
constexpr size_t kTpSmem = 128 + (size_t)kTpStages * kTpPiece;
#ifndef SYMM_TP_UNROLL
#define SYMM_TP_UNROLL 8
#endif
constexpr int kTpUnroll = SYMM_TP_UNROLL;  // vectors in flight per thread in a tile copy
#ifndef SYMM_TP_ROW_MIN_BLOCKS  // CTAs per SM of the instances that copy by rows
#define SYMM_TP_ROW_MIN_BLOCKS 2
#endif
#ifndef SYMM_TP_MIN_BLOCKS
#define SYMM_TP_MIN_BLOCKS 1
#endif

struct TpArgs {
  const uint8_t* in;  // PE 0 copies of the symmetric objects; PE k at +k*slab
  uint8_t* out;
  uint8_t* bulk;      // rank slots [W][S][H][D] per PE
  uint8_t* signals;   // region A [nbs][W], then region B [buffer_num][nbd*H], 64 B apart
  size_t slab;
  size_t row;         // bytes of one [H][D] row
  uint32_t W, S, H, D, es, tile_s, block_d, nbd, nbs, buffer_num;
  uint64_t budget_ns;
  Control* ctl;
  const uint8_t* heap_base;
};

__device__ __forceinline__ int64_t* sig_a(const TpArgs& a, uint32_t d, uint32_t b, uint32_t r) {
  return reinterpret_cast<int64_t*>(a.signals + d * a.slab +
                                    ((size_t)b * a.W + r) * SYMM_SIGNAL_STRIDE_BYTES);
}
__device__ __forceinline__ int64_t* sig_b(const TpArgs& a, uint32_t d, uint32_t buf,
                                          uint32_t task) {
  const size_t slot = (size_t)a.nbs * a.W + (size_t)buf * a.H * a.nbd + task;
  return reinterpret_cast<int64_t*>(a.signals + d * a.slab + slot * SYMM_SIGNAL_STRIDE_BYTES);
}

// Sender unit u = b * W(W-1) + p: S block b of the segment PE r holds for
// PE d != r (p = d*(W-1) + k, r = k, skipping d).  Rows d*S + s0 .. of r's
// input land at rows r*S + s0 .. of d's rank slots; both are contiguous.
struct TpChunk {
  const uint8_t* src;
  uint8_t* dst;
  size_t len;
  int64_t* sig;
};
__device__ __forceinline__ TpChunk tp_chunk(const TpArgs& a, uint64_t u) {
  const uint32_t pairs = a.W * (a.W - 1);
  const uint32_t b = (uint32_t)(u / pairs), p = (uint32_t)(u % pairs);
  const uint32_t d = p / (a.W - 1), k = p % (a.W - 1), r = k < d ? k : k + 1;
  const uint32_t s0 = b * a.tile_s, rows = min(a.tile_s, a.S - s0);
  return TpChunk{a.in + r * a.slab + ((size_t)d * a.S + s0) * a.row,
                 a.bulk + d * a.slab + ((size_t)r * a.S + s0) * a.row, (size_t)rows * a.row,
                 sig_a(a, d, b, r)};
}

// Phase 1 with bulk copies: one thread keeps kTpStages pieces of its chunks
// in flight (load cursor ahead of the store cursor); a chunk's signal is
// released once all its stores have completed.
__device__ __noinline__ void tp_send_bulk(const TpArgs& a, uint8_t* smem) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + 128;
  for (int i = 0; i < kTpStages; ++i) symm::mbar_init(&bars[i], 1);
  symm::fence_mbar_init();
  const uint64_t units = (uint64_t)a.nbs * a.W * (a.W - 1);
  uint64_t lu = blockIdx.x, su = blockIdx.x;  // load / store cursors: unit ...
  size_t loff = 0, soff = 0;                  // ... and byte offset inside it
  uint64_t issued = 0, done = 0;              // pieces
  for (;;) {
    while (issued - done < (uint64_t)kTpStages && lu < units) {  // refill the ring
      const TpChunk c = tp_chunk(a, lu);
      const uint32_t n = (uint32_t)min((size_t)kTpPiece, c.len - loff);
      const int st = (int)(issued % kTpStages);
      symm::mbar_arrive_expect_tx(&bars[st], n);
      symm::bulk_load(ring + (size_t)st * kTpPiece, c.src + loff, n, &bars[st]);
      ++issued;
      loff += n;
      if (loff == c.len) {
        loff = 0;
        lu += gridDim.x;
      }
    }
    if (done == issued) break;
    const int st = (int)(done % kTpStages);
    if (!symm::mbar_wait(&bars[st], (uint32_t)(done / kTpStages) & 1u, a.budget_ns)) {
      symm::record_error(a.ctl, symm::kErrTimedOut, -1);
      for (uint64_t i = done; i < issued; ++i)  // let the loads in flight land (bounded)
        symm::mbar_wait(&bars[i % kTpStages], (uint32_t)(i / kTpStages) & 1u, a.budget_ns);
      break;
    }
    const TpChunk c = tp_chunk(a, su);
    const uint32_t n = (uint32_t)min((size_t)kTpPiece, c.len - soff);
    symm::bulk_store(c.dst + soff, ring + (size_t)st * kTpPiece, n);
    symm::bulk_commit();
    ++done;
    soff += n;
    if (soff == c.len) {  // the chunk has been sent: publish it
      symm::bulk_wait<0>();
      symm::fence_proxy_async_global();
      symm::st_release(c.sig, 1);
      soff = 0;
      su += gridDim.x;
    }
    symm::bulk_wait_read<0>();  // this stage's store has read it before a refill
  }
  symm::bulk_wait<0>();
}

// Phase 1 with 16-byte vector copies (layouts that bulk copies cannot take):
// sender warp `sw` of `nsw` in each CTA takes every (G * nsw)-th chunk.
__device__ __noinline__ void tp_send_vector(const TpArgs& a, int sw, int nsw, int lane) {
  const uint64_t units = (uint64_t)a.nbs * a.W * (a.W - 1);
  for (uint64_t u = (uint64_t)blockIdx.x * nsw + sw; u < units; u += (uint64_t)gridDim.x * nsw) {
    const TpChunk c = tp_chunk(a, u);
    symm::warp_copy<SYMM_TP_ROW_UNROLL, symm::kRO, symm::kST>(c.dst, c.src, c.len, lane);
    __syncwarp();  // the lanes' stores precede lane 0's release
    if (lane == 0) symm::st_release(c.sig, 1);
  }
}

// A group of n threads copies a tile of `rows` rows of `nv` 16-byte vectors
// (both sides 16-byte aligned; the tile spans less than 4 GiB on each side).
// Vector k of the tile is row k / nv, column k % nv; a thread takes vectors
// tid, tid + n, ..., kTpUnroll of them in flight, walking (row, column)
// incrementally so no division is left in the loop.
template <int LK, int SK>
__device__ __forceinline__ void tp_group_copy(uint8_t* dst, uint32_t dstride, const uint8_t* src,
                                              uint32_t sstride, uint32_t rows, uint32_t nv,
                                              int tid, int n) {
  const uint32_t total = rows * nv;
  const uint32_t di = (uint32_t)n / nv, dc = (uint32_t)n % nv;
  uint32_t i = (uint32_t)tid / nv, c = (uint32_t)tid % nv;
  for (uint32_t k0 = tid; k0 < total; k0 += (uint32_t)n * kTpUnroll) {
    uint4 v[kTpUnroll];
    uint32_t ii = i, cc = c;
#pragma unroll
    for (int u = 0; u < kTpUnroll; ++u) {
      if (k0 + (uint32_t)(u * n) < total) v[u] = symm::ld16<LK>(src + (ii * sstride + 16 * cc));
      cc += dc;
      ii += di + (cc >= nv);
      cc -= cc >= nv ? nv : 0;
    }
#pragma unroll
    for (int u = 0; u < kTpUnroll; ++u) {
      if (k0 + (uint32_t)(u * n) < total) symm::st16k<SK>(dst + (i * dstride + 16 * c), v[u]);
      c += dc;
      i += di + (c >= nv);
      c -= c >= nv ? nv : 0;
    }
  }
}

// The self-loop producer group or the consumer group of a CTA.
struct TpGroup {
  int gtid, gwarp, nwarps, nthreads, bar_id;
  int* status;  // [2], indexed by the group's task parity
  bool producer;
};

// One tile: thread 0 waits for the tile's slot, the group copies up to
// tile_s rows of block_d elements, and -- for a producer, or a consumer of a
// self tile -- thread 0 then releases the slot (1: filled, 0: credit
// returned).  Returns false when the wait gave up.
template <bool ALIGNED>
__device__ __forceinline__ bool tp_tile(const TpArgs& a, const TpGroup& g, uint32_t t, uint32_t b,
                                        uint32_t d, uint32_t r, uint32_t h, uint32_t bd,
                                        int lane) {
  const bool self = r == d;
  const uint32_t buf = b % a.buffer_num, s0 = b * a.tile_s;
  const uint32_t rows = min(a.tile_s, a.S - s0);
  int64_t* slot = self ? sig_b(a, d, buf, bd * a.H + h) : sig_a(a, d, b, r);
  if (g.gtid == 0)
    g.status[t & 1] = symm::spin_wait(slot, symm::kCmpEq, g.producer ? 0 : 1, a.budget_ns, a.ctl,
                                      a.heap_base);
  symm::group_sync(g.bar_id, g.nthreads);
  if (g.status[t & 1] != symm::kSpinOk) return false;  // uniform across the group
  const uint32_t x0 = bd * a.block_d;
  const size_t len = (size_t)min(a.block_d, a.D - x0) * a.es;
  const size_t col = ((size_t)h * a.D + x0) * a.es;
  // PE d's rank slot r (self: the double buffer at the start of slot d)
  uint8_t* slot_row0 = a.bulk + d * a.slab +
                       ((size_t)r * a.S + (self ? (size_t)buf * a.tile_s : s0)) * a.row + col;
  const uint8_t* src;
  uint8_t* dst;
  size_t sstride, dstride;
  if (g.producer) {
    src = a.in + d * a.slab + ((size_t)d * a.S + s0) * a.row + col;
    dst = slot_row0;
    sstride = dstride = a.row;
  } else {
    src = slot_row0;
    dst = a.out + d * a.slab + (size_t)s0 * a.row * a.W + (size_t)r * a.row + col;
    sstride = a.row;
    dstride = a.row * a.W;
  }
  if (ALIGNED) {
    // every row segment 16-byte aligned: the group's threads share the
    // tile's vectors, kTpUnroll in flight per thread
    if (g.producer)
      tp_group_copy<symm::kRO, symm::kST>(dst, (uint32_t)dstride, src, (uint32_t)sstride, rows,
                                          (uint32_t)(len >> 4), g.gtid, g.nthreads);
    else
      tp_group_copy<symm::kCG, symm::kCS>(dst, (uint32_t)dstride, src, (uint32_t)sstride, rows,
                                          (uint32_t)(len >> 4), g.gtid, g.nthreads);
  } else if (g.producer) {
    for (uint32_t i = g.gwarp; i < rows; i += g.nwarps)
      symm::warp_copy<SYMM_TP_ROW_UNROLL, symm::kRO, symm::kST>(dst + i * dstride,
                                                                src + i * sstride, len, lane);
  } else {
    for (uint32_t i = g.gwarp; i < rows; i += g.nwarps)
      symm::warp_copy<SYMM_TP_ROW_UNROLL, symm::kCG, symm::kCS>(dst + i * dstride,
                                                                src + i * sstride, len, lane);
  }
  if (g.producer || self) {
    symm::group_sync(g.bar_id, g.nthreads);  // the group's copies precede the release
    if (g.gtid == 0) symm::st_release(slot, g.producer ? 1 : 0);
  }
  return true;
}

// BULK: sender chunks are 16-byte aligned (bulk copies); ALIGNED (implies
// BULK): every tile row segment is too (group-wide vector tile copies).
template <bool BULK, bool ALIGNED>
__global__ void __launch_bounds__(kTpThreads,
                                  ALIGNED ? SYMM_TP_MIN_BLOCKS : SYMM_TP_ROW_MIN_BLOCKS)
    a2a_two_phase_kernel(const TpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int status[2][2];
  using R = TpRoles<BULK>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < R::kSender) {
    if (BULK) {
      if (lane == 0) tp_send_bulk(a, smem);
    } else {
      tp_send_vector(a, warp, R::kSender, lane);
    }
    return;
  }
  TpGroup g;
  g.producer = warp < R::kSender + R::kProducer;
  g.gtid = threadIdx.x - 32 * (g.producer ? R::kSender : R::kSender + R::kProducer);
  g.gwarp = g.gtid >> 5;
  g.nwarps = g.producer ? R::kProducer : R::kConsumer;
  g.nthreads = 32 * g.nwarps;
  g.bar_id = g.producer ? 1 : 2;
  g.status = status[g.producer ? 0 : 1];
  const uint32_t G = gridDim.x;
  const size_t ht = (size_t)a.H * a.nbd;     // tiles per (PE, source) and S block
  const size_t qs = a.W * ht;                // self tiles per S block
  const size_t qr = (size_t)(a.W - 1) * qs;  // remote tiles per S block
  uint32_t t = 0;
  for (uint32_t b = 0; b < a.nbs; ++b) {
    // self tiles, q = (d*nbd + bd)*H + h: the same CTA for every S block
    for (size_t q = blockIdx.x; q < qs; q += G, ++t) {
      const uint32_t d = (uint32_t)(q / ht), h = (uint32_t)(q % a.H);
      const uint32_t bd = (uint32_t)((q % ht) / a.H);
      if (!tp_tile<ALIGNED>(a, g, t, b, d, d, h, bd, lane)) return;
    }
    if (g.producer) continue;
    // remote tiles, q = ((d*(W-1) + k)*H + h)*nbd + bd: dealt round robin
    // over all CTAs in (S block, q) order
    const uint64_t base = (uint64_t)b * qr;
    for (uint64_t gq = base + (blockIdx.x + G - base % G) % G; gq < base + qr; gq += G, ++t) {
      uint64_t v = gq - base;
      const uint32_t bd = (uint32_t)(v % a.nbd);
      v /= a.nbd;
      const uint32_t h = (uint32_t)(v % a.H);
      v /= a.H;
      const uint32_t k = (uint32_t)(v % (a.W - 1)), d = (uint32_t)(v / (a.W - 1));
      if (!tp_tile<ALIGNED>(a, g, t, b, d, k < d ? k : k + 1, h, bd, lane)) return;
    }
  }
}

__global__ void tp_signal_reset_kernel(uint8_t* signals, size_t slab, uint32_t W, size_t nslots) {
  const size_t per_pe = nslots * (SYMM_SIGNAL_STRIDE_BYTES / 8);
  const size_t n = (size_t)W * per_pe;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    reinterpret_cast<int64_t*>(signals + (i / per_pe) * slab)[i % per_pe] = 0;
}

// The kernel instance for a layout: 0 = vector copies everywhere, 1 = bulk
// sender chunks, 2 = bulk chunks and group-wide tile copies.
const void* tp_kernel(int mode) {
  if (mode == 2) return (const void*)a2a_two_phase_kernel<true, true>;
  if (mode == 1) return (const void*)a2a_two_phase_kernel<true, false>;
  return (const void*)a2a_two_phase_kernel<false, false>;
}

// Co-resident CTAs of an instance on the current device (cached).
int tp_capacity(int mode) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({dev, mode});
  if (it != cache.end()) return it->second;
  const void* k = tp_kernel(mode);
  const size_t smem = mode ? kTpSmem : 0;
  if (mode && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                  cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTpThreads, smem) != cudaSuccess)
    return 0;
  const int n = per_sm * sm_count();
  cache[{dev, mode}] = n;
  return n;
}

struct TpShape {
  size_t row, nbytes, bulk_bytes, signal_bytes, nslots;
  uint32_t nbs, nbd, block_d;
};

int tp_shape(int W, int S, int H, int D, int es, int tile_s, int block_d, int buffer_num,
             const char* what, TpShape* o) {
  if (W < 1 || S < 0 || H < 0 || D < 0 || es < 1)
    return fail(SYMM_EINVAL, std::string(what) + ": W < 1, a negative extent or elem_bytes < 1");
  if (tile_s < 1 || block_d < 0 || buffer_num < 1)
    return fail(SYMM_EINVAL, std::string(what) + ": tile_s < 1, block_d < 0 or buffer_num < 1");
  if ((uint64_t)S * W > 0x7fffffffull || (uint64_t)H * D > 0x7fffffffull || W > 65536)
    return fail(SYMM_EINVAL, std::string(what) + ": extents too large");
  o->block_d = (uint32_t)(block_d == 0 || block_d > D ? (D > 0 ? D : 1) : block_d);
  o->nbs = (uint32_t)((S + tile_s - 1) / tile_s);
  o->nbd = (uint32_t)((D + o->block_d - 1) / o->block_d);
  o->row = (size_t)H * D * es;
  if (o->row && (size_t)S * W > SIZE_MAX / 4 / o->row)
    return fail(SYMM_EINVAL, std::string(what) + ": size overflow");
  o->nbytes = (size_t)S * W * o->row;
  o->bulk_bytes = o->nbytes;
  o->nslots = (size_t)o->nbs * W + (size_t)buffer_num * H * o->nbd;
  o->signal_bytes = o->nslots * SYMM_SIGNAL_STRIDE_BYTES;
  return SYMM_OK;
}

}  // namespace

extern "C" int all2all_two_phase_workspace(int W, int S, int H, int D, int elem_bytes, int tile_s,
                                           int block_d, int buffer_num, size_t* bulk_bytes,
                                           size_t* signal_bytes) {
  TpShape sh;
  int rc = tp_shape(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num,
                    "all2all_two_phase_workspace", &sh);
  if (rc) return rc;
  if (bulk_bytes) *bulk_bytes = sh.bulk_bytes;
  if (signal_bytes) *signal_bytes = sh.signal_bytes;
  return SYMM_OK;
}

extern "C" int all2all_combine_two_phase(symm_heap_t* h, const void* in, void* out, int W, int S,
                                         int H, int D, int elem_bytes, int tile_s, int block_d,
                                         int buffer_num, void* bulk, int64_t* signals,
                                         void* stream) {
  const char* what = "all2all_combine_two_phase";
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  TpShape sh;
  int rc = tp_shape(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num, what, &sh);
  if (rc) return rc;
  if (W != h->npes) return fail(SYMM_EINVAL, std::string(what) + ": W differs from the heap's PEs");
  size_t off[4];
  const void* ptr[4] = {in, out, bulk, signals};
  const size_t len[4] = {sh.nbytes, sh.nbytes, sh.bulk_bytes, sh.signal_bytes};
  const char* names[4] = {"in", "out", "bulk", "signals"};
  for (int i = 0; i < 4; ++i) {
    rc = check_range(h, ptr[i], len[i], (std::string(what) + ": " + names[i]).c_str(), &off[i]);
    if (rc) return rc;
  }
  if (off[3] & 7) return fail(SYMM_EINVAL, std::string(what) + ": signals not 8-byte aligned");
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (len[i] && len[j] && off[i] < off[j] + len[j] && off[j] < off[i] + len[i])
        return fail(SYMM_EINVAL, std::string(what) + ": " + names[i] + " and " + names[j] +
                                     " overlap");
  if (sh.nbytes == 0) return SYMM_OK;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  uint8_t* sig = h->base + off[3];
  const size_t words = (size_t)W * sh.nslots * (SYMM_SIGNAL_STRIDE_BYTES / 8);
  tp_signal_reset_kernel<<<(unsigned)std::min<size_t>((words + 255) / 256, 1024), 256, 0, s>>>(
      sig, h->slab, (uint32_t)W, sh.nslots);
  rc = cuda_check(cudaGetLastError(), "all2all_combine_two_phase: signal reset");
  if (rc) return rc;

  TpArgs a;
  a.in = h->base + off[0];
  a.out = h->base + off[1];
  a.bulk = h->base + off[2];
  a.signals = sig;
  a.slab = h->slab;
  a.row = sh.row;
  a.W = (uint32_t)W;
  a.S = (uint32_t)S;
  a.H = (uint32_t)H;
  a.D = (uint32_t)D;
  a.es = (uint32_t)elem_bytes;
  a.tile_s = (uint32_t)tile_s;
  a.block_d = sh.block_d;
  a.nbd = sh.nbd;
  a.nbs = sh.nbs;
  a.buffer_num = (uint32_t)buffer_num;
  a.budget_ns = h->spin_budget;
  a.ctl = reinterpret_cast<Control*>(h->base);
  a.heap_base = h->base;
  const bool bulk_ok = sh.row % 16 == 0 && off[0] % 16 == 0 && off[2] % 16 == 0;
  const bool aligned = bulk_ok && off[1] % 16 == 0 &&
                       ((size_t)sh.block_d * elem_bytes) % 16 == 0 &&
                       ((size_t)D * elem_bytes) % 16 == 0 &&
                       (size_t)tile_s * sh.row * W < (1ull << 32);
  const int mode = aligned ? 2 : bulk_ok ? 1 : 0;
  const int cap = tp_capacity(mode);
  if (cap <= 0) return fail(SYMM_ECUDA, std::string(what) + ": occupancy query failed");
  const size_t work = std::max<size_t>((size_t)sh.nbs * W * W * sh.nbd * H,
                                       (size_t)sh.nbs * W * (W - 1) /
                                           (mode ? 1 : SYMM_TP_VEC_SENDERS));
  const int grid = (int)std::min<size_t>((size_t)cap, std::max<size_t>(work, 1));
  void* args[] = {&a};
  return cuda_check(cudaLaunchCooperativeKernel(tp_kernel(mode), grid, kTpThreads, args,
                                                mode ? kTpSmem : 0, s),
                    "all2all_combine_two_phase: launch");
}
