// ag_gemm.cu -- fused AllGather + MatMul on the emulated symmetric heap.
//
// Source: HyperParallel RFC "Symmetric Memory (one-sided communication)",
// section 10 (fused_all_gather_matmul: every rank pushes its rows block by
// block to all ranks, and the matmul of a block starts as soon as that
// block's signal has arrived) and its example 2 (a: m_local x k per rank, b:
// k x n per rank, gather_out: m_total x k, result m_total x n per rank).
// The result on PE d is gather_out_d @ b_d, the gathered rows stacked in rank
// order.
//
// GB300 design: one persistent cooperative launch runs every PE's push and
// matmul at once, 256 threads per CTA, one CTA per SM:
//   warp 0      TMA producer: per output tile (PE d, 128 rows, 256 columns)
//               it waits (acquire, bounded) for the signal of the 128-row
//               block the tile reads (tiles of PE d's own rows read a_d and
//               wait for nothing), then streams 64-wide K slices of A
//               (the gathered rows, K-major) and B (b_d as stored: N-major,
//               in 64-column boxes) into a 4-stage shared-memory ring,
//               128-byte swizzled;
//   warp 1      MMA issuer: owns 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and issues tcgen05.mma kind::f16
//               (M 128, N 256, K 16) from the ring, committing each stage
//               back to the producer and each finished tile to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp its 32 TMEM
//               lanes), rounding to the input type, 128-byte-swizzled boxes
//               in shared memory and TMA stores to c_d; the other
//               accumulator is filled meanwhile;
//   warps 6-7   push: 16 KB pieces of every rank's 128-row blocks, each read
//               once and stored to all W PEs' gather_out; the warp that
//               completes a block (acquire/release count) sets that block's
//               signal on every PE.
// Every CTA works alone (no thread-block clusters): each loads its own A and
// B slices into its own shared memory.
// b is read in place (row-major k x n) as an MN-major operand.  Every wait
// is bounded; a role that gives up
// records the error, and the CTA drains its in-flight copies and MMAs before
// it frees TMEM.
#include <cuda.h>  // CUtensorMap and its enums (types only)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

namespace {

#ifndef SYMM_AG_BN
#define SYMM_AG_BN 256
#endif
#ifndef SYMM_AG_STAGES
#define SYMM_AG_STAGES 4
#endif
// tile: kBM x kBN outputs, kBK-wide K slices (64 x 2 bytes = one 128-byte swizzle span)
constexpr int kBM = 128, kBN = SYMM_AG_BN, kBK = 64;
constexpr int kStages = SYMM_AG_STAGES;

constexpr uint32_t kATile = kBM * kBK * 2;
constexpr uint32_t kBTile = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kATile + kBTile;
#ifndef SYMM_AG_PUSH_WARPS
#define SYMM_AG_PUSH_WARPS 2
#endif
constexpr int kPushWarps = SYMM_AG_PUSH_WARPS;
constexpr int kAgThreads = 32 * (6 + kPushWarps);  // TMA, MMA, 4 epilogue, push
constexpr uint32_t kTmemCols = 2 * kBN;  // two accumulators of kBN fp32 columns
// epilogue staging: per epilogue warp two 32-row x 64-column output boxes
// (4 KB each, 128-byte swizzled) for TMA stores
constexpr uint32_t kOutBox = 32 * 64 * 2;
constexpr uint32_t kOutBytes = 4 * 2 * kOutBox;
constexpr size_t kAgSmem = 1024 + (size_t)kStages * kStageBytes + kOutBytes + 256;
constexpr uint32_t kPushPiece = 16384;
constexpr int kPushUnroll = 4;

struct AgArgs {
  const uint8_t* a;  // PE 0 copies of the symmetric objects; PE k at +k*slab
  uint8_t* gather;
  uint8_t* c;
  uint8_t* signals;  // per PE: W*nblk slots, 64 B apart; then (PE 0) W*nblk counters
  size_t slab;
  uint32_t W, m_local, k, n, nblk, ktiles, ntiles_n;
  uint64_t tiles;
  uint32_t pe_major;  // tile order after the self tiles (see ag_tile)
  uint64_t budget_ns;
  Control* ctl;
  const uint8_t* heap_base;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(symm::smem_addr(bar)) : "memory");
}
// Bounded wait that also gives up once any waiter of the heap has given up.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t* bar, uint32_t parity, uint64_t budget_ns,
                                             const Control* ctl) {
  const uint64_t t0 = symm::globaltimer_ns();
  const uint64_t max_iters = budget_ns / 32 + (1u << 20);
  for (uint64_t it = 0;; ++it) {
    if (symm::mbar_try_wait(bar, parity)) return true;
    if ((it & 255) == 255 &&
        (symm::ld_relaxed_u32(&ctl->abort) || symm::globaltimer_ns() - t0 > budget_ns ||
         it > max_iters))
      return false;
  }
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(symm::smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(symm::smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(symm::smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   symm::smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, kind::f16.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   symm::smem_addr(bar))
               : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per lane).
// The load and its wait are one asm statement, so no use of the registers
// can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(const void* tile) {
  const uint64_t addr = symm::smem_addr(tile);
  return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of one type
// (fmt 0 = fp16, 1 = bf16), A K-major, B MN-major (bit 16), N = kBN, M = kBM.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t fmt) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) | ((uint32_t)(kBN >> 3) << 17) |
         ((uint32_t)(kBM >> 4) << 24);
}

// Shared-memory descriptor of an MN-major B tile written by TMA in boxes of
// 64 N-elements (one 128-byte swizzled row) x kBK K-rows: 8-row K groups are
// 1024 bytes apart, 64-column N groups one box (kBK * 128 bytes) apart.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(const void* tile) {
  const uint64_t addr = symm::smem_addr(tile);
  return ((addr & 0x3FFFFull) >> 4) | ((uint64_t)((kBK * 128) >> 4) << 16) |
         ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ uint64_t atom_add_acq_rel_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ int64_t* ag_signal(const AgArgs& a, uint32_t d, uint32_t r,
                                              uint32_t blk) {
  return reinterpret_cast<int64_t*>(a.signals + d * a.slab +
                                    ((size_t)r * a.nblk + blk) * SYMM_SIGNAL_STRIDE_BYTES);
}
__device__ __forceinline__ int64_t* ag_counter(const AgArgs& a, uint32_t r, uint32_t blk) {
  return reinterpret_cast<int64_t*>(a.signals + (size_t)a.W * a.nblk * SYMM_SIGNAL_STRIDE_BYTES +
                                    ((size_t)r * a.nblk + blk) * 8);
}

// Output tile t: PE d, source rank r = (d + jr) % W, its 128-row block jb,
// columns nt*kBN ..  Every PE's own rows (jr = 0) come first, all PEs
// together: they are read from a_d itself and wait for no signal (the
// page's "start with local data") while the push delivers the other ranks'
// blocks.  Within a row block the kBN-column tiles are consecutive, so the
// block is read from L2.  The remaining tiles come in one of two orders:
//   pe_major = 0: (jr, jb, d, nt) -- every PE advances through the blocks in
//                 push order, so few tiles wait for the push; used when all
//                 W b matrices fit in L2 together;
//   pe_major = 1: (d, jr, jb, nt) -- one PE's tiles are consecutive, so b_d
//                 stays in L2 while the row blocks stream past it (when the
//                 b matrices do not fit, the first order re-reads them from
//                 DRAM: 1010 against 1550 TFLOP/s at k = n = 4096).
struct AgTile {
  uint32_t d, r, jb, m0, n0;
  bool self;
};
__device__ __forceinline__ AgTile ag_tile(const AgArgs& a, uint64_t t) {
  AgTile x;
  const uint32_t nb = a.nblk, ntn = a.ntiles_n;
  const uint64_t n_self = (uint64_t)a.W * nb * ntn;
  const bool self = t < n_self;
  uint64_t v = self ? t : t - n_self;
  const uint32_t nt = (uint32_t)(v % ntn);
  v /= ntn;
  uint32_t jr = 0;
  if (self) {  // (d, jb, nt)
    x.jb = (uint32_t)(v % nb);
    x.d = (uint32_t)(v / nb);
  } else if (a.pe_major) {  // (d, jr - 1, jb, nt)
    x.jb = (uint32_t)(v % nb);
    v /= nb;
    jr = 1 + (uint32_t)(v % (a.W - 1));
    x.d = (uint32_t)(v / (a.W - 1));
  } else {  // (jr - 1, jb, d, nt)
    x.d = (uint32_t)(v % a.W);
    v /= a.W;
    x.jb = (uint32_t)(v % nb);
    jr = 1 + (uint32_t)(v / nb);
  }
  x.self = self;
  x.r = (x.d + jr) % a.W;
  x.m0 = x.r * a.m_local + x.jb * kBM;
  x.n0 = nt * kBN;
  return x;
}

template <int FMT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if (FMT == 1) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// The tensor maps are __grid_constant__ parameters.
template <int FMT>
__global__ void __launch_bounds__(kAgThreads, 1)
    ag_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                   const __grid_constant__ CUtensorMap tma_local,
                   const __grid_constant__ CUtensorMap tma_b,
                   const __grid_constant__ CUtensorMap tma_c, const AgArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (symm::smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* out_stage = smem + kStages * kStageBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + kOutBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      symm::mbar_init(&full[s], 1);
      symm::mbar_init(&empty[s], 1);  // freed by this CTA's MMAs
    }
    for (int b = 0; b < 2; ++b) {
      symm::mbar_init(&tfull[b], 1);
      symm::mbar_init(&tempty[b], 128);
    }
    symm::mbar_init(drain, 1);
    symm::fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t G = gridDim.x;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------- TMA producer
      uint64_t it = 0;
      bool ok = true;
      for (uint64_t t = blockIdx.x; ok && t < a.tiles; t += G) {
        const AgTile x = ag_tile(a, t);
        if (!x.self && symm::spin_wait(ag_signal(a, x.d, x.r, x.jb), symm::kCmpEq, 1, a.budget_ns,
                                       a.ctl, a.heap_base) != symm::kSpinOk) {
          ok = false;
          break;
        }
        symm::fence_proxy_async_global();  // the pushed rows, for the async-proxy loads
        for (uint32_t kt = 0; kt < a.ktiles; ++kt, ++it) {
          const int s = (int)(it % kStages);
          if (!mbar_wait_ab(&empty[s], (uint32_t)((it / kStages) & 1) ^ 1u, a.budget_ns, a.ctl)) {
            symm::record_error(a.ctl, symm::kErrTimedOut, -3);
            ok = false;
            break;
          }
          uint8_t* st = smem + (size_t)s * kStageBytes;
          symm::mbar_arrive_expect_tx(&full[s], kStageBytes);
          // A: rows jb*128 .. of a_d itself (own rows) or of the gathered rows
          const CUtensorMap* amap = x.self ? &tma_local : &tma_a;
          const int ay = (int)(x.self ? x.jb * kBM : x.m0);
          tma_load_3d(st, amap, (int)(kt * kBK), ay, (int)x.d, &full[s]);
          // B: b itself, row-major, in 64 N x kBK K boxes
          for (int i = 0; i < kBN / 64; ++i)
            tma_load_3d(st + kATile + i * (kBK * 128), &tma_b, (int)(x.n0 + 64 * i),
                        (int)(kt * kBK), (int)x.d, &full[s]);
        }
      }
      // every load issued lands before the CTA may leave (bounded)
      for (uint64_t i = it > (uint64_t)kStages ? it - kStages : 0; i < it; ++i)
        symm::mbar_wait(&full[i % kStages], (uint32_t)((i / kStages) & 1), a.budget_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // -------------------------------------- MMA issuer
      const uint32_t idesc = mma_idesc(FMT);
      uint64_t it = 0, tc = 0;
      bool ok = true;
      for (uint64_t t = blockIdx.x; ok && t < a.tiles; t += G, ++tc) {
        const uint32_t buf = (uint32_t)(tc & 1);
        if (!mbar_wait_ab(&tempty[buf], (uint32_t)((tc >> 1) & 1) ^ 1u, a.budget_ns, a.ctl)) {
          symm::record_error(a.ctl, symm::kErrTimedOut, -4);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * kBN;
        for (uint32_t kt = 0; kt < a.ktiles; ++kt, ++it) {
          const int s = (int)(it % kStages);
          if (!mbar_wait_ab(&full[s], (uint32_t)((it / kStages) & 1), a.budget_ns, a.ctl)) {
            symm::record_error(a.ctl, symm::kErrTimedOut, -5);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + (size_t)s * kStageBytes;
          const uint64_t ad = sw128_kmajor_desc(st);
          const uint64_t bd = sw128_mnmajor_desc(st + kATile);
          constexpr uint64_t kBStep = (16 * 128) >> 4;  // B: 16 K-rows of 128 bytes
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)  // K = 16 per instruction (A: +32 bytes)
            tc_mma(acc, ad + 2 * j, bd + kBStep * j, idesc, (kt | j) != 0);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&tfull[buf]);
      }
      tc_commit(drain);  // all MMAs issued above are complete before TMEM is freed
      symm::mbar_wait(drain, 0, a.budget_ns);
    }
  } else if (warp < 6) {  // ------------------------------------ epilogue
    // Each warp owns TMEM lanes 32q .. 32q + 31 (its 32 rows of the tile).
    // Per 64-column chunk: two tcgen05.ld of 32 columns, rounding to the
    // input type, 16-byte rows of a 128-byte-swizzled 32 x 64 box in this
    // warp's shared staging (chunk j of row r at (j ^ (r & 7)) * 16), and
    // one TMA store of the box (rows and columns past c's edge are
    // dropped by the copy).  Two boxes per warp alternate.
    const uint32_t q = (uint32_t)(warp & 3);
    uint8_t* my_stage = out_stage + (size_t)q * 2 * kOutBox;
    uint64_t tc = 0, chunks = 0;
    for (uint64_t t = blockIdx.x; t < a.tiles; t += G, ++tc) {
      const AgTile x = ag_tile(a, t);
      const uint32_t buf = (uint32_t)(tc & 1);
      if (!mbar_wait_ab(&tfull[buf], (uint32_t)((tc >> 1) & 1), a.budget_ns, a.ctl)) {
        symm::record_error(a.ctl, symm::kErrTimedOut, -6);
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < kBN / 64; ++ch, ++chunks) {
        uint32_t v0[32], v1[32];
        const uint32_t col = tmem + ((32 * q) << 16) + buf * kBN + ch * 64;
        tmem_ld32(col, v0);
        tmem_ld32(col + 32, v1);
        if (ch == kBN / 64 - 1) {  // the accumulator is free for the next tile
          tc_fence_before();
          mbar_arrive(&tempty[buf]);
        }
        uint8_t* box = my_stage + (chunks & 1) * kOutBox;
        if (chunks >= 2) {  // the store issued from this box two chunks ago has read it
          if (lane == 0) symm::bulk_wait_read<1>();
          __syncwarp();
        }
        uint8_t* row = box + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t* vv = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
          uint4 o;
          o.x = pack2<FMT>(__uint_as_float(vv[0]), __uint_as_float(vv[1]));
          o.y = pack2<FMT>(__uint_as_float(vv[2]), __uint_as_float(vv[3]));
          o.z = pack2<FMT>(__uint_as_float(vv[4]), __uint_as_float(vv[5]));
          o.w = pack2<FMT>(__uint_as_float(vv[6]), __uint_as_float(vv[7]));
          *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = o;
        }
        symm::fence_proxy_async_shared();  // the box, for the async-proxy store
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tma_c, box, (int)(x.n0 + 64 * ch), (int)(x.m0 + 32 * q), (int)x.d);
          symm::bulk_commit();
        }
      }
    }
    if (lane == 0) symm::bulk_wait<0>();  // stores complete before the CTA leaves
    __syncwarp();
  } else {  // ------------------------------------------------------ push
    const uint32_t block_bytes = kBM * a.k * 2;
    const uint32_t npieces = (block_bytes + kPushPiece - 1) / kPushPiece;
    const uint64_t units = (uint64_t)a.nblk * a.W * npieces;
    const uint64_t gw = (uint64_t)blockIdx.x * kPushWarps + (warp - 6);
    for (uint64_t u = gw; u < units; u += (uint64_t)G * kPushWarps) {
      const uint32_t p = (uint32_t)(u % npieces);
      const uint64_t v = u / npieces;  // = jb*W + r: block 0 of every rank first
      const uint32_t r = (uint32_t)(v % a.W), jb = (uint32_t)(v / a.W);
      const uint32_t off = p * kPushPiece;
      const uint32_t nvec = (min(kPushPiece, block_bytes - off)) >> 4;
      const uint8_t* src = a.a + r * a.slab + (size_t)jb * block_bytes + off;
      uint8_t* dst0 = a.gather + ((size_t)r * a.m_local * a.k * 2) + (size_t)jb * block_bytes + off;
      for (uint32_t base = 0; base < nvec; base += 32 * kPushUnroll) {
        uint4 vv[kPushUnroll];
#pragma unroll
        for (int i = 0; i < kPushUnroll; ++i) {
          const uint32_t j = base + 32 * i + lane;
          if (j < nvec) vv[i] = symm::ld16_ro(src + 16 * (size_t)j);
        }
        for (uint32_t d = 0; d < a.W; ++d) {
#pragma unroll
          for (int i = 0; i < kPushUnroll; ++i) {
            const uint32_t j = base + 32 * i + lane;
            if (j < nvec) symm::st16(dst0 + d * a.slab + 16 * (size_t)j, vv[i]);
          }
        }
      }
      __syncwarp();  // the lanes' stores precede lane 0's acquire/release count
      int last = 0;
      if (lane == 0)
        last = atom_add_acq_rel_u64(reinterpret_cast<uint64_t*>(ag_counter(a, r, jb)), 1) +
                   1 == npieces;
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (last)
        for (uint32_t d = lane; d < a.W; d += 32) symm::st_release(ag_signal(a, d, r, jb), 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void ag_reset_kernel(uint8_t* signals, size_t slab, uint32_t W, uint32_t slots) {
  const size_t per_pe = (size_t)slots * (SYMM_SIGNAL_STRIDE_BYTES / 8);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)W * per_pe;
       i += (size_t)gridDim.x * blockDim.x)
    reinterpret_cast<int64_t*>(signals + (i / per_pe) * slab)[i % per_pe] = 0;
  int64_t* counters =
      reinterpret_cast<int64_t*>(signals + (size_t)slots * SYMM_SIGNAL_STRIDE_BYTES);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < slots;
       i += (size_t)gridDim.x * blockDim.x)
    counters[i] = 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-d tensor map over one object of every PE: [W][rows][inner] 2-byte
// elements, PE stride = the slab; boxes of box_inner x box_rows, 128-byte
// swizzled.
int make_map(CUtensorMap* map, void* base, int fmt, uint32_t inner, uint32_t rows, uint32_t W,
             size_t slab, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(SYMM_ECUDA, "shmem_fused_all_gather_matmul: no cuTensorMapEncodeTiled");
  const cuuint64_t dims[3] = {inner, rows, W};
  const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)slab};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      fn(map, fmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
         base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SYMM_ECUDA, "shmem_fused_all_gather_matmul: tensor map rejected (CUresult " +
                                std::to_string((int)r) + ")");
  return SYMM_OK;
}

struct AgShape {
  uint32_t nblk, slots;
  size_t a_bytes, b_bytes, gather_bytes, c_bytes, signal_bytes;
};

int ag_shape(int W, int m_local, int k, int n, int block_size, const char* what, AgShape* o) {
  if (W < 1 || W > 4096 || m_local < 0 || k < 1 || n < 1)
    return fail(SYMM_EINVAL,
                std::string(what) + ": W outside [1, 4096], m_local < 0, k < 1 or n < 1");
  if (block_size != kBM)
    return fail(SYMM_EINVAL, std::string(what) + ": block_size must be 128 (the MMA tile height)");
  if (m_local % kBM)
    return fail(SYMM_EINVAL, std::string(what) + ": m_local must be a multiple of block_size");
  if (k % 8 || n % 8)
    return fail(SYMM_EINVAL, std::string(what) + ": k and n must be multiples of 8 (16-byte rows)");
  if ((uint64_t)W * m_local > (1u << 30) || (uint64_t)k * kBM * 2 > 0xffffffffull ||
      (uint64_t)k > (1u << 20) || (uint64_t)n > (1u << 20))
    return fail(SYMM_EINVAL, std::string(what) + ": extents too large");
  o->nblk = (uint32_t)(m_local / kBM);
  o->slots = (uint32_t)W * o->nblk;
  o->a_bytes = (size_t)m_local * k * 2;
  o->b_bytes = (size_t)k * n * 2;
  o->gather_bytes = (size_t)W * o->a_bytes;
  o->c_bytes = (size_t)W * m_local * n * 2;
  o->signal_bytes = ((size_t)o->slots * (SYMM_SIGNAL_STRIDE_BYTES + 8) + 63) & ~(size_t)63;
  return SYMM_OK;
}

const void* ag_kernel(int fmt) {
  return fmt ? (const void*)ag_gemm_kernel<1> : (const void*)ag_gemm_kernel<0>;
}

// CTAs resident at once (one per SM: the kernel takes all of TMEM).
int ag_capacity(int fmt) {
  static std::mutex mu;
  static int cached[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& slot = cached[fmt][dev];
  if (slot) return slot;
  const void* k = ag_kernel(fmt);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAgSmem) !=
      cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAgThreads, kAgSmem) !=
      cudaSuccess)
    return 0;
  slot = std::min(per_sm, 1) * sm_count();
  return slot;
}

}  // namespace

extern "C" int shmem_fused_ag_matmul_workspace(int W, int m_local, int k, int n, int block_size,
                                               size_t* signal_bytes) {
  AgShape sh;
  int rc = ag_shape(W, m_local, k, n, block_size, "shmem_fused_ag_matmul_workspace", &sh);
  if (rc) return rc;
  if (signal_bytes) *signal_bytes = sh.signal_bytes;
  return SYMM_OK;
}

extern "C" int shmem_fused_all_gather_matmul(symm_heap_t* h, const void* a, const void* b,
                                             void* c, void* gather_out, int W, int m_local, int k,
                                             int n, int dtype, int block_size, int64_t* signals,
                                             void* stream) {
  const char* what = "shmem_fused_all_gather_matmul";
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  if (dtype != SYMM_DTYPE_F16 && dtype != SYMM_DTYPE_BF16)
    return fail(SYMM_EINVAL, std::string(what) + ": dtype must be SYMM_DTYPE_F16 or _BF16");
  AgShape sh;
  int rc = ag_shape(W, m_local, k, n, block_size, what, &sh);
  if (rc) return rc;
  if (W != h->npes) return fail(SYMM_EINVAL, std::string(what) + ": W differs from the heap's PEs");
  constexpr int kObj = 5;
  size_t off[kObj];
  const void* ptr[kObj] = {a, b, c, gather_out, signals};
  const size_t len[kObj] = {sh.a_bytes, sh.b_bytes, sh.c_bytes, sh.gather_bytes, sh.signal_bytes};
  const char* names[kObj] = {"a", "b", "c", "gather_out", "signals"};
  for (int i = 0; i < kObj; ++i) {
    rc = check_range(h, ptr[i], len[i], (std::string(what) + ": " + names[i]).c_str(), &off[i]);
    if (rc) return rc;
    if (off[i] % 16)
      return fail(SYMM_EINVAL, std::string(what) + ": " + names[i] + " not 16-byte aligned");
  }
  for (int i = 0; i < kObj; ++i)
    for (int j = i + 1; j < kObj; ++j)
      if (len[i] && len[j] && off[i] < off[j] + len[j] && off[j] < off[i] + len[i])
        return fail(SYMM_EINVAL, std::string(what) + ": " + names[i] + " and " + names[j] +
                                     " overlap");
  if (m_local == 0) return SYMM_OK;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  const int fmt = dtype == SYMM_DTYPE_BF16 ? 1 : 0;
  CUtensorMap map_a, map_local, map_b, map_c;
  rc = make_map(&map_a, h->base + off[3], fmt, (uint32_t)k, (uint32_t)(W * m_local), (uint32_t)W,
                h->slab, kBK, kBM);
  if (rc) return rc;
  rc = make_map(&map_local, h->base + off[0], fmt, (uint32_t)k, (uint32_t)m_local, (uint32_t)W,
                h->slab, kBK, kBM);
  if (rc) return rc;
  rc = make_map(&map_b, h->base + off[1], fmt, (uint32_t)n, (uint32_t)k, (uint32_t)W, h->slab, 64,
                kBK);
  if (rc) return rc;
  rc = make_map(&map_c, h->base + off[2], fmt, (uint32_t)n, (uint32_t)(W * m_local), (uint32_t)W,
                h->slab, 64, 32);
  if (rc) return rc;
  const int cap = ag_capacity(fmt);
  if (cap < 1) return fail(SYMM_ECUDA, std::string(what) + ": kernel set-up failed");

  ag_reset_kernel<<<(unsigned)std::min<size_t>(((size_t)W * sh.slots * 8 + 255) / 256 + 1, 1024),
                    256, 0, s>>>(h->base + off[4], h->slab, (uint32_t)W, sh.slots);
  rc = cuda_check(cudaGetLastError(), "shmem_fused_all_gather_matmul: signal reset");
  if (rc) return rc;

  AgArgs args;
  args.a = h->base + off[0];
  args.gather = h->base + off[3];
  args.c = h->base + off[2];
  args.signals = h->base + off[4];
  args.slab = h->slab;
  args.W = (uint32_t)W;
  args.m_local = (uint32_t)m_local;
  args.k = (uint32_t)k;
  args.n = (uint32_t)n;
  args.nblk = sh.nblk;
  args.ktiles = (uint32_t)((k + kBK - 1) / kBK);
  args.ntiles_n = (uint32_t)((n + kBN - 1) / kBN);
  args.tiles = (uint64_t)W * (W * sh.nblk) * args.ntiles_n;
  // all W b matrices well inside L2 (126 MB): keep every PE on the push's
  // block order; otherwise keep one PE's b in L2 at a time
  args.pe_major = (uint64_t)W * sh.b_bytes > (48ull << 20) ? 1u : 0u;
  args.budget_ns = h->spin_budget;
  args.ctl = reinterpret_cast<Control*>(h->base);
  args.heap_base = h->base;
  const int grid = (int)std::min<uint64_t>((uint64_t)cap, std::max<uint64_t>(args.tiles, 1));
  void* kargs[] = {&map_a, &map_local, &map_b, &map_c, &args};
  // cooperative: every CTA resident at once, since tiles wait on blocks that
  // other CTAs push
  return cuda_check(
      cudaLaunchCooperativeKernel(ag_kernel(fmt), grid, kAgThreads, kargs, kAgSmem, s),
      "shmem_fused_all_gather_matmul: launch");
}
