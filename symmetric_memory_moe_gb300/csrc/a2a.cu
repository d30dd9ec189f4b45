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
//    like the page's cores, each CTA owns a fixed set of tasks and walks the
//    S blocks in order, its consumer group consuming exactly the tiles its own
//    producer group staged.  Every wait is thus satisfied by the same CTA,
//    and successive producers of a slot are ordered.  The page's target
//    rotation (rank + i) % W staggers one PE's producers across
//    destinations; here every (r, d) pair is in flight at once, so it has
//    nothing left to stagger.
//  * Copies move 16-byte vectors per lane (funnel-shifted when source and
//    destination disagree mod 16) instead of masked 2-D tile loads; ragged
//    S and D blocks are bounds in the row loop and the byte count.
//  * The direct variant is one pass with no staging: every contiguous run of
//    H*D elements (fixed r, d, s) is copied once, the minimum traffic.
#include <stdio.h>

#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

namespace {

constexpr int kRunThreads = 256;
constexpr int kPcThreads = 256;  // 4 producer warps + 4 consumer warps
constexpr int kPcGroup = 128;
constexpr int kPcMinBlocks = 3;

// --------------------------------------------------------------- direct ---
// One warp per run of R = H*D*elem_bytes contiguous bytes, destination-major.
// INVERSE = false (combine, dispatch with Sb = S/W):
//   run k = (d*Sb + s)*W + r : in slab r row d*Sb + s  ->  out slab d row s*W + r
// INVERSE = true (combine_back):
//   run k = (r*W + d)*Sb + s : in slab d row s*W + r   ->  out slab r row d*Sb + s
// (a "row" here is one run of R bytes).
template <bool INVERSE>
__global__ void __launch_bounds__(kRunThreads)
    a2a_runs_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, size_t slab,
                    uint32_t W, uint32_t Sb, size_t R, uint32_t nruns) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * kRunThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kRunThreads) >> 5;
  for (uint32_t k = warp; k < nruns; k += nwarps) {
    const uint8_t* src;
    uint8_t* dst;
    if (!INVERSE) {
      const uint32_t r = k % W, t = k / W, s = t % Sb, d = t / Sb;
      src = in + r * slab + (size_t)(d * Sb + s) * R;
      dst = out + d * slab + (size_t)(s * W + r) * R;
    } else {
      const uint32_t s = k % Sb, t = k / Sb, d = t % W, r = t / W;
      src = in + d * slab + (size_t)(s * W + r) * R;
      dst = out + r * slab + (size_t)(d * Sb + s) * R;
    }
    symm::warp_copy<4, symm::kRO, symm::kCS>(dst, src, R, lane);
  }
}

// ------------------------------------------------ producer / consumer ---
struct PcArgs {
  const uint8_t* in;   // PE 0 copies of the symmetric objects; PE k at +k*slab
  uint8_t* out;
  uint8_t* staging;
  uint8_t* signals;
  size_t slab;
  uint32_t W, H, S, D, es;
  uint32_t tile_s, block_d, nbd, nbs, buffer_num;
  uint64_t budget_ns;
  Control* ctl;
  const uint8_t* heap_base;
};

__global__ void __launch_bounds__(kPcThreads, kPcMinBlocks) a2a_pc_kernel(const PcArgs a) {
  __shared__ int status[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int role = warp >> 2;          // 0 = producer group, 1 = consumer group
  const int gwarp = warp & 3;          // warp inside its group
  const int gtid = threadIdx.x & (kPcGroup - 1);
  const int bar_id = 1 + role;         // named barrier of the group
  const size_t tasks_per_block = (size_t)a.W * a.W * a.H * a.nbd;
  const size_t stage_row = (size_t)a.H * a.W * a.D * a.es;  // one staging row, bytes

  // As on the page, a task (one signal slot) belongs to one CTA for every S
  // block and the CTA walks the S blocks in order: the producer of S block b
  // and the consumer of S block b - buffer_num on the same slot are this
  // CTA's own two groups, so no wait depends on another CTA.
  for (uint32_t b = 0; b < a.nbs; ++b)
  for (size_t q0 = blockIdx.x; q0 < tasks_per_block; q0 += gridDim.x) {
    size_t q = q0;  // q = ((d*W + r)*H + h)*nbd + bd
    const uint32_t bd = (uint32_t)(q % a.nbd);
    q /= a.nbd;
    const uint32_t h = (uint32_t)(q % a.H);
    q /= a.H;
    const uint32_t r = (uint32_t)(q % a.W);
    const uint32_t d = (uint32_t)(q / a.W);
    const uint32_t buf = b % a.buffer_num;
    // slot (buf, r, bd, h) of destination d, one 64-byte line each
    int64_t* slot = reinterpret_cast<int64_t*>(
        a.signals + d * a.slab +
        ((((size_t)buf * a.W + r) * a.nbd + bd) * a.H + h) * SYMM_SIGNAL_STRIDE_BYTES);
    const uint32_t s0 = b * a.tile_s;
    const uint32_t rows = min(a.tile_s, a.S - s0);
    const uint32_t x0 = bd * a.block_d;
    const size_t len = (size_t)min(a.block_d, a.D - x0) * a.es;
    const size_t stage_col = ((size_t)(r * a.H + h) * a.D + x0) * a.es;
    uint8_t* stage = a.staging + d * a.slab + (size_t)buf * a.tile_s * stage_row + stage_col;

    if (gtid == 0)
      status[role] =
          symm::spin_wait(slot, symm::kCmpEq, role == 0 ? 0 : 1, a.budget_ns, a.ctl, a.heap_base);
    symm::group_sync(bar_id, kPcGroup);
    if (status[role] != symm::kSpinOk) return;  // uniform across the group

    if (role == 0) {
      // producer: input rows d*S + s0 + i of source r -> destination d's slot
      const uint8_t* src =
          a.in + r * a.slab + (((size_t)(d * a.S + s0) * a.H + h) * a.D + x0) * a.es;
      const size_t src_row = (size_t)a.H * a.D * a.es;
      for (uint32_t i = gwarp; i < rows; i += 4)
        symm::warp_copy<4, symm::kRO, symm::kST>(stage + i * stage_row, src + i * src_row, len,
                                                  lane);
    } else {
      // consumer: staged tile -> output rows s0 + i, column r*H + h
      uint8_t* dst = a.out + d * a.slab + ((size_t)s0 * a.H * a.W * a.D) * a.es + stage_col;
      for (uint32_t i = gwarp; i < rows; i += 4)
        symm::warp_copy<4, symm::kCG, symm::kCS>(dst + i * stage_row, stage + i * stage_row, len,
                                                  lane);
    }
    symm::group_sync(bar_id, kPcGroup);  // the group's copies precede the release
    if (gtid == 0) symm::st_release(slot, role == 0 ? 1 : 0);
  }
}

// Zeroes the `slots` signal lines of every PE (the page's host-side reset
// before each launch, done in-stream).
__global__ void a2a_signal_reset_kernel(uint8_t* signals, size_t slab, uint32_t W, size_t slots) {
  const size_t n = (size_t)W * slots;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t pe = i / slots, k = i % slots;
    *reinterpret_cast<int64_t*>(signals + pe * slab + k * SYMM_SIGNAL_STRIDE_BYTES) = 0;
  }
}

// ------------------------------------------------------------ launching ---
// CTAs of `kernel` (launched with `threads` threads, no dynamic shared
// memory) that are resident on the current device at once; cached.
int resident_ctas(const void* kernel, int threads) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({dev, kernel});
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess)
    return 0;
  const int n = per_sm * sm_count();
  cache[{dev, kernel}] = n;
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

int launch_runs(symm_heap* h, size_t in_off, size_t out_off, uint32_t W, uint32_t Sb, size_t R,
                bool inverse, cudaStream_t s, const char* what) {
  const size_t nruns = (size_t)W * W * Sb;
  if (nruns == 0 || R == 0) return SYMM_OK;
  if (nruns > 0x7fffffffull)
    return fail(SYMM_EINVAL, std::string(what) + ": more than 2^31 runs");
  const void* kfn = inverse ? (const void*)a2a_runs_kernel<true> : (const void*)a2a_runs_kernel<false>;
  int cap = resident_ctas(kfn, kRunThreads);
  if (cap <= 0) cap = 4 * (sm_count() > 0 ? sm_count() : 1);
  const size_t need = (nruns + kRunThreads / 32 - 1) / (kRunThreads / 32);
  const int grid = (int)(need < (size_t)cap ? need : (size_t)cap);
  const uint8_t* in = h->base + in_off;
  uint8_t* out = h->base + out_off;
  if (inverse)
    a2a_runs_kernel<true><<<grid, kRunThreads, 0, s>>>(in, out, h->slab, W, Sb, R, (uint32_t)nruns);
  else
    a2a_runs_kernel<false><<<grid, kRunThreads, 0, s>>>(in, out, h->slab, W, Sb, R,
                                                        (uint32_t)nruns);
  return cuda_check(cudaGetLastError(), what);
}

}  // namespace

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

  const uint32_t bd = block_d ? (uint32_t)block_d : (uint32_t)D;
  const uint32_t nbd = (D + bd - 1) / bd;
  const size_t slots = sg_bytes / SYMM_SIGNAL_STRIDE_BYTES;
  if (!(flags & SYMM_A2A_FLAG_NO_RESET)) {
    const size_t n = slots * W;
    const int grid = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    a2a_signal_reset_kernel<<<grid, 256, 0, s>>>(h->base + sg_off, h->slab, W, slots);
    rc = cuda_check(cudaGetLastError(), "all2all_combine: signal reset");
    if (rc) return rc;
  }
  PcArgs a;
  a.in = h->base + in_off;
  a.out = h->base + out_off;
  a.staging = h->base + st_off;
  a.signals = h->base + sg_off;
  a.slab = h->slab;
  a.W = W;
  a.H = H;
  a.S = S;
  a.D = D;
  a.es = es;
  a.tile_s = tile_s;
  a.block_d = bd;
  a.nbd = nbd;
  a.nbs = (S + tile_s - 1) / tile_s;
  a.buffer_num = buffer_num;
  a.budget_ns = h->spin_budget;
  a.ctl = reinterpret_cast<Control*>(h->base);
  a.heap_base = h->base;
  // tasks of one S block, dealt evenly: k per CTA, ceil(tasks / k) CTAs, never
  // more CTAs than are resident at once
  const size_t tasks = (size_t)W * W * H * nbd;
  int cap = resident_ctas((const void*)a2a_pc_kernel, kPcThreads);
  if (cap <= 0) return fail(SYMM_ECUDA, "all2all_combine: occupancy query failed");
  const size_t per_cta = (tasks + cap - 1) / cap;
  const int grid = (int)((tasks + per_cta - 1) / per_cta);
  a2a_pc_kernel<<<grid, kPcThreads, 0, s>>>(a);
  return cuda_check(cudaGetLastError(), "all2all_combine: PC launch");
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
  if (flags & ~SYMM_A2A_FLAG_NO_RESET) return fail(SYMM_EINVAL, "all2all_combine: unknown flag");
  cudaStream_t s = as_stream(stream);
  if (kind == SYMM_A2A_DIRECT)
    return launch_runs(h, in_off, out_off, W, S, (size_t)H * D * elem_bytes, false, s,
                       "all2all_combine");
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
  return launch_runs(h, in_off, out_off, W, S / W, (size_t)H * D * elem_bytes, false,
                     as_stream(stream), "all2all_dispatch");
}

extern "C" int all2all_combine_back(symm_heap_t* h, const void* in, void* out, int W, int Sp,
                                    int H, int D, int elem_bytes, void* stream) {
  if (Sp < 0 || W < 1) return fail(SYMM_EINVAL, "all2all_combine_back: Sp < 0 or W < 1");
  size_t in_off, out_off, nbytes;
  int rc = check_perm(h, in, out, W, (size_t)Sp * W, H, D, elem_bytes, "all2all_combine_back",
                      &in_off, &out_off, &nbytes);
  if (rc) return rc;
  return launch_runs(h, in_off, out_off, W, Sp, (size_t)H * D * elem_bytes, true,
                     as_stream(stream), "all2all_combine_back");
}

extern "C" int all2all_combine_host(symm_heap_t* h, const void* host_in, void* host_out,
                                    const void* in, void* out, int W, int S, int H, int D,
                                    int elem_bytes, int variant, int tile_s, int block_d,
                                    int buffer_num, void* staging, int64_t* signals,
                                    void* stream) {
  if (S < 0 || W < 1) return fail(SYMM_EINVAL, "all2all_combine_host: S < 0 or W < 1");
  size_t in_off, out_off, nbytes;
  int rc = check_perm(h, in, out, W, (size_t)S * W, H, D, elem_bytes, "all2all_combine_host",
                      &in_off, &out_off, &nbytes);
  if (rc) return rc;
  if (nbytes && (!host_in || !host_out))
    return fail(SYMM_EINVAL, "all2all_combine_host: NULL host buffer");
  cudaStream_t s = as_stream(stream);
  for (int r = 0; r < W && nbytes; ++r) {
    rc = cuda_check(cudaMemcpyAsync(h->base + (size_t)r * h->slab + in_off,
                                    static_cast<const uint8_t*>(host_in) + (size_t)r * nbytes,
                                    nbytes, cudaMemcpyHostToDevice, s),
                    "all2all_combine_host: host-to-device copy");
    if (rc) return rc;
  }
  rc = all2all_combine(h, in, out, W, S, H, D, elem_bytes, variant, tile_s, block_d, buffer_num,
                       staging, signals, stream);
  if (rc) return rc;
  for (int d = 0; d < W && nbytes; ++d) {
    rc = cuda_check(cudaMemcpyAsync(static_cast<uint8_t*>(host_out) + (size_t)d * nbytes,
                                    h->base + (size_t)d * h->slab + out_off, nbytes,
                                    cudaMemcpyDeviceToHost, s),
                    "all2all_combine_host: device-to-host copy");
    if (rc) return rc;
  }
  return SYMM_OK;
}
