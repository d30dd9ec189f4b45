// pc_noalloc.cu -- all2all_combine_pc_noalloc: the producer/consumer combine
// for callers that cannot allocate device memory.
//
// Who needs it: code that must not call cudaMalloc/cudaFree (or any
// allocator) on its hot path -- for example a serving loop whose device
// memory is all handed out up front by another allocator, or a latency-bound
// caller that cannot afford the device-wide synchronisation those calls
// imply -- yet still wants the staged, signalled combine.  The regular
// all2all_combine(SYMM_A2A_PC) takes its staging ring and signal slots from
// the caller's symmetric heap; this variant takes them from one fixed
// array that the library itself declares, so the caller provides only the
// input and output.
//
// The array is a file-scope __device__ object of SYMM_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Every
// call shares it and it keeps the last call's contents, so each call zeroes
// its signal slots first, and calls that overlap on the GPU race on it.
// Host code cannot use the array's name as a device address (there it is a
// host-side stand-in), so the first call on each device looks the address
// up with cudaGetSymbolAddress, with that device current, and caches it;
// make that first call before any stream capture.
#include <map>
#include <mutex>
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

static __device__ __align__(256) uint8_t g_noalloc_scratch[SYMM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kThreads = 256;  // 4 producer warps + 4 consumer warps
constexpr int kGroup = 128;

struct NoallocArgs {
  const uint8_t* in;   // PE 0 copies of the heap objects; PE k at +k*slab
  uint8_t* out;
  size_t slab;
  uint8_t* staging;    // scratch: PE k's staging ring at +k*stage_stride
  uint8_t* signals;    // scratch: PE k's signal slots at +k*sig_stride
  size_t stage_stride, sig_stride;
  uint32_t W, H, S, D, es;
  uint32_t tile_s, block_d, nbd, nbs, buffer_num;
  uint64_t budget_ns;
  Control* ctl;
  const uint8_t* heap_base;
};

__global__ void noalloc_signal_reset_kernel(uint8_t* signals, size_t stride, uint32_t W,
                                            size_t slots) {
  const size_t n = (size_t)W * slots;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    *reinterpret_cast<int64_t*>(signals + (i / slots) * stride +
                                (i % slots) * SYMM_SIGNAL_STRIDE_BYTES) = 0;
}

// Same task loop as the heap-workspace kernel: a CTA owns fixed (d, r, h,
// D-block) slots for every S block; its producer warps stage a tile and
// release the slot, its consumer warps acquire it, copy the tile out and
// release it back to 0.  FLAT: tile rows, bases and row strides are 16-byte
// aligned and a tile spans less than 4 GiB, so each group copies whole tiles
// flattened to 16-byte vectors; otherwise row by row with warp_copy.
template <bool FLAT>
__global__ void __launch_bounds__(kThreads, 3) a2a_pc_noalloc_kernel(const NoallocArgs a) {
  __shared__ int status[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int role = warp >> 2;
  const int gwarp = warp & 3;
  const int gtid = threadIdx.x & (kGroup - 1);
  const int bar_id = 1 + role;
  const size_t tasks = (size_t)a.W * a.W * a.H * a.nbd;
  const size_t stage_row = (size_t)a.H * a.W * a.D * a.es;

  for (uint32_t b = 0; b < a.nbs; ++b)
    for (size_t q0 = blockIdx.x; q0 < tasks; q0 += gridDim.x) {
      size_t q = q0;  // q = ((d*W + r)*H + h)*nbd + bd
      const uint32_t bd = (uint32_t)(q % a.nbd);
      q /= a.nbd;
      const uint32_t h = (uint32_t)(q % a.H);
      q /= a.H;
      const uint32_t r = (uint32_t)(q % a.W);
      const uint32_t d = (uint32_t)(q / a.W);
      const uint32_t buf = b % a.buffer_num;
      int64_t* slot = reinterpret_cast<int64_t*>(
          a.signals + d * a.sig_stride +
          ((((size_t)buf * a.W + r) * a.nbd + bd) * a.H + h) * SYMM_SIGNAL_STRIDE_BYTES);
      const uint32_t s0 = b * a.tile_s;
      const uint32_t rows = min(a.tile_s, a.S - s0);
      const uint32_t x0 = bd * a.block_d;
      const size_t len = (size_t)min(a.block_d, a.D - x0) * a.es;
      const size_t stage_col = ((size_t)(r * a.H + h) * a.D + x0) * a.es;
      uint8_t* stage =
          a.staging + d * a.stage_stride + (size_t)buf * a.tile_s * stage_row + stage_col;

      if (gtid == 0)
        status[role] = symm::spin_wait(slot, symm::kCmpEq, role == 0 ? 0 : 1, a.budget_ns,
                                       a.ctl, a.heap_base);
      symm::group_sync(bar_id, kGroup);
      if (status[role] != symm::kSpinOk) return;

      if (role == 0) {
        const uint8_t* src =
            a.in + r * a.slab + (((size_t)(d * a.S + s0) * a.H + h) * a.D + x0) * a.es;
        const size_t src_row = (size_t)a.H * a.D * a.es;
        if (FLAT)
          symm::group_copy_tile<kGroup, 4, symm::kRO, symm::kST>(
              stage, (uint32_t)stage_row, src, (uint32_t)src_row, rows, (uint32_t)(len >> 4),
              gtid);
        else
          for (uint32_t i = gwarp; i < rows; i += 4)
            symm::warp_copy<4, symm::kRO, symm::kST>(stage + i * stage_row, src + i * src_row,
                                                      len, lane);
      } else {
        uint8_t* dst = a.out + d * a.slab + ((size_t)s0 * a.H * a.W * a.D) * a.es + stage_col;
        if (FLAT)
          symm::group_copy_tile<kGroup, 4, symm::kCG, symm::kCS>(
              dst, (uint32_t)stage_row, stage, (uint32_t)stage_row, rows, (uint32_t)(len >> 4),
              gtid);
        else
          for (uint32_t i = gwarp; i < rows; i += 4)
            symm::warp_copy<4, symm::kCG, symm::kCS>(dst + i * stage_row, stage + i * stage_row,
                                                      len, lane);
      }
      symm::group_sync(bar_id, kGroup);
      if (gtid == 0) symm::st_release(slot, role == 0 ? 1 : 0);
    }
}

// Device address of the scratch array on the current device, looked up once
// per device with cudaGetSymbolAddress (with that device current).
int scratch_address(uint8_t** out) {
  static std::mutex mu;
  static std::map<int, uint8_t*> addr;
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "all2all_combine_pc_noalloc: cudaGetDevice");
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it == addr.end()) {
    void* p = nullptr;
    rc = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                    "all2all_combine_pc_noalloc: cudaGetSymbolAddress of the scratch array");
    if (rc) return rc;
    it = addr.emplace(dev, static_cast<uint8_t*>(p)).first;
  }
  *out = it->second;
  return SYMM_OK;
}

int resident(int threads) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  // both instances have the same launch bounds (256 threads, 3 CTAs per SM)
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, a2a_pc_noalloc_kernel<false>, threads,
                                                    0) != cudaSuccess)
    return 0;
  return cache[dev] = per_sm * sm_count();
}

size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

}  // namespace

extern "C" int all2all_combine_pc_noalloc(symm_heap_t* h, const void* in, void* out, int W, int S,
                                          int H, int D, int elem_bytes, int tile_s, int block_d,
                                          int buffer_num, void* stream) {
  static const char* what = "all2all_combine_pc_noalloc";
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  if (W != h->npes) return fail(SYMM_EINVAL, std::string(what) + ": W differs from the heap's PEs");
  if (S < 0 || H < 0 || D < 0 || elem_bytes < 1 || tile_s < 1 || block_d < 0 || buffer_num < 1)
    return fail(SYMM_EINVAL, std::string(what) + ": bad shape or tiling arguments");
  if ((size_t)S * W > 0x7fffffffull || (size_t)H * W > 0x7fffffffull)
    return fail(SYMM_EINVAL, std::string(what) + ": more than 2^31 rows or columns per PE");
  const size_t nbytes = (size_t)S * W * H * D * elem_bytes;
  size_t in_off, out_off;
  int rc = check_range(h, in, nbytes, "all2all_combine_pc_noalloc: in", &in_off);
  if (rc) return rc;
  rc = check_range(h, out, nbytes, "all2all_combine_pc_noalloc: out", &out_off);
  if (rc) return rc;
  if (nbytes && in_off < out_off + nbytes && out_off < in_off + nbytes)
    return fail(SYMM_EINVAL, std::string(what) + ": input and output ranges overlap");
  if (nbytes == 0) return SYMM_OK;

  const uint32_t bd = block_d ? (uint32_t)block_d : (uint32_t)D;
  const uint32_t nbd = (D + bd - 1) / bd;
  size_t stage_bytes = (size_t)buffer_num;
  for (size_t f : {(size_t)tile_s, (size_t)H, (size_t)W, (size_t)D, (size_t)elem_bytes})
    if (__builtin_mul_overflow(stage_bytes, f, &stage_bytes) ||
        stage_bytes > (size_t)SYMM_NOALLOC_SCRATCH_BYTES)
      return fail(SYMM_EINVAL, std::string(what) + ": the staging ring exceeds the static "
                                                   "scratch (SYMM_NOALLOC_SCRATCH_BYTES); lower "
                                                   "tile_s or buffer_num");
  const size_t slots = (size_t)buffer_num * W * nbd * H;
  const size_t stage_stride = up256(stage_bytes);
  const size_t sig_stride = up256(slots * SYMM_SIGNAL_STRIDE_BYTES);
  const size_t need = (size_t)W * (stage_stride + sig_stride);
  if (need > (size_t)SYMM_NOALLOC_SCRATCH_BYTES)
    return fail(SYMM_EINVAL, std::string(what) + ": needs " + std::to_string(need) +
                                 " bytes of staging and signals but the static scratch holds " +
                                 std::to_string((size_t)SYMM_NOALLOC_SCRATCH_BYTES) +
                                 " (SYMM_NOALLOC_SCRATCH_BYTES); lower tile_s or buffer_num");

  uint8_t* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;

  NoallocArgs a;
  a.in = h->base + in_off;
  a.out = h->base + out_off;
  a.slab = h->slab;
  a.staging = scratch;
  a.signals = scratch + (size_t)W * stage_stride;
  a.stage_stride = stage_stride;
  a.sig_stride = sig_stride;
  a.W = W;
  a.H = H;
  a.S = S;
  a.D = D;
  a.es = elem_bytes;
  a.tile_s = tile_s;
  a.block_d = bd;
  a.nbd = nbd;
  a.nbs = (S + tile_s - 1) / tile_s;
  a.buffer_num = buffer_num;
  a.budget_ns = h->spin_budget;
  a.ctl = reinterpret_cast<Control*>(h->base);
  a.heap_base = h->base;

  // the scratch keeps the previous call's signals: zero this call's slots
  const size_t n = slots * W;
  const int rgrid = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  noalloc_signal_reset_kernel<<<rgrid, 256, 0, s>>>(a.signals, sig_stride, W, slots);
  rc = cuda_check(cudaGetLastError(), "all2all_combine_pc_noalloc: signal reset");
  if (rc) return rc;

  const size_t tasks = (size_t)W * W * H * nbd;
  const int cap = resident(kThreads);
  if (cap <= 0) return fail(SYMM_ECUDA, std::string(what) + ": occupancy query failed");
  const size_t per_cta = (tasks + cap - 1) / cap;
  const int grid = (int)((tasks + per_cta - 1) / per_cta);
  const bool flat = ((size_t)D * elem_bytes) % 16 == 0 && ((size_t)bd * elem_bytes) % 16 == 0 &&
                    in_off % 16 == 0 && out_off % 16 == 0 &&
                    (uint64_t)tile_s * H * W * D * elem_bytes < (1ull << 32);
  if (flat)
    a2a_pc_noalloc_kernel<true><<<grid, kThreads, 0, s>>>(a);
  else
    a2a_pc_noalloc_kernel<false><<<grid, kThreads, 0, s>>>(a);
  return cuda_check(cudaGetLastError(), "all2all_combine_pc_noalloc: launch");
}
