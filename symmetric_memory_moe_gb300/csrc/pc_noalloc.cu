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
// host-side stand-in), so its address is looked up with cudaGetSymbolAddress,
// with the device current, and cached per device: symm_heap_init does this
// for its device (which also loads the module that holds the array, so the
// array is reserved at set-up rather than in the first call), and a first
// call on any other device does it itself -- make that call before any
// stream capture.
//
// The protocol, the kernels and their launch are the ones of
// all2all_combine(SYMM_A2A_PC) (symm_host::launch_pc); this file only
// places the staging ring and the signal slots in the array.
#include <map>
#include <mutex>
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

static __device__ __align__(256) uint8_t g_noalloc_scratch[SYMM_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_addr_mu;
std::map<int, uint8_t*> g_addr;  // device -> address of the array on it

size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

}  // namespace

// Device address of the array on the current device, looked up once per
// device with cudaGetSymbolAddress (that device being current).
int symm_host::noalloc_scratch_address(uint8_t** out) {
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "all2all_combine_pc_noalloc: cudaGetDevice");
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  auto it = g_addr.find(dev);
  if (it == g_addr.end()) {
    void* p = nullptr;
    rc = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                    "all2all_combine_pc_noalloc: cudaGetSymbolAddress of the scratch array");
    if (rc) return rc;
    it = g_addr.emplace(dev, static_cast<uint8_t*>(p)).first;
  }
  *out = it->second;
  return SYMM_OK;
}

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
  size_t nbytes = (size_t)S * W;
  for (size_t f : {(size_t)H, (size_t)D, (size_t)elem_bytes})
    if (__builtin_mul_overflow(nbytes, f, &nbytes))
      return fail(SYMM_EINVAL, std::string(what) + ": size overflow");
  size_t in_off, out_off;
  int rc = check_range(h, in, nbytes, "all2all_combine_pc_noalloc: in", &in_off);
  if (rc) return rc;
  rc = check_range(h, out, nbytes, "all2all_combine_pc_noalloc: out", &out_off);
  if (rc) return rc;
  if (nbytes && in_off < out_off + nbytes && out_off < in_off + nbytes)
    return fail(SYMM_EINVAL, std::string(what) + ": input and output ranges overlap");
  if (nbytes == 0) return SYMM_OK;

  size_t stage_bytes, sig_bytes;
  rc = all2all_pc_workspace(W, S, H, D, elem_bytes, tile_s, block_d, buffer_num, &stage_bytes,
                            &sig_bytes);
  if (rc) return rc;
  const size_t cap = (size_t)SYMM_NOALLOC_SCRATCH_BYTES;
  if (stage_bytes > cap || sig_bytes > cap)
    return fail(SYMM_EINVAL, std::string(what) + ": the staging ring exceeds the static scratch "
                                                 "(SYMM_NOALLOC_SCRATCH_BYTES); lower tile_s or "
                                                 "buffer_num");
  const size_t stage_stride = up256(stage_bytes);
  const size_t sig_stride = up256(sig_bytes);
  const size_t need = (size_t)W * (stage_stride + sig_stride);
  if (need > cap)
    return fail(SYMM_EINVAL, std::string(what) + ": needs " + std::to_string(need) +
                                 " bytes of staging and signals but the static scratch holds " +
                                 std::to_string(cap) +
                                 " (SYMM_NOALLOC_SCRATCH_BYTES); lower tile_s or buffer_num");

  uint8_t* scratch = nullptr;
  rc = noalloc_scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;

  PcPlan p;
  p.in = h->base + in_off;
  p.out = h->base + out_off;
  p.slab = h->slab;
  p.staging = scratch;  // PE k's ring at + k*stage_stride
  p.stage_pe = stage_stride;
  p.signals = scratch + (size_t)W * stage_stride;  // PE k's slots at + k*sig_stride
  p.sig_pe = sig_stride;
  p.W = W;
  p.S = S;
  p.H = H;
  p.D = D;
  p.es = elem_bytes;
  p.tile_s = tile_s;
  p.block_d = block_d;
  p.buffer_num = buffer_num;
  p.reset = true;  // the array keeps the previous call's signals
  p.vector_only = false;
  p.budget_ns = h->spin_budget;
  p.ctl = h->base;
  // a slot that times out is reported by its offset in the signal area of
  // the array, marked by SYMM_INFO_NOALLOC_SIGNAL
  p.err_base = p.signals;
  p.err_bias = SYMM_INFO_NOALLOC_SIGNAL;
  return launch_pc(p, s, what);
}
