// heap.cu -- the emulated symmetric heap (W slabs of one caller-owned device
// allocation) and the one-sided primitives on it: put, get, signal_op,
// wait_for_signal and put_with_signal.
//
// Sources: "Distributed Architecture Design" sections 5 (symmetric heap,
// 5.3 remote address = target PE's heap base + the pointer's offset from the
// local base) and 6 (signal SET/ADD, wait as a local spin, fence before
// signal); HyperParallel RFC "Symmetric Memory", sections 4 and 6 (API and
// semantics of shmem_put/get/signal_op/wait_for_signal/put_with_signal) and 8
// (put_mem_signal: data copy on all cores, fence, core sync, one signal).
//
// Differences from the pages' design, all deliberate: offsets and sizes are
// kernel arguments by value (the pages pass them as device tensors only
// because their kernels read parameters from global memory); the copy runs on
// every SM with 16-byte vectors instead of one or four AI cores through a
// ping-pong buffer; the fence + core sync + single signal of put_mem_signal
// becomes "last CTA to arrive signals" with acquire/release atomics.
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;

namespace symm_host {

static thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SYMM_OK;
  return fail(SYMM_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                              cudaGetErrorString(e) + ")");
}

int64_t slab_offset(const symm_heap* h, const void* p) {
  const uint8_t* q = static_cast<const uint8_t*>(p);
  if (!h || q < h->base || q >= h->base + h->slab * (size_t)h->npes) return -1;
  return (int64_t)((size_t)(q - h->base) % h->slab);
}

int check_range(const symm_heap* h, const void* p, size_t bytes, const char* what, size_t* off) {
  const int64_t o = slab_offset(h, p);
  if (o < 0) return fail(SYMM_EINVAL, std::string(what) + ": not a symmetric-heap pointer");
  if ((size_t)o < SYMM_HEAP_HEADER_BYTES)
    return fail(SYMM_EINVAL, std::string(what) + ": points into the heap header");
  if (bytes > h->slab - (size_t)o)
    return fail(SYMM_EINVAL, std::string(what) + ": range runs past the end of its slab");
  *off = (size_t)o;
  return SYMM_OK;
}

__global__ void ctrl_zero_kernel(Control* ctl) {
  int64_t* w = reinterpret_cast<int64_t*>(ctl);
  if (threadIdx.x < sizeof(Control) / 8) w[threadIdx.x] = 0;
}

int ensure_ctrl(symm_heap* h, cudaStream_t stream) {
  if (h->ctrl_ready) return SYMM_OK;
  ctrl_zero_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<Control*>(h->base));
  int rc = cuda_check(cudaGetLastError(), "heap header init");
  if (rc == SYMM_OK) h->ctrl_ready = true;
  return rc;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace symm_host

using namespace symm_host;

// ------------------------------------------------------------- kernels ---
namespace {

constexpr int kCopyThreads = 256;
constexpr size_t kPiece = 16384;  // bytes per warp task, cut at dst-aligned boundaries

// Copies n bytes with every warp of the grid; pieces end on kPiece-aligned
// destination addresses so that all but the first start 16-byte aligned.
__device__ __forceinline__ void grid_copy(uint8_t* dst, const uint8_t* src, size_t n) {
  if (n == 0) return;
  const int lane = threadIdx.x & 31;
  const size_t warp = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = (gridDim.x * (size_t)blockDim.x) >> 5;
  const uintptr_t d0 = (uintptr_t)dst;
  const uintptr_t first = (d0 / kPiece + 1) * kPiece;  // first cut after d0
  const uintptr_t end = d0 + n;
  const size_t npieces = end > first ? 1 + (end - first + kPiece - 1) / kPiece : 1;
  for (size_t k = warp; k < npieces; k += nwarps) {
    const uintptr_t lo = k == 0 ? d0 : first + (k - 1) * kPiece;
    uintptr_t hi = k == 0 ? first : lo + kPiece;
    if (hi > end) hi = end;
    symm::warp_copy<4, symm::kCG, symm::kST>(dst + (lo - d0), src + (lo - d0), hi - lo, lane);
  }
}

__global__ void __launch_bounds__(kCopyThreads) put_kernel(uint8_t* dst, const uint8_t* src,
                                                           size_t n) {
  grid_copy(dst, src, n);
}

__device__ __forceinline__ void apply_signal(int64_t* sig, int64_t value, int op) {
  if (op == SYMM_SIGNAL_SET)
    symm::st_release(sig, value);
  else
    symm::red_add_release(sig, value);
}

__global__ void __launch_bounds__(kCopyThreads)
    put_signal_kernel(uint8_t* dst, const uint8_t* src, size_t n, int64_t* sig, int64_t value,
                      int op, Control* ctl) {
  grid_copy(dst, src, n);
  __syncthreads();  // this CTA's stores are ordered before thread 0's release below
  if (threadIdx.x == 0) {
    symm::fence_acq_rel();
    const uint32_t prev = symm::atom_add_acq_rel_u32(&ctl->done, 1u);
    if (prev == gridDim.x - 1) {  // last arrival: every CTA's bytes are visible
      symm::st_relaxed_u32(&ctl->done, 0u);
      apply_signal(sig, value, op);
    }
  }
}

__global__ void signal_kernel(int64_t* sig, int64_t value, int op) {
  if (threadIdx.x == 0) apply_signal(sig, value, op);
}

__global__ void wait_kernel(const int64_t* sig, int cmp, int64_t value, uint64_t budget_ns,
                            Control* ctl, const void* heap_base) {
  if (threadIdx.x == 0) symm::spin_wait(sig, cmp, value, budget_ns, ctl, heap_base);
}

__global__ void ctrl_clear_kernel(Control* ctl) {
  if (threadIdx.x == 0) {
    ctl->error = 0;
    ctl->abort = 0;
    ctl->error_info = 0;
  }
}

int copy_grid(size_t n) {
  const size_t pieces = n / kPiece + 2;
  const size_t warps_per_cta = kCopyThreads / 32;
  size_t ctas = (pieces + warps_per_cta - 1) / warps_per_cta;
  const size_t cap = (size_t)(sm_count() > 0 ? sm_count() : 1) * 8;
  if (ctas > cap) ctas = cap;
  return (int)(ctas ? ctas : 1);
}

}  // namespace

// ------------------------------------------------------------ C ABI: heap --
extern "C" int symm_heap_init(void* base, size_t slab_stride, int npes, symm_heap_t** heap) {
  if (!heap) return fail(SYMM_EINVAL, "symm_heap_init: heap out-pointer is NULL");
  *heap = nullptr;
  if (!base || ((uintptr_t)base & 255))
    return fail(SYMM_EINVAL, "symm_heap_init: base must be non-NULL and 256-byte aligned");
  if (npes < 1) return fail(SYMM_EINVAL, "symm_heap_init: npes must be >= 1");
  if (slab_stride % 256 || slab_stride <= SYMM_HEAP_HEADER_BYTES)
    return fail(SYMM_EINVAL,
                "symm_heap_init: slab_stride must be a multiple of 256 above the header size");
  symm_heap* h = new symm_heap();
  h->base = static_cast<uint8_t*>(base);
  h->slab = slab_stride;
  h->npes = npes;
  h->next = SYMM_HEAP_HEADER_BYTES;
  h->spin_budget = 2000000000ull;
  h->device = -1;
  if (cudaGetDevice(&h->device) == cudaSuccess) {
    // set-up of all2all_combine_pc_noalloc on this device: look up its static
    // array now (this loads the module that holds it), not in its first call
    uint8_t* scratch = nullptr;
    (void)symm_host::noalloc_scratch_address(&scratch);
  }
  cudaGetLastError();  // no device is not an error for host-only use
  h->ctrl_ready = false;
  *heap = h;
  return SYMM_OK;
}

extern "C" int symm_heap_destroy(symm_heap_t* heap) {
  delete heap;
  return SYMM_OK;
}

extern "C" int symm_malloc(symm_heap_t* h, size_t bytes, size_t align, void** ptr) {
  if (!h || !ptr) return fail(SYMM_EINVAL, "symm_malloc: NULL heap or out-pointer");
  *ptr = nullptr;
  if (align == 0) align = 256;
  if (align & (align - 1)) return fail(SYMM_EINVAL, "symm_malloc: align must be a power of two");
  if (align < 256) align = 256;
  if (align > h->slab) return fail(SYMM_ENOMEM, "symm_malloc: alignment exceeds the slab");
  const size_t off = (h->next + align - 1) & ~(align - 1);
  if (off > h->slab || bytes > h->slab - off)
    return fail(SYMM_ENOMEM, "symm_malloc: " + std::to_string(bytes) + " bytes do not fit in " +
                                 std::to_string(h->slab - h->next) + " free bytes per slab");
  const size_t padded = (bytes + 255) & ~(size_t)255;
  h->next = (padded > h->slab - off) ? h->slab : off + padded;
  *ptr = h->base + off;
  return SYMM_OK;
}

extern "C" int symm_heap_reset(symm_heap_t* h) {
  if (!h) return fail(SYMM_EINVAL, "symm_heap_reset: NULL heap");
  h->next = SYMM_HEAP_HEADER_BYTES;
  return SYMM_OK;
}

extern "C" void* symm_at(symm_heap_t* h, const void* ptr, int pe) {
  if (!h || pe < 0 || pe >= h->npes) return nullptr;
  const int64_t off = slab_offset(h, ptr);
  if (off < 0) return nullptr;
  return h->base + (size_t)pe * h->slab + (size_t)off;
}

extern "C" int symm_set_spin_budget(symm_heap_t* h, uint64_t budget_ns) {
  if (!h || budget_ns == 0) return fail(SYMM_EINVAL, "symm_set_spin_budget: bad arguments");
  h->spin_budget = budget_ns;
  return SYMM_OK;
}

extern "C" int symm_check_error(symm_heap_t* h, void* stream, int64_t* info) {
  if (!h) return fail(SYMM_EINVAL, "symm_check_error: NULL heap");
  if (info) *info = 0;
  cudaStream_t s = as_stream(stream);
  int rc = ensure_ctrl(h, s);
  if (rc) return rc;
  Control ctl;
  rc = cuda_check(cudaMemcpyAsync(&ctl, h->base, sizeof(ctl), cudaMemcpyDeviceToHost, s),
                  "symm_check_error: read header");
  if (rc) return rc;
  rc = cuda_check(cudaStreamSynchronize(s), "symm_check_error: synchronize");
  if (rc) return rc;
  if (ctl.error == 0 && ctl.abort == 0) return SYMM_OK;
  ctrl_clear_kernel<<<1, 32, 0, s>>>(reinterpret_cast<Control*>(h->base));
  rc = cuda_check(cudaGetLastError(), "symm_check_error: clear");
  if (rc) return rc;
  if (info) *info = ctl.error_info;
  const int code = ctl.error ? ctl.error : SYMM_ETIMEDOUT;
  if (code == SYMM_ERANGE)
    return fail(code, "device-side sizes exceed a buffer (nothing was copied)");
  if (ctl.error_info >= SYMM_INFO_NOALLOC_SIGNAL)
    return fail(code, "device wait gave up (signal at byte offset " +
                          std::to_string(ctl.error_info - SYMM_INFO_NOALLOC_SIGNAL) +
                          " of the signal area of all2all_combine_pc_noalloc's static array)");
  return fail(code, "device wait gave up (signal at heap byte offset " +
                        std::to_string(ctl.error_info) + ")");
}

extern "C" const char* symm_last_error(void) { return g_last_error.c_str(); }

// ------------------------------------------------------ C ABI: primitives --
static int check_pe(const symm_heap* h, int pe, const char* what) {
  if (pe < 0 || pe >= h->npes)
    return fail(SYMM_EINVAL, std::string(what) + ": PE " + std::to_string(pe) + " out of range");
  return SYMM_OK;
}

static int signal_address(symm_heap* h, const int64_t* signal, size_t signal_off, int pe,
                          const char* what, int64_t** out) {
  int rc = check_pe(h, pe, what);
  if (rc) return rc;
  if (signal_off > (SIZE_MAX / 8) - 1) return fail(SYMM_EINVAL, std::string(what) + ": offset");
  const uint8_t* p = reinterpret_cast<const uint8_t*>(signal) + signal_off * 8;
  size_t off;
  rc = check_range(h, p, 8, what, &off);
  if (rc) return rc;
  if (off & 7) return fail(SYMM_EINVAL, std::string(what) + ": signal not 8-byte aligned");
  *out = reinterpret_cast<int64_t*>(h->base + (size_t)pe * h->slab + off);
  return SYMM_OK;
}

static int remote_range(symm_heap* h, const void* obj, size_t obj_off, size_t bytes, int pe,
                        const char* what, uint8_t** out) {
  int rc = check_pe(h, pe, what);
  if (rc) return rc;
  const int64_t base_off = slab_offset(h, obj);
  if (base_off < 0) return fail(SYMM_EINVAL, std::string(what) + ": not a symmetric-heap pointer");
  if (obj_off > h->slab) return fail(SYMM_EINVAL, std::string(what) + ": offset past the slab");
  size_t off;
  rc = check_range(h, static_cast<const uint8_t*>(obj) + obj_off, bytes, what, &off);
  if (rc) return rc;
  *out = h->base + (size_t)pe * h->slab + off;
  return SYMM_OK;
}

extern "C" int shmem_put(symm_heap_t* h, void* target, size_t target_off, const void* src,
                         size_t src_off, size_t bytes, int target_pe, void* stream) {
  if (!h) return fail(SYMM_EINVAL, "shmem_put: NULL heap");
  uint8_t* dst;
  int rc = remote_range(h, target, target_off, bytes, target_pe, "shmem_put: target", &dst);
  if (rc) return rc;
  if (bytes == 0) return SYMM_OK;
  if (!src) return fail(SYMM_EINVAL, "shmem_put: NULL src");
  const uint8_t* s = static_cast<const uint8_t*>(src) + src_off;
  put_kernel<<<copy_grid(bytes), kCopyThreads, 0, as_stream(stream)>>>(dst, s, bytes);
  return cuda_check(cudaGetLastError(), "shmem_put: launch");
}

extern "C" int shmem_get(symm_heap_t* h, void* dst, size_t dst_off, const void* src,
                         size_t src_off, size_t bytes, int src_pe, void* stream) {
  if (!h) return fail(SYMM_EINVAL, "shmem_get: NULL heap");
  uint8_t* s;
  int rc = remote_range(h, src, src_off, bytes, src_pe, "shmem_get: src", &s);
  if (rc) return rc;
  if (bytes == 0) return SYMM_OK;
  if (!dst) return fail(SYMM_EINVAL, "shmem_get: NULL dst");
  uint8_t* d = static_cast<uint8_t*>(dst) + dst_off;
  put_kernel<<<copy_grid(bytes), kCopyThreads, 0, as_stream(stream)>>>(d, s, bytes);
  return cuda_check(cudaGetLastError(), "shmem_get: launch");
}

extern "C" int shmem_signal_op(symm_heap_t* h, int64_t* signal, size_t signal_off, int64_t value,
                               int op, int target_pe, void* stream) {
  if (!h) return fail(SYMM_EINVAL, "shmem_signal_op: NULL heap");
  if (op != SYMM_SIGNAL_SET && op != SYMM_SIGNAL_ADD)
    return fail(SYMM_EINVAL, "shmem_signal_op: op must be SET (0) or ADD (1)");
  int64_t* sig;
  int rc = signal_address(h, signal, signal_off, target_pe, "shmem_signal_op", &sig);
  if (rc) return rc;
  signal_kernel<<<1, 32, 0, as_stream(stream)>>>(sig, value, op);
  return cuda_check(cudaGetLastError(), "shmem_signal_op: launch");
}

extern "C" int shmem_wait_for_signal(symm_heap_t* h, const int64_t* signal, size_t signal_off,
                                     int64_t cmp_value, int cmp, int pe, uint64_t budget_ns,
                                     void* stream) {
  if (!h) return fail(SYMM_EINVAL, "shmem_wait_for_signal: NULL heap");
  if (cmp != SYMM_CMP_EQ && cmp != SYMM_CMP_GT && cmp != SYMM_CMP_LT)
    return fail(SYMM_EINVAL, "shmem_wait_for_signal: cmp must be EQ (0), GT (1) or LT (2)");
  int64_t* sig;
  int rc = signal_address(h, signal, signal_off, pe, "shmem_wait_for_signal", &sig);
  if (rc) return rc;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  wait_kernel<<<1, 32, 0, s>>>(sig, cmp, cmp_value, budget_ns ? budget_ns : h->spin_budget,
                               reinterpret_cast<Control*>(h->base), h->base);
  return cuda_check(cudaGetLastError(), "shmem_wait_for_signal: launch");
}

extern "C" int shmem_put_with_signal(symm_heap_t* h, void* target, size_t target_off,
                                     const void* src, size_t src_off, size_t bytes,
                                     int64_t* signal, size_t signal_off, int64_t value, int op,
                                     int target_pe, void* stream) {
  if (!h) return fail(SYMM_EINVAL, "shmem_put_with_signal: NULL heap");
  if (op != SYMM_SIGNAL_SET && op != SYMM_SIGNAL_ADD)
    return fail(SYMM_EINVAL, "shmem_put_with_signal: op must be SET (0) or ADD (1)");
  uint8_t* dst;
  int rc = remote_range(h, target, target_off, bytes, target_pe, "shmem_put_with_signal: target",
                        &dst);
  if (rc) return rc;
  int64_t* sig;
  rc = signal_address(h, signal, signal_off, target_pe, "shmem_put_with_signal: signal", &sig);
  if (rc) return rc;
  if (bytes && !src) return fail(SYMM_EINVAL, "shmem_put_with_signal: NULL src");
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  const uint8_t* sp = static_cast<const uint8_t*>(src) + (bytes ? src_off : 0);
  put_signal_kernel<<<copy_grid(bytes), kCopyThreads, 0, s>>>(
      dst, sp, bytes, sig, value, op, reinterpret_cast<Control*>(h->base));
  return cuda_check(cudaGetLastError(), "shmem_put_with_signal: launch");
}
