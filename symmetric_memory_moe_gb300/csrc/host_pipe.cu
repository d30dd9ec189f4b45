// host_pipe.cu -- the combine on host buffers.
//
// Page-locked host buffers are mapped into the device's address space, and
// on GB300 the GPU reaches host memory over the coherent chip-to-chip link.
// So for the direct variant the run kernel reads host_in and writes host_out
// in place: one pass, both link directions busy at once, no copy engine and
// no staging in device memory (measured 340 GB/s over the link against 341
// for copy-engine copies in both directions at once).  Otherwise (pageable
// buffers, or the producer/consumer variant, which stages through the
// symmetric heap by design) the work goes through copies, pipelined by
// chunks of S rows over three streams:
//
// The combine keeps every row s of the output independent: out_d rows
// s0 .. s1 need exactly the input rows d*S + s0 .. d*S + s1 of every PE r.
// So a chunk of cs rows is (1) gathered from the host into a compact device
// buffer [d][cs] per PE with one 2-D copy per PE (W strided pieces of the
// host input), (2) combined with S = cs, and (3) copied back with one copy
// per destination PE.  Two buffers (inside the caller's `in` and `out`
// objects) alternate, so the host-to-device copy of chunk c + 1, the
// combine of chunk c and the device-to-host copy of chunk c - 1 overlap.
#include <cuda.h>  // CUpointer_attribute (types only)
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <string>

#include "symm_internal.h"

using namespace symm_host;

#ifndef SYMM_HOST_CHUNKS
#define SYMM_HOST_CHUNKS 8  // chunks of S rows in the pipeline
#endif

namespace {

// Two copy streams and the events of the pipeline, per device, kept for the
// process's lifetime.
struct Pipe {
  std::mutex mu;  // one enqueue at a time: event waits take the state at enqueue
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr, in_ready[2] = {}, computed[2] = {}, drained[2] = {};
};

int pipe_for_device(Pipe** out) {
  static std::mutex mu;
  static std::map<int, Pipe> pipes;  // node-based: entries never move
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "all2all_combine_host: device");
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(mu);
  auto it = pipes.find(dev);
  if (it == pipes.end()) {
    it = pipes.try_emplace(dev).first;
    Pipe& p = it->second;
    rc = cuda_check(cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking), "stream");
    if (!rc) rc = cuda_check(cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking), "stream");
    cudaEvent_t* evs[7] = {&p.entry,       &p.in_ready[0], &p.in_ready[1], &p.computed[0],
                           &p.computed[1], &p.drained[0],  &p.drained[1]};
    for (int i = 0; i < 7 && !rc; ++i)
      rc = cuda_check(cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming), "event");
    if (rc) {
      pipes.erase(it);
      return rc;
    }
  }
  *out = &it->second;
  return SYMM_OK;
}

// The device address of [p, p + bytes) when the whole range lies inside one
// page-locked, device-mapped host allocation (else nullptr): the kernel must
// not run past the caller's allocation.
void* mapped_host_range(const void* p, size_t bytes) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory may report an error here: not sticky
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  static PFN_cuPointerGetAttribute_v4000 get_attr = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 4000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuPointerGetAttribute_v4000) nullptr;
    return reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(f);
  }();
  if (!get_attr) return nullptr;
  CUdeviceptr start = 0;
  size_t size = 0;
  const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(at.devicePointer);
  if (get_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
      get_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS)
    return nullptr;
  if (dp < start || dp - start > size || bytes > size - (dp - start)) return nullptr;
  return at.devicePointer;
}

}  // namespace

extern "C" int all2all_combine_host(symm_heap_t* h, const void* host_in, void* host_out,
                                    const void* in, void* out, int W, int S, int H, int D,
                                    int elem_bytes, int variant, int tile_s, int block_d,
                                    int buffer_num, void* staging, int64_t* signals,
                                    void* stream) {
  const char* what = "all2all_combine_host";
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  if (S < 0 || W < 1 || W != h->npes || H < 0 || D < 0 || elem_bytes < 1)
    return fail(SYMM_EINVAL, std::string(what) + ": bad W, S, H, D or elem_bytes");
  const size_t R = (size_t)H * D * elem_bytes;  // one input row
  if (R && (size_t)S * W > SIZE_MAX / R)
    return fail(SYMM_EINVAL, std::string(what) + ": size overflow");
  const size_t nbytes = (size_t)S * W * R;  // per PE, in and out
  size_t in_off, out_off;
  int rc = check_range(h, in, nbytes, (std::string(what) + ": in").c_str(), &in_off);
  if (rc) return rc;
  rc = check_range(h, out, nbytes, (std::string(what) + ": out").c_str(), &out_off);
  if (rc) return rc;
  if (nbytes && in_off < out_off + nbytes && out_off < in_off + nbytes)
    return fail(SYMM_EINVAL, std::string(what) + ": input and output ranges overlap");
  if (nbytes == 0)  // nothing to move; the combine still validates its arguments
    return all2all_combine(h, in, out, W, S, H, D, elem_bytes, variant, tile_s, block_d,
                           buffer_num, staging, signals, stream);
  if (!host_in || !host_out) return fail(SYMM_EINVAL, std::string(what) + ": NULL host buffer");
  const int kind = variant & 0xff, flags = variant & ~0xff;
  if ((kind != SYMM_A2A_DIRECT && kind != SYMM_A2A_PC) ||
      (flags & ~(SYMM_A2A_FLAG_NO_RESET | SYMM_A2A_FLAG_VECTOR | SYMM_A2A_FLAG_BULK)))
    return fail(SYMM_EINVAL, std::string(what) + ": unknown variant or flag");
  cudaStream_t s = as_stream(stream);
  const uint8_t* hin = static_cast<const uint8_t*>(host_in);
  uint8_t* hout = static_cast<uint8_t*>(host_out);
  const size_t host_bytes = (size_t)W * nbytes;
  if (kind == SYMM_A2A_DIRECT && !(flags & SYMM_A2A_FLAG_BULK) &&
      (hin + host_bytes <= hout || hout + host_bytes <= hin)) {
    const void* din = mapped_host_range(hin, host_bytes);
    void* dout = din ? mapped_host_range(hout, host_bytes) : nullptr;
    if (din && dout)  // the combine in place on the host buffers
      return launch_runs_raw(static_cast<const uint8_t*>(din), static_cast<uint8_t*>(dout),
                             nbytes, nbytes, (uint32_t)W, (uint32_t)S, R, false, s, what,
                             /*device_mem=*/false);
  }

  // chunks of cs rows, two buffers of W*cs rows inside each object
  const int chunks = S >= 2 * SYMM_HOST_CHUNKS ? SYMM_HOST_CHUNKS : 1;
  const int cs = (S + chunks - 1) / chunks;
  if (chunks == 1) {  // one chunk: the plain sequence on the caller's stream
    for (int r = 0; r < W; ++r) {
      rc = cuda_check(cudaMemcpyAsync(h->base + (size_t)r * h->slab + in_off, hin + r * nbytes,
                                      nbytes, cudaMemcpyHostToDevice, s),
                      "all2all_combine_host: host-to-device copy");
      if (rc) return rc;
    }
    rc = all2all_combine(h, in, out, W, S, H, D, elem_bytes, variant, tile_s, block_d,
                         buffer_num, staging, signals, stream);
    if (rc) return rc;
    for (int d = 0; d < W; ++d) {
      rc = cuda_check(cudaMemcpyAsync(hout + d * nbytes, h->base + (size_t)d * h->slab + out_off,
                                      nbytes, cudaMemcpyDeviceToHost, s),
                      "all2all_combine_host: device-to-host copy");
      if (rc) return rc;
    }
    return SYMM_OK;
  }

  Pipe* p;
  rc = pipe_for_device(&p);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(p->mu);
  // everything enqueued on the caller's stream before this call comes first
  rc = cuda_check(cudaEventRecord(p->entry, s), "all2all_combine_host: event");
  if (!rc) rc = cuda_check(cudaStreamWaitEvent(p->h2d, p->entry, 0), "all2all_combine_host: wait");
  if (!rc) rc = cuda_check(cudaStreamWaitEvent(p->d2h, p->entry, 0), "all2all_combine_host: wait");
  if (rc) return rc;
  const size_t buf_bytes = (size_t)W * cs * R;  // one chunk, per PE (input or output)
  for (int c = 0; c < chunks; ++c) {
    const int s0 = c * cs;
    const int rows = std::min(cs, S - s0);
    if (rows <= 0) break;
    const int b = c & 1;
    const size_t boff = b * buf_bytes;
    // (1) gather: in_r[d*S + s0 .. + rows] -> buffer b of PE r, laid out [d][rows]
    if (c >= 2) {  // the combine of chunk c - 2 has read this buffer
      rc = cuda_check(cudaStreamWaitEvent(p->h2d, p->computed[b], 0), "all2all_combine_host");
      if (rc) return rc;
    }
    for (int r = 0; r < W; ++r) {
      rc = cuda_check(cudaMemcpy2DAsync(h->base + (size_t)r * h->slab + in_off + boff,
                                        (size_t)rows * R, hin + r * nbytes + (size_t)s0 * R,
                                        (size_t)S * R, (size_t)rows * R, (size_t)W,
                                        cudaMemcpyHostToDevice, p->h2d),
                      "all2all_combine_host: host-to-device copy");
      if (rc) return rc;
    }
    rc = cuda_check(cudaEventRecord(p->in_ready[b], p->h2d), "all2all_combine_host: event");
    if (rc) return rc;
    // (2) combine the chunk on the caller's stream
    rc = cuda_check(cudaStreamWaitEvent(s, p->in_ready[b], 0), "all2all_combine_host: wait");
    if (!rc && c >= 2)  // the copy-out of chunk c - 2 has read this output buffer
      rc = cuda_check(cudaStreamWaitEvent(s, p->drained[b], 0), "all2all_combine_host: wait");
    if (rc) return rc;
    rc = all2all_combine(h, static_cast<const uint8_t*>(in) + boff,
                         static_cast<uint8_t*>(out) + boff, W, rows, H, D, elem_bytes, variant,
                         tile_s, block_d, buffer_num, staging, signals, stream);
    if (rc) return rc;
    rc = cuda_check(cudaEventRecord(p->computed[b], s), "all2all_combine_host: event");
    if (rc) return rc;
    // (3) copy out: rows s0 .. of out_d, one copy per destination PE
    rc = cuda_check(cudaStreamWaitEvent(p->d2h, p->computed[b], 0), "all2all_combine_host: wait");
    if (rc) return rc;
    for (int d = 0; d < W; ++d) {
      rc = cuda_check(cudaMemcpyAsync(hout + d * nbytes + (size_t)s0 * W * R,
                                      h->base + (size_t)d * h->slab + out_off + boff,
                                      (size_t)rows * W * R, cudaMemcpyDeviceToHost, p->d2h),
                      "all2all_combine_host: device-to-host copy");
      if (rc) return rc;
    }
    rc = cuda_check(cudaEventRecord(p->drained[b], p->d2h), "all2all_combine_host: event");
    if (rc) return rc;
  }
  // the caller's stream continues once the last copies have landed
  for (int b = 0; b < 2 && !rc; ++b)
    rc = cuda_check(cudaStreamWaitEvent(s, p->drained[b], 0), "all2all_combine_host: wait");
  return rc;
}
