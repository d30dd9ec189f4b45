// collectives.cu -- push-mode AllToAll with uneven per-pair row counts, and
// push-mode AllGather, on the emulated symmetric heap.
//
// Source: HyperParallel RFC "Symmetric Memory (one-sided communication)",
// section 10 (advanced algorithms):
//  * AllToAll, push mode: the receive offsets are exchanged first
//    (metadata), then every rank pushes its segment for each destination, and
//    each destination's signal is ADDed to until it reaches world_size.
//  * AllGather, push mode: every rank pushes its data to
//    output[rank * size] of every rank and ADDs 1 to that rank's signal; a
//    receiver waits for its signal to reach world_size.
//
// GB300 design: all W PEs run in one launch per step.  The metadata step is
// one small kernel (prefix sums over the W x W counts on the device, so the
// host never synchronises to learn them); the push is one grid-stride kernel
// in which the warp that completes a unit of signalling -- counted with an
// acquire/release atomic -- ADDs 1 to the destination's signal with release
// semantics; a last one-thread kernel performs the receivers' waits
// (bounded).  Segments with no rows are signalled by the metadata kernel.
// AllToAll: one warp per output row; a (source, destination) segment is the
// unit of signalling.  AllGather: one warp per 8 KB piece of a PE's input,
// read once and stored to all W outputs (W reads of the same input would
// cost W times its bytes in DRAM reads); all W segments of a source complete
// together.  The page's 16-stream pool
// and the separate metadata all_to_all collapse into these in-stream kernels.
#include <string>

#include "symm_device.cuh"
#include "symm_internal.h"

using symm::Control;
using namespace symm_host;

namespace {

constexpr int kThreads = 256;
#ifndef SYMM_A2AV_UNROLL
#define SYMM_A2AV_UNROLL 4  // 16-byte vectors in flight per lane in the AllToAll push (8: -3 %)
#endif
#ifndef SYMM_AG_BCAST_UNROLL
#define SYMM_AG_BCAST_UNROLL 8  // 16-byte vectors in flight per lane in the AllGather push
#endif
constexpr size_t kGatherPiece = 8192;  // AllGather work unit (bytes of one PE's input)
enum { kErrRange = -5 };

// Workspace (int64 words): send_off[W*W] | recv_off[W*W] | done[W*W] |
// recv_total[W] | valid[1]
struct Ws {
  int64_t *send_off, *recv_off, *done, *recv_total, *valid;
};
__host__ __device__ inline Ws ws_of(int64_t* w, int W) {
  const size_t ww = (size_t)W * W;
  return Ws{w, w + ww, w + 2 * ww, w + 3 * ww, w + 3 * ww + W};
}
size_t ws_words(int W) { return 3 * (size_t)W * W + W + 1; }

__device__ __forceinline__ uint64_t atom_add_acq_rel_u64(int64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}

// One CTA: prefix sums, capacity checks, zeroed counters and signals, and
// the signal of every empty segment.  counts == nullptr means every segment
// has `uniform` rows (AllGather: pieces of one segment).
__global__ void collective_meta_kernel(const int64_t* counts, int64_t uniform, int W,
                                       int64_t in_rows, int64_t out_rows, int64_t* wsp,
                                       int64_t* signals, size_t slab, Control* ctl) {
  const Ws ws = ws_of(wsp, W);
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int t = threadIdx.x; t < W; t += blockDim.x) {
    int64_t acc = 0;  // rank t as sender: offsets of its segment for each d
    for (int d = 0; d < W; ++d) {
      const int64_t c = counts ? counts[(size_t)t * W + d] : uniform;
      if (c < 0 || c > in_rows || c > out_rows) bad = 1;  // also keeps the sums from overflowing
      ws.send_off[(size_t)t * W + d] = acc;
      acc += c;
    }
    if (acc > in_rows) bad = 1;
    acc = 0;  // rank t as receiver: where each sender's segment lands
    for (int r = 0; r < W; ++r) {
      const int64_t c = counts ? counts[(size_t)r * W + t] : uniform;
      ws.recv_off[(size_t)r * W + t] = acc;
      acc += c;
    }
    ws.recv_total[t] = acc;
    if (acc > out_rows) bad = 1;
    *reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(signals) + (size_t)t * slab) = 0;
  }
  for (size_t i = threadIdx.x; i < (size_t)W * W; i += blockDim.x) ws.done[i] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    *ws.valid = bad ? 0 : 1;
    if (bad) symm::record_error(ctl, kErrRange, -1);
  }
  if (bad) return;
  for (size_t i = threadIdx.x; i < (size_t)W * W; i += blockDim.x) {
    const int64_t c = counts ? counts[i] : uniform;
    if (c == 0)  // an empty segment is complete at once
      symm::red_add_release(
          reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(signals) + (i % W) * slab), 1);
  }
}

// Marks one more unit of segment (r, d) done; the unit that completes it
// ADDs 1 to PE d's signal.  The acquire/release count chains every unit's
// writes (ordered before the count by __syncwarp) into the final release.
__device__ __forceinline__ void unit_done(int64_t* done, int64_t total, int64_t* sig_d, int lane) {
  __syncwarp();
  if (lane == 0) {
    const uint64_t prev = atom_add_acq_rel_u64(done, 1);
    if ((int64_t)prev + 1 == total) symm::red_add_release(sig_d, 1);
  }
}

// AllToAll push: one warp per output row (d, j); the owner r of row j is the
// last sender whose receive offset is <= j.
__global__ void __launch_bounds__(kThreads)
    alltoall_push_kernel(const uint8_t* in, uint8_t* out, const int64_t* counts, int W,
                         size_t row_bytes, int64_t out_rows, int64_t* wsp, int64_t* signals,
                         size_t slab) {
  const Ws ws = ws_of(wsp, W);
  if (*ws.valid != 1) return;
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (blockIdx.x * (uint64_t)kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  const uint64_t nunits = (uint64_t)W * out_rows;
  for (uint64_t k = warp; k < nunits; k += nwarps) {
    const int d = (int)(k / out_rows);
    const int64_t j = (int64_t)(k % out_rows);
    if (j >= ws.recv_total[d]) continue;
    int r = 0;
    for (int rr = 1; rr < W; ++rr)
      if (ws.recv_off[(size_t)rr * W + d] <= j) r = rr;
    const size_t seg = (size_t)r * W + d;
    const int64_t src_row = ws.send_off[seg] + (j - ws.recv_off[seg]);
    symm::warp_copy<SYMM_A2AV_UNROLL, symm::kRO, symm::kST>(
        out + d * slab + (size_t)j * row_bytes, in + r * slab + (size_t)src_row * row_bytes,
        row_bytes, lane);
    unit_done(&ws.done[seg], counts[seg],
              reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(signals) + d * slab), lane);
  }
}

// One warp copies n bytes from src to nd destinations dst + i * dstride
// (i < nd), reading src once.  dstride is a multiple of 16, so every
// destination has dst's alignment and one plan serves all of them: bytes up
// to dst's 16-byte boundary one per lane, then 16-byte stores (loads
// funnel-shifted when src and dst disagree mod 16, as in symm::warp_copy;
// a block read past the end of src stays in its 16-byte-aligned block), then
// the last < 16 bytes one per lane.
template <int U>
__device__ __forceinline__ void warp_copy_bcast(uint8_t* dst, size_t dstride, int nd,
                                                const uint8_t* src, size_t n, int lane) {
  if (n == 0) return;
  size_t head = (16 - ((uintptr_t)dst & 15)) & 15;
  if (head > n) head = n;
  if ((size_t)lane < head) {
    const uint8_t b = symm::ld1_ro(src + lane);
    for (int i = 0; i < nd; ++i) symm::st1(dst + i * dstride + lane, b);
  }
  const size_t nvec = (n - head) >> 4;
  uint8_t* d = dst + head;
  const uint8_t* s = src + head;
  const unsigned m = (unsigned)((uintptr_t)s & 15);
  for (size_t base = 0; base < nvec; base += 32 * U) {  // warp-uniform loop
    uint4 v[U];
    if (m == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t j = base + 32 * u + lane;
        if (j < nvec) v[u] = symm::ld16_ro(s + 16 * j);
      }
    } else {
      const uint8_t* a0 = s - m;  // aligned blocks a0[0..nvec] cover the body
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t j = base + 32 * u + lane;
        const uint4 a = j <= nvec ? symm::ld16_ro(a0 + 16 * j) : make_uint4(0, 0, 0, 0);
        uint4 b;
        b.x = __shfl_down_sync(0xffffffffu, a.x, 1);
        b.y = __shfl_down_sync(0xffffffffu, a.y, 1);
        b.z = __shfl_down_sync(0xffffffffu, a.z, 1);
        b.w = __shfl_down_sync(0xffffffffu, a.w, 1);
        if (lane == 31 && j + 1 <= nvec) b = symm::ld16_ro(a0 + 16 * (j + 1));
        v[u] = symm::funnel16(a, b, m);
      }
    }
    for (int i = 0; i < nd; ++i) {
      uint8_t* di = d + i * dstride;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t j = base + 32 * u + lane;
        if (j < nvec) symm::st16(di + 16 * j, v[u]);
      }
    }
  }
  const size_t done = head + (nvec << 4);
  if ((size_t)lane < n - done) {
    const uint8_t b = symm::ld1_ro(src + done + lane);
    for (int i = 0; i < nd; ++i) symm::st1(dst + i * dstride + done + lane, b);
  }
}

// AllGather push: one warp per piece p of PE r's input, read once and
// written to byte r*bytes + p*kGatherPiece of every PE's output.  The unit
// that completes PE r's input ADDs 1 to every PE's signal (one per lane
// stride; __syncwarp orders the lanes' releases after lane 0's acquire).
__global__ void __launch_bounds__(kThreads)
    allgather_push_kernel(const uint8_t* in, uint8_t* out, int W, size_t bytes, int64_t pieces,
                          int64_t* wsp, int64_t* signals, size_t slab) {
  const Ws ws = ws_of(wsp, W);
  if (*ws.valid != 1) return;
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (blockIdx.x * (uint64_t)kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  const uint64_t nunits = (uint64_t)W * pieces;
  for (uint64_t k = warp; k < nunits; k += nwarps) {
    const int r = (int)(k / pieces);
    const size_t off = (size_t)(k % pieces) * kGatherPiece;
    const size_t len = bytes - off < kGatherPiece ? bytes - off : kGatherPiece;
    warp_copy_bcast<SYMM_AG_BCAST_UNROLL>(out + (size_t)r * bytes + off, slab, W,
                                          in + r * slab + off, len, lane);
    __syncwarp();
    int last = 0;
    if (lane == 0) last = (int64_t)atom_add_acq_rel_u64(&ws.done[r], 1) + 1 == pieces;
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();
    if (last)
      for (int d = lane; d < W; d += 32)
        symm::red_add_release(
            reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(signals) + d * slab), 1);
  }
}

// The receivers' waits: every PE's signal reaches W (bounded spin).
__global__ void collective_wait_kernel(int W, int64_t* wsp, int64_t* signals, size_t slab,
                                       uint64_t budget_ns, Control* ctl, const void* heap_base) {
  const Ws ws = ws_of(wsp, W);
  if (threadIdx.x != 0 || *ws.valid != 1) return;
  for (int d = 0; d < W; ++d) {
    const int64_t* sig =
        reinterpret_cast<const int64_t*>(reinterpret_cast<const uint8_t*>(signals) + d * slab);
    if (symm::spin_wait(sig, symm::kCmpEq, W, budget_ns, ctl, heap_base) != symm::kSpinOk) return;
  }
}

int push_grid(size_t units) {
  const size_t ctas = (units + kThreads / 32 - 1) / (kThreads / 32);
  const size_t cap = (size_t)(sm_count() > 0 ? sm_count() : 1) * 8;
  return (int)(ctas < cap ? (ctas ? ctas : 1) : cap);
}

// Shared argument checks: in/out ranges, disjointness, signals, workspace.
int check_collective(symm_heap* h, const void* in, size_t in_bytes, const void* out,
                     size_t out_bytes, const int64_t* signals, const void* workspace, int W,
                     const char* what, size_t* in_off, size_t* out_off, size_t* sig_off) {
  if (!h) return fail(SYMM_EINVAL, std::string(what) + ": NULL heap");
  if (W != h->npes) return fail(SYMM_EINVAL, std::string(what) + ": W differs from the heap's PEs");
  if (!workspace || ((uintptr_t)workspace & 7))
    return fail(SYMM_EINVAL, std::string(what) + ": workspace NULL or not 8-byte aligned");
  int rc = check_range(h, in, in_bytes, (std::string(what) + ": in").c_str(), in_off);
  if (rc) return rc;
  rc = check_range(h, out, out_bytes, (std::string(what) + ": out").c_str(), out_off);
  if (rc) return rc;
  rc = check_range(h, signals, 8, (std::string(what) + ": signals").c_str(), sig_off);
  if (rc) return rc;
  if (*sig_off & 7) return fail(SYMM_EINVAL, std::string(what) + ": signals not 8-byte aligned");
  const size_t offs[3] = {*in_off, *out_off, *sig_off};
  const size_t lens[3] = {in_bytes, out_bytes, 8};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (lens[i] && lens[j] && offs[i] < offs[j] + lens[j] && offs[j] < offs[i] + lens[i])
        return fail(SYMM_EINVAL, std::string(what) + ": in/out/signals ranges overlap");
  return SYMM_OK;
}

}  // namespace

extern "C" int shmem_collective_workspace(int W, size_t* bytes) {
  if (W < 1 || W > 4096 || !bytes)
    return fail(SYMM_EINVAL, "shmem_collective_workspace: W must be in [1, 4096]");
  *bytes = (ws_words(W) * 8 + 255) & ~(size_t)255;
  return SYMM_OK;
}

extern "C" int shmem_alltoall(symm_heap_t* h, const void* in, void* out, const int64_t* counts,
                              int W, size_t row_bytes, size_t in_rows, size_t out_rows,
                              void* workspace, int64_t* signals, void* stream) {
  const char* what = "shmem_alltoall";
  if (!counts) return fail(SYMM_EINVAL, "shmem_alltoall: NULL counts");
  if (W < 1 || W > 4096) return fail(SYMM_EINVAL, "shmem_alltoall: W must be in [1, 4096]");
  size_t in_bytes, out_bytes;
  if (in_rows > (1ull << 40) || out_rows > (1ull << 40) ||
      __builtin_mul_overflow(in_rows, row_bytes, &in_bytes) ||
      __builtin_mul_overflow(out_rows, row_bytes, &out_bytes))
    return fail(SYMM_EINVAL, "shmem_alltoall: rows or row_bytes too large");
  size_t in_off, out_off, sig_off;
  int rc = check_collective(h, in, in_bytes, out, out_bytes, signals, workspace, W, what, &in_off,
                            &out_off, &sig_off);
  if (rc) return rc;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  Control* ctl = reinterpret_cast<Control*>(h->base);
  int64_t* wsp = static_cast<int64_t*>(workspace);
  int64_t* sig = reinterpret_cast<int64_t*>(h->base + sig_off);
  collective_meta_kernel<<<1, 256, 0, s>>>(counts, 0, W, (int64_t)in_rows, (int64_t)out_rows, wsp,
                                           sig, h->slab, ctl);
  rc = cuda_check(cudaGetLastError(), "shmem_alltoall: metadata");
  if (rc) return rc;
  if (out_rows) {  // rows of zero bytes still complete their segments
    alltoall_push_kernel<<<push_grid((size_t)W * out_rows), kThreads, 0, s>>>(
        h->base + in_off, h->base + out_off, counts, W, row_bytes, (int64_t)out_rows, wsp, sig,
        h->slab);
    rc = cuda_check(cudaGetLastError(), "shmem_alltoall: push");
    if (rc) return rc;
  }
  collective_wait_kernel<<<1, 32, 0, s>>>(W, wsp, sig, h->slab, h->spin_budget, ctl, h->base);
  return cuda_check(cudaGetLastError(), "shmem_alltoall: wait");
}

extern "C" int shmem_allgather(symm_heap_t* h, const void* in, void* out, int W, size_t bytes,
                               void* workspace, int64_t* signals, void* stream) {
  const char* what = "shmem_allgather";
  if (W < 1 || W > 4096) return fail(SYMM_EINVAL, "shmem_allgather: W must be in [1, 4096]");
  if (bytes > (1ull << 40) / (size_t)W)
    return fail(SYMM_EINVAL, "shmem_allgather: bytes too large");
  size_t in_off, out_off, sig_off;
  int rc = check_collective(h, in, bytes, out, (size_t)W * bytes, signals, workspace, W, what,
                            &in_off, &out_off, &sig_off);
  if (rc) return rc;
  cudaStream_t s = as_stream(stream);
  rc = ensure_ctrl(h, s);
  if (rc) return rc;
  Control* ctl = reinterpret_cast<Control*>(h->base);
  int64_t* wsp = static_cast<int64_t*>(workspace);
  int64_t* sig = reinterpret_cast<int64_t*>(h->base + sig_off);
  const int64_t pieces = (int64_t)((bytes + kGatherPiece - 1) / kGatherPiece);
  collective_meta_kernel<<<1, 256, 0, s>>>(nullptr, pieces, W, (int64_t)W * pieces,
                                           (int64_t)W * pieces, wsp, sig, h->slab, ctl);
  rc = cuda_check(cudaGetLastError(), "shmem_allgather: metadata");
  if (rc) return rc;
  if (pieces) {
    allgather_push_kernel<<<push_grid((size_t)W * pieces), kThreads, 0, s>>>(
        h->base + in_off, h->base + out_off, W, bytes, pieces, wsp, sig, h->slab);
    rc = cuda_check(cudaGetLastError(), "shmem_allgather: push");
    if (rc) return rc;
  }
  collective_wait_kernel<<<1, 32, 0, s>>>(W, wsp, sig, h->slab, h->spin_budget, ctl, h->base);
  return cuda_check(cudaGetLastError(), "shmem_allgather: wait");
}
