// symm_device.cuh -- device-side building blocks of the symmetric-heap library
// (sm_103a): scoped release/acquire on int64 signals, a bounded spin, and
// warp-cooperative byte copies that keep 16-byte vector loads and stores on
// any source/destination alignment.
//
// Memory-model notes.  All W emulated PEs live on one GPU, so ".gpu" scope is
// the scope of every signal.  A signal is released by one thread after a
// named barrier of its group (the group's stores are ordered before the
// release through the barrier, then the release fence), and acquired by one
// thread before a named barrier (the group's later loads are ordered after
// the acquire).  Data that may change while a kernel runs (staging slots,
// one-sided put/get sources) is read with ld.global.cg (L2 only), never
// through the non-coherent path; inputs that are read-only for the whole
// launch use ld.global.nc with L1::no_allocate.
#pragma once

#include <stdint.h>

namespace symm {

// ---------------------------------------------------------------- scalars --
__device__ __forceinline__ int64_t ld_acquire(const int64_t* p) {
  int64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int64_t ld_relaxed(const int64_t* p) {
  int64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int64_t* p, int64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_release(int64_t* p, int64_t v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Named barrier over `nthreads` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------ control block ------
// Lives in the first bytes of slab 0 of every heap (the heap header).
struct Control {
  int32_t error;       // 0 or a negative SYMM_E* code (first error wins)
  uint32_t abort;      // set once any waiter gives up; every spin then returns
  int64_t error_info;  // byte offset (from the heap base) of the signal that timed out
  uint32_t done;       // CTA arrival counter of shmem_put_with_signal
  uint32_t pad0;
  int64_t reserved[5];
};

enum { kCmpEq = 0, kCmpGt = 1, kCmpLt = 2 };
enum { kSpinOk = 0, kSpinTimeout = 1, kSpinAborted = 2 };
enum { kErrTimedOut = -3 };

__device__ __forceinline__ bool cmp_holds(int64_t cur, int cmp, int64_t v) {
  return cmp == kCmpEq ? cur == v : (cmp == kCmpGt ? cur > v : cur < v);
}

__device__ __forceinline__ void record_error(Control* ctl, int code, int64_t info) {
  if (atomicCAS(reinterpret_cast<int*>(&ctl->error), 0, code) == 0) ctl->error_info = info;
  st_relaxed_u32(&ctl->abort, 1u);
}
// A wait on `sig` gave up: records its byte offset from `base`, plus `bias`
// (0 for signals in the heap, whose base is the heap's).
__device__ __forceinline__ void record_timeout(Control* ctl, const void* base, const int64_t* sig,
                                               int64_t bias = 0) {
  record_error(ctl, kErrTimedOut, (int64_t)((const char*)sig - (const char*)base) + bias);
}

// Longest sleep between two polls of a spin, in ns (0: poll without sleeping).
#ifndef SYMM_SPIN_MAX_SLEEP_NS
#define SYMM_SPIN_MAX_SLEEP_NS 256
#endif

// Spin (one thread) until `*sig cmp v` holds, with acquire semantics.  Gives
// up after `budget_ns` of %globaltimer time, or after an iteration cap that
// bounds the wait even if the timer stood still, or as soon as another waiter
// has raised the abort flag.  Never traps.  A give-up is recorded as the
// signal's offset from heap_base plus info_bias.
__device__ __forceinline__ int spin_wait(const int64_t* sig, int cmp, int64_t v, uint64_t budget_ns,
                                         Control* ctl, const void* heap_base,
                                         int64_t info_bias = 0) {
  if (cmp_holds(ld_acquire(sig), cmp, v)) return kSpinOk;
  const uint64_t t0 = globaltimer_ns();
  // a poll takes >= ~16 ns, so this cap is >= ~budget/4 of wall time even if
  // the timer stood still
  const uint64_t max_iters = budget_ns / 64 + 4096;
  uint32_t backoff = 16;
  for (uint64_t it = 0;; ++it) {
    if (cmp_holds(ld_acquire(sig), cmp, v)) return kSpinOk;
    if (ld_relaxed_u32(&ctl->abort)) return kSpinAborted;
    if (globaltimer_ns() - t0 > budget_ns || it > max_iters) {
      record_timeout(ctl, heap_base, sig, info_bias);
      return kSpinTimeout;
    }
    if (SYMM_SPIN_MAX_SLEEP_NS > 0) {
      __nanosleep(backoff);
      if (backoff < SYMM_SPIN_MAX_SLEEP_NS) backoff <<= 1;
    }
  }
}

// -------------------------------------------------------------- vectors ---
// Read-only-for-the-launch input: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld16_ro(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// Data another thread may have written during this launch: L2 only.
__device__ __forceinline__ uint4 ld16_cg(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// Streaming store (evict-first): final outputs that nothing re-reads soon.
__device__ __forceinline__ void st16_cs(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint8_t ld1_ro(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return (uint8_t)v;
}
__device__ __forceinline__ uint8_t ld1_cg(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return (uint8_t)v;
}
__device__ __forceinline__ void st1(uint8_t* p, uint8_t v) {
  asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "h"((uint16_t)v) : "memory");
}

// L2 cache policies (createpolicy) and accesses that carry one.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st16_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// Load policy: kRO for launch-constant inputs, kCG for data written in-launch.
enum LoadKind { kRO = 0, kCG = 1 };
// Store policy: plain, or streaming (evict-first) for final outputs.
enum StoreKind { kST = 0, kCS = 1 };

template <int LK>
__device__ __forceinline__ uint4 ld16(const void* p) {
  if (LK == kRO) return ld16_ro(p);
  return ld16_cg(p);
}
template <int SK>
__device__ __forceinline__ void st16k(void* p, uint4 v) {
  if (SK == kCS)
    st16_cs(p, v);
  else
    st16(p, v);
}
template <int LK>
__device__ __forceinline__ uint8_t ld1(const uint8_t* p) {
  if (LK == kRO) return ld1_ro(p);
  return ld1_cg(p);
}

// One warp copies nvec 16-byte vectors; src and dst are 16-byte aligned.
template <int U, int LK, int SK>
__device__ __forceinline__ void warp_copy_aligned(uint8_t* dst, const uint8_t* src, size_t nvec,
                                                  int lane) {
  size_t j = lane;
  for (; j + 32 * (U - 1) < nvec; j += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld16<LK>(src + 16 * (j + 32 * u));
#pragma unroll
    for (int u = 0; u < U; ++u) st16k<SK>(dst + 16 * (j + 32 * u), v[u]);
  }
  uint4 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (j + 32 * u < nvec) v[u] = ld16<LK>(src + 16 * (j + 32 * u));
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (j + 32 * u < nvec) st16k<SK>(dst + 16 * (j + 32 * u), v[u]);
}

// A step of `g` vectors through a tile of rows of `vrow` vectors, as whole
// rows plus vectors (vrow > 0): advance() moves a (row, vector) position by
// it with two adds and a compare.
struct TileStep {
  uint32_t rows, vecs;  // g = rows * vrow + vecs, vecs < vrow
  __device__ __forceinline__ void advance(uint32_t& i, uint32_t& c, uint32_t vrow) const {
    i += rows;
    c += vecs;
    if (c >= vrow) {
      c -= vrow;
      ++i;
    }
  }
};
__device__ __forceinline__ TileStep tile_step(uint32_t g, uint32_t vrow) {
  TileStep t;
  t.rows = g / vrow;
  t.vecs = g - t.rows * vrow;
  return t;
}

// One tile (rows x vrow 16-byte vectors, rows dst_row / src_row bytes apart)
// copied by a group of G threads (gtid = 0 .. G-1) with the tile flattened
// to vectors, so narrow rows still keep every thread busy; U vectors in
// flight per thread.  Offsets inside the tile are 32-bit: the caller keeps
// rows * max(dst_row, src_row) below 4 GiB.
template <int G, int U, int LK, int SK>
__device__ __forceinline__ void group_copy_tile(uint8_t* dst, uint32_t dst_row,
                                                const uint8_t* src, uint32_t src_row,
                                                uint32_t rows, uint32_t vrow, int gtid) {
  const uint32_t nv = rows * vrow;
  if (nv == 0) return;
  // (row, vector) of this thread's next vector, and the step of G vectors,
  // kept by adds: two divisions per call instead of one per vector, so the
  // loads of a round do not wait on a division chain
  const TileStep step = tile_step(G, vrow);
  uint32_t i = (uint32_t)gtid / vrow, c = (uint32_t)gtid - i * vrow;
  for (uint32_t v0 = gtid; v0 < nv; v0 += G * U) {
    uint4 x[U];
    uint32_t off_d[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      off_d[u] = i * dst_row + 16 * c;
      if (v0 + u * G < nv) x[u] = ld16<LK>(src + (i * src_row + 16 * c));
      step.advance(i, c, vrow);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + u * G < nv) st16k<SK>(dst + off_d[u], x[u]);
  }
}

// Bytes m..m+15 (1 <= m <= 15) of the 32-byte little-endian concatenation a|b.
__device__ __forceinline__ uint4 funnel16(uint4 a, uint4 b, unsigned m) {
  uint64_t w0 = (uint64_t)a.x | ((uint64_t)a.y << 32);
  uint64_t w1 = (uint64_t)a.z | ((uint64_t)a.w << 32);
  uint64_t w2 = (uint64_t)b.x | ((uint64_t)b.y << 32);
  if (m >= 8) {
    w0 = w1;
    w1 = w2;
    w2 = (uint64_t)b.z | ((uint64_t)b.w << 32);
    m -= 8;
  }
  uint64_t lo = w0, hi = w1;
  if (m) {
    const unsigned sh = m * 8;
    lo = (w0 >> sh) | (w1 << (64 - sh));
    hi = (w1 >> sh) | (w2 << (64 - sh));
  }
  return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
}

// One tile of rows x len bytes at any alignment, copied by a group of G
// threads (gtid = 0 .. G-1, whole warps) with the tile flattened to 16-byte
// output vectors, U in flight per thread.  dst_row must be a multiple of 16,
// so every row has the same head (bytes before dst's next 16-byte boundary),
// the same nvec aligned body vectors and the same tail; the source phase may
// differ from row to row.  A body vector is the funnel shift of the two
// 16-byte-aligned source blocks under it: the first is loaded, the second
// comes from the next lane by shuffle when that lane holds the next vector
// of the same row, and is loaded otherwise (lane 31 and row ends), in the
// same round as the first.  A block read past a row's last byte stays inside
// that byte's 16-byte granule.  Head and tail bytes are copied one per
// thread.  Offsets inside the tile are 32-bit: rows * max(dst_row, src_row)
// stays below 4 GiB.
template <int G, int U, int LK, int SK>
__device__ __forceinline__ void group_copy_tile_any(uint8_t* dst, uint32_t dst_row,
                                                    const uint8_t* src, uint32_t src_row,
                                                    uint32_t rows, uint32_t len, int gtid) {
  uint32_t head = (uint32_t)((16 - ((uintptr_t)dst & 15)) & 15);
  if (head > len) head = len;
  const uint32_t nvec = (len - head) >> 4;
  const uint32_t tail = len - head - (nvec << 4);
  const uint32_t nv = rows * nvec;
  const int lane = gtid & 31;
  // (row, vector) of this thread's next vector, advanced by adds (see group_copy_tile)
  const TileStep step = nvec ? tile_step(G, nvec) : TileStep{0, 0};
  uint32_t i = nvec ? (uint32_t)gtid / nvec : 0, c = nvec ? (uint32_t)gtid - i * nvec : 0;
  for (uint32_t v0 = 0; v0 < nv; v0 += G * U) {  // uniform across the group
    uint4 a[U], b[U];
    uint32_t off_d[U], m[U];
    bool from_next[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t v = v0 + u * G + gtid;
      const bool valid = v < nv;
      const uint8_t* s = src + (i * src_row + head) + 16 * c;  // first source byte (if valid)
      m[u] = (uint32_t)((uintptr_t)s & 15);
      const uint8_t* blk = s - m[u];
      off_d[u] = i * dst_row + head + 16 * c;
      // the next lane holds (i, c + 1) when c + 1 < nvec; lane 31 never does
      from_next[u] = lane < 31 && c + 1 < nvec;
      a[u] = valid ? ld16<LK>(blk) : make_uint4(0, 0, 0, 0);
      b[u] = (valid && m[u] && !from_next[u]) ? ld16<LK>(blk + 16) : make_uint4(0, 0, 0, 0);
      step.advance(i, c, nvec);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t v = v0 + u * G + gtid;
      uint4 n;
      n.x = __shfl_down_sync(0xffffffffu, a[u].x, 1);
      n.y = __shfl_down_sync(0xffffffffu, a[u].y, 1);
      n.z = __shfl_down_sync(0xffffffffu, a[u].z, 1);
      n.w = __shfl_down_sync(0xffffffffu, a[u].w, 1);
      if (from_next[u]) b[u] = n;
      if (v < nv) st16k<SK>(dst + off_d[u], m[u] ? funnel16(a[u], b[u], m[u]) : a[u]);
    }
  }
  // head and tail bytes (at most 15 + 15): row e >> 5, byte e & 31 of the
  // row's head | tail
  const uint32_t edge = head + tail;
  if (edge)
    for (uint32_t e = gtid; e < rows * 32; e += G) {
      const uint32_t i = e >> 5, k = e & 31;
      if (k >= edge) continue;
      const uint32_t x = k < head ? k : head + (nvec << 4) + (k - head);
      st1(dst + i * dst_row + x, ld1<LK>(src + i * src_row + x));
    }
}

// Head and tail bytes of a tile whose rows all have the same head (bytes
// before dst's next 16-byte boundary), nvec body vectors and tail; source
// byte x of row i at src_of(i) + x, read with load kind LK (kRO or kCG), or
// plainly when LK < 0 (shared memory).  One byte per thread-step.
template <int G, int LK, typename SrcOf>
__device__ __forceinline__ void group_copy_edges(uint8_t* dst, uint32_t dst_row, SrcOf src_of,
                                                 uint32_t rows, uint32_t head, uint32_t nvec,
                                                 uint32_t tail, int gtid) {
  const uint32_t edge = head + tail;  // at most 15 + 15
  if (!edge) return;
  for (uint32_t e = gtid; e < rows * 32; e += G) {
    const uint32_t i = e >> 5, k = e & 31;
    if (k >= edge) continue;
    const uint32_t x = k < head ? k : head + (nvec << 4) + (k - head);
    const uint8_t* s = src_of(i) + x;
    if constexpr (LK < 0)
      st1(dst + i * dst_row + x, *s);
    else
      st1(dst + i * dst_row + x, ld1<LK>(s));
  }
}

// A tile of rows x len bytes whose source and destination rows share one
// 16-byte phase ((dst - src) % 16 == 0, both row strides multiples of 16),
// at any alignment: byte heads and tails, and a body of aligned 16-byte
// vectors copied with the whole tile flattened over the group
// (group_copy_tile).
template <int G, int U, int LK, int SK>
__device__ __forceinline__ void group_copy_tile_phase(uint8_t* dst, uint32_t dst_row,
                                                      const uint8_t* src, uint32_t src_row,
                                                      uint32_t rows, uint32_t len, int gtid) {
  uint32_t head = (uint32_t)((16 - ((uintptr_t)dst & 15)) & 15);
  if (head > len) head = len;
  const uint32_t nvec = (len - head) >> 4;
  const uint32_t tail = len - head - (nvec << 4);
  group_copy_tile<G, U, LK, SK>(dst + head, dst_row, src + head, src_row, rows, nvec, gtid);
  group_copy_edges<G, LK>(
      dst, dst_row, [&](uint32_t i) { return src + i * src_row; }, rows, head, nvec, tail, gtid);
}

// Rows of len bytes from a shared-memory ring to global memory, any
// alignment.  Ring row i (pitch bytes apart, 16-byte aligned) holds the
// 16-byte-aligned block range covering source row i, whose first byte sits
// at ring offset m_i = (m0 + i * msrc) % 16 (the source rows' addresses mod
// 16 step by msrc).  Destination rows are dst_row bytes apart, dst_row a
// multiple of 16, so they share one head, nvec body vectors and one tail.  A
// body vector is the funnel shift of the two aligned ring blocks under it;
// stores carry the L2 policy `pol`.  A warp copies a row, its lanes taking
// the row's vectors in turn, U at a time.
template <int G, int U>
__device__ __forceinline__ void group_copy_ring_any(uint8_t* dst, uint32_t dst_row,
                                                    const uint8_t* ring, uint32_t pitch,
                                                    uint32_t m0, uint32_t msrc, uint32_t rows,
                                                    uint32_t len, int gtid, uint64_t pol) {
  uint32_t head = (uint32_t)((16 - ((uintptr_t)dst & 15)) & 15);
  if (head > len) head = len;
  const uint32_t nvec = (len - head) >> 4;
  const uint32_t tail = len - head - (nvec << 4);
  // a warp per row, its lanes along the row, U vectors in flight per lane
  for (uint32_t i = (uint32_t)gtid >> 5; i < rows; i += G / 32) {
    const uint32_t q0 = ((m0 + i * msrc) & 15) + head;  // ring byte of the row's first vector
    const uint8_t* rrow = ring + i * pitch;
    uint8_t* drow = dst + i * dst_row + head;
    for (uint32_t c0 = gtid & 31; c0 < nvec; c0 += 32 * U) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t q = q0 + 16 * (c0 + 32 * u);
        const uint8_t* p = rrow + (q & ~15u);
        if (c0 + 32 * u < nvec) {
          x[u] = *reinterpret_cast<const uint4*>(p);
          if (q & 15) x[u] = funnel16(x[u], *reinterpret_cast<const uint4*>(p + 16), q & 15);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c0 + 32 * u < nvec) st16_hint(drow + 16 * (c0 + 32 * u), x[u], pol);
    }
  }
  group_copy_edges<G, -1>(
      dst, dst_row, [&](uint32_t i) { return ring + i * pitch + ((m0 + i * msrc) & 15); }, rows,
      head, nvec, tail, gtid);
}

// Drops the 128-byte L2 line at p (128-byte aligned) without writing it
// back: its contents become undefined.
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// ------------------------------------------------------- warp byte copy ---
// One warp copies n bytes src -> dst (any alignments, non-overlapping).
//  * head: bytes up to dst's next 16-byte boundary, one byte per lane;
//  * body: 16-byte aligned stores; loads are 16-byte aligned too -- when src
//    and dst disagree mod 16, each lane loads the aligned block under its
//    output, takes the next block from its right neighbour by shuffle, and
//    funnel-shifts the pair (a block read past the end of src stays inside
//    src's 16-byte-aligned, 16-byte-padded allocation);
//  * tail: the last < 16 bytes, one byte per lane.
// U = 16-byte vectors in flight per lane on the aligned path, V on the
// shift-merge path (default U/2: each output needs two source blocks).
template <int U, int LK, int SK, int V = (U > 1 ? U / 2 : 1)>
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, size_t n, int lane) {
  if (n == 0) return;
  size_t head = (16 - ((uintptr_t)dst & 15)) & 15;
  if (head > n) head = n;
  if ((size_t)lane < head) st1(dst + lane, ld1<LK>(src + lane));
  const size_t nvec = (n - head) >> 4;
  uint8_t* d = dst + head;
  const uint8_t* s = src + head;
  const unsigned m = (unsigned)((uintptr_t)s & 15);
  if (m == 0) {
    size_t j = lane;
    for (; j + 32 * (U - 1) < nvec; j += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = ld16<LK>(s + 16 * (j + 32 * u));
#pragma unroll
      for (int u = 0; u < U; ++u) st16k<SK>(d + 16 * (j + 32 * u), v[u]);
    }
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (j + 32 * u < nvec) v[u] = ld16<LK>(s + 16 * (j + 32 * u));
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (j + 32 * u < nvec) st16k<SK>(d + 16 * (j + 32 * u), v[u]);
  } else if (nvec) {
    // aligned source blocks a[0..nvec] (nvec+1 of them) cover the body
    const uint8_t* a0 = s - m;
    for (size_t base = 0; base < nvec; base += 32 * V) {  // warp-uniform loop
      uint4 a[V];
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const size_t j = base + 32 * u + lane;
        a[u] = j <= nvec ? ld16<LK>(a0 + 16 * j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const size_t j = base + 32 * u + lane;
        uint4 b;
        b.x = __shfl_down_sync(0xffffffffu, a[u].x, 1);
        b.y = __shfl_down_sync(0xffffffffu, a[u].y, 1);
        b.z = __shfl_down_sync(0xffffffffu, a[u].z, 1);
        b.w = __shfl_down_sync(0xffffffffu, a[u].w, 1);
        if (lane == 31 && j + 1 <= nvec) b = ld16<LK>(a0 + 16 * (j + 1));
        if (j < nvec) st16k<SK>(d + 16 * j, funnel16(a[u], b, m));
      }
    }
  }
  const size_t done = head + (nvec << 4);
  if ((size_t)lane < n - done) st1(dst + done + lane, ld1<LK>(src + done + lane));
}

// ------------------------------------------------ bulk (TMA) copies -------
// Bulk copies run in the async proxy: a global->shared copy completes on an
// mbarrier (complete_tx), a shared->global copy in a bulk group.  Both need
// 16-byte-aligned addresses and a size that is a multiple of 16.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// Makes mbarrier initialisation visible to the async proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with `parity` of an mbarrier, at most budget_ns (or
// an iteration cap if the timer stood still).  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = globaltimer_ns();
  const uint64_t max_iters = budget_ns / 64 + (1u << 20);
  for (uint64_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > budget_ns || it > max_iters) return false;
  }
}
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gsrc, uint32_t bytes,
                                               uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// All but the newest N bulk groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// All but the newest N bulk groups have completed their global writes.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Orders generic-proxy accesses to this CTA's shared memory before later
// async-proxy (bulk copy) accesses to it, and vice versa.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Orders generic-proxy and async-proxy accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace symm
