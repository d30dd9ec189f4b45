// symm_internal.h -- host-side state and helpers shared by the library's
// translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/symm_a2a.h"

struct symm_heap {
  uint8_t* base;         // device; caller-owned
  size_t slab;           // bytes per PE
  int npes;              // W
  size_t next;           // bump offset inside every slab
  uint64_t spin_budget;  // ns
  int device;            // CUDA device that was current at init
  bool ctrl_ready;       // header zeroed on the device
};

namespace symm_host {

// Records `msg` as this thread's last error and returns `code`.
int fail(int code, const std::string& msg);
// Maps a CUDA error to SYMM_ECUDA (with its name and `what`), or SYMM_OK.
int cuda_check(cudaError_t e, const char* what);

// Offset of `p` inside its slab when p lies in the heap, else -1.
int64_t slab_offset(const symm_heap* h, const void* p);
// Validates that [p, p + bytes) names a range of one slab past the header
// and returns its slab offset in *off.
int check_range(const symm_heap* h, const void* p, size_t bytes, const char* what, size_t* off);

// Zeroes the header of slab 0 on `stream` the first time it is needed.
int ensure_ctrl(symm_heap* h, cudaStream_t stream);

// SMs of the current device, cached per device.
int sm_count();

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// The direct run permutation (combine when !inverse, its inverse otherwise)
// between two device-accessible buffers with PE strides in_pe and out_pe.
// device_mem: both buffers are device memory, so bulk (TMA) copies may read
// them (page-locked host memory is read with plain loads only); ctl (a heap
// header, zeroed) and budget_ns: where a kernel with bounded waits records a
// give-up -- without them only kernels that never wait are used.
int launch_runs_raw(const uint8_t* in, uint8_t* out, size_t in_pe, size_t out_pe, uint32_t W,
                    uint32_t Sb, size_t R, bool inverse, cudaStream_t s, const char* what,
                    bool device_mem = true, void* ctl = nullptr, uint64_t budget_ns = 0);

// One producer/consumer combine (all2all_combine's SYMM_A2A_PC and the
// allocation-free entry point share it): PE k's input and output at
// in/out + k*slab, its staging ring at staging + k*stage_pe and its signal
// slots at signals + k*sig_pe.  Shapes as for all2all_combine; the caller
// has validated them and the ranges.
struct PcPlan {
  const uint8_t* in;
  uint8_t* out;
  size_t slab;
  uint8_t* staging;
  size_t stage_pe;
  uint8_t* signals;
  size_t sig_pe;
  int W, S, H, D, es, tile_s, block_d, buffer_num;
  bool reset;        // zero the signal slots first (inside the launch, each CTA its own)
  bool vector_only;  // 16-byte vector copies only (SYMM_A2A_FLAG_VECTOR)
  uint64_t budget_ns;
  void* ctl;                // the heap header (device) that records errors
  const uint8_t* err_base;  // a slot that times out is reported as its byte
  int64_t err_bias;         // offset from err_base plus err_bias
};
int launch_pc(const PcPlan& p, cudaStream_t s, const char* what);

// Device address, on the current device, of the static array of
// all2all_combine_pc_noalloc (looked up once per device and cached).
int noalloc_scratch_address(uint8_t** out);

}  // namespace symm_host
