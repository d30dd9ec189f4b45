// release_latency.cu -- latency of one gpu-scope release store
// (st.release.gpu) by one thread, alone and while the other warps of its
// CTAs stream copies through HBM, and what those releases cost the streams.
// Three CTAs of 256 threads per SM; warp 0 of each CTA times `kReleases`
// releases with clock64 (after writing `own` KB itself, or not) and then
// stops the streaming warps of its CTA through a shared flag; every loop is
// bounded.  Measurement tool for the producer/consumer combine's handshake
// cost.
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include <cuda_runtime.h>

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      std::printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      std::exit(1);                                                            \
    }                                                                          \
  } while (0)

constexpr int kReleases = 2000;
constexpr long kMaxStreamIters = 20000000;  // bound on a streaming warp's loop

// mode 0: warp 0 alone, releases only; 1: warp 0 writes `own_kb` KB before
// each release; 2: warps 1-7 stream, warp 0 releases only; 3: warps 1-7
// stream, warp 0 writes own_kb KB before each release; 4: warps 1-7 stream,
// warp 0 makes cta-scope releases; 5: warps 1-7 stream, warp 0 idles for
// `idle_cycles` (no releases)
__global__ void __launch_bounds__(256) release_kernel(uint8_t* src, uint8_t* dst, size_t per_warp,
                                                      int64_t* flags, int mode, int own_kb,
                                                      long long idle_cycles,
                                                      unsigned long long* cycles,
                                                      unsigned long long* streamed) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t gw = blockIdx.x * 8ull + warp;
  uint8_t* s = src + gw * per_warp;
  uint8_t* d = dst + gw * per_warp;
  int64_t* flag = flags + blockIdx.x * 16;  // one 128-byte line per CTA
  __shared__ volatile int stop;
  if (threadIdx.x == 0) stop = 0;
  __syncthreads();
  if (warp == 0) {
    unsigned long long acc = 0;
    if (mode == 5) {
      const long long t0 = clock64();
      while (clock64() - t0 < idle_cycles) __nanosleep(1000);
    } else {
      for (int it = 0; it < kReleases; ++it) {
        if (mode == 1 || mode == 3) {
          const size_t nvec = (size_t)own_kb * 1024 / 16;
          for (size_t j = lane; j < nvec; j += 32)
            asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(d + 16 * j), "r"(it),
                         "r"((uint32_t)j), "r"(1), "r"(2)
                         : "memory");
          __syncwarp();
        }
        if (lane == 0) {
          const long long t0 = clock64();
          if (mode == 4)
            asm volatile("st.release.cta.global.b64 [%0], %1;" ::"l"(flag), "l"((int64_t)it)
                         : "memory");
          else
            asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(flag), "l"((int64_t)it)
                         : "memory");
          acc += (unsigned long long)(clock64() - t0);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      cycles[blockIdx.x] = acc;
      stop = 1;
    }
  } else if (mode >= 2) {
    const size_t nvec = per_warp / 16;
    size_t j = lane;
    unsigned long long n = 0;
    for (long k = 0; k < kMaxStreamIters && !stop; ++k, ++n) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                     : "l"(s + 16 * ((j + 32 * u) % nvec)));
#pragma unroll
      for (int u = 0; u < 4; ++u)
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(d + 16 * ((j + 32 * u) % nvec)),
                     "r"(v[u].x), "r"(v[u].y), "r"(v[u].z), "r"(v[u].w)
                     : "memory");
      j = (j + 128) % nvec;
    }
    if (lane == 0) atomicAdd(streamed, n * 128ull * 16 * 2);  // bytes read + written
  }
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  const int ctas = 3 * nsm;
  const size_t per_warp = 1 << 20;  // 1 MB per warp: 3.6 GB per buffer in all
  uint8_t *a, *b;
  int64_t* flags;
  unsigned long long *cyc, *streamed;
  CK(cudaMalloc(&a, per_warp * ctas * 8));
  CK(cudaMalloc(&b, per_warp * ctas * 8));
  CK(cudaMalloc(&flags, ctas * 16 * sizeof(int64_t)));
  CK(cudaMalloc(&cyc, ctas * sizeof(unsigned long long)));
  CK(cudaMalloc(&streamed, sizeof(unsigned long long)));
  CK(cudaMemset(a, 1, per_warp * ctas * 8));
  unsigned long long* host = (unsigned long long*)std::malloc(ctas * sizeof(unsigned long long));
  struct Case {
    int mode, own_kb;
    const char* what;
  } cases[] = {{0, 0, "gpu release, alone"},
               {1, 8, "gpu release after 8 KB of own stores"},
               {1, 32, "gpu release after 32 KB of own stores"},
               {2, 0, "gpu release, 7 warps per CTA streaming"},
               {3, 32, "gpu release after 32 KB, 7 warps streaming"},
               {4, 0, "cta release, 7 warps streaming"},
               {5, 0, "no releases, 7 warps streaming"}};
  std::printf("# %d CTAs of 256 threads (3 per SM); %d releases per CTA\n", ctas, kReleases);
  for (const Case& c : cases) {
    release_kernel<<<ctas, 256>>>(a, b, per_warp, flags, c.mode, c.own_kb, 100000, cyc,
                                  streamed);  // warm-up
    CK(cudaDeviceSynchronize());
    CK(cudaMemset(streamed, 0, sizeof(unsigned long long)));
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    CK(cudaEventRecord(e0));
    release_kernel<<<ctas, 256>>>(a, b, per_warp, flags, c.mode, c.own_kb, 10000000ll, cyc,
                                  streamed);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaGetLastError());
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    CK(cudaMemcpy(host, cyc, ctas * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
    unsigned long long st = 0;
    CK(cudaMemcpy(&st, streamed, sizeof(st), cudaMemcpyDeviceToHost));
    double sum = 0;
    for (int i = 0; i < ctas; ++i) sum += (double)host[i];
    const double per = c.mode == 5 ? 0.0 : sum / ctas / kReleases;
    std::printf("%-44s %7.0f cycles per release   streams %7.1f GB/s   launch %.2f ms\n", c.what,
                per, st / (ms * 1e-3) / 1e9, ms);
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
  }
  std::free(host);
  return 0;
}
