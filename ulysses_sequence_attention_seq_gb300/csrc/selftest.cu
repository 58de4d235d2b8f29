// selftest.cu -- ulysses_selftest_wait_timeout: exercises the kernels' bounded
// pipeline wait and its status reporting without a fault;
// ulysses_selftest_ex2_rate: measures the SM's base-2 exponential (MUFU)
// throughput, the secondary bound of the softmax.
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for it
// with the same bounded wait the attention kernels use (sm100::mbar_wait_bounded),
// here with a caller-chosen limit.  When the limit passes the wait returns false,
// the CTA sets the forward-timeout bit of the workspace status word (as an
// attention CTA that gave up would) and exits normally: no trap, the context
// stays usable, and the host reads the bit with ulysses_read_status.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace {

__global__ void wait_timeout_kernel(uint32_t *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ulysses::sm100::mbar_init(ulysses::sm100::smem_u32(&bar), 1);
    abort_flag = 0;
    ulysses::sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // parity 0: the first phase, which never completes (no arrivals)
    const bool ok = ulysses::sm100::mbar_wait_bounded(ulysses::sm100::smem_u32(&bar), 0, &abort_flag, nullptr,
                                                      limit_ns);
    if (!ok) atomicOr(status, (uint32_t)ULYSSES_STATUS_FWD_TIMEOUT);
  }
}

// Every thread runs 8 independent chains x <- 2^(-x) (x stays in [1/2, 1]) for
// `iters` steps; thread 0 of each block records the block's elapsed SM cycles.
// All blocks are resident at once (2 per SM), so the largest is the launch's.
__global__ void __launch_bounds__(512) ex2_rate_kernel(unsigned long long *cycles, int iters) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = 0.5f + 0.01f * c + 1e-6f * threadIdx.x;
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = ulysses::sm100::ex2(-x[c]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) acc += x[c];
  if (threadIdx.x == 0) atomicMax(cycles, (unsigned long long)(t1 - t0) + (acc < 0.f ? 1ull : 0ull));
}

}  // namespace

extern "C" int ulysses_selftest_ex2_rate(void *cycles, size_t bytes, long long *ex2_per_launch, int *sms,
                                         ulysses_stream_t stream) {
  if (!cycles || bytes < 8 || !ex2_per_launch || !sms) return ULYSSES_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(cycles) % 8 != 0) return ULYSSES_ERR_ALIGN;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || n <= 0)
    return ULYSSES_ERR_CUDA;
  constexpr int kIters = 4096, kThreads = 512, kPerSm = 2;
  if (cudaMemsetAsync(cycles, 0, 8, (cudaStream_t)stream) != cudaSuccess) return ULYSSES_ERR_CUDA;
  ex2_rate_kernel<<<n * kPerSm, kThreads, 0, (cudaStream_t)stream>>>(static_cast<unsigned long long *>(cycles),
                                                                     kIters);
  *ex2_per_launch = (long long)n * kPerSm * kThreads * kIters * 8;
  *sms = n;
  return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

extern "C" int ulysses_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned long long limit_ns,
                                             ulysses_stream_t stream) {
  if (!ws || ws_bytes < 256 || limit_ns == 0 || limit_ns > 2000000000ull) return ULYSSES_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return ULYSSES_ERR_ALIGN;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<uint32_t *>(ws), limit_ns);
  return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}
