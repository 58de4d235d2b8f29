// selftest.cu -- ulysses_selftest_wait_timeout: exercises the kernels' bounded
// pipeline wait and its status reporting without a fault.
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

}  // namespace

extern "C" int ulysses_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned long long limit_ns,
                                             ulysses_stream_t stream) {
  if (!ws || ws_bytes < 256 || limit_ns == 0 || limit_ns > 2000000000ull) return ULYSSES_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return ULYSSES_ERR_ALIGN;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<uint32_t *>(ws), limit_ns);
  return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}
