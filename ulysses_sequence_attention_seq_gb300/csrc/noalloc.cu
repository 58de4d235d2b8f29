// noalloc.cu -- ulysses_attn_bwd_noalloc: the backward without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code that runs under an allocator they do not control (a host
// framework that owns every cudaMalloc and forbids side allocations), code
// paths that must not synchronise (cudaMalloc/cudaFree can serialise the
// device), or embedders whose memory budget is fixed before the first call.
// For them this entry point takes the backward's scratch (RoPE table, delta,
// dO in head layout, status word) from a fixed array that lives in the
// library's own device memory instead of from a workspace argument.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// cannot use its name as a device address; the address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.  All calls share the one array: two calls whose
// kernels overlap on the GPU (different streams, or different host threads
// without ordering) race on it.  The kernels that run first in every call
// rebuild the RoPE table and clear the status word, so nothing carries over
// from an earlier call except bytes that are always rewritten before use.
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

using ulysses::check_bwd_call;

namespace {

constexpr size_t kNoAllocScratchBytes = 32ull << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns nullptr if the lookup fails.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int ulysses_attn_bwd_noalloc(const ulysses_problem *prob, const void *q_head,
                                        const void *k_head, const void *v_head,
                                        const void *o_head, const float *lse, const void *do_seq,
                                        void *dq_seq, void *dk_seq, void *dv_seq,
                                        ulysses_stream_t stream) {
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  if (prob->dtype != ULYSSES_BF16 || (prob->head_dim != 64 && prob->head_dim != 128))
    return ULYSSES_ERR_UNSUPPORTED;  // the backward's kernels are bf16, head_dim 64 or 128
  const size_t need = ulysses_workspace_bytes(prob, 1);
  if (need == 0 || need > kNoAllocScratchBytes) return ULYSSES_ERR_WORKSPACE;
  void *scratch = scratch_on_current_device();
  if (!scratch) return ULYSSES_ERR_CUDA;
  // Every check the backward makes, with the scratch array in the place of the
  // workspace, before anything is enqueued: a refused call leaves the array
  // (and any earlier call still running on it) untouched.
  rc = check_bwd_call(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, scratch,
                      kNoAllocScratchBytes);
  if (rc) return rc;
  // Rebuild the RoPE table and clear the status word for this problem, then
  // run the ordinary backward on the fixed scratch.
  rc = ulysses_workspace_init(prob, scratch, kNoAllocScratchBytes, stream);
  if (rc) return rc;
  return ulysses_attn_bwd(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq,
                          scratch, kNoAllocScratchBytes, stream);
}

extern "C" int ulysses_noalloc_read_status(uint32_t *status, ulysses_stream_t stream) {
  if (!status) return ULYSSES_ERR_ARG;
  void *scratch = scratch_on_current_device();
  if (!scratch) return ULYSSES_ERR_CUDA;
  return ulysses_read_status(scratch, status, stream);
}
