// ulysses_abi.cu -- the extern "C" entry points of include/ulysses.h.
//
// Host side only: argument validation (the head-count bound of plain Ulysses,
// "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention", §4,
// and the shape contract of "Comparing Ulysses and Megatron Sequence
// Parallelism", "DeepSpeed Attention"), workspace layout, and kernel launches.
// Nothing here computes on the host and nothing allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace ulysses {

// An NVTX range around an entry point's host work (validation and launches),
// named after the entry point: a profiler's timeline shows which call enqueued
// which kernels.  Header-only NVTX: without a tool attached it costs a branch.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WorkspaceLayout workspace_layout(const ulysses_problem &p) {
  WorkspaceLayout L;
  const size_t es = elem_size(p);
  L.status = 0;
  L.rope = 256;
  L.rope_bytes = p.use_rope ? (size_t)p.S * p.head_dim * 4 : 0;
  L.total_fwd = align256(L.rope + L.rope_bytes);
  L.delta = L.total_fwd;
  // rows of P*B*hp = B*n_head*ring, each delta_ld floats
  L.delta_bytes = (size_t)p.B * p.n_head * ring_of(p) * delta_ld(p) * 4;
  L.nlse = align256(L.delta + L.delta_bytes);
  L.nlse_bytes = L.delta_bytes;
  L.dohead = align256(L.nlse + L.nlse_bytes);
  L.dohead_bytes = (size_t)p.B * p.S * p.n_head * p.head_dim * es;
  L.part_bytes = kv_replicas(p) > 1 ? (size_t)p.P * p.B * chunk_len(p) * p.head_dim * 4 : 0;
  L.dkpart = align256(L.dohead + L.dohead_bytes);
  L.dvpart = align256(L.dkpart + L.part_bytes);
  L.total_bwd = align256(L.dvpart + L.part_bytes);
  L.dqacc = L.total_bwd;
  L.dqacc_bytes = (size_t)p.B * p.n_head * ((p.S + 127) / 128 * 128) * p.head_dim * 4;
  L.total_fused = align256(L.dqacc + L.dqacc_bytes);
  const size_t n_kt = (size_t)(p.S + 127) / 128;
  L.ds = L.total_bwd;
  const size_t tiles = p.causal ? n_kt * (n_kt + 1) / 2 : n_kt * n_kt;  // per q-head
  L.ds_bytes = (size_t)p.B * p.n_head * tiles * 128 * 128 * 2;
  L.total_ds = align256(L.ds + L.ds_bytes);
  // a kv-head's q-heads on one rank: n_head / n_kv_head, or with replicated
  // kv-heads (fewer than the ranks of a group) all n_head / Pu of the rank's
  L.ds_kv_bytes = (size_t)(p.n_head / group_ranks(p) / kv_per_rank(p)) * tiles * 128 * 128 * 2;
  L.total_ds_min = align256(L.ds + L.ds_kv_bytes);
  return L;
}

uint32_t rope_key(const ulysses_problem &p) {
  uint32_t bits = 0;
  const float base = p.use_rope ? p.rope_base : 0.f;
  memcpy(&bits, &base, 4);
  uint32_t h = 2166136261u;
  const uint32_t words[4] = {(uint32_t)p.S, (uint32_t)p.head_dim, bits, (uint32_t)p.use_rope};
  for (uint32_t w : words) {
    h ^= w;
    h *= 16777619u;
  }
  return h | 1u;  // never 0, so a zeroed workspace never matches
}

bool get_tma_encoder(TmaEncoder *enc) {
  static const TmaEncoder cached = [] {
    TmaEncoder e;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      e.encode = reinterpret_cast<decltype(e.encode)>(fn);
    else
      cudaGetLastError();
    return e;
  }();
  *enc = cached;
  return cached.encode != nullptr;
}

}  // namespace ulysses

using namespace ulysses;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  const void *p;
  size_t n;
};

bool overlaps(Span a, Span b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a.n && b.n && a0 < b0 + b.n && b0 < a0 + a.n;
}

// Every output must be disjoint from every input and from every other output.
int check_spans(const Span *in, int nin, const Span *out, int nout) {
  for (int i = 0; i < nin; ++i)
    if (!in[i].p) return ULYSSES_ERR_ARG;
  for (int i = 0; i < nout; ++i)
    if (!out[i].p) return ULYSSES_ERR_ARG;
  for (int i = 0; i < nin; ++i)
    if (!aligned16(in[i].p)) return ULYSSES_ERR_ALIGN;
  for (int i = 0; i < nout; ++i)
    if (!aligned16(out[i].p)) return ULYSSES_ERR_ALIGN;
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < nin; ++i)
      if (overlaps(out[o], in[i])) return ULYSSES_ERR_ALIAS;
    for (int o2 = o + 1; o2 < nout; ++o2)
      if (overlaps(out[o], out[o2])) return ULYSSES_ERR_ALIAS;
  }
  return ULYSSES_OK;
}

int check_ws(const ulysses_problem &p, const void *ws, size_t ws_bytes, int phase) {
  if (!ws) return ULYSSES_ERR_WORKSPACE;
  if (!aligned16(ws)) return ULYSSES_ERR_ALIGN;
  const WorkspaceLayout L = workspace_layout(p);
  if (ws_bytes < (phase == 4   ? L.total_ds_min
                  : phase == 3 ? L.total_ds
                  : phase == 2 ? L.total_fused
                  : phase      ? L.total_bwd
                               : L.total_fwd))
    return ULYSSES_ERR_WORKSPACE;
  return ULYSSES_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA; }

size_t act_bytes(const ulysses_problem &p, int heads) {
  return (size_t)p.B * p.S * heads * p.head_dim * elem_size(p);
}

// K or V in head layout [P][B][Cs][kv-heads per rank][D]: with replicated
// kv-heads P copies of one kv-head's rows, else the same size as the tensor.
size_t kv_head_bytes(const ulysses_problem &p) {
  return (size_t)p.P * p.B * chunk_len(p) * kv_per_rank(p) * p.head_dim * elem_size(p);
}


// Shared checks of the backward entry points: a bf16 problem with a tensor-core
// kernel, a phase-1 workspace.
int bwd_common(const ulysses_problem *prob, const void *ws, size_t ws_bytes) {
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.dtype != ULYSSES_BF16 || (p.head_dim != 64 && p.head_dim != 128)) return ULYSSES_ERR_UNSUPPORTED;
  return check_ws(p, ws, ws_bytes, 1);
}

// Step 2 of the backward, with or without the dS store (phase-3 workspace):
// dK, dV (with replicated kv-heads, each rank's float partials and then
// their sum) in sequence layout.
int dkdv_call(const ulysses_problem *prob, const void *q_head, const void *k_head, const void *v_head,
              void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream, bool store_ds) {
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (store_ds && (rc = check_ws(p, ws, ws_bytes, 3))) return rc;
  const size_t nk = act_bytes(p, p.n_kv_head), nkh = kv_head_bytes(p);
  const Span in[3] = {{q_head, act_bytes(p, p.n_head)}, {k_head, nkh}, {v_head, nkh}};
  const Span out[3] = {{dk_seq, nk}, {dv_seq, nk}, {ws, ws_bytes}};
  if ((rc = check_spans(in, 3, out, 3))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
  const float *nlse = reinterpret_cast<const float *>(w + L.nlse), *delta = reinterpret_cast<const float *>(w + L.delta);
  void *ds = store_ds ? static_cast<void *>(w + L.ds) : nullptr;
  if (kv_replicas(p) > 1) {
    // each rank's partial dK, dV (its own q-heads) into the workspace, then the
    // sum over every kv-head's replicas into sequence layout
    float *dkp = reinterpret_cast<float *>(w + L.dkpart), *dvp = reinterpret_cast<float *>(w + L.dvpart);
    cudaError_t e = launch_attn_bwd_dkdv(p, enc, q_head, k_head, v_head, w + L.dohead, nlse, delta, ws, dkp, dvp,
                                         status, st, false, ds);
    if (e == cudaSuccess) {
      const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
      e = launch_kv_reduce(p, dkp, dvp, dk_seq, dv_seq, scale, ws, st);
    }
    return cuda_rc(e);
  }
  return cuda_rc(launch_attn_bwd_dkdv(p, enc, q_head, k_head, v_head, w + L.dohead, nlse, delta, ws, dk_seq, dv_seq,
                                      status, st, false, ds));
}

}  // namespace

extern "C" {

int ulysses_validate(const ulysses_problem *prob) {
  if (!prob) return ULYSSES_ERR_ARG;
  const ulysses_problem &p = *prob;
  if (p.B <= 0 || p.S <= 0 || p.hidden <= 0 || p.n_head <= 0 || p.n_kv_head <= 0 ||
      p.head_dim <= 0 || p.P <= 0)
    return ULYSSES_ERR_ARG;
  if ((p.causal != 0 && p.causal != 1) || (p.use_rope != 0 && p.use_rope != 1))
    return ULYSSES_ERR_ARG;
  if (!(p.softmax_scale >= 0.f) || isinf(p.softmax_scale)) return ULYSSES_ERR_ARG;
  if (p.use_rope && (!(p.rope_base > 0.f) || isinf(p.rope_base))) return ULYSSES_ERR_ARG;
  if (p.ring < 0) return ULYSSES_ERR_ARG;
  const int Pu = p.P / ring_of(p);  // ranks of one ring position
  if (p.P % ring_of(p) || p.S % p.P || p.n_head % Pu || p.n_head % p.n_kv_head ||
      (p.n_kv_head % Pu != 0 && Pu % p.n_kv_head != 0))
    return ULYSSES_ERR_DIVISIBILITY;
  if ((long long)p.n_head * p.head_dim != p.hidden) return ULYSSES_ERR_HIDDEN;
  if (p.dtype != ULYSSES_BF16 && p.dtype != ULYSSES_FP32) return ULYSSES_ERR_UNSUPPORTED;
  if (p.head_dim != 32 && p.head_dim != 64 && p.head_dim != 128) return ULYSSES_ERR_UNSUPPORTED;
  // Index arithmetic inside the kernels keeps per-tensor element counts in
  // 64 bits and per-row quantities in 32 bits.
  if ((long long)p.B * p.P > (1ll << 30) || (long long)p.S * p.n_head > (1ll << 31))
    return ULYSSES_ERR_UNSUPPORTED;
  // The hybrid runs on the tensor-core kernels, whose tiles must not straddle
  // two ring positions' chunks.
  if (ring_of(p) > 1 && (p.dtype != ULYSSES_BF16 || (p.head_dim != 64 && p.head_dim != 128) ||
                         chunk_len(p) % 128 != 0))
    return ULYSSES_ERR_UNSUPPORTED;
  return ULYSSES_OK;
}

size_t ulysses_workspace_bytes(const ulysses_problem *prob, int phase) {
  if (phase < 0 || phase > 4 || ulysses_validate(prob) != ULYSSES_OK) return 0;
  const WorkspaceLayout L = workspace_layout(*prob);
  return phase == 4 ? L.total_ds_min
         : phase == 3 ? L.total_ds
         : phase == 2 ? L.total_fused
         : phase      ? L.total_bwd
                      : L.total_fwd;
}

int ulysses_workspace_init(const ulysses_problem *prob, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream) {
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  if ((rc = check_ws(*prob, ws, ws_bytes, 0))) return rc;
  return cuda_rc(launch_rope_table(*prob, ws, (cudaStream_t)stream));
}

int ulysses_read_status_async(const void *ws, uint32_t *status, ulysses_stream_t stream) {
  if (!ws || !status) return ULYSSES_ERR_ARG;
  return cuda_rc(cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream));
}

int ulysses_read_status(const void *ws, uint32_t *status, ulysses_stream_t stream) {
  if (!ws || !status) return ULYSSES_ERR_ARG;
  cudaError_t e = cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return cuda_rc(e);
}

int ulysses_pack_qkv(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                     const void *v_seq, void *q_head, void *k_head, void *v_head, void *ws,
                     size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_pack_qkv");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  const size_t nq = act_bytes(p, p.n_head), nk = act_bytes(p, p.n_kv_head), nkh = kv_head_bytes(p);
  const Span in[4] = {{q_seq, nq}, {k_seq, nk}, {v_seq, nk}, {ws, ws_bytes}};
  const Span out[3] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}};
  if ((rc = check_ws(p, ws, ws_bytes, 0))) return rc;
  if ((rc = check_spans(in, 4, out, 3))) return rc;
  return cuda_rc(launch_pack_qkv(p, q_seq, k_seq, v_seq, q_head, k_head, v_head, ws,
                                 (cudaStream_t)stream));
}

int ulysses_qkv_proj_pack(const ulysses_problem *prob, const void *x_seq, const void *w_qkv, const void *b_qkv,
                          void *q_head, void *k_head, void *v_head, void *ws, size_t ws_bytes,
                          ulysses_stream_t stream) {
  const NvtxRange range("ulysses_qkv_proj_pack");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.dtype != ULYSSES_BF16 || (p.head_dim != 64 && p.head_dim != 128) || ring_of(p) > 1)
    return ULYSSES_ERR_UNSUPPORTED;
  if (!x_seq || !w_qkv) return ULYSSES_ERR_ARG;
  const size_t n_out = (size_t)(p.n_head + 2 * p.n_kv_head) * p.head_dim;
  const size_t nx = (size_t)p.B * p.S * p.hidden * 2, nw = n_out * p.hidden * 2, nb = n_out * 2;
  const size_t nq = act_bytes(p, p.n_head), nkh = kv_head_bytes(p);
  const Span in[4] = {{x_seq, nx}, {w_qkv, nw}, {b_qkv ? b_qkv : x_seq, b_qkv ? nb : nx}, {ws, ws_bytes}};
  const Span out[3] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}};
  if ((rc = check_ws(p, ws, ws_bytes, 0))) return rc;
  if ((rc = check_spans(in, 4, out, 3))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  return cuda_rc(launch_qkv_proj_pack(p, enc, x_seq, w_qkv, b_qkv, q_head, k_head, v_head, ws,
                                      (cudaStream_t)stream));
}

int ulysses_out_proj_unpack(const ulysses_problem *prob, const void *o_head, const void *w_o, const void *b_o,
                            void *y_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_out_proj_unpack");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.dtype != ULYSSES_BF16 || (p.head_dim != 64 && p.head_dim != 128) || (p.S / p.P) % 128 != 0 ||
      ring_of(p) > 1)
    return ULYSSES_ERR_UNSUPPORTED;
  if (!o_head || !w_o) return ULYSSES_ERR_ARG;
  const size_t no = act_bytes(p, p.n_head), nw = (size_t)p.hidden * p.hidden * 2, nb = (size_t)p.hidden * 2;
  const size_t ny = (size_t)p.B * p.S * p.hidden * 2;
  const Span in[3] = {{o_head, no}, {w_o, nw}, {b_o ? b_o : o_head, b_o ? nb : no}};
  const Span out[2] = {{y_seq, ny}, {ws, ws_bytes}};
  if ((rc = check_ws(p, ws, ws_bytes, 0))) return rc;
  if ((rc = check_spans(in, 3, out, 2))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  return cuda_rc(launch_out_proj_unpack(p, enc, o_head, w_o, b_o, y_seq, ws, (cudaStream_t)stream));
}

int ulysses_attn_fwd(const ulysses_problem *prob, const void *q_head, const void *k_head,
                     const void *v_head, void *o_head, float *lse, void *ws, size_t ws_bytes,
                     ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_fwd");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.dtype == ULYSSES_BF16 && p.head_dim != 64 && p.head_dim != 128) return ULYSSES_ERR_UNSUPPORTED;
  const size_t nq = act_bytes(p, p.n_head), nkh = kv_head_bytes(p);
  const size_t nl = (size_t)p.B * p.n_head * p.S * sizeof(float);
  const Span in[3] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}};
  const Span out[3] = {{o_head, nq}, {lse, nl}, {ws, ws_bytes}};
  if ((rc = check_ws(p, ws, ws_bytes, 0))) return rc;
  if ((rc = check_spans(in, 3, out, 3))) return rc;
  uint32_t *status = static_cast<uint32_t *>(ws);
  if (p.dtype == ULYSSES_FP32)
    return cuda_rc(launch_attn_fwd_simt(p, static_cast<const float *>(q_head),
                                        static_cast<const float *>(k_head),
                                        static_cast<const float *>(v_head),
                                        static_cast<float *>(o_head), lse, status, (cudaStream_t)stream));
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  return cuda_rc(launch_attn_fwd_tc(p, enc, q_head, k_head, v_head, o_head, lse, status, false,
                                    (cudaStream_t)stream));
}

int ulysses_attn_fwd_folded(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                            const void *v_seq, void *o_seq, float *lse, void *ws, size_t ws_bytes,
                            ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_fwd_folded");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.dtype != ULYSSES_BF16 || (p.head_dim != 64 && p.head_dim != 128) || p.use_rope ||
      (p.S / p.P) % 128 != 0 || ring_of(p) > 1)
    return ULYSSES_ERR_UNSUPPORTED;
  const size_t nq = act_bytes(p, p.n_head), nk = act_bytes(p, p.n_kv_head);
  const size_t nl = (size_t)p.B * p.n_head * p.S * sizeof(float);
  const Span in[3] = {{q_seq, nq}, {k_seq, nk}, {v_seq, nk}};
  const Span out[3] = {{o_seq, nq}, {lse, nl}, {ws, ws_bytes}};
  if ((rc = check_ws(p, ws, ws_bytes, 0))) return rc;
  if ((rc = check_spans(in, 3, out, 3))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  return cuda_rc(launch_attn_fwd_tc(p, enc, q_seq, k_seq, v_seq, o_seq, lse, static_cast<uint32_t *>(ws),
                                    true, (cudaStream_t)stream));
}

int ulysses_unpack_out(const ulysses_problem *prob, const void *o_head, void *o_seq,
                       ulysses_stream_t stream) {
  const NvtxRange range("ulysses_unpack_out");
  int rc = ulysses_validate(prob);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  const size_t n = act_bytes(p, p.n_head);
  const Span in[1] = {{o_head, n}};
  const Span out[1] = {{o_seq, n}};
  if ((rc = check_spans(in, 1, out, 1))) return rc;
  return cuda_rc(launch_unpack(p, o_head, o_seq, (cudaStream_t)stream));
}

int ulysses_attn_bwd_prepare(const ulysses_problem *prob, const void *o_head, const float *lse,
                             const void *do_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_prepare");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  const size_t nq = act_bytes(p, p.n_head);
  const size_t nl = (size_t)p.B * p.n_head * p.S * sizeof(float);
  const Span in[3] = {{o_head, nq}, {lse, nl}, {do_seq, nq}};
  const Span out[1] = {{ws, ws_bytes}};
  if ((rc = check_spans(in, 3, out, 1))) return rc;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  return cuda_rc(launch_pack_do_delta(p, do_seq, o_head, lse, w + L.dohead, reinterpret_cast<float *>(w + L.delta),
                                      reinterpret_cast<float *>(w + L.nlse), reinterpret_cast<uint32_t *>(w + L.status),
                                      (cudaStream_t)stream));
}

int ulysses_attn_bwd_dkdv(const ulysses_problem *prob, const void *q_head, const void *k_head,
                          const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                          ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dkdv");
  return dkdv_call(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, ws_bytes, stream, false);
}

int ulysses_attn_bwd_dq(const ulysses_problem *prob, const void *q_head, const void *k_head,
                        const void *v_head, void *dq_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dq");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  const size_t nq = act_bytes(p, p.n_head), nkh = kv_head_bytes(p);
  const Span in[3] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}};
  const Span out[2] = {{dq_seq, nq}, {ws, ws_bytes}};
  if ((rc = check_spans(in, 3, out, 2))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  return cuda_rc(launch_attn_bwd_dq(p, enc, q_head, k_head, v_head, w + L.dohead,
                                    reinterpret_cast<const float *>(w + L.nlse),
                                    reinterpret_cast<const float *>(w + L.delta), ws, dq_seq,
                                    reinterpret_cast<uint32_t *>(w + L.status), (cudaStream_t)stream));
}

}  // extern "C"

int ulysses::check_bwd_call(const ulysses_problem *prob, const void *q_head, const void *k_head,
                            const void *v_head, const void *o_head, const float *lse, const void *do_seq,
                            const void *dq_seq, const void *dk_seq, const void *dv_seq, const void *ws,
                            size_t ws_bytes) {
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  const size_t nq = act_bytes(p, p.n_head), nk = act_bytes(p, p.n_kv_head), nkh = kv_head_bytes(p);
  const size_t nl = (size_t)p.B * p.n_head * p.S * sizeof(float);
  const Span in[6] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}, {o_head, nq}, {lse, nl}, {do_seq, nq}};
  const Span out[4] = {{dq_seq, nq}, {dk_seq, nk}, {dv_seq, nk}, {ws, ws_bytes}};
  return check_spans(in, 6, out, 4);
}

extern "C" {

int ulysses_attn_bwd_dkdvq(const ulysses_problem *prob, const void *q_head, const void *k_head,
                           const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dkdvq");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if ((rc = check_ws(p, ws, ws_bytes, 2))) return rc;
  const size_t nq = act_bytes(p, p.n_head), nk = act_bytes(p, p.n_kv_head), nkh = kv_head_bytes(p);
  const Span in[3] = {{q_head, nq}, {k_head, nkh}, {v_head, nkh}};
  const Span out[3] = {{dk_seq, nk}, {dv_seq, nk}, {ws, ws_bytes}};
  if ((rc = check_spans(in, 3, out, 3))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  float *acc = reinterpret_cast<float *>(w + L.dqacc);
  uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
  const float *nlse = reinterpret_cast<const float *>(w + L.nlse), *delta = reinterpret_cast<const float *>(w + L.delta);
  // the dQ shares are added into a zeroed accumulator
  if (launch_zero(acc, L.dqacc_bytes / 4, st) != cudaSuccess) return ULYSSES_ERR_CUDA;
  if (kv_replicas(p) > 1) {
    float *dkp = reinterpret_cast<float *>(w + L.dkpart), *dvp = reinterpret_cast<float *>(w + L.dvpart);
    cudaError_t e = launch_attn_bwd_fused(p, enc, q_head, k_head, v_head, w + L.dohead, nlse, delta, ws, acc, dkp,
                                          dvp, status, st);
    if (e == cudaSuccess) {
      const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
      e = launch_kv_reduce(p, dkp, dvp, dk_seq, dv_seq, scale, ws, st);
    }
    return cuda_rc(e);
  }
  return cuda_rc(launch_attn_bwd_fused(p, enc, q_head, k_head, v_head, w + L.dohead, nlse, delta, ws, acc, dk_seq,
                                       dv_seq, status, st));
}

int ulysses_attn_bwd_dq_finish(const ulysses_problem *prob, void *dq_seq, void *ws, size_t ws_bytes,
                               ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dq_finish");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if ((rc = check_ws(p, ws, ws_bytes, 2))) return rc;
  const Span out[2] = {{dq_seq, act_bytes(p, p.n_head)}, {ws, ws_bytes}};
  if ((rc = check_spans(nullptr, 0, out, 2))) return rc;
  TmaEncoder enc;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  return cuda_rc(launch_dq_finish(p, enc, ws, reinterpret_cast<float *>(w + L.dqacc), dq_seq,
                                  reinterpret_cast<uint32_t *>(w + L.status), (cudaStream_t)stream));
}

int ulysses_attn_bwd_fused(const ulysses_problem *prob, const void *q_head, const void *k_head,
                           const void *v_head, const void *o_head, const float *lse, const void *do_seq,
                           void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_fused");
  int rc = check_bwd_call(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                          ws_bytes);
  if (rc) return rc;
  if ((rc = check_ws(*prob, ws, ws_bytes, 2))) return rc;
  if ((rc = ulysses_attn_bwd_prepare(prob, o_head, lse, do_seq, ws, ws_bytes, stream))) return rc;
  if ((rc = ulysses_attn_bwd_dkdvq(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, ws_bytes, stream))) return rc;
  return ulysses_attn_bwd_dq_finish(prob, dq_seq, ws, ws_bytes, stream);
}

int ulysses_attn_bwd_dkdv_ds(const ulysses_problem *prob, const void *q_head, const void *k_head,
                             const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                             ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dkdv_ds");
  return dkdv_call(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, ws_bytes, stream, true);
}

int ulysses_attn_bwd_dq_ds(const ulysses_problem *prob, const void *k_head, void *dq_seq, void *ws,
                           size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_dq_ds");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if ((rc = check_ws(p, ws, ws_bytes, 3))) return rc;
  const Span in[1] = {{k_head, kv_head_bytes(p)}};
  const Span out[2] = {{dq_seq, act_bytes(p, p.n_head)}, {ws, ws_bytes}};
  if ((rc = check_spans(in, 1, out, 2))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  return cuda_rc(launch_dq_from_ds(p, enc, k_head, ws, w + L.ds, dq_seq, reinterpret_cast<uint32_t *>(w + L.status),
                                   (cudaStream_t)stream));
}

int ulysses_attn_bwd_ds(const ulysses_problem *prob, const void *q_head, const void *k_head,
                        const void *v_head, const void *o_head, const float *lse, const void *do_seq,
                        void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                        ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_ds");
  int rc = check_bwd_call(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                          ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if ((rc = check_ws(p, ws, ws_bytes, 4))) return rc;
  if ((rc = ulysses_attn_bwd_prepare(prob, o_head, lse, do_seq, ws, ws_bytes, stream))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
  const float *nlse = reinterpret_cast<const float *>(w + L.nlse), *delta = reinterpret_cast<const float *>(w + L.delta);
  const bool rep = kv_replicas(p) > 1;
  void *dkk = rep ? static_cast<void *>(w + L.dkpart) : dk_seq, *dvv = rep ? static_cast<void *>(w + L.dvpart) : dv_seq;
  // As many kv-heads' tiles as the workspace holds at a time (all of them with
  // a phase-3 workspace): dK/dV storing that chunk's dS, then its dQ.
  const int all_kv = group_ranks(p) * p.B * kv_per_rank(p);
  const size_t fit = (ws_bytes - L.ds) / L.ds_kv_bytes;
  const int chunk = fit >= (size_t)all_kv ? all_kv : (int)fit;
  cudaError_t e = cudaSuccess;
  for (int h0 = 0; h0 < all_kv && e == cudaSuccess; h0 += chunk) {
    const int hn = all_kv - h0 < chunk ? all_kv - h0 : chunk;
    e = launch_attn_bwd_dkdv(p, enc, q_head, k_head, v_head, w + L.dohead, nlse, delta, ws, dkk, dvv, status, st,
                             false, w + L.ds, h0, hn);
    if (e == cudaSuccess) e = launch_dq_from_ds(p, enc, k_head, ws, w + L.ds, dq_seq, status, st, h0, hn);
  }
  if (e == cudaSuccess && rep) {
    // the sum over every kv-head's replicas of the ranks' partials
    const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
    e = launch_kv_reduce(p, reinterpret_cast<float *>(dkk), reinterpret_cast<float *>(dvv), dk_seq, dv_seq, scale, ws,
                         st);
  }
  return cuda_rc(e);
}

int ulysses_attn_bwd(const ulysses_problem *prob, const void *q_head, const void *k_head,
                     const void *v_head, const void *o_head, const float *lse,
                     const void *do_seq, void *dq_seq, void *dk_seq, void *dv_seq, void *ws,
                     size_t ws_bytes, ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd");
  int rc = check_bwd_call(prob, q_head, k_head, v_head, o_head, lse, do_seq, dq_seq, dk_seq, dv_seq, ws,
                          ws_bytes);
  if (rc) return rc;
  if ((rc = ulysses_attn_bwd_prepare(prob, o_head, lse, do_seq, ws, ws_bytes, stream))) return rc;
  if ((rc = ulysses_attn_bwd_dkdv(prob, q_head, k_head, v_head, dk_seq, dv_seq, ws, ws_bytes, stream))) return rc;
  return ulysses_attn_bwd_dq(prob, q_head, k_head, v_head, dq_seq, ws, ws_bytes, stream);
}

int ulysses_attn_bwd_folded(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                            const void *v_seq, const void *o_seq, const float *lse, const void *do_seq,
                            void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                            ulysses_stream_t stream) {
  const NvtxRange range("ulysses_attn_bwd_folded");
  int rc = bwd_common(prob, ws, ws_bytes);
  if (rc) return rc;
  const ulysses_problem &p = *prob;
  if (p.use_rope || (p.S / p.P) % 128 != 0 || ring_of(p) > 1) return ULYSSES_ERR_UNSUPPORTED;
  const size_t nq = act_bytes(p, p.n_head), nk = act_bytes(p, p.n_kv_head);
  const size_t nl = (size_t)p.B * p.n_head * p.S * sizeof(float);
  const Span in[6] = {{q_seq, nq}, {k_seq, nk}, {v_seq, nk}, {o_seq, nq}, {lse, nl}, {do_seq, nq}};
  const Span out[4] = {{dq_seq, nq}, {dk_seq, nk}, {dv_seq, nk}, {ws, ws_bytes}};
  if ((rc = check_spans(in, 6, out, 4))) return rc;
  TmaEncoder enc;
  if (!get_tma_encoder(&enc)) return ULYSSES_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(p);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
  const float *nlse = reinterpret_cast<const float *>(w + L.nlse);
  const float *delta = reinterpret_cast<const float *>(w + L.delta);
  // delta and the base-2 LSE from O and dO in sequence layout (no dO pack)
  cudaError_t e = launch_pack_do_delta(p, do_seq, o_seq, lse, nullptr, reinterpret_cast<float *>(w + L.delta),
                                       reinterpret_cast<float *>(w + L.nlse), status, st, true);
  if (e != cudaSuccess) return cuda_rc(e);
  if (kv_replicas(p) > 1) {
    float *dkp = reinterpret_cast<float *>(w + L.dkpart), *dvp = reinterpret_cast<float *>(w + L.dvpart);
    e = launch_attn_bwd_dkdv(p, enc, q_seq, k_seq, v_seq, do_seq, nlse, delta, ws, dkp, dvp, status, st, true);
    if (e == cudaSuccess) {
      const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
      e = launch_kv_reduce(p, dkp, dvp, dk_seq, dv_seq, scale, ws, st);
    }
  } else {
    e = launch_attn_bwd_dkdv(p, enc, q_seq, k_seq, v_seq, do_seq, nlse, delta, ws, dk_seq, dv_seq, status, st,
                             true);
  }
  if (e != cudaSuccess) return cuda_rc(e);
  return cuda_rc(launch_attn_bwd_dq(p, enc, q_seq, k_seq, v_seq, do_seq, nlse, delta, ws, dq_seq, status, st, true));
}

const char *ulysses_status_string(int code) {
  switch (code) {
    case ULYSSES_OK: return "ok";
    case ULYSSES_ERR_ARG: return "invalid argument (NULL pointer or non-positive size)";
    case ULYSSES_ERR_DIVISIBILITY:
      return "divisibility: S and n_head must be multiples of P, n_head a multiple of n_kv_head, and one of "
             "n_kv_head, P a multiple of the other";
    case ULYSSES_ERR_HIDDEN: return "hidden must equal n_head * head_dim";
    case ULYSSES_ERR_UNSUPPORTED: return "unsupported head_dim / dtype / pass combination";
    case ULYSSES_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case ULYSSES_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case ULYSSES_ERR_WORKSPACE: return "workspace missing or too small";
    case ULYSSES_ERR_CUDA: return "a CUDA call failed";
    default: return "unknown status code";
  }
}

}  // extern "C"
