// internal.h -- declarations shared by the translation units of libulysses.
// Host-side launch helpers; no public API (that is include/ulysses.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ulysses.h"

namespace ulysses {

// Workspace layout (byte offsets, 256-aligned).  The first 256 bytes hold the
// device status word (uint32 at 0) and the RoPE table key (uint32 at 4).
struct WorkspaceLayout {
  size_t status = 0;
  size_t rope = 0, rope_bytes = 0;    // float cos[S][D/2], then float sin[S][D/2]
  size_t delta = 0, delta_bytes = 0;  // float [P][B][hp][delta_ld]    (backward)
  size_t nlse = 0, nlse_bytes = 0;    // float [P][B][hp][delta_ld], -lse*log2(e) (backward)
  size_t dohead = 0, dohead_bytes = 0;  // dO in head layout [P][B][S][hp][D] (backward)
  // With replicated kv-heads (n_kv_head < P): each rank's partial dK and dV,
  // float [P][B][S][D] each, summed over the replicas afterwards (backward).
  size_t dkpart = 0, dvpart = 0, part_bytes = 0;
  size_t total_fwd = 0, total_bwd = 0;
  // The fused backward's float dQ accumulator [B*n_head][Sp][D] (Sp = S rounded
  // up to 128), behind the phase-1 workspace (phase 2 only).
  size_t dqacc = 0, dqacc_bytes = 0, total_fused = 0;
  // phase 3 (dS-store backward): every causal (or, unmasked, every) 128 x 128
  // tile pair's bf16 dS, at the same offset as the fused mode's accumulator
  size_t ds = 0, ds_bytes = 0, total_ds = 0;
  // phase 4: room for the tiles of one kv-head's q-heads at a time (the
  // dS-store backward then runs the kv-heads in chunks)
  size_t ds_kv_bytes = 0, total_ds_min = 0;
};
WorkspaceLayout workspace_layout(const ulysses_problem &p);

// A 32-bit key of (S, D, base) written next to the RoPE table by the init;
// kernels that read the table compare it with the key of their own problem.
uint32_t rope_key(const ulysses_problem &p);

inline size_t elem_size(const ulysses_problem &p) { return p.dtype == ULYSSES_BF16 ? 2 : 4; }

// The Ulysses x ring hybrid: `ring` ring positions of Pu ranks each.  The
// All-to-All runs inside a ring position (over Pu ranks) and a head-layout
// buffer holds the Cs = S / ring tokens of its ring position; ring = 1 is
// plain Ulysses (Pu = P, Cs = S).
inline int ring_of(const ulysses_problem &p) { return p.ring > 1 ? p.ring : 1; }
inline int group_ranks(const ulysses_problem &p) { return p.P / ring_of(p); }  // Pu
inline int chunk_len(const ulysses_problem &p) { return p.S / ring_of(p); }    // Cs
// Row stride, in floats, of the backward's delta and rescaled-LSE rows in the
// workspace: Cs rounded up to 4 so that every row starts on 16 bytes (a TMA
// tensor map's row stride must be a multiple of 16 bytes).  The pad is never
// read or written.
inline int delta_ld(const ulysses_problem &p) { return (chunk_len(p) + 3) & ~3; }

// KV-head replication: with fewer kv-heads than ranks (P a multiple of
// n_kv_head) the q-heads of rank r all read kv-head r / R, R = P / n_kv_head,
// so the seq -> head All-to-All hands each kv-head to R ranks and every rank
// holds one kv-head in head layout.  (Ranks here: the Pu of a ring position.)
inline int kv_replicas(const ulysses_problem &p) {
  return p.n_kv_head < group_ranks(p) ? group_ranks(p) / p.n_kv_head : 1;
}
inline int kv_per_rank(const ulysses_problem &p) {
  return p.n_kv_head >= group_ranks(p) ? p.n_kv_head / group_ranks(p) : 1;
}

// Every host check of ulysses_attn_bwd (problem, bf16 / head_dim, phase-1
// workspace size and alignment, pointers, alignment, overlaps) without
// enqueueing anything; ULYSSES_OK or the code ulysses_attn_bwd would return.
int check_bwd_call(const ulysses_problem *prob, const void *q_head, const void *k_head, const void *v_head,
                   const void *o_head, const float *lse, const void *do_seq, const void *dq_seq,
                   const void *dk_seq, const void *dv_seq, const void *ws, size_t ws_bytes);

// ---- permutation kernels (permute.cu) ----
cudaError_t launch_rope_table(const ulysses_problem &p, void *ws, cudaStream_t st);
cudaError_t launch_pack_qkv(const ulysses_problem &p, const void *q, const void *k, const void *v,
                            void *qh, void *kh, void *vh, void *ws, cudaStream_t st);
cudaError_t launch_unpack(const ulysses_problem &p, const void *o_head, void *o_seq,
                          cudaStream_t st);
// dO seq -> head, delta[i] = sum_e dO[i][e] * O[i][e] and nlse[i] = -lse[i] * log2(e)
// per (rank, b, head, row).  Folded: `o` is O in sequence layout and dO is not
// packed (do_head unused); delta and nlse are the same.
cudaError_t launch_pack_do_delta(const ulysses_problem &p, const void *do_seq, const void *o,
                                 const float *lse, void *do_head, float *delta, float *nlse,
                                 uint32_t *status, cudaStream_t st, bool folded = false);
// Replicated kv-heads: dk_seq/dv_seq (bf16, sequence layout) = the sum over
// each kv-head's replicas of their float partials, in rank order; dK also
// scaled by `scale` and rotated back by the RoPE angle of its position.
cudaError_t launch_kv_reduce(const ulysses_problem &p, const float *dk_part, const float *dv_part,
                             void *dk_seq, void *dv_seq, float scale, const void *ws, cudaStream_t st);

// ---- attention kernels ----
struct TmaEncoder {
  // cuTensorMapEncodeTiled, fetched from the driver at run time.
  CUresult (*encode)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                     CUtensorMapFloatOOBfill) = nullptr;
};
bool get_tma_encoder(TmaEncoder *enc);

cudaError_t launch_attn_fwd_simt(const ulysses_problem &p, const float *q, const float *k,
                                 const float *v, float *o, float *lse, uint32_t *status, cudaStream_t st);
// folded: q/k/v are the sequence-sharded buffers and o is written in sequence
// layout (requires S/P % 128 == 0).
cudaError_t launch_attn_fwd_tc(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                               const void *k, const void *v, void *o, float *lse,
                               uint32_t *status, bool folded, cudaStream_t st);
// QKV projection of the sequence-sharded activations with the pack and RoPE in
// the epilogue (qkv_proj_tc.cu); bias may be null.
cudaError_t launch_qkv_proj_pack(const ulysses_problem &p, const TmaEncoder &enc, const void *x, const void *w,
                                 const void *bias, void *q, void *k, void *v, const void *ws, cudaStream_t st);
// Output projection with the head -> seq unpack folded into its operand loads
// (qkv_proj_tc.cu); needs S/P % 128 == 0; bias may be null.
cudaError_t launch_out_proj_unpack(const ulysses_problem &p, const TmaEncoder &enc, const void *o_head,
                                   const void *w, const void *bias, void *y, const void *ws, cudaStream_t st);
// The two tensor-core kernels of the backward (attn_bwd_tc.cu): dK/dV, then dQ,
// reading the delta / nlse rows the dO step wrote into the workspace.
// folded: q/k/v/do are the sequence-sharded buffers (plain Ulysses, S/P % 128
// == 0); the gradients are written in sequence layout either way.
cudaError_t launch_attn_bwd_dkdv(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                                 const void *k, const void *v, const void *do_head, const float *nlse,
                                 const float *delta, const void *ws, void *dk_seq, void *dv_seq,
                                 uint32_t *status, cudaStream_t st, bool folded = false, void *ds = nullptr,
                                 int head0 = 0, int head_n = -1);
cudaError_t launch_attn_bwd_dq(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                               const void *k, const void *v, const void *do_head, const float *nlse,
                               const float *delta, const void *ws, void *dq_seq, uint32_t *status,
                               cudaStream_t st, bool folded = false);
// dS-store backward (attn_bwd_tc.cu): the dK/dV kernel above with `ds` set
// also writes every step's bf16 dS tile there; this computes dQ = scale *
// sum dS K from those tiles (no recomputation) and writes it in sequence
// layout.  Head layout only (not folded).  Both can be limited to the
// kv-heads [head0, head0 + head_n) of (member * B + batch) * kvp + local
// kv-head and their q-heads (head_n < 0: all of them); `ds` then holds the
// tiles of those q-heads only.
cudaError_t launch_dq_from_ds(const ulysses_problem &p, const TmaEncoder &enc, const void *k, const void *ws,
                              const void *ds, void *dq_seq, uint32_t *status, cudaStream_t st, int head0 = 0,
                              int head_n = -1);
// The fused backward (attn_bwd_tc.cu): dK / dV as the dK/dV kernel writes
// them, and every step's dQ share added into the float accumulator dq_acc
// (which must hold zeros); then dq_finish scales, unrotates and writes dQ in
// sequence layout.
cudaError_t launch_attn_bwd_fused(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                                  const void *v, const void *do_head, const float *nlse, const float *delta,
                                  const void *ws, float *dq_acc, void *dk_seq, void *dv_seq, uint32_t *status,
                                  cudaStream_t st, bool folded = false);
cudaError_t launch_dq_finish(const ulysses_problem &p, const TmaEncoder &enc, const void *ws, float *dq_acc,
                             void *dq_seq, uint32_t *status, cudaStream_t st);
// n floats from `p` (16-byte aligned) set to zero.
cudaError_t launch_zero(float *p, size_t n, cudaStream_t st);

// Heads per CTA group (see grouped_order): as many heads as keep the tiles
// their CTAs stream (per_head_bytes each) within `budget` bytes of L2 (48 MiB
// unless the kernel asks for less).  A grid
// with fewer than 16 CTAs per SM keeps one group (plain longest-first order):
// there a late group's longest CTAs would start near the end and lengthen the
// tail by more than the L2 misses cost.
inline int l2_head_group(size_t per_head_bytes, int n_heads, long long n_ctas,
                         size_t budget = (size_t)48 << 20) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || sms <= 0)
    sms = 152;
  if (n_ctas < 16LL * sms) return n_heads;
  size_t g = per_head_bytes ? budget / per_head_bytes : (size_t)n_heads;
  if (g < 1) g = 1;
  if (g > (size_t)n_heads) g = (size_t)n_heads;
  return (int)g;
}

}  // namespace ulysses
