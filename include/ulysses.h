/*
 * ulysses.h -- C ABI of the single-GPU Ulysses attention path (sm_103a).
 *
 * The method ("Sequence Parallelism II: DeepSpeed Ulysses and All-to-All
 * Attention", §1-§3 and §6; "Comparing Ulysses and Megatron Sequence
 * Parallelism", "DeepSpeed Attention"): activations are sharded by sequence
 * over P ranks; an All-to-All turns "all heads for my tokens" into "all tokens
 * for my heads"; every rank runs ordinary attention over the full sequence
 * for its n_head/P heads; a second All-to-All turns the output back.  Here
 * the P ranks are virtual: all of their buffers live in one GPU's memory, the
 * All-to-All is an on-device permutation kernel and attention runs on the
 * tensor cores.
 *
 * Notation: hp = n_head/P, kvp = n_kv_head/P, Sl = S/P, D = head_dim,
 * H = n_head*D.  Every multi-rank tensor is ONE allocation, rank-major,
 * row-major, innermost index last:
 *   sequence-sharded   X[P][B][Sl][heads][D]   (rank r holds tokens [r*Sl,(r+1)*Sl))
 *   head-sharded       Y[P][B][S][hp or kvp][D] (rank r holds q-heads [r*hp,(r+1)*hp)
 *                                                and kv-heads [r*kvp,(r+1)*kvp))
 *   log-sum-exp        LSE[P][B][hp][S]  float, natural log
 * Element type is bf16 (dtype 0) or fp32 (dtype 1), the same for every
 * activation tensor of a call.  Query head g reads kv-head g/(n_head/n_kv_head).
 *
 * Ownership and execution.  The caller allocates and frees every buffer,
 * including the workspace; the library allocates no device memory and keeps no
 * state between calls.  Every entry point that takes a stream only enqueues
 * work on it (no host synchronisation) and returns once the launches are
 * queued; the outputs are valid when the stream reaches that point.  A NULL
 * stream is the legacy default stream.  Inputs are never written.  Input and
 * output byte ranges of one call must not overlap (ULYSSES_ERR_ALIAS).  Every
 * device pointer must be 16-byte aligned (ULYSSES_ERR_ALIGN).
 *
 * Errors.  Entry points return ULYSSES_OK (0) or a negative code; on an error
 * nothing has been enqueued, except ULYSSES_ERR_CUDA (a launch failed; the
 * CUDA error is also left in cudaGetLastError).  Faults found while kernels
 * run (a bounded wait that timed out, a workspace whose RoPE table does not
 * match the problem) set bits in the workspace's status word, which
 * ulysses_read_status() returns; kernels never trap.
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ulysses_stream_t; /* the same type as cudaStream_t */

enum ulysses_dtype { ULYSSES_BF16 = 0, ULYSSES_FP32 = 1 };

enum ulysses_status_code {
  ULYSSES_OK = 0,
  ULYSSES_ERR_ARG = -1,          /* NULL pointer, or a size <= 0 */
  ULYSSES_ERR_DIVISIBILITY = -2, /* S%P, n_head%Pu, n_head%n_kv_head or P%ring != 0, or
                                    neither of n_kv_head, Pu divides the other (Pu = P/ring):
                                    the head-count bound of Ulysses */
  ULYSSES_ERR_HIDDEN = -3,       /* hidden != n_head * head_dim */
  ULYSSES_ERR_UNSUPPORTED = -4,  /* head_dim / dtype / pass with no kernel */
  ULYSSES_ERR_ALIGN = -5,        /* a pointer is not 16-byte aligned */
  ULYSSES_ERR_ALIAS = -6,        /* an output overlaps an input or another output */
  ULYSSES_ERR_WORKSPACE = -7,    /* workspace NULL or smaller than ulysses_workspace_bytes() */
  ULYSSES_ERR_CUDA = -8          /* a CUDA launch or query failed */
};

/* Bits of the device status word (ulysses_read_status). */
enum ulysses_device_status {
  ULYSSES_STATUS_FWD_TIMEOUT = 1u << 0,  /* attention forward: a pipeline wait gave up */
  ULYSSES_STATUS_BWD_TIMEOUT = 1u << 1,  /* attention backward: a pipeline wait gave up */
  ULYSSES_STATUS_ROPE_TABLE = 1u << 2,   /* RoPE table missing or built for another problem */
  ULYSSES_STATUS_SMEM_ALIGN = 1u << 3,   /* a kernel's dynamic shared memory did not start on a
                                            1024-byte boundary and its tiles did not fit behind
                                            the padding: that kernel wrote nothing */
  ULYSSES_STATUS_BOUNDS = 1u << 4        /* range-checked builds only (compiled with
                                            ULYSSES_CHECK_BOUNDS): a global load or store fell
                                            outside its buffer and was skipped */
};

/*
 * The problem statement of "Comparing Ulysses and Megatron Sequence
 * Parallelism" ("A simple attention skeleton" and the constants of "Megatron
 * Attention costs"): batch B, sequence length S, hidden size, n_head,
 * n_kv_head, head_dim and the sequence-parallel group size P; plus the causal
 * flag, the element type, RoPE on/off with its base, and the softmax scale
 * (0 selects 1/sqrt(head_dim)).
 *
 * `ring` (0 or 1: plain Ulysses) selects the Ulysses x ring hybrid that
 * "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention" points
 * to when P exceeds what the heads allow (§4: a head-sharded group cannot have
 * more ranks than heads; §8: Ring Attention keeps query blocks and circulates
 * key/value blocks).  The P ranks form `ring` ring positions of Pu = P/ring
 * ranks: rank p = r*Pu + u still owns tokens [p*S/P, (p+1)*S/P) in sequence
 * layout, and the All-to-All runs inside each ring position, so in head layout
 * rank (r, u) holds chunk r (tokens [r*Cs, (r+1)*Cs), Cs = S/ring) of heads
 * [u*hp, (u+1)*hp), hp = n_head/Pu (kv-heads likewise).  Attention for those
 * query rows runs over the key/value chunks of every ring position (the
 * ring's circulation), so O, dQ, dK, dV are those of plain attention.  Head
 * layouts below then read [P][B][Cs][...] instead of [P][B][S][...], the LSE
 * [P][B][hp][Cs].  With fewer kv-heads than Pu (Pu a multiple of n_kv_head)
 * each kv-head goes to the Pu/n_kv_head members whose q-heads read it, as in
 * plain Ulysses.  ring > 1 needs bf16, head_dim 64 or 128 and Cs a multiple of
 * 128 (ULYSSES_ERR_UNSUPPORTED otherwise); the folded forward and the two
 * projections take ring <= 1 only.
 */
typedef struct ulysses_problem {
  int B, S, hidden, n_head, n_kv_head, head_dim, P;
  int causal;   /* 1: key k attends for query i iff k <= i (global positions) */
  int dtype;    /* enum ulysses_dtype */
  int use_rope; /* 1: rotate q and k by their global position inside the pack */
  float rope_base;
  float softmax_scale;
  int ring;     /* ring positions of the Ulysses x ring hybrid; 0 or 1: plain Ulysses */
} ulysses_problem;

/* Checks the problem statement alone.  Returns ULYSSES_OK or the first failing
 * code among ERR_ARG, ERR_DIVISIBILITY, ERR_HIDDEN, ERR_UNSUPPORTED.
 * Host only; needs no GPU. */
int ulysses_validate(const ulysses_problem *prob);

/* Workspace bytes for a phase: 0 = forward (pack + attention + unpack),
 * 1 = backward (also valid for the forward), 2 = the fused backward
 * (ulysses_attn_bwd_fused; the phase-1 workspace followed by a float dQ
 * accumulator of B*n_head*ceil(S/128)*128*head_dim*4 bytes; valid for every
 * call), 3 = the dS-store backward (ulysses_attn_bwd_ds; the phase-1
 * workspace followed by B*n_head*T tiles of 128*128 bf16, T = n(n+1)/2 causal
 * or n*n unmasked, n = ceil(S/128); valid for every call but the fused
 * backward's when smaller than phase 2), 4 = the least workspace the
 * dS-store backward takes (the phase-1 workspace followed by the tiles of one
 * kv-head's q-heads on one rank; ulysses_attn_bwd_ds then runs the kv-heads in
 * chunks, as many at a time as the workspace holds).  Returns 0 for an invalid
 * problem or a phase outside 0..4.
 * Host only; needs no GPU. */
size_t ulysses_workspace_bytes(const ulysses_problem *prob, int phase);

/* Prepares a workspace for `prob`: clears the status word and, when use_rope
 * is set, fills the RoPE table (cos and sin of p*base^(-2i/D), p < S,
 * i < D/2, computed in double precision and rounded to float).  Call once
 * per (workspace, problem) before any call that takes `ws`; calls with a
 * workspace prepared for another problem flag ULYSSES_STATUS_ROPE_TABLE and
 * leave their outputs unwritten. */
int ulysses_workspace_init(const ulysses_problem *prob, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream);

/* Copies the workspace status word to *status (synchronises `stream`). */
int ulysses_read_status(const void *ws, uint32_t *status, ulysses_stream_t stream);

/* Enqueues the same copy on `stream` without synchronising: *status holds the
 * word once the stream has reached this point (the caller waits on the stream
 * or an event recorded after this call).  `status` should be pinned host
 * memory (cudaHostAlloc / torch pin_memory) for the copy to stay asynchronous.
 * Errors: ULYSSES_ERR_ARG (NULL pointer), ULYSSES_ERR_CUDA. */
int ulysses_read_status_async(const void *ws, uint32_t *status, ulysses_stream_t stream);

/*
 * Seq -> head All-to-All of Q, K and V, RoPE fused ("Sequence Parallelism II",
 * §1 ownership example and §3; "Comparing Ulysses and Megatron Sequence
 * Parallelism", skeleton: rope, then transpose):
 *   q_head[d][b][s*Sl+t][j][:] = rope(q_seq[s][b][t][d*hp+j][:], s*Sl+t)
 *   k_head likewise with kvp, v_head without rope.
 * q_seq [P][B][Sl][n_head][D], k_seq/v_seq [P][B][Sl][n_kv_head][D];
 * q_head [P][B][S][hp][D], k_head/v_head [P][B][S][kvp][D].
 * RoPE: rotate-half, x'_i = x_i cos - x_{i+D/2} sin, x'_{i+D/2} = x_{i+D/2} cos
 * + x_i sin, angle p*base^(-2i/D); float arithmetic on the input values, one
 * rounding to the element type.  Without RoPE the result is a bit-exact copy.
 * `ws` (phase 0) must have been prepared by ulysses_workspace_init.
 */
int ulysses_pack_qkv(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                     const void *v_seq, void *q_head, void *k_head, void *v_head, void *ws,
                     size_t ws_bytes, ulysses_stream_t stream);

/*
 * Per-rank attention over the full sequence for the rank's heads
 * ("Sequence Parallelism II", §2 fourth step): for rank r, batch b, local
 * head j (global g = r*hp+j, kv-head g/(n_head/n_kv_head)):
 *   o[i] = sum_k softmax_k(scale * q_i.k_k [+ causal mask]) v_k,
 *   lse[i] = log sum_k exp(scale * q_i.k_k).
 * bf16: tensor-core kernel, head_dim 64 or 128, fp32 accumulation and softmax.
 * fp32: CUDA-core kernel, head_dim 32, 64 or 128.
 * o_head [P][B][S][hp][D] (element type), lse [P][B][hp][S] float.
 */
int ulysses_attn_fwd(const ulysses_problem *prob, const void *q_head, const void *k_head,
                     const void *v_head, void *o_head, float *lse, void *ws, size_t ws_bytes,
                     ulysses_stream_t stream);

/*
 * Folded forward: pack, attention and unpack in one kernel, with both
 * All-to-Alls turned into addressing ("Sequence Parallelism II", §1: the
 * All-to-All is a distributed transpose of ownership).  The tensor-core kernel
 * reads the 128-row tiles of rank r's heads straight out of the
 * sequence-sharded buffers (the tile at global position p comes from rank
 * p/Sl, row p%Sl) and writes O straight into sequence layout.  Results are
 * identical to ulysses_pack_qkv + ulysses_attn_fwd + ulysses_unpack_out.
 * q_seq [P][B][Sl][n_head][D], k_seq/v_seq [P][B][Sl][n_kv_head][D] ->
 * o_seq [P][B][Sl][H], lse [P][B][hp][S] float.
 * Requires bf16, head_dim 64 or 128, use_rope == 0 (q and k must already be
 * rotated by their producer) and S/P a multiple of 128, else
 * ULYSSES_ERR_UNSUPPORTED.  `ws` (phase 0) carries the status word.
 */
int ulysses_attn_fwd_folded(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                            const void *v_seq, void *o_seq, float *lse, void *ws, size_t ws_bytes,
                            ulysses_stream_t stream);

/*
 * The QKV projection with the seq -> head All-to-All and RoPE fused into it
 * ("Sequence Parallelism II", §2 second and third steps: each rank projects
 * its own tokens with the complete, replicated weights, then the All-to-All;
 * "Comparing Ulysses and Megatron Sequence Parallelism", "A simple attention
 * skeleton": q, k, v projections, viewed as heads, RoPE on q and k).
 *   x_seq  [P][B][Sl][hidden] bf16 (the sequence-sharded activations);
 *   w_qkv  [(n_head + 2 n_kv_head) * head_dim][hidden] bf16: the q, k and v
 *          projection weights stacked in that order, each in the Linear
 *          layout [out_features][in_features];
 *   b_qkv  [(n_head + 2 n_kv_head) * head_dim] bf16, or NULL for no bias.
 * Writes q_head/k_head/v_head exactly as ulysses_pack_qkv would from the
 * projected q, k, v: q = x W_q^T + b_q etc. accumulated in fp32, RoPE applied
 * in fp32, rounded once to bf16 (KV-head replication included).  `ws` (phase
 * 0, prepared by ulysses_workspace_init) supplies the RoPE table and the
 * status word.  bf16 and head_dim 64 or 128, else ULYSSES_ERR_UNSUPPORTED;
 * other errors as ulysses_pack_qkv.
 */
int ulysses_qkv_proj_pack(const ulysses_problem *prob, const void *x_seq, const void *w_qkv,
                          const void *b_qkv, void *q_head, void *k_head, void *v_head, void *ws,
                          size_t ws_bytes, ulysses_stream_t stream);

/*
 * Head -> seq All-to-All of the attention output ("Sequence Parallelism II",
 * §2 fifth step; "Comparing Ulysses and Megatron Sequence Parallelism",
 * "DeepSpeed Attention": [B,S,heads/P,D] back to [B,S/P,heads,D] = [B,S/P,H]):
 *   o_seq[d][b][t][(s*hp+j)*D+e] = o_head[s][b][d*Sl+t][j][e]   (bit-exact copy)
 * o_head [P][B][S][hp][D] -> o_seq [P][B][Sl][H].
 */
int ulysses_unpack_out(const ulysses_problem *prob, const void *o_head, void *o_seq,
                       ulysses_stream_t stream);

/*
 * The output projection with the head -> seq All-to-All folded into its
 * operand loads ("Sequence Parallelism II", §2 fifth step: the inverse
 * All-to-All gives every rank [B, S/P, H] back, and each rank applies the
 * complete output projection to its own tokens; "Comparing Ulysses and
 * Megatron Sequence Parallelism", skeleton: y = output_proj(y)).
 *   o_head [P][B][S][hp][D] bf16 (as written by ulysses_attn_fwd);
 *   w_o    [hidden][n_head * head_dim] bf16, the Linear layout [out][in];
 *   b_o    [hidden] bf16, or NULL for no bias;
 *   y_seq  [P][B][Sl][hidden] bf16: y = unpack(o) w_o^T + b_o, accumulated in
 *          fp32 and rounded once.
 * Requires bf16, head_dim 64 or 128 and S/P a multiple of 128 (a 128-token
 * tile then lies in one rank's shard), else ULYSSES_ERR_UNSUPPORTED.  `ws`
 * (phase 0) carries the status word.
 */
int ulysses_out_proj_unpack(const ulysses_problem *prob, const void *o_head, const void *w_o,
                            const void *b_o, void *y_seq, void *ws, size_t ws_bytes,
                            ulysses_stream_t stream);

/*
 * Backward of the whole path ("Sequence Parallelism II", §6; "Comparing
 * Ulysses and Megatron Sequence Parallelism", "DeepSpeed Attention costs":
 * the inverse All-to-All for each tensor): dO_seq [P][B][Sl][H] goes seq ->
 * head, per-head attention backward, dQ/dK/dV go head -> seq with the RoPE
 * rotation undone on dQ and dK (gradients w.r.t. the pre-rope q, k; dK and dV
 * summed over the q-heads that share a kv-head).
 * Inputs: the head-layout q/k/v written by ulysses_pack_qkv, o_head and lse
 * written by ulysses_attn_fwd, do_seq.  Outputs: dq_seq [P][B][Sl][n_head][D],
 * dk_seq/dv_seq [P][B][Sl][n_kv_head][D].  bf16, head_dim 64 or 128.
 * `ws` must be sized for phase 1 and prepared by ulysses_workspace_init.
 */
int ulysses_attn_bwd(const ulysses_problem *prob, const void *q_head, const void *k_head,
                     const void *v_head, const void *o_head, const float *lse,
                     const void *do_seq, void *dq_seq, void *dk_seq, void *dv_seq, void *ws,
                     size_t ws_bytes, ulysses_stream_t stream);

/*
 * The backward in its three steps, for callers that schedule or time them
 * separately; ulysses_attn_bwd is exactly these three calls in this order on
 * one stream, and the results are identical.
 *
 * ulysses_attn_bwd_prepare: the seq -> head All-to-All of the output gradient
 * ("Sequence Parallelism II", §6) together with delta_i = dO_i . O_i and the
 * rescaled log-sum-exp, written into the workspace `ws` (phase 1, prepared by
 * ulysses_workspace_init).  Reads o_head and lse from ulysses_attn_fwd and
 * do_seq [P][B][Sl][H].
 *
 * ulysses_attn_bwd_dkdv: dK and dV per kv-head (summed over the q-heads that
 * share it), then head -> seq into dk_seq / dv_seq [P][B][Sl][n_kv_head][D],
 * with the RoPE rotation undone on dK.  Reads the head-layout q/k/v from
 * ulysses_pack_qkv and what ulysses_attn_bwd_prepare left in `ws`.
 *
 * ulysses_attn_bwd_dq: dQ per q-head, then head -> seq into dq_seq
 * [P][B][Sl][n_head][D] with the RoPE rotation undone.  Same inputs as the
 * dK/dV step; the two may run in either order after the prepare step.
 *
 * bf16 and head_dim 64 or 128 (else ULYSSES_ERR_UNSUPPORTED); the errors and
 * ownership rules of ulysses_attn_bwd apply to each.
 */
int ulysses_attn_bwd_prepare(const ulysses_problem *prob, const void *o_head, const float *lse,
                             const void *do_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream);
int ulysses_attn_bwd_dkdv(const ulysses_problem *prob, const void *q_head, const void *k_head,
                          const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                          ulysses_stream_t stream);
int ulysses_attn_bwd_dq(const ulysses_problem *prob, const void *q_head, const void *k_head,
                        const void *v_head, void *dq_seq, void *ws, size_t ws_bytes, ulysses_stream_t stream);

/*
 * The backward with dQ accumulated inside the dK/dV loop ("Sequence
 * Parallelism II", §6, the same gradients as ulysses_attn_bwd; "Comparing
 * Ulysses and Megatron Sequence Parallelism", "DeepSpeed Attention costs":
 * the backward does about twice the forward's products).  ulysses_attn_bwd
 * runs two tensor-core kernels, the second recomputing the scores and dP for
 * dQ: seven matrix products per (128-key, 128-query) tile pair.  Here one
 * kernel forms dV, dK and each tile pair's dQ share from the same scores:
 * five products per pair.  The dQ shares of one query tile come from the
 * CTAs of different key tiles and are added into a float accumulator in the
 * workspace by the copy engine's reduce-add, in an order that varies from run
 * to run: dQ is reproducible to float rounding, not bit for bit (dK and dV
 * are bit-identical to ulysses_attn_bwd's).  Same arguments, layouts and
 * results (within the stated tolerance) as ulysses_attn_bwd; `ws` must be
 * sized for phase 2 and prepared by ulysses_workspace_init.  bf16, head_dim
 * 64 or 128; the errors of ulysses_attn_bwd, and ULYSSES_ERR_WORKSPACE for a
 * workspace smaller than phase 2.
 *
 * Its steps, for callers that time or schedule them: ulysses_attn_bwd_prepare
 * (above), then ulysses_attn_bwd_dkdvq (zeroes the accumulator, then dK, dV
 * into dk_seq / dv_seq as ulysses_attn_bwd_dkdv writes them and every dQ
 * share added into the accumulator), then ulysses_attn_bwd_dq_finish (dQ
 * from the accumulator: scaled, RoPE rotation undone, rounded to bf16 into
 * dq_seq [P][B][Sl][n_head][D]).
 */
int ulysses_attn_bwd_fused(const ulysses_problem *prob, const void *q_head, const void *k_head,
                           const void *v_head, const void *o_head, const float *lse, const void *do_seq,
                           void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream);
int ulysses_attn_bwd_dkdvq(const ulysses_problem *prob, const void *q_head, const void *k_head,
                           const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                           ulysses_stream_t stream);
int ulysses_attn_bwd_dq_finish(const ulysses_problem *prob, void *dq_seq, void *ws, size_t ws_bytes,
                               ulysses_stream_t stream);

/*
 * The backward with dS stored ("Sequence Parallelism II", §6, the same
 * gradients as ulysses_attn_bwd).  The dK/dV kernel, which forms every
 * (128-key, 128-query) tile pair's dS as the operand of its dK product, also
 * writes that bf16 tile to the workspace; a second tensor-core kernel then
 * sums dQ = scale * dS K over the stored tiles instead of recomputing the
 * scores and dP: five matrix products per tile pair, deterministic (every
 * call gives the same bits), at the price of writing and reading 32 KB per
 * tile pair (B*n_head*T*32 KB in all, T as under ulysses_workspace_bytes).
 * dK and dV are bit-identical to ulysses_attn_bwd's; dQ is the sum of the
 * same bf16 dS values the dK product uses (within the stated tolerance of
 * ulysses_attn_bwd's).  Same arguments, layouts and results as
 * ulysses_attn_bwd; `ws` must be sized for at least phase 4 and prepared by
 * ulysses_workspace_init.  With less than phase 3 the kv-heads are processed
 * in chunks (each: the dK/dV step storing its q-heads' tiles, then their dQ),
 * as many kv-heads at a time as the workspace holds tiles for; the results
 * are the same bits either way.  bf16, head_dim 64 or 128; the errors of
 * ulysses_attn_bwd, and ULYSSES_ERR_WORKSPACE for a workspace smaller than
 * phase 4.
 *
 * Its steps, with a phase-3 workspace (all the tiles at once):
 * ulysses_attn_bwd_prepare (above), then ulysses_attn_bwd_dkdv_ds
 * (dK, dV into dk_seq / dv_seq as ulysses_attn_bwd_dkdv writes them, and the
 * dS tiles into the workspace), then ulysses_attn_bwd_dq_ds (dQ from the
 * tiles and k_head: scaled, RoPE rotation undone, rounded to bf16 into dq_seq
 * [P][B][Sl][n_head][D]; reads no q, v or dO).
 */
int ulysses_attn_bwd_ds(const ulysses_problem *prob, const void *q_head, const void *k_head,
                        const void *v_head, const void *o_head, const float *lse, const void *do_seq,
                        void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                        ulysses_stream_t stream);
int ulysses_attn_bwd_dkdv_ds(const ulysses_problem *prob, const void *q_head, const void *k_head,
                             const void *v_head, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                             ulysses_stream_t stream);
int ulysses_attn_bwd_dq_ds(const ulysses_problem *prob, const void *k_head, void *dq_seq, void *ws,
                           size_t ws_bytes, ulysses_stream_t stream);

/*
 * Folded backward: the backward of ulysses_attn_fwd_folded with every
 * All-to-All turned into addressing ("Sequence Parallelism II", §6: the
 * backward makes the forward's layout changes in reverse).  The dK/dV and dQ
 * kernels read the 128-row tiles of q, k, v and dO straight out of the
 * sequence-sharded buffers (the tile at global position p of head g comes from
 * rank p/Sl, row p%Sl, head g) and write dQ, dK, dV straight into sequence
 * layout; a first kernel forms delta_i = dO_i . O_i from o_seq and do_seq in
 * place (no dO pack).  Results are identical to ulysses_attn_bwd on the packed
 * buffers of the same problem.
 * Inputs: q_seq [P][B][Sl][n_head][D], k_seq/v_seq [P][B][Sl][n_kv_head][D]
 * (the already-rotated q, k the folded forward read), o_seq [P][B][Sl][H] and
 * lse [P][B][hp][S] from the folded forward, do_seq [P][B][Sl][H].  Outputs
 * dq_seq [P][B][Sl][n_head][D], dk_seq/dv_seq [P][B][Sl][n_kv_head][D] (the
 * gradients with respect to the rotated q, k: no rotation is undone).
 * Requires bf16, head_dim 64 or 128, use_rope == 0, ring <= 1 and S/P a
 * multiple of 128, else ULYSSES_ERR_UNSUPPORTED.  `ws` must be sized for
 * phase 1 and prepared by ulysses_workspace_init; other errors and the
 * ownership rules as for ulysses_attn_bwd.
 */
int ulysses_attn_bwd_folded(const ulysses_problem *prob, const void *q_seq, const void *k_seq,
                            const void *v_seq, const void *o_seq, const float *lse, const void *do_seq,
                            void *dq_seq, void *dk_seq, void *dv_seq, void *ws, size_t ws_bytes,
                            ulysses_stream_t stream);

/*
 * Self-test of failure detection (no counterpart in the pages): one CTA waits,
 * with the bounded wait every pipeline wait of the attention kernels uses, on a
 * barrier that nothing ever completes.  After `limit_ns` (1 ns .. 2 s) the wait
 * gives up, the CTA sets ULYSSES_STATUS_FWD_TIMEOUT in the status word at the
 * start of `ws` (any workspace prepared by ulysses_workspace_init, at least 256
 * bytes) and exits normally; the context stays usable.  Asynchronous on
 * `stream`; read the bit with ulysses_read_status, clear it with
 * ulysses_workspace_init.  Errors: ULYSSES_ERR_ARG (NULL or too small `ws`,
 * limit out of range), ULYSSES_ERR_ALIGN, ULYSSES_ERR_CUDA (launch failed).
 */
int ulysses_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned long long limit_ns,
                                  ulysses_stream_t stream);

/*
 * Throughput of the SM's base-2 exponential (the MUFU unit's ex2), the
 * secondary bound of the softmax: the attention forward takes one exponential
 * per (query, key) pair it computes ("Sequence Parallelism II: DeepSpeed
 * Ulysses and All-to-All Attention", §8: causal attention keeps its triangular
 * work), B*n_head*S(S+1)/2 for a causal pass.
 *
 * Launches, on `stream`, 2 blocks of 512 threads per SM, every thread running 8
 * independent dependent chains of ex2 for 4096 steps, and writes the largest
 * block's elapsed SM cycles (uint64) to the device pointer `cycles` (8 bytes,
 * 8-byte aligned; the caller reads it after the stream completes).  Sets
 * *ex2_per_launch to the exponentials the launch computes and *sms to the SM
 * count, so ex2 per SM per cycle = *ex2_per_launch / (*sms * cycles).
 * Errors: ULYSSES_ERR_ARG (NULL pointer, bytes < 8), ULYSSES_ERR_ALIGN,
 * ULYSSES_ERR_CUDA.
 */
int ulysses_selftest_ex2_rate(void *cycles, size_t bytes, long long *ex2_per_launch, int *sms,
                              ulysses_stream_t stream);

/*
 * The backward for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point (the pages describe no
 * allocation policy).  It exists for callers that cannot hand the library a
 * workspace: code running under an allocator it does not own (a host framework
 * that owns every device allocation), paths that must not call cudaMalloc or
 * cudaFree because those can synchronise the device, or embedders with a memory
 * budget fixed up front.
 *
 * Same arguments, layouts and results as ulysses_attn_bwd, without `ws`.  The
 * scratch (RoPE table, delta, dO in head layout, status word) comes from a
 * 32 MiB array in the library's own device memory, which every GPU that loads
 * the library holds until the process exits.  A problem whose phase-1
 * workspace (ulysses_workspace_bytes(prob, 1)) exceeds 32 MiB is rejected with
 * ULYSSES_ERR_WORKSPACE before anything is enqueued; so are problems and
 * pointers ulysses_attn_bwd would refuse (same codes, checked before the array
 * is touched).  No device memory is allocated by this call.  Faults the
 * kernels find are flagged in the array's status word: read it with
 * ulysses_noalloc_read_status.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every call
 * rebuilds the RoPE table and clears the status word in the array before the
 * backward kernels run.  All calls share the one array: calls whose kernels
 * overlap on the GPU (other streams, other host threads) race on it and must
 * be ordered by the caller.
 */
int ulysses_attn_bwd_noalloc(const ulysses_problem *prob, const void *q_head, const void *k_head,
                             const void *v_head, const void *o_head, const float *lse,
                             const void *do_seq, void *dq_seq, void *dk_seq, void *dv_seq,
                             ulysses_stream_t stream);

/* The status word of the scratch array ulysses_attn_bwd_noalloc uses on the
 * current device (the bits of enum ulysses_device_status, as
 * ulysses_read_status returns them for a workspace): waits for `stream`, then
 * copies the word written by the noalloc calls enqueued before this point.
 * Like that entry point, it has no counterpart in the pages.
 * Errors: ULYSSES_ERR_ARG (NULL status), ULYSSES_ERR_CUDA. */
int ulysses_noalloc_read_status(uint32_t *status, ulysses_stream_t stream);

/* A static English description of a return code. */
const char *ulysses_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
