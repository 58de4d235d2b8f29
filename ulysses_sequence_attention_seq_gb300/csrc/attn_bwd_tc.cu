// attn_bwd_tc.cu -- bf16 attention backward on the 5th-generation tensor cores,
// with the reverse All-to-All of the gradients fused into the epilogues.
//
// "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention", §6:
// the output gradient is All-to-All'd into head layout (done before these
// kernels, together with delta = rowsum(dO * O)); the Q, K, V gradients are
// produced per head and All-to-All'd back to sequence layout.  The gradient
// formulas of softmax(scale q k^T) v, with P = exp(scale q.k - lse):
//   dV = P^T dO          dP = dO V^T          dS = P * (dP - delta)
//   dQ = scale dS K      dK = scale dS^T Q    (dK, dV summed over the q-heads
//                                              that share a kv-head)
// Two kernels, each deterministic (no atomics), every MMA 128x128x16:
//   dkdv: one CTA per 128-key tile of one kv-head.  K and V stay in shared
//         memory; the loop runs over the q-heads of the group and the
//         128-query tiles at or after the key tile (causal).  Per step:
//         S^T = K Q^T and dP^T = V dO^T into TMEM, the softmax warps form
//         P^T and dS^T (bf16) in TMEM, then dV += P^T dO and dK += dS^T Q
//         (A operand read from TMEM) accumulate in TMEM across the loop.
//   dq:   one CTA per 128-query tile of one head.  Q and dO stay in TMEM
//         (the A operand of S and dP); the loop runs over 128-key tiles at or
//         before the query tile.  Per step: S = Q K^T and dP = dO V^T into
//         TMEM, dS (bf16) over dP, dQ += dS K in TMEM.
// Epilogues: the thread that owns a row of the accumulator writes it straight
// to its place in the sequence-sharded output (the inverse All-to-All as
// addressing) after undoing the RoPE rotation on dQ and dK (both elements of
// every rotation pair are in the same thread's row).
// Warp roles: warps 0-7 softmax / epilogue (two warpgroups, each owns half of
// the tile's columns; warp w reads TMEM lanes 32*(w%4)...), warp 8 TMA
// producer, warp 9 MMA issuer; the dq kernel adds warps 10-11 to complete a
// third warpgroup for its per-warpgroup register split.  All waits are bounded.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "check.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace ulysses {
namespace {

using namespace sm100;
using dev::warp_wait;

constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, S, P, Sl, hp, kvp, group, causal;
  int n_head, n_kv;                    // global head counts (row widths of the seq layout)
  int group_kv, group_q;               // heads per CTA group (grouped_order) of the two kernels
  float scale, scale_log2;
  const float *nlse, *delta;           // [P][B][hp] rows of Cs values, Ld apart; nlse = -lse * log2(e)
  const float *rope_cos, *rope_sin;    // [S][D/2], or null without RoPE
  const __nv_bfloat16 *q, *dout;       // head layout [P][B][S][hp][D] (the dQ kernel's TMEM operands)
  __nv_bfloat16 *dq, *dk, *dv;         // sequence-sharded outputs
  int kv_rep;                          // > 1: replicated kv-heads; dk/dv then point to float
                                       // per-rank partials [P*B][Cs][D] (unscaled, not rotated)
  uint32_t *status;                    // status word; the RoPE table key follows it
  uint32_t rope_key;
  // Ulysses x ring hybrid: Pu ranks per ring position, Cs tokens per chunk
  // (plain Ulysses: P, S).  A CTA works on one (group member, batch, head)
  // over the full sequence; the rows at global position pos live in the
  // head-layout buffer of rank (pos / Cs) * Pu + member, row pos % Cs.
  int Pu, Cs;
  int Ld;                              // row stride of nlse / delta (Cs rounded up to 4)
  int Sp;                              // S rounded up to 128: rows per head of the fused kernel's
                                       // float dQ accumulator [Pu*B][hp][Sp][D]
  // Folded addressing: q, dout and the K / V maps cover the sequence-sharded
  // buffers [P*B][Sl][heads][D] instead of the head-layout ones (plain Ulysses,
  // Sl a multiple of 128); nlse / delta keep their head-layout rows.
  int folded;
  // Elements of the buffers the kernels read or write with plain loads and
  // stores (range checks of a checked build): dQ, dK / dV (or their float
  // partials), Q / dO in head layout, the nlse / delta rows, the RoPE table.
  long long dq_n, dkv_n, qo_n, rows_n, rope_n;
  // dS-store mode: the dK/dV kernel also writes every step's dS tile (bf16,
  // [128 keys][128 queries]) to `ds` (null: not stored); `ds_pairs` tiles per
  // q-head (see ds_tile).
  __nv_bfloat16 *ds;
  long long ds_pairs;
  // The kv-heads ((member * B + batch) * kvp + local kv-head) a dK/dV or
  // dQ-from-dS launch covers, [head0, head0 + head_n), with their q-heads; the
  // dS store then holds the tiles of those q-heads only, the first q-head's at
  // its start.
  int head0, head_n;
};

// Head-layout (rank * B + batch) of the rows at global position `pos` for the
// CTA of member*B + batch = `rb`.
__device__ __forceinline__ int hl_outer(const BwdParams &p, int rb, int pos) {
  return (pos / p.Cs) * p.Pu * p.B + rb;
}

// TMA coordinates (head, row, outer) of the 128 rows at position `pos` (a
// multiple of 128) of local head `h` of the CTA's (member, batch) `rb`: in the
// head-layout buffers, or, folded, in the sequence shard that holds them (rank
// pos / Sl, row pos % Sl, the global head: member * heads_local + h, or
// member / rep for a kv-head replicated over rep ranks).
struct ActCoord {
  int head, row, outer;
};
__device__ __forceinline__ ActCoord act_coord(const BwdParams &p, int rb, int h, int heads_local, int pos,
                                              int rep) {
  if (!p.folded) return {h, pos % p.Cs, hl_outer(p, rb, pos)};
  const int u = rb / p.B, b = rb - u * p.B;
  return {rep > 1 ? u / rep : u * heads_local + h, pos % p.Sl, (pos / p.Sl) * p.B + b};
}

// One key row's 64 dS values of a warpgroup's half tile (see ds_tile): four
// 32-byte streaming stores, 2048 elements apart; read by another kernel.
__device__ __forceinline__ void store_ds_row(__nv_bfloat16 *dst, const uint32_t (&x)[32]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_global_cs_v8(dst + u * 2048, x[8 * u], x[8 * u + 1], x[8 * u + 2], x[8 * u + 3], x[8 * u + 4], x[8 * u + 5],
                    x[8 * u + 6], x[8 * u + 7]);
}

// Tile index of (q-head hq, query tile m, key tile n) in the dS store: the
// causal pairs n <= m of a head in query-tile order (m(m+1)/2 + n), or all
// n_kt * n_kt pairs without the mask; a head's pairs are contiguous.  A tile
// is 8 chunks of 16 queries, each chunk the 128 keys' 32-byte rows, the two
// 8-query halves of a row swapped in every other group of 4 keys: element
// (key k, query q) at (q / 16 * 128 + k) * 16 + ((q / 8 % 2) ^ (k / 4 % 2)) * 8
// + q % 8.  Read back whole, that is the 32-byte-swizzled MN-major operand
// layout, and the dK/dV kernel's lanes (one key each) write it with 32-byte
// stores, 1 KB contiguous per warp.
__device__ __forceinline__ long long ds_tile(const BwdParams &p, int hq, int m, int n) {
  const int n_kt = (p.S + 127) / 128;
  const long long t = p.causal ? (long long)m * (m + 1) / 2 + n : (long long)m * n_kt + n;
  return (long long)(hq - p.head0 * p.group) * p.ds_pairs + t;
}

// Element offset of row `pos` of local q-head j of the CTA's (member, batch)
// `rb` in q / dout (head layout, or folded the sequence-sharded buffer).
__device__ __forceinline__ size_t q_row_offset(const BwdParams &p, int rb, int j, int pos, int D) {
  if (!p.folded) return (((size_t)hl_outer(p, rb, pos) * p.Cs + pos % p.Cs) * p.hp + j) * D;
  const int u = rb / p.B, b = rb - u * p.B, s = pos / p.Sl;
  return ((((size_t)s * p.B + b) * p.Sl + (pos - s * p.Sl)) * p.n_head + u * p.hp + j) * D;
}

// True (and the status bit set) when the workspace's RoPE table was built for
// another problem: the kernel then writes nothing.
__device__ __forceinline__ bool stale_rope_table(const BwdParams &p) {
  if (p.rope_cos && p.status[1] != p.rope_key) {
    if (threadIdx.x == 0) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_ROPE_TABLE);
    return true;
  }
  return false;
}

// 32 fp32 accumulator columns -> scaled bf16 in global memory.
__device__ __forceinline__ void store_plain(__nv_bfloat16 *dst, const uint32_t (&x)[32], float scale) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    w[e] = pack_bf16x2(__uint_as_float(x[2 * e]) * scale, __uint_as_float(x[2 * e + 1]) * scale);
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) d[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
}

// The cos / sin of rotation pairs [i0, i0+32) at one position, read ahead of
// the epilogue that undoes the rotation: `rope_prefetch` asks L2 for the two
// 128-byte rows (kept with evict-last priority: every head's CTAs over the
// same rows read them) when a CTA starts, `rope_load` brings them into
// registers while the last products are still running.
struct RopeRow {
  float4 c[8], s[8];
};
__device__ __forceinline__ void rope_prefetch(const float *cs, const float *sn) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(cs));
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(sn));
}
__device__ __forceinline__ void rope_load(RopeRow &a, const float *cs, const float *sn) {
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    a.c[v] = __ldg(reinterpret_cast<const float4 *>(cs) + v);
    a.s[v] = __ldg(reinterpret_cast<const float4 *>(sn) + v);
  }
}

// Columns [i0, i0+32) (x) and [i0+D/2, i0+D/2+32) (y) of a gradient row:
// scale, undo the rotation by the position's angle (x' = x cos + y sin,
// y' = y cos - x sin) when `rot`, round to bf16 and store.
__device__ __forceinline__ void store_unrotated(__nv_bfloat16 *dx, __nv_bfloat16 *dy, uint32_t (&x)[32],
                                                uint32_t (&y)[32], float scale, bool rot, const RopeRow &a) {
  if (rot) {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 c4 = a.c[e / 4];
      const float4 s4 = a.s[e / 4];
      const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = __uint_as_float(x[e + q]), b = __uint_as_float(y[e + q]);
        x[e + q] = __float_as_uint(a * cc[q] + b * ss[q]);
        y[e + q] = __float_as_uint(b * cc[q] - a * ss[q]);
      }
    }
  }
  store_plain(dx, x, scale);
  store_plain(dy, y, scale);
}

// ============================================================= dK / dV kernel
// One CTA per 128-key tile of one kv-head; 128-query steps over the group's
// q-heads, every MMA 128x128x16.  TMEM: S^T [0,128), dP^T [128,256),
// dV [256, 256+D), dK [256+D, 256+2D).  Warpgroup g owns query columns
// [64g, 64g+64) of a step: it reads its S^T columns and writes P^T (bf16, two
// per column) over the first half of them, then reads its dP^T columns and
// writes dS^T likewise; the dV/dK MMAs read them from there as their A
// operand (columns [0,32) and [64,96) of each region).
// The tensor core runs dV(i), S^T(i+1), dK(i), dP^T(i+1), ...: S^T(i+1)
// overwrites P^T(i) only after dV(i) (one issuer's MMAs run in order) and is
// computed while the softmax warps form dS^T(i); dP^T(i+1) likewise follows
// dK(i) and runs while they form P^T(i+1).  So the tensor core never waits for
// the softmax of its own step as long as each softmax phase is shorter than
// two MMA groups.  A thread with MMAs in flight stalls on its next
// shared-memory access (such as a barrier wait, ~100 cycles each even on a
// completed phase) until they have been taken by the tensor core, which leaves
// a gap in the pipe, so the issuer waits once per burst: for PFull(i) before
// dV(i) S^T(i+1) and for DSFull(i) before dK(i) dP^T(i+1).  The softmax warps
// wait for the ring tiles in its place before arriving: at the end of step
// i's dS phase for dO tile i+1 and Q tile i+2 (off the P phase, on which the
// tensor core waits), so each arrival vouches for every tile the bursts after
// it read.
// Q tiles stream through a 3-slot ring released after dK (their last reader),
// dO tiles through a 2-slot ring released after dV; each step's delta rides in
// its Q slot (read in the dS phase, before dK) and its LSE in its dO slot (read
// in the P phase, before dV).  The third Q slot covers the L2 latency of a
// tile load, which is longer than the two MMA groups between dK(i) and S^T(i+2).
constexpr int kQSlots = 3, kOSlots = 2;
constexpr int kThreadsKV = 320;  // 8 softmax warps, TMA warp, MMA warp (160 registers, no split)

enum : uint32_t {
  kKBarIn = 0,
  kKBarQFull = 8,    // [3]
  kKBarQEmpty = 32,  // [3]
  kKBarOFull = 56,   // [2]
  kKBarOEmpty = 72,  // [2]
  kKBarSFull = 88,
  kKBarDPFull = 96,
  kKBarPFull = 104,  // 256 arrivals
  kKBarDSFull = 112, // 256 arrivals
  kKBarAcc = 120,
  kKBarDrain = 128,
  kKTmemSlot = 136,
  kKAbortSlot = 140,
  kKBarBytes = 144
};

// P = exp2(scale*log2(e)*s - lse*log2(e)) for the 64 columns of S^T a
// thread holds (query c's -lse*log2(e) at nl[c/2]); with kMask, columns
// outside [lo, hi) are 0.  P is kept in fp32 for dS and packed to bf16.
template <bool kMask>
__device__ __forceinline__ void p_columns(const uint32_t (&s)[2][32], const float2 *nl, float sl, int lo,
                                          int hi, float2 (&pf)[32], uint32_t (&w)[2][16]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t *sh = s[c >> 4];
    const float2 x = fma2(make_float2(__uint_as_float(sh[2 * (c & 15)]), __uint_as_float(sh[2 * (c & 15) + 1])),
                          make_float2(sl, sl), nl[c]);
    float2 pe = make_float2(ex2(x.x), ex2(x.y));
    if (kMask) {
      if (2 * c < lo || 2 * c >= hi) pe.x = 0.f;
      if (2 * c + 1 < lo || 2 * c + 1 >= hi) pe.y = 0.f;
    }
    pf[c] = pe;
    w[c >> 4][c & 15] = pack_bf16x2(pe.x, pe.y);
  }
}

// dS = P * (dP - delta) for the same 64 columns (query c's delta at dl[c/2]).
__device__ __forceinline__ void ds_columns(const uint32_t (&d)[2][32], const float2 *dl, const float2 (&pf)[32],
                                           uint32_t (&w)[2][16]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t *dh = d[c >> 4];
    const float2 x = sub2(make_float2(__uint_as_float(dh[2 * (c & 15)]), __uint_as_float(dh[2 * (c & 15) + 1])),
                          dl[c]);
    const float2 ds = mul2(pf[c], x);
    w[c >> 4][c & 15] = pack_bf16x2(ds.x, ds.y);
  }
}

constexpr uint32_t kMaxDynSmem = 232448;  // 227 KB per block

template <int D>
struct KVLayout {
  static constexpr uint32_t kT = 128u * D * 2;  // one 128-row tile
  static constexpr uint32_t oK = 0, oV = kT, oQ = 2 * kT, odO = oQ + kQSlots * kT,
                            oDl = odO + kOSlots * kT,  // delta rows, one per Q slot
                            oL = oDl + kQSlots * 512,  // -LSE*log2(e) rows, one per dO slot
                            oBar = oL + kOSlots * 512;
  static constexpr uint32_t kUsed = oBar + kKBarBytes;
  // Room for aligning the base to 1024 bytes where it fits; at D = 128 it
  // does not, and the kernel checks the base it was given.
  static constexpr uint32_t kAlloc = kUsed + 1024 <= kMaxDynSmem ? kUsed + 1024 : kMaxDynSmem;
  static_assert(kUsed <= kMaxDynSmem, "dK/dV tiles exceed shared memory");
};

template <int D>
__global__ void __launch_bounds__(kThreadsKV, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmDl,
                const BwdParams p) {
  using L = KVLayout<D>;
  constexpr int kCh = D / 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + L::oK, sV = sb + L::oV, sQ = sb + L::oQ, sdO = sb + L::odO,
                 sL = sb + L::oL, sDl = sb + L::oDl, bar = sb + L::oBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::oBar + kKAbortSlot);
  const volatile uint32_t *gst = p.status;
  if ((*gst & 3u) || stale_rope_table(p)) return;
  if (pad + L::kUsed > L::kAlloc) {  // uniform over the block: nobody has touched a barrier yet
    if (threadIdx.x == 0) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_SMEM_ALIGN);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kt_all = (p.S + 127) / 128;
  const dev::HeadTile ht = dev::grouped_order((int)blockIdx.x, p.head_n, n_kt_all, p.group_kv);
  const int n = ht.rank;  // key tile; low tiles have the most work
  const int hid = p.head0 + ht.head;
  const int kl = hid % p.kvp, rb = hid / p.kvp;
  const int n_qt = (p.S + 127) / 128;
  const int m0 = p.causal ? n : 0;
  const int n_m = n_qt - m0;
  const int n_iter = p.group * n_m;

  if (threadIdx.x == 0) {
    mbar_init(bar + kKBarIn, 1);
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(bar + kKBarQFull + 8 * i, 1);
      mbar_init(bar + kKBarQEmpty + 8 * i, 1);
    }
    for (int i = 0; i < kOSlots; ++i) {
      mbar_init(bar + kKBarOFull + 8 * i, 1);
      mbar_init(bar + kKBarOEmpty + 8 * i, 1);
    }
    mbar_init(bar + kKBarSFull, 1);
    mbar_init(bar + kKBarDPFull, 1);
    mbar_init(bar + kKBarPFull, 256);
    mbar_init(bar + kKBarDSFull, 256);
    mbar_init(bar + kKBarAcc, 1);
    mbar_init(bar + kKBarDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kKTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::oBar + kKTmemSlot);
  const uint32_t tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp >= 8) {
    if (warp == kTmaWarp) {
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmQ);
        mbar_arrive_expect_tx(bar + kKBarIn, 2 * L::kT);
        const ActCoord kc = act_coord(p, rb, kl, p.kvp, n * 128, p.kv_rep);
        for (int c = 0; c < kCh; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, bar + kKBarIn, c * 64, kc.head, kc.row, kc.outer);
          tma_load_4d(sV + c * 16384, &tmV, bar + kKBarIn, c * 64, kc.head, kc.row, kc.outer);
        }
        int issued_q = -1, issued_o = -1;
        for (int i = 0; i < n_iter; ++i) {
          const int qs = i % kQSlots, os = i % kOSlots;
          const int gi = i / n_m, m = m0 + i % n_m, j = kl * p.group + gi;
          // the delta / nlse rows are in head layout in either mode
          const int mrow = m * 128 % p.Cs, mo = hl_outer(p, rb, m * 128);
          const ActCoord qc = act_coord(p, rb, j, p.hp, m * 128, 1);
          if (!mbar_wait_bounded(bar + kKBarQEmpty + 8 * qs, ((i / kQSlots) & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kKBarQFull + 8 * qs, L::kT + 512);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sQ + qs * L::kT + c * 16384, &tmQ, bar + kKBarQFull + 8 * qs, c * 64, qc.head, qc.row,
                        qc.outer);
          dev::tma_load_2d(sDl + qs * 512, &tmDl, bar + kKBarQFull + 8 * qs, mrow, mo * p.hp + j);
          issued_q = i;
          if (!mbar_wait_bounded(bar + kKBarOEmpty + 8 * os, ((i / kOSlots) & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kKBarOFull + 8 * os, L::kT + 512);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sdO + os * L::kT + c * 16384, &tmdO, bar + kKBarOFull + 8 * os, c * 64, qc.head, qc.row,
                        qc.outer);
          dev::tma_load_2d(sL + os * 512, &tmL, bar + kKBarOFull + 8 * os, mrow, mo * p.hp + j);
          issued_o = i;
        }
        if (*abort_flag) {
          volatile int never = 0;
          mbar_wait_bounded(bar + kKBarIn, 0, &never, nullptr, 500000000ull);
          for (int i = issued_q - (kQSlots - 1); i <= issued_q; ++i)
            if (i >= 0)
              mbar_wait_bounded(bar + kKBarQFull + 8 * (i % kQSlots), (i / kQSlots) & 1, &never, nullptr,
                                500000000ull);
          for (int i = issued_o - (kOSlots - 1); i <= issued_o; ++i)
            if (i >= 0)
              mbar_wait_bounded(bar + kKBarOFull + 8 * (i % kOSlots), (i / kOSlots) & 1, &never, nullptr,
                                500000000ull);
        }
      }
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: both operands K-major
        constexpr uint32_t idA = idesc_bf16_f32(128, D, 0, 1);    // dV, dK: B (dO, Q) MN-major
        auto q_ready = [&](int i) -> bool {
          return mbar_wait_bounded(bar + kKBarQFull + 8 * (i % kQSlots), (i / kQSlots) & 1, abort_flag, gst);
        };
        auto o_ready = [&](int i) -> bool {
          return mbar_wait_bounded(bar + kKBarOFull + 8 * (i % kOSlots), (i / kOSlots) & 1, abort_flag, gst);
        };
        // S^T(i) = K Q_i^T (Q tile i has landed: the caller waited).
        auto issue_s = [&](int i) {
          const int qs = i % kQSlots;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem, smem_desc_sw128(sK + o, 16, 1024),
                        smem_desc_sw128(sQ + qs * L::kT + o, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kKBarSFull);
        };
        // dP^T(i) = V dO_i^T (dO tile i has landed: the caller waited).
        auto issue_dp = [&](int i) {
          const int os = i % kOSlots;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + 128, smem_desc_sw128(sV + o, 16, 1024),
                        smem_desc_sw128(sdO + os * L::kT + o, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kKBarDPFull);
        };
        // Q tile 1 as well: the burst dV(0) S^T(1) follows the P phase of step 0,
        // and later Q tiles are vouched for by the softmax's arrivals.
        bool ok = mbar_wait_bounded(bar + kKBarIn, 0, abort_flag, gst) && q_ready(0) && o_ready(0) &&
                  (n_iter < 2 || q_ready(1));
        if (ok && n_iter > 0) {
          tc_fence_after_sync();
          issue_s(0);
          issue_dp(0);
        }
        for (int i = 0; ok && i < n_iter; ++i) {
          const int qs = i % kQSlots, os = i % kOSlots;
          // burst 1: dV(i), S^T(i+1).  P^T / dS^T: queries 16kk..16kk+15 are
          // columns 8kk.. of warpgroup 0's half (kk < 4) or of warpgroup 1's
          // half at +64 (kk >= 4).
          if (!(ok = mbar_wait_bounded(bar + kKBarPFull, i & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = (kk < 4 ? 0u : 64u) + (uint32_t)(kk & 3) * 8;
            mma_bf16_ts(tdV, tmem + ac, smem_desc_sw128(sdO + os * L::kT + kk * 2048, 16384, 1024), idA,
                        (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar + kKBarOEmpty + 8 * os);
          if (i + 1 < n_iter) issue_s(i + 1);
          // burst 2: dK(i), dP^T(i+1)
          if (!(ok = mbar_wait_bounded(bar + kKBarDSFull, i & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = (kk < 4 ? 0u : 64u) + (uint32_t)(kk & 3) * 8;
            mma_bf16_ts(tdK, tmem + 128 + ac, smem_desc_sw128(sQ + qs * L::kT + kk * 2048, 16384, 1024), idA,
                        (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar + kKBarQEmpty + 8 * qs);
          if (i + 1 < n_iter) issue_dp(i + 1);
        }
        mma_commit(bar + kKBarAcc);
        mma_commit(bar + kKBarDrain);
        volatile int never = 0;
        mbar_wait_bounded(bar + kKBarDrain, 0, &never, nullptr);
      }
    }
  } else {
    // ---------------------------------------------- softmax warpgroups
    const int g = warp >> 2, w4 = warp & 3;
    const int r = w4 * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const int kvr = n * 128 + r;
    // dK's epilogue undoes the rotation of key row kvr: pairs [g*32, g*32+32)
    // (warpgroup 0 alone for D = 64)
    const bool rot = p.rope_cos && p.kv_rep == 1 && (D == 128 || g == 0) && kvr < p.S &&
                     in_range(p.status, (long long)kvr * (D / 2), D / 2, p.rope_n);
    const float *rcs = rot ? p.rope_cos + (size_t)kvr * (D / 2) + g * 32 : nullptr;
    const float *rsn = rot ? p.rope_sin + (size_t)kvr * (D / 2) + g * 32 : nullptr;
    if (rot) rope_prefetch(rcs, rsn);
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const int qs = i % kQSlots, os = i % kOSlots;
      if (!warp_wait(bar + kKBarSFull, i & 1, abort_flag, gst)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t sr[2][32];
      tmem_ld32(tmem + lane_base + g * 64, sr[0]);
      tmem_ld32(tmem + lane_base + g * 64 + 32, sr[1]);
      // This step's LSE rides in its dO slot; after step 0 these threads
      // waited for that slot at the end of the previous step.
      if (i == 0 && !warp_wait(bar + kKBarOFull, 0, abort_flag, gst)) { ok = false; break; }
      tmem_wait_ld();
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      const int q0 = (m0 + i % n_m) * 128 + g * 64;
      // Query q0 + c sees key kvr iff q0 + c >= kvr (causal) and q0 + c < S:
      // columns [lo, hi) of this warpgroup's 64 are valid.
      const int lo = p.causal ? kvr - q0 : 0, hi = p.S - q0;
      const float2 *nl2 = reinterpret_cast<const float2 *>(smem + L::oL + os * 512) + g * 32;
      const float2 *dl2 = reinterpret_cast<const float2 *>(smem + L::oDl + qs * 512) + g * 32;
      float2 pf[32];  // P of this thread's 64 columns, kept for dS
      uint32_t w[2][16];
      if (__all_sync(0xffffffffu, lo <= 0 && hi >= 64))
        p_columns<false>(sr, nl2, p.scale_log2, lo, hi, pf, w);
      else
        p_columns<true>(sr, nl2, p.scale_log2, lo, hi, pf, w);
      tmem_st16(tmem + lane_base + g * 64, w[0]);
      tmem_st16(tmem + lane_base + g * 64 + 16, w[1]);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar + kKBarPFull);

      if (!warp_wait(bar + kKBarDPFull, i & 1, abort_flag, gst)) { ok = false; break; }
      // ... and its delta in its Q slot, which these threads waited for at the
      // end of step i-2 (steps 0 and 1: here).
      if (i < 2 && !warp_wait(bar + kKBarQFull + 8 * qs, 0, abort_flag, gst)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t dr[2][32];
      tmem_ld32(tmem + lane_base + 128 + g * 64, dr[0]);
      tmem_ld32(tmem + lane_base + 128 + g * 64 + 32, dr[1]);
      tmem_wait_ld();
      reg_fence(dr[0]);
      reg_fence(dr[1]);
      ds_columns(dr, dl2, pf, w);
      tmem_st16(tmem + lane_base + 128 + g * 64, w[0]);
      tmem_st16(tmem + lane_base + 128 + g * 64 + 16, w[1]);
      tmem_wait_st();
      tc_fence_before_sync();
      // The issuer waits for this arrival alone before dK(i) dP^T(i+1) and
      // (as the last wait before it) dV(i+1) S^T(i+2), so it also vouches for
      // dO tile i+1 and Q tile i+2 having landed.  Waiting here, a step ahead
      // of S^T(i+2), keeps these waits off the softmax's P phase, which the
      // tensor core waits for.
      if (i + 1 < n_iter &&
          !warp_wait(bar + kKBarOFull + 8 * ((i + 1) % kOSlots), ((i + 1) / kOSlots) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      if (i + 2 < n_iter &&
          !warp_wait(bar + kKBarQFull + 8 * ((i + 2) % kQSlots), ((i + 2) / kQSlots) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      mbar_arrive(bar + kKBarDSFull);
      if (p.ds) {
        // dS-store mode: this row's 64 dS values (queries 64g..) into the tile of
        // (q-head, query tile, key tile n), as four 16-query chunks (see ds_tile);
        // issued after the arrival that releases dK(i), they drain while these
        // threads wait for the next scores
        const int gi = i / n_m, j = kl * p.group + gi;
        const long long e = ds_tile(p, rb * p.hp + j, m0 + i % n_m, n) * 16384 + (g * 4 * 128 + r) * 16;
        if (in_range(p.status, e, 3 * 2048 + 16, p.ds_pairs * 16384LL * p.head_n * p.group)) {
          const bool sw = (r >> 2) & 1;  // the halves' swap: words 4..7 first
          uint32_t x[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = sw ? w[k >> 4][(k & 15) ^ 4] : w[k >> 4][k & 15];
          store_ds_row(p.ds + e, x);
        }
      }
    }
    // ------------------------------------------------------------ epilogue
    RopeRow angles;
    if (ok && rot) rope_load(angles, rcs, rsn);
    if (ok) ok = warp_wait(bar + kKBarAcc, 0, abort_flag, gst);
    if (ok && p.kv_rep > 1) {
      // Replicated kv-head: this rank's q-heads give only part of dK, dV; the
      // raw fp32 accumulators go to the per-rank partial buffers and the sum
      // over the replicas (with scale and inverse rotation) follows.
      tc_fence_after_sync();
      const bool live = kvr < p.S;
      // partials [P*B][Cs][D]: the row of key kvr in this member's head layout
      const int kr = live ? kvr : 0;
      const size_t prow = (size_t)hl_outer(p, rb, kr) * p.Cs + kr % p.Cs;
      float *pv = reinterpret_cast<float *>(p.dv) + prow * D;
      float *pk = reinterpret_cast<float *>(p.dk) + prow * D;
      const bool put = live && in_range(p.status, (long long)(prow * D), D, p.dkv_n);
      // warpgroup g owns columns [g*D/2, (g+1)*D/2) of both accumulators; the
      // TMEM loads are warp-wide, only the stores depend on the row
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t x[32], y[32];
        tmem_ld32(tdV + lane_base + col, x);
        tmem_ld32(tdK + lane_base + col, y);
        tmem_wait_ld();
        if (put) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            reinterpret_cast<uint4 *>(pv + col)[v] = make_uint4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
            reinterpret_cast<uint4 *>(pk + col)[v] = make_uint4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
          }
        }
      }
    } else if (ok) {
      tc_fence_after_sync();
      const bool live = kvr < p.S;
      const int s_rank = kvr / p.Sl, t = kvr - s_rank * p.Sl;
      const int rr = rb / p.B, bb = rb - rr * p.B;
      const size_t row = (((size_t)(s_rank * p.B + bb) * p.Sl + t) * p.n_kv + (rr * p.kvp + kl)) * D;
      const bool put = live && in_range(p.status, (long long)row, D, p.dkv_n) &&
                       (!p.rope_cos || in_range(p.status, (long long)kvr * (D / 2), D / 2, p.rope_n));
      // dV: warpgroup g owns columns [g*D/2, (g+1)*D/2)
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t x[32];
        const int col = g * (D / 2) + c * 32;
        tmem_ld32(tdV + lane_base + col, x);
        tmem_wait_ld();
        if (put) store_plain(p.dv + row + col, x, 1.0f);
      }
      // dK: rotation pairs (i, i + D/2); warpgroup g owns i in [g*32, g*32+32)
      // for D = 128, warpgroup 0 owns all 32 pairs for D = 64.
      if (D == 128 || g == 0) {
        const int i0 = g * 32;
        uint32_t x[32], y[32];
        tmem_ld32(tdK + lane_base + i0, x);
        tmem_ld32(tdK + lane_base + D / 2 + i0, y);
        tmem_wait_ld();
        if (put) store_unrotated(p.dk + row + i0, p.dk + row + D / 2 + i0, x, y, p.scale, rot, angles);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_BWD_TIMEOUT);
}

// ================================================================== dQ kernel
// 128-key tiles, every MMA 128x128x16.  Q and dO are the same for the whole
// loop, so the softmax warps copy them once into TMEM (bf16, two per column),
// where S = Q K^T and dP = dO V^T read them as their A operand: the shared
// memory port then carries only the K and V tiles.  TMEM: S [0,128),
// dP [128,256), dQ [256, 256+D), Q [384, 384+D/2), dO [448, 448+D/2).
// Warpgroup g owns key columns [64g, 64g+64) of S and dP; it writes dS (bf16,
// two per column) over the first half of its dP columns ([128+64g, 160+64g)),
// where the dQ MMA reads it as its A operand.
// The softmax runs in two phases per tile: it loads S_i and releases it at
// once (P_i stays in registers), then waits for dP_i and forms dS_i.  The
// tensor core runs S_{i+1}, dQ_i, dP_{i+1}, ...: S_{i+1} overlaps the P phase
// of tile i+1's predecessor, dP_{i+1} overwrites dS_i only after dQ_i has read
// it (one issuer's MMAs run in order).
// K tiles stream through a 3-slot ring (released after the dQ MMA), V tiles
// through a 3-slot ring (released after the dP MMA).
constexpr int kThreadsQ = 384;  // warpgroups 0-1 softmax, warpgroup 2: TMA, MMA, 2 idle warps
constexpr uint32_t kRegsQProducer = 72, kRegsQSoftmax = 216;
static_assert(128 * kRegsQProducer + 256 * kRegsQSoftmax <= 384 * 168, "register split over budget");
constexpr int kKSlots = 3, kVSlots = 3;

enum : uint32_t {
  kQBarQReady = 0,                         // 256 arrivals: Q and dO are in TMEM
  kQBarKFull = 8,                          // [kKSlots]
  kQBarKEmpty = kQBarKFull + 8 * kKSlots,  // [kKSlots]
  kQBarVFull = kQBarKEmpty + 8 * kKSlots,  // [kVSlots]
  kQBarVEmpty = kQBarVFull + 8 * kVSlots,  // [kVSlots]
  kQBarSFull = kQBarVEmpty + 8 * kVSlots,
  kQBarSFree = kQBarSFull + 8,             // 256 arrivals
  kQBarDPFull = kQBarSFree + 8,
  kQBarDSFull = kQBarDPFull + 8,           // 256 arrivals
  kQBarAcc = kQBarDSFull + 8,
  kQBarDrain = kQBarAcc + 8,
  kQTmemSlot = kQBarDrain + 8,
  kQAbortSlot = kQTmemSlot + 4
};
static_assert(kQAbortSlot + 4 <= 256, "dQ barrier block");

template <int D>
struct QLayout {
  static constexpr uint32_t kT = 128u * D * 2;  // one 128-row tile of K or V
  static constexpr uint32_t oK = 0, oV = kKSlots * kT, oBar = oV + kVSlots * kT;
  static constexpr uint32_t kAlloc = oBar + 256 + 1024;
};

// P = exp2(scale*log2(e)*s - lse*log2(e)) for the 64 key columns of one query
// row a thread holds; with kMask, columns at or past hi are 0.
template <bool kMask>
__device__ __forceinline__ void p_row(const uint32_t (&s)[2][32], float sl, float nl, int hi, float2 (&pf)[32]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t *sh = s[c >> 4];
    const int e = 2 * (c & 15);
    const float2 x = fma2(make_float2(__uint_as_float(sh[e]), __uint_as_float(sh[e + 1])), make_float2(sl, sl),
                          make_float2(nl, nl));
    float2 pe = make_float2(ex2(x.x), ex2(x.y));
    if (kMask) {
      if (2 * c >= hi) pe.x = 0.f;
      if (2 * c + 1 >= hi) pe.y = 0.f;
    }
    pf[c] = pe;
  }
}

// dS = P * (dP - delta) for the same 64 columns, packed to bf16.
__device__ __forceinline__ void ds_row(const uint32_t (&d)[2][32], const float2 (&pf)[32], float dlt,
                                       uint32_t (&w)[2][16]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t *dh = d[c >> 4];
    const int e = 2 * (c & 15);
    const float2 y = sub2(make_float2(__uint_as_float(dh[e]), __uint_as_float(dh[e + 1])), make_float2(dlt, dlt));
    const float2 ds = mul2(pf[c], y);
    w[c >> 4][c & 15] = pack_bf16x2(ds.x, ds.y);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsQ, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const BwdParams p) {
  using L = QLayout<D>;
  constexpr int kCh = D / 64;
  constexpr uint32_t kColDP = 128, kColDQ = 256, kColQ = 384, kColDO = 448;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + L::oK, sV = sb + L::oV, bar = sb + L::oBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::oBar + kQAbortSlot);
  const volatile uint32_t *gst = p.status;
  if ((*gst & 3u) || stale_rope_table(p)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads_total = p.Pu * p.B * p.hp;
  const int n_qt = (p.S + 127) / 128;
  const dev::HeadTile ht = dev::grouped_order((int)blockIdx.x, heads_total, n_qt, p.group_q);
  const int m = n_qt - 1 - ht.rank;  // longest tiles first
  const int hid = ht.head;
  const int j = hid % p.hp, rb = hid / p.hp;
  const int kl = j / p.group;
  const int n_kt = (p.S + 127) / 128;
  const int n_kv = p.causal ? min(n_kt, m + 1) : n_kt;

  if (threadIdx.x == 0) {
    mbar_init(bar + kQBarQReady, 256);
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(bar + kQBarKFull + 8 * i, 1);
      mbar_init(bar + kQBarKEmpty + 8 * i, 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bar + kQBarVFull + 8 * i, 1);
      mbar_init(bar + kQBarVEmpty + 8 * i, 1);
    }
    mbar_init(bar + kQBarSFull, 1);
    mbar_init(bar + kQBarSFree, 256);
    mbar_init(bar + kQBarDPFull, 1);
    mbar_init(bar + kQBarDSFull, 256);
    mbar_init(bar + kQBarAcc, 1);
    mbar_init(bar + kQBarDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kQTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::oBar + kQTmemSlot);
  const uint32_t tdQ = tmem + kColDQ;

  if (warp >= 8) {
    regs_dec<kRegsQProducer>();
    if (warp == kTmaWarp) {
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        int issued_k = -1, issued_v = -1;
        for (int i = 0; i < n_kv; ++i) {
          const int ks = i % kKSlots, vs = i % kVSlots;
          if (!mbar_wait_bounded(bar + kQBarKEmpty + 8 * ks, ((i / kKSlots) & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kQBarKFull + 8 * ks, L::kT);
          const ActCoord kc = act_coord(p, rb, kl, p.kvp, i * 128, p.kv_rep);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sK + ks * L::kT + c * 16384, &tmK, bar + kQBarKFull + 8 * ks, c * 64, kc.head, kc.row,
                        kc.outer);
          issued_k = i;
          if (!mbar_wait_bounded(bar + kQBarVEmpty + 8 * vs, ((i / kVSlots) & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kQBarVFull + 8 * vs, L::kT);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sV + vs * L::kT + c * 16384, &tmV, bar + kQBarVFull + 8 * vs, c * 64, kc.head, kc.row,
                        kc.outer);
          issued_v = i;
        }
        if (*abort_flag) {
          volatile int never = 0;
          for (int i = issued_k - (kKSlots - 1); i <= issued_k; ++i)
            if (i >= 0)
              mbar_wait_bounded(bar + kQBarKFull + 8 * (i % kKSlots), (i / kKSlots) & 1, &never, nullptr,
                                500000000ull);
          for (int i = issued_v - (kVSlots - 1); i <= issued_v; ++i)
            if (i >= 0)
              mbar_wait_bounded(bar + kQBarVFull + 8 * (i % kVSlots), (i / kVSlots) & 1, &never, nullptr,
                                500000000ull);
        }
      }
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: A (TMEM) and K, V K-major
        constexpr uint32_t idQ = idesc_bf16_f32(128, D, 0, 1);    // dQ: B (K tile) MN-major
        auto k_ready = [&](int i) -> bool {
          return mbar_wait_bounded(bar + kQBarKFull + 8 * (i % kKSlots), (i / kKSlots) & 1, abort_flag, gst);
        };
        auto v_ready = [&](int i) -> bool {
          return mbar_wait_bounded(bar + kQBarVFull + 8 * (i % kVSlots), (i / kVSlots) & 1, abort_flag, gst);
        };
        // S_i = Q K_i^T (Q: D elements 16kk.. are TMEM columns kColQ + 8kk ..);
        // K_i has landed (the caller waited).
        auto issue_s = [&](int i) {
          const int ks = i % kKSlots;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ts(tmem, tmem + kColQ + kk * 8, smem_desc_sw128(sK + ks * L::kT + o, 16, 1024), idS,
                        kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kQBarSFull);
        };
        // dP_i = dO V_i^T (V_i has landed: the caller waited).
        auto issue_dp = [&](int i) {
          const int vs = i % kVSlots;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ts(tmem + kColDP, tmem + kColDO + kk * 8, smem_desc_sw128(sV + vs * L::kT + o, 16, 1024),
                        idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kQBarDPFull);
          mma_commit(bar + kQBarVEmpty + 8 * vs);
        };
        // One wait per burst (a thread with MMAs in flight stalls on its next
        // shared-memory access): the softmax's SFree and DSFull arrivals also
        // vouch for K tile i+1 and V tile i+1.
        bool ok = mbar_wait_bounded(bar + kQBarQReady, 0, abort_flag, gst) && (n_kv == 0 || (k_ready(0) && v_ready(0)));
        if (ok && n_kv > 0) {
          tc_fence_after_sync();
          issue_s(0);
          issue_dp(0);
        }
        for (int i = 0; ok && i < n_kv; ++i) {
          // burst 1: S_{i+1}, once the softmax has loaded S_i
          if (i + 1 < n_kv) {
            if (!(ok = mbar_wait_bounded(bar + kQBarSFree, i & 1, abort_flag, gst))) break;
            tc_fence_after_sync();
            issue_s(i + 1);
          }
          // burst 2: dQ += dS_i K_i, dP_{i+1}.  Keys 16kk.. of dS_i are columns
          // 8kk.. of warpgroup 0's half (kk < 4) or of warpgroup 1's half at +64.
          if (!(ok = mbar_wait_bounded(bar + kQBarDSFull, i & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
          const int ks = i % kKSlots;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = kColDP + (kk < 4 ? 0u : 64u) + (uint32_t)(kk & 3) * 8;
            mma_bf16_ts(tdQ, tmem + ac, smem_desc_sw128(sK + ks * L::kT + kk * 2048, 16384, 1024), idQ,
                        (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar + kQBarKEmpty + 8 * ks);
          if (i + 1 < n_kv) issue_dp(i + 1);
        }
        mma_commit(bar + kQBarAcc);
        mma_commit(bar + kQBarDrain);
        volatile int never = 0;
        mbar_wait_bounded(bar + kQBarDrain, 0, &never, nullptr);
      }
    }
  } else {
    regs_inc<kRegsQSoftmax>();
    // ---------------------------------------- softmax warpgroups: warpgroup g
    // owns key columns [64g, 64g+64) of every tile.
    const int g = warp >> 2, w4 = warp & 3;
    const int r = w4 * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const int qi = m * 128 + r;
    const bool live = qi < p.S;
    // dQ's epilogue undoes the rotation of query row qi: pairs [g*32, g*32+32)
    // (warpgroup 0 alone for D = 64)
    const bool rot = p.rope_cos && (D == 128 || g == 0) && live &&
                     in_range(p.status, (long long)qi * (D / 2), D / 2, p.rope_n);
    const float *rcs = rot ? p.rope_cos + (size_t)qi * (D / 2) + g * 32 : nullptr;
    const float *rsn = rot ? p.rope_sin + (size_t)qi * (D / 2) + g * 32 : nullptr;
    if (rot) rope_prefetch(rcs, rsn);
    {
      // Warpgroup 0 copies this thread's Q row, warpgroup 1 its dO row, into
      // TMEM (rows past S are zero).
      const int qr = live ? qi : 0;
      const size_t qoff = q_row_offset(p, rb, j, qr, D);
      const __nv_bfloat16 *src = (g == 0 ? p.q : p.dout) + qoff;
      const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
      const bool get = live && in_range(p.status, (long long)qoff, D, p.qo_n);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t x[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 u = get ? __ldg(s4 + c * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
          x[4 * v] = u.x;
          x[4 * v + 1] = u.y;
          x[4 * v + 2] = u.z;
          x[4 * v + 3] = u.w;
        }
        tmem_st32(tmem + lane_base + (g == 0 ? kColQ : kColDO) + c * 32, x);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar + kQBarQReady);
    }
    const int qr = live ? qi : 0;
    const size_t lrow = ((size_t)hl_outer(p, rb, qr) * p.hp + j) * p.Ld + qr % p.Cs;
    const bool get_row = live && in_range(p.status, (long long)lrow, 1, p.rows_n);
    const float nl2 = get_row ? p.nlse[lrow] : 0.f;
    const float dlt = get_row ? p.delta[lrow] : 0.f;
    bool ok = true;
    for (int i = 0; i < n_kv; ++i) {
      if (!warp_wait(bar + kQBarSFull, i & 1, abort_flag, gst)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t sr[2][32];
      tmem_ld32(tmem + lane_base + g * 64, sr[0]);
      tmem_ld32(tmem + lane_base + g * 64 + 32, sr[1]);
      tmem_wait_ld();
      tc_fence_before_sync();
      // The issuer waits for this arrival alone before S_{i+1}, so it also
      // vouches for K tile i+1 having landed.
      if (i + 1 < n_kv &&
          !warp_wait(bar + kQBarKFull + 8 * ((i + 1) % kKSlots), ((i + 1) / kKSlots) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      mbar_arrive(bar + kQBarSFree);
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      const int k0 = i * 128 + g * 64;
      // Key k0 + c is seen by query qi iff k0 + c <= qi (causal) and k0 + c < S:
      // columns [0, hi) of this warpgroup's 64 are valid.
      const int hi = min(p.causal ? qi - k0 + 1 : 64, p.S - k0);
      float2 pf[32];
      if (__all_sync(0xffffffffu, hi >= 64))
        p_row<false>(sr, p.scale_log2, nl2, hi, pf);
      else
        p_row<true>(sr, p.scale_log2, nl2, hi, pf);

      if (!warp_wait(bar + kQBarDPFull, i & 1, abort_flag, gst)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t dr[2][32];
      tmem_ld32(tmem + lane_base + kColDP + g * 64, dr[0]);
      tmem_ld32(tmem + lane_base + kColDP + g * 64 + 32, dr[1]);
      tmem_wait_ld();
      reg_fence(dr[0]);
      reg_fence(dr[1]);
      uint32_t wd[2][16];
      ds_row(dr, pf, dlt, wd);
      tmem_st16(tmem + lane_base + kColDP + g * 64, wd[0]);
      tmem_st16(tmem + lane_base + kColDP + g * 64 + 16, wd[1]);
      tmem_wait_st();
      tc_fence_before_sync();
      // ... and this one alone before dQ(i) and dP_{i+1}: V tile i+1 too.
      if (i + 1 < n_kv &&
          !warp_wait(bar + kQBarVFull + 8 * ((i + 1) % kVSlots), ((i + 1) / kVSlots) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      mbar_arrive(bar + kQBarDSFull);
    }
    RopeRow angles;
    if (ok && rot) rope_load(angles, rcs, rsn);
    if (ok) ok = warp_wait(bar + kQBarAcc, 0, abort_flag, gst);
    if (ok && (D == 128 || g == 0)) {
      tc_fence_after_sync();
      const int s_rank = qi / p.Sl, t = qi - s_rank * p.Sl;
      const int rr = rb / p.B, bb = rb - rr * p.B;
      const size_t row = (((size_t)(s_rank * p.B + bb) * p.Sl + t) * p.n_head + (rr * p.hp + j)) * D;
      const int i0 = g * 32;
      uint32_t x[32], y[32];
      tmem_ld32(tdQ + lane_base + i0, x);
      tmem_ld32(tdQ + lane_base + D / 2 + i0, y);
      tmem_wait_ld();
      if (live && in_range(p.status, (long long)row, D, p.dq_n) &&
          (!p.rope_cos || in_range(p.status, (long long)qi * (D / 2), D / 2, p.rope_n)))
        store_unrotated(p.dq + row + i0, p.dq + row + D / 2 + i0, x, y, p.scale, rot, angles);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_BWD_TIMEOUT);
}

// ======================================================= fused dK / dV / dQ kernel
// The dK/dV kernel's loop with dQ added to it: besides dV += P^T dO and
// dK += dS^T Q, every step also forms its query tile's dQ share dS K (the
// step's 128 keys' part of dQ) and adds it into a float accumulator in the
// workspace with the copy engine's reduce-add (cp.reduce.async.bulk.tensor
// .add): five products per (key tile, query tile) pair instead of the seven
// the two-kernel backward executes (which recomputes S and dP for dQ).  The
// float additions of one dQ row arrive from several CTAs in an order that
// varies from run to run, so dQ is reproducible only to float rounding; dK
// and dV are accumulated exactly as the dK/dV kernel does (bit-identical).
//
// TMEM: S^T [0,128) with P^T (bf16) over the first half of each softmax
// warpgroup's columns; dP^T [128,256) with dS^T (bf16) likewise, and after
// the dK MMA has read it the step's dQ share [128, 128+D) (query rows as
// lanes); dV [256, 256+D), dK [256+D, 256+2D).
// Shared memory: K, V resident; Q in a 2-slot ring (its delta and -LSE*log2e
// rows ride in the slot), dO in one slot; dS (bf16, [key][query] in two
// 128-byte-swizzled 64-query chunks: the MN-major A operand of dQ = dS K); a
// float staging area X for half of a dQ share's columns.  A warpgroup of its
// own drains each dQ share: TMEM into registers (which frees the TMEM for the
// next dP), then columns [D/2, D) through the dS area (free once the dQ MMA
// has read it, until the next dS) and [0, D/2) through X, one reduce-add per
// [128 x 32] box.  The copy engine's reduce-adds run at the L2's pace (about
// 6 TB/s over the whole chip).
// Warps: 0-7 softmax (two warpgroups, each half of a step's 128 queries),
// 8-11 dQ drain, 12 TMA producer, 13 MMA issuer, 14-15 idle; registers split
// 160 / 144 / 48 per thread by warpgroup.
// Tensor-core order, one wait per burst:
//   prologue   S(0) dP(0) | PFull(0): dV(0)
//   step i     DSFull(i): S(i+1) dK(i) dQ(i)  | XGo(i): dP(i+1) dV(i+1)
// XGo(i) is arrived by the softmax warps after P(i+1) and by the drain warps
// once dQ(i) is out of TMEM and dO tile i+1 has landed, so it vouches for
// everything dP(i+1) and dV(i+1) use; DSFull(i) after Q tile i+1 has landed.
// What bounds it (measured at the pages' sizing, clock64 traces of one CTA): a
// step takes ~5,500 cycles against 2,560 of tensor-core work.  Its chain is
// DSFull -> S dK dQ (24 MMAs, ~1,970) -> dQ out of TMEM -> dP -> dS phase ->
// DSFull, with every other phase hidden behind it; the dS phase waits for the
// reduce-adds to read the dS area back, because each step's dQ share (64 KB of
// floats) leaves at the L2's reduce rate, ~20 bytes per SM-cycle, ~3,200
// cycles per step.  Shared memory carries ~480 KB per step (the SS products
// read 64 KB each, the staging writes and reads 128 KB), close to its 128
// bytes per cycle over a step.  The five products per pair then take about as
// long as the two-kernel backward's seven.
constexpr int kFQSlots = 2;
constexpr int kThreadsF = 512;
constexpr int kFTmaWarp = 12, kFMmaWarp = 13;
constexpr uint32_t kRegsFSoftmax = 160, kRegsFDrain = 144, kRegsFProducer = 48;
static_assert(128 * (2 * kRegsFSoftmax + kRegsFDrain + kRegsFProducer) <= 65536, "register split over budget");

enum : uint32_t {
  kFBarIn = 0,
  kFBarQFull = 8,     // [2]
  kFBarQEmpty = 24,   // [2]
  kFBarOFull = 40,
  kFBarOEmpty = 48,
  kFBarSFull = 56,
  kFBarDPFull = 64,
  kFBarPFull = 72,    // 256 arrivals (step 0 only)
  kFBarDSFull = 80,   // 256 arrivals
  kFBarDQFull = 88,
  kFBarXGo = 96,      // 384 arrivals: softmax after P(i+1), drain after dQ(i) left TMEM
  kFBarStage = 104,   // 128 arrivals: the drain warps have staged a half of dQ(i)
  kFBarBufFree = 112, // 1 arrival: the reduce-adds of dQ(i) have read the dS area
  kFBarXFree = 120,   // 1 arrival: ... and X
  kFBarAcc = 128,
  kFBarDrain = 136,
  kFTmemSlot = 144,
  kFAbortSlot = 148,
  kFBarBytes = 152
};

template <int D>
struct FLayout {
  static constexpr uint32_t kT = 128u * D * 2;        // one 128-row tile of K, V, Q or dO
  static constexpr uint32_t kDS = 128u * 128u * 2;    // dS: 128 keys x 128 queries, bf16
  static constexpr uint32_t kStage = 128u * (D / 2) * 4;  // half of a dQ share's columns, float
  static constexpr uint32_t oK = 0, oV = kT, oQ = 2 * kT, odO = oQ + kFQSlots * kT, oDS = odO + kT,
                            oX = oDS + kDS,
                            oRows = oX + kStage,  // per Q slot: delta row, then -LSE*log2(e) row
                            oBar = oRows + kFQSlots * 1024;
  static constexpr uint32_t kUsed = oBar + kFBarBytes;
  static constexpr uint32_t kAlloc = kUsed + 1024 <= kMaxDynSmem ? kUsed + 1024 : kMaxDynSmem;
  static_assert(kUsed <= kMaxDynSmem, "fused backward tiles exceed shared memory");
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Reduce-add of a float box in shared memory into the global tensor of `m`
// at (c0, c1), tracked by this thread's bulk async-groups.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *m, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// D/2 floats of a thread's row (`x`) into a staging area: D/64 boxes of
// [128 rows][32 floats], 128-byte swizzled (the 16-byte unit c of row r at
// unit c ^ (r % 8)), so the 8 rows a quarter-warp writes land in distinct
// banks; the reduce-add's tensor map has the same swizzle.
template <int D>
__device__ __forceinline__ void stage_half(uint8_t *area, int r, const uint32_t *x) {
#pragma unroll
  for (int b = 0; b < D / 64; ++b) {
    uint8_t *row = area + b * 16384 + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) * 16)) =
          make_uint4(x[32 * b + 4 * c], x[32 * b + 4 * c + 1], x[32 * b + 4 * c + 2], x[32 * b + 4 * c + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsF, 1)
    dkdvq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                 const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmDl,
                 const __grid_constant__ CUtensorMap tmAcc, const BwdParams p) {
  using L = FLayout<D>;
  constexpr int kCh = D / 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + L::oK, sV = sb + L::oV, sQ = sb + L::oQ, sdO = sb + L::odO, sDS = sb + L::oDS,
                 sX = sb + L::oX, sRows = sb + L::oRows, bar = sb + L::oBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::oBar + kFAbortSlot);
  const volatile uint32_t *gst = p.status;
  if ((*gst & 3u) || stale_rope_table(p)) return;
  if (pad + L::kUsed > L::kAlloc) {  // uniform over the block: nobody has touched a barrier yet
    if (threadIdx.x == 0) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_SMEM_ALIGN);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads_total = p.Pu * p.B * p.kvp;
  const int n_kt_all = (p.S + 127) / 128;
  const dev::HeadTile ht = dev::grouped_order((int)blockIdx.x, heads_total, n_kt_all, p.group_kv);
  const int n = ht.rank;  // key tile; low tiles have the most work
  const int hid = ht.head;
  const int kl = hid % p.kvp, rb = hid / p.kvp;
  const int n_qt = (p.S + 127) / 128;
  const int m0 = p.causal ? n : 0;
  const int n_m = n_qt - m0;
  const int n_iter = p.group * n_m;

  if (threadIdx.x == 0) {
    mbar_init(bar + kFBarIn, 1);
    for (int i = 0; i < kFQSlots; ++i) {
      mbar_init(bar + kFBarQFull + 8 * i, 1);
      mbar_init(bar + kFBarQEmpty + 8 * i, 1);
    }
    mbar_init(bar + kFBarOFull, 1);
    mbar_init(bar + kFBarOEmpty, 1);
    mbar_init(bar + kFBarSFull, 1);
    mbar_init(bar + kFBarDPFull, 1);
    mbar_init(bar + kFBarPFull, 256);
    mbar_init(bar + kFBarDSFull, 256);
    mbar_init(bar + kFBarDQFull, 1);
    mbar_init(bar + kFBarXGo, 384);
    mbar_init(bar + kFBarStage, 128);
    mbar_init(bar + kFBarBufFree, 1);
    mbar_init(bar + kFBarXFree, 1);
    mbar_init(bar + kFBarAcc, 1);
    mbar_init(bar + kFBarDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kFMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kFTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::oBar + kFTmemSlot);
  const uint32_t tdQ = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp >= 12) {
    regs_dec<kRegsFProducer>();
    if (warp == kFTmaWarp) {
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmQ);
        mbar_arrive_expect_tx(bar + kFBarIn, 2 * L::kT);
        const ActCoord kc = act_coord(p, rb, kl, p.kvp, n * 128, p.kv_rep);
        for (int c = 0; c < kCh; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, bar + kFBarIn, c * 64, kc.head, kc.row, kc.outer);
          tma_load_4d(sV + c * 16384, &tmV, bar + kFBarIn, c * 64, kc.head, kc.row, kc.outer);
        }
        // Loads in the order the slots free up: dO(i) after dV(i-1), Q(i) after dK(i-2).
        int issued_q = -1, issued_o = -1;
        for (int i = 0; i < n_iter; ++i) {
          const int qs = i % kFQSlots;
          const int gi = i / n_m, m = m0 + i % n_m, j = kl * p.group + gi;
          // the delta / nlse rows are in head layout in either mode
          const int mrow = m * 128 % p.Cs, mo = hl_outer(p, rb, m * 128);
          const ActCoord qc = act_coord(p, rb, j, p.hp, m * 128, 1);
          if (!mbar_wait_bounded(bar + kFBarQEmpty + 8 * qs, ((i / kFQSlots) & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kFBarQFull + 8 * qs, L::kT + 1024);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sQ + qs * L::kT + c * 16384, &tmQ, bar + kFBarQFull + 8 * qs, c * 64, qc.head, qc.row,
                        qc.outer);
          dev::tma_load_2d(sRows + qs * 1024, &tmDl, bar + kFBarQFull + 8 * qs, mrow, mo * p.hp + j);
          dev::tma_load_2d(sRows + qs * 1024 + 512, &tmL, bar + kFBarQFull + 8 * qs, mrow, mo * p.hp + j);
          issued_q = i;
          if (!mbar_wait_bounded(bar + kFBarOEmpty, (i & 1) ^ 1, abort_flag, gst)) break;
          mbar_arrive_expect_tx(bar + kFBarOFull, L::kT);
          for (int c = 0; c < kCh; ++c)
            tma_load_4d(sdO + c * 16384, &tmdO, bar + kFBarOFull, c * 64, qc.head, qc.row, qc.outer);
          issued_o = i;
        }
        if (*abort_flag) {
          volatile int never = 0;
          mbar_wait_bounded(bar + kFBarIn, 0, &never, nullptr, 500000000ull);
          for (int i = issued_q - (kFQSlots - 1); i <= issued_q; ++i)
            if (i >= 0)
              mbar_wait_bounded(bar + kFBarQFull + 8 * (i % kFQSlots), (i / kFQSlots) & 1, &never, nullptr,
                                500000000ull);
          if (issued_o >= 0) mbar_wait_bounded(bar + kFBarOFull, issued_o & 1, &never, nullptr, 500000000ull);
        }
      }
    } else if (warp == kFMmaWarp) {
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: both operands K-major
        constexpr uint32_t idA = idesc_bf16_f32(128, D, 0, 1);    // dV, dK: B (dO, Q) MN-major
        constexpr uint32_t idQ = idesc_bf16_f32(128, D, 1, 1);    // dQ: A (dS) and B (K) MN-major
        const uint32_t sK_ = sK, sV_ = sV, sQ_ = sQ, sdO_ = sdO, sDS_ = sDS;
        // The shared-memory bases pass through an empty asm in each helper, so
        // the descriptors are formed when a burst is issued instead of all
        // being held in registers across the loop (this warpgroup runs on 48).
        auto opaque = [](uint32_t v) {
          asm volatile("" : "+r"(v));
          return v;
        };
        // S^T(i) = K Q_i^T.
        auto issue_s = [&](int i) {
          const int qs = i % kFQSlots;
          const uint32_t sK = opaque(sK_), sQ = opaque(sQ_);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem, smem_desc_sw128(sK + o, 16, 1024), smem_desc_sw128(sQ + qs * L::kT + o, 16, 1024),
                        idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kFBarSFull);
        };
        // dP^T(i) = V dO_i^T.
        auto issue_dp = [&]() {
          const uint32_t sV = opaque(sV_), sdO = opaque(sdO_);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + 128, smem_desc_sw128(sV + o, 16, 1024), smem_desc_sw128(sdO + o, 16, 1024), idS,
                        kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kFBarDPFull);
        };
        // dV += P^T(i) dO_i (P^T from TMEM: queries 16kk.. are columns 8kk.. of
        // warpgroup 0's half (kk < 4) or of warpgroup 1's half at +64); releases dO.
        auto issue_dv = [&](int i) {
          const uint32_t sdO = opaque(sdO_);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = (kk < 4 ? 0u : 64u) + (uint32_t)(kk & 3) * 8;
            mma_bf16_ts(tdV, tmem + ac, smem_desc_sw128(sdO + kk * 2048, 16384, 1024), idA,
                        (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar + kFBarOEmpty);
        };
        // The two waits of each step are on the critical path and usually not
        // yet complete when reached, so the issuer polls them (a suspended
        // try_wait resumed ~500 cycles after the phase completed); the softmax
        // warps keep sleeping waits (polling there cost more issue slots than
        // it saved).
        bool ok = mbar_wait_bounded(bar + kFBarIn, 0, abort_flag, gst) &&
                  mbar_wait_bounded(bar + kFBarQFull, 0, abort_flag, gst) &&
                  mbar_wait_bounded(bar + kFBarOFull, 0, abort_flag, gst);
        if (ok) {
          tc_fence_after_sync();
          issue_s(0);
          issue_dp();
          if ((ok = mbar_wait_bounded(bar + kFBarPFull, 0, abort_flag, gst))) {
            tc_fence_after_sync();
            issue_dv(0);
          }
        }
        for (int i = 0; ok && i < n_iter; ++i) {
          const int qs = i % kFQSlots;
          // burst 1: S^T(i+1), dK(i), dQ(i)
          if (!(ok = mbar_wait_spin_bounded(bar + kFBarDSFull, i & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
          if (i + 1 < n_iter) issue_s(i + 1);
          const uint32_t sQ = opaque(sQ_), sDS = opaque(sDS_), sK = opaque(sK_);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = (kk < 4 ? 0u : 64u) + (uint32_t)(kk & 3) * 8;
            mma_bf16_ts(tdK, tmem + 128 + ac, smem_desc_sw128(sQ + qs * L::kT + kk * 2048, 16384, 1024), idA,
                        (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar + kFBarQEmpty + 8 * qs);
          // dQ share = dS K over this tile's keys (16kk.. per MMA): A = dS [key][query]
          // (MN-major, two 64-query chunks), B = K [key][d] (MN-major, D/64 chunks)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tdQ, smem_desc_sw128(sDS + kk * 2048, 16384, 1024),
                        smem_desc_sw128(sK + kk * 2048, 16384, 1024), idQ, kk > 0 ? 1u : 0u);
          mma_commit(bar + kFBarDQFull);
          if (i + 1 >= n_iter) break;
          // burst 2: dP^T(i+1), dV(i+1), once dQ(i) is out of TMEM and P^T(i+1) is in
          if (!(ok = mbar_wait_spin_bounded(bar + kFBarXGo, i & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
          issue_dp();
          issue_dv(i + 1);
        }
        mma_commit(bar + kFBarAcc);
        mma_commit(bar + kFBarDrain);
        volatile int never = 0;
        mbar_wait_bounded(bar + kFBarDrain, 0, &never, nullptr);
      }
    }
  } else if (warp >= 8) {
    regs_inc<kRegsFDrain>();
    // ------------------------------------------------------- dQ drain warpgroup
    const int w4 = warp & 3;
    const int r = w4 * 32 + lane;  // query row of the dQ share == TMEM lane
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const bool elected = w4 == 0 && lane == 0;  // issues the reduce-adds
    for (int i = 0; i < n_iter; ++i) {
      if (!dev::warp_wait(bar + kFBarDQFull, i & 1, abort_flag, gst)) break;
      tc_fence_after_sync();
      uint32_t x[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tdQ + lane_base + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(x + 32 * c));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(x + 32 * c));
      if (i + 1 < n_iter) {
        // dP(i+1) and dV(i+1) read dO tile i+1
        if (!dev::warp_wait(bar + kFBarOFull, (i + 1) & 1, abort_flag, gst)) break;
        tc_fence_before_sync();
        mbar_arrive(bar + kFBarXGo);
      }
      // Columns [D/2, D) go through the dS area (the dQ MMA is done with it;
      // the softmax writes the next dS there only after BufFree), their
      // reduce-adds first, so that area is read back soonest; columns
      // [0, D/2) through X (free once the last step's X reduce-adds have read it).
      bool ok = true;
      const int gi = i / n_m, m = m0 + i % n_m, j = kl * p.group + gi;
      const int row0 = (rb * p.hp + j) * p.Sp + m * 128;
#pragma unroll
      for (int h = 1; h >= 0; --h) {
        if (h == 0 && i > 0 && !dev::warp_wait(bar + kFBarXFree, (i - 1) & 1, abort_flag, gst)) {
          ok = false;
          break;
        }
        stage_half<D>(smem + (h ? L::oDS : L::oX), r, x + h * (D / 2));
        fence_proxy_async_smem();
        mbar_arrive(bar + kFBarStage);
        if (elected) {
          if (!mbar_wait_bounded(bar + kFBarStage, (2 * i + (1 - h)) & 1, abort_flag, gst)) {
            ok = false;
          } else {
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx)
              tma_reduce_add_2d(&tmAcc, (h ? sDS : sX) + bx * 16384, h * (D / 2) + 32 * bx, row0);
            bulk_commit();
          }
        }
        __syncwarp();
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (elected && ok) {
        bulk_wait_read_1();  // the dS area's group (the older one) has been read
        mbar_arrive(bar + kFBarBufFree);
        bulk_wait_read_all();
        mbar_arrive(bar + kFBarXFree);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    // every reduce-add this warpgroup issued is complete before the CTA ends
    if (elected) bulk_wait_all();
  } else {
    regs_inc<kRegsFSoftmax>();
    // ------------------------------------------------- softmax warpgroups
    const int g = warp >> 2, w4 = warp & 3;
    const int r = w4 * 32 + lane;  // key row of S^T, dP^T == TMEM lane
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const int kvr = n * 128 + r;
    const bool rot = p.rope_cos && p.kv_rep == 1 && (D == 128 || g == 0) && kvr < p.S &&
                     in_range(p.status, (long long)kvr * (D / 2), D / 2, p.rope_n);
    const float *rcs = rot ? p.rope_cos + (size_t)kvr * (D / 2) + g * 32 : nullptr;
    const float *rsn = rot ? p.rope_sin + (size_t)kvr * (D / 2) + g * 32 : nullptr;
    if (rot) rope_prefetch(rcs, rsn);
    float2 pf[32];  // P of this thread's 64 columns, kept for dS
    uint32_t w[2][16];
    // P phase of step s: S^T(s) -> P^T (bf16) over the first half of this
    // warpgroup's S^T columns; P kept in pf.
    auto p_phase = [&](int s) -> bool {
      if (!dev::warp_wait(bar + kFBarSFull, s & 1, abort_flag, gst)) return false;
      tc_fence_after_sync();
      uint32_t sr[2][32];
      tmem_ld32(tmem + lane_base + g * 64, sr[0]);
      tmem_ld32(tmem + lane_base + g * 64 + 32, sr[1]);
      // this step's -LSE*log2(e) rides in its Q slot (step 0: waited here;
      // later steps: waited in the dS phase before)
      if (s == 0 && !dev::warp_wait(bar + kFBarQFull, 0, abort_flag, gst)) return false;
      tmem_wait_ld();
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      const int q0 = (m0 + s % n_m) * 128 + g * 64;
      const int lo = p.causal ? kvr - q0 : 0, hi = p.S - q0;
      const float2 *nl2 = reinterpret_cast<const float2 *>(smem + L::oRows + (s % kFQSlots) * 1024 + 512) + g * 32;
      if (__all_sync(0xffffffffu, lo <= 0 && hi >= 64))
        p_columns<false>(sr, nl2, p.scale_log2, lo, hi, pf, w);
      else
        p_columns<true>(sr, nl2, p.scale_log2, lo, hi, pf, w);
      tmem_st16(tmem + lane_base + g * 64, w[0]);
      tmem_st16(tmem + lane_base + g * 64 + 16, w[1]);
      tmem_wait_st();
      tc_fence_before_sync();
      return true;
    };
    bool ok = p_phase(0);
    if (ok) mbar_arrive(bar + kFBarPFull);
    for (int i = 0; ok && i < n_iter; ++i) {
      const int qs = i % kFQSlots;
      // ---------------- dS phase of step i
      if (!dev::warp_wait(bar + kFBarDPFull, i & 1, abort_flag, gst)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t dr[2][32];
      tmem_ld32(tmem + lane_base + 128 + g * 64, dr[0]);
      tmem_ld32(tmem + lane_base + 128 + g * 64 + 32, dr[1]);
      tmem_wait_ld();
      reg_fence(dr[0]);
      reg_fence(dr[1]);
      const float2 *dl2 = reinterpret_cast<const float2 *>(smem + L::oRows + qs * 1024) + g * 32;
      ds_columns(dr, dl2, pf, w);
      tmem_st16(tmem + lane_base + 128 + g * 64, w[0]);
      tmem_st16(tmem + lane_base + 128 + g * 64 + 16, w[1]);
      // the dS area held columns [D/2, D) of dQ(i-1) for their reduce-adds
      if (i > 0 && !dev::warp_wait(bar + kFBarBufFree, (i - 1) & 1, abort_flag, gst)) { ok = false; break; }
      {
        // dS [key r][queries 64g..64g+63] into chunk g of the dS area, 128-byte swizzle
        uint8_t *row = smem + L::oDS + g * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4 *>(row + ((u ^ (r & 7)) * 16)) =
              make_uint4(w[u >> 2][(u & 3) * 4], w[u >> 2][(u & 3) * 4 + 1], w[u >> 2][(u & 3) * 4 + 2],
                         w[u >> 2][(u & 3) * 4 + 3]);
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before_sync();
      // The issuer waits for this arrival alone before S^T(i+1) dK(i) dQ(i):
      // Q tile i+1 (and the rows riding with it) must have landed.
      if (i + 1 < n_iter &&
          !dev::warp_wait(bar + kFBarQFull + 8 * ((i + 1) % kFQSlots), ((i + 1) / kFQSlots) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      mbar_arrive(bar + kFBarDSFull);
      // ---------------- P phase of step i+1 (overlaps dK(i), dQ(i))
      if (i + 1 < n_iter) {
        if (!(ok = p_phase(i + 1))) break;
        mbar_arrive(bar + kFBarXGo);
      }
    }
    // ------------------------------------------------------------ epilogue
    RopeRow angles;
    if (ok && rot) rope_load(angles, rcs, rsn);
    if (ok) ok = dev::warp_wait(bar + kFBarAcc, 0, abort_flag, gst);
    if (ok && p.kv_rep > 1) {
      tc_fence_after_sync();
      const bool live = kvr < p.S;
      const int kr = live ? kvr : 0;
      const size_t prow = (size_t)hl_outer(p, rb, kr) * p.Cs + kr % p.Cs;
      float *pv = reinterpret_cast<float *>(p.dv) + prow * D;
      float *pk = reinterpret_cast<float *>(p.dk) + prow * D;
      const bool put = live && in_range(p.status, (long long)(prow * D), D, p.dkv_n);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t xv[32], yk[32];
        tmem_ld32(tdV + lane_base + col, xv);
        tmem_ld32(tdK + lane_base + col, yk);
        tmem_wait_ld();
        if (put) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            reinterpret_cast<uint4 *>(pv + col)[v] =
                make_uint4(xv[4 * v], xv[4 * v + 1], xv[4 * v + 2], xv[4 * v + 3]);
            reinterpret_cast<uint4 *>(pk + col)[v] =
                make_uint4(yk[4 * v], yk[4 * v + 1], yk[4 * v + 2], yk[4 * v + 3]);
          }
        }
      }
    } else if (ok) {
      tc_fence_after_sync();
      const bool live = kvr < p.S;
      const int s_rank = kvr / p.Sl, t = kvr - s_rank * p.Sl;
      const int rr = rb / p.B, bb = rb - rr * p.B;
      const size_t row = (((size_t)(s_rank * p.B + bb) * p.Sl + t) * p.n_kv + (rr * p.kvp + kl)) * D;
      const bool put = live && in_range(p.status, (long long)row, D, p.dkv_n) &&
                       (!p.rope_cos || in_range(p.status, (long long)kvr * (D / 2), D / 2, p.rope_n));
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t xv[32];
        const int col = g * (D / 2) + c * 32;
        tmem_ld32(tdV + lane_base + col, xv);
        tmem_wait_ld();
        if (put) store_plain(p.dv + row + col, xv, 1.0f);
      }
      if (D == 128 || g == 0) {
        const int i0 = g * 32;
        uint32_t xk[32], yk[32];
        tmem_ld32(tdK + lane_base + i0, xk);
        tmem_ld32(tdK + lane_base + D / 2 + i0, yk);
        tmem_wait_ld();
        if (put) store_unrotated(p.dk + row + i0, p.dk + row + D / 2 + i0, xk, yk, p.scale, rot, angles);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kFMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_BWD_TIMEOUT);
}

// dQ from the fused kernel's float accumulator: scale, undo the rotation,
// round to bf16 and write to its sequence-layout row (nothing is written when
// the status word reports a fault).  Accumulator rows [Pu*B][hp][Sp][D]
// (Sp = S rounded up to 128).  One thread per (token, head, 4 rotation pairs:
// x at c*4.., y at D/2 + c*4..), consecutive threads along the token's heads,
// so a token's dQ row in sequence layout (n_head*D values) is written
// contiguously.  (Zeroing each accumulator row right behind its load here ran
// at a seventh of the memory rate; the fused step zeroes the accumulator with
// a plain fill before its kernel instead.)
template <int D>
__global__ void __launch_bounds__(256) dq_finish_kernel(const float *__restrict__ acc, const BwdParams p) {
  constexpr int half = D / 2, q4 = half / 4;
  const long long task = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_tok = p.n_head * q4;
  if (task >= (long long)p.B * p.S * per_tok) return;
  const int tok = (int)(task / per_tok), rest = (int)(task - (long long)tok * per_tok);
  const int g = rest / q4, c = rest - g * q4;
  const int bb = tok / p.S, pos = tok - bb * p.S;
  const int rr = g / p.hp, j = g - rr * p.hp;  // group member holding global head g, its local head
  const long long arow = ((long long)(rr * p.B + bb) * p.hp + j) * p.Sp + pos;
  const long long acc_n = (long long)p.Pu * p.B * p.hp * p.Sp * D;
  if (!in_range(p.status, arow * D + c * 4, half + 4, acc_n)) return;
  if ((*p.status & 3u) != 0u || (p.rope_cos && p.status[1] != p.rope_key)) return;
  const float *a = acc + arow * D + c * 4;
  const float4 x4 = *reinterpret_cast<const float4 *>(a);
  const float4 y4 = *reinterpret_cast<const float4 *>(a + half);
  float xs[4] = {x4.x, x4.y, x4.z, x4.w}, ys[4] = {y4.x, y4.y, y4.z, y4.w};
  if (p.rope_cos) {
    if (!in_range(p.status, (long long)pos * half + c * 4, 4, p.rope_n)) return;
    const float4 c4 = *reinterpret_cast<const float4 *>(p.rope_cos + (size_t)pos * half + c * 4);
    const float4 s4 = *reinterpret_cast<const float4 *>(p.rope_sin + (size_t)pos * half + c * 4);
    const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // x' = x cos + y sin, y' = y cos - x sin
      const float xq = xs[q], yq = ys[q];
      xs[q] = xq * cc[q] + yq * ss[q];
      ys[q] = yq * cc[q] - xq * ss[q];
    }
  }
  const int s_rank = pos / p.Sl, t = pos - s_rank * p.Sl;
  const size_t o = ((((size_t)s_rank * p.B + bb) * p.Sl + t) * p.n_head + g) * D + c * 4;
  if (!in_range(p.status, (long long)o, half + 4, p.dq_n)) return;
  const uint32_t w0 = pack_bf16x2(xs[0] * p.scale, xs[1] * p.scale);
  const uint32_t w1 = pack_bf16x2(xs[2] * p.scale, xs[3] * p.scale);
  const uint32_t w2 = pack_bf16x2(ys[0] * p.scale, ys[1] * p.scale);
  const uint32_t w3 = pack_bf16x2(ys[2] * p.scale, ys[3] * p.scale);
  *reinterpret_cast<uint2 *>(p.dq + o) = make_uint2(w0, w1);
  *reinterpret_cast<uint2 *>(p.dq + o + half) = make_uint2(w2, w3);
}

// ============================================== dQ from stored dS (dS-store mode)
// The dK/dV kernel can also write every step's dS tile (bf16, 128 keys x 128
// queries, the values it feeds its dK MMA, in the layout described at
// ds_tile) to the workspace.  dQ is then a plain sum of products over the
// stored tiles, dQ_m = sum_n dS_{m,n} K_n, and the scores and dP need not be
// recomputed: five products per tile pair in all (S^T, dP^T, dV, dK; dQ)
// instead of seven, deterministic, at the price of writing and reading the dS
// tiles once (32 KB per pair).
// One CTA per (q-head, 128-query tile m), longest first; a 3-stage ring of
// (dS tile, K tile) pairs, the dS tile by one bulk copy (stored as the
// 32-byte-swizzled MN-major operand) and K by TMA; dQ += dS K with A = dS and
// B = K both MN-major, accumulated in TMEM in key-tile order; the epilogue
// (one warpgroup, thread = query row) scales, undoes the RoPE rotation and
// writes sequence layout, as the dQ kernel does.
constexpr int kDSStages = 3;
constexpr int kThreadsDS = 192;  // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kDSTmaWarp = 4, kDSMmaWarp = 5;
enum : uint32_t {
  kDBarFull = 0,                          // [kDSStages]
  kDBarEmpty = 8 * kDSStages,             // [kDSStages]
  kDBarAcc = 16 * kDSStages,
  kDBarDrain = kDBarAcc + 8,
  kDTmemSlot = kDBarDrain + 8,
  kDAbortSlot = kDTmemSlot + 4,
  kDBarBytes = kDAbortSlot + 4
};

template <int D>
struct DSLayout {
  static constexpr uint32_t kDS = 128u * 128u * 2;  // one dS tile
  static constexpr uint32_t kT = 128u * D * 2;      // one K tile
  static constexpr uint32_t kStage = kDS + kT;
  static constexpr uint32_t oBar = kDSStages * kStage;
  static constexpr uint32_t kAlloc = oBar + 256 + 1024;
  static_assert(kAlloc <= kMaxDynSmem, "dS-store dQ tiles exceed shared memory");
};

template <int D>
__global__ void __launch_bounds__(kThreadsDS, 1)
    dq_ds_kernel(const __grid_constant__ CUtensorMap tmK, const BwdParams p) {
  using L = DSLayout<D>;
  constexpr int kCh = D / 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t bar = sb + L::oBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::oBar + kDAbortSlot);
  const volatile uint32_t *gst = p.status;
  if ((*gst & 3u) || stale_rope_table(p)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.S + 127) / 128;
  const dev::HeadTile ht = dev::grouped_order((int)blockIdx.x, p.head_n * p.group, n_qt, p.group_q);
  const int m = n_qt - 1 - ht.rank;            // longest tiles first
  const int hq = p.head0 * p.group + ht.head;  // (member * B + batch) * hp + local q-head
  const int j = hq % p.hp, rb = hq / p.hp;
  const int kl = j / p.group;
  const int n_kv = p.causal ? m + 1 : n_qt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDSStages; ++s) {
      mbar_init(bar + kDBarFull + 8 * s, 1);
      mbar_init(bar + kDBarEmpty + 8 * s, 1);
    }
    mbar_init(bar + kDBarAcc, 1);
    mbar_init(bar + kDBarDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kDSMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kDTmemSlot, D < 32 ? 32 : D);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::oBar + kDTmemSlot);

  if (warp == kDSTmaWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      int issued = -1;
      for (int n = 0; n < n_kv; ++n) {
        const int s = n % kDSStages;
        if (!mbar_wait_bounded(bar + kDBarEmpty + 8 * s, ((n / kDSStages) & 1) ^ 1, abort_flag, gst)) break;
        const uint32_t full = bar + kDBarFull + 8 * s, st = sb + s * L::kStage;
        const long long e = ds_tile(p, hq, m, n) * 16384;
        if (!in_range(p.status, e, 16384, p.ds_pairs * 16384LL * p.head_n * p.group)) {  // checked build only
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(full, L::kStage);
        bulk_load(st, p.ds + e, L::kDS, full);
        const ActCoord kc = act_coord(p, rb, kl, p.kvp, n * 128, p.kv_rep);
        for (int c = 0; c < kCh; ++c)
          tma_load_4d(st + L::kDS + c * 16384, &tmK, full, c * 64, kc.head, kc.row, kc.outer);
        issued = n;
      }
      if (*abort_flag) {
        volatile int never = 0;
        for (int n = issued - (kDSStages - 1); n <= issued; ++n)
          if (n >= 0)
            mbar_wait_bounded(bar + kDBarFull + 8 * (n % kDSStages), (n / kDSStages) & 1, &never, nullptr,
                              500000000ull);
      }
    }
  } else if (warp == kDSMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idQ = idesc_bf16_f32(128, D, 1, 1);  // A (dS) and B (K) MN-major
      bool ok = true;
      for (int n = 0; ok && n < n_kv; ++n) {
        const int s = n % kDSStages;
        if (!(ok = mbar_wait_bounded(bar + kDBarFull + 8 * s, (n / kDSStages) & 1, abort_flag, gst))) break;
        tc_fence_after_sync();
        const uint32_t st = sb + s * L::kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // keys 16kk..: two 8-row groups of 32-byte rows
          mma_bf16_ss(tmem, smem_desc_sw32(st + kk * 512, 4096, 256),
                      smem_desc_sw128(st + L::kDS + kk * 2048, 16384, 1024), idQ, (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar + kDBarEmpty + 8 * s);
      }
      mma_commit(bar + kDBarAcc);
      mma_commit(bar + kDBarDrain);
      volatile int never = 0;
      mbar_wait_bounded(bar + kDBarDrain, 0, &never, nullptr);
    }
  } else if (warp < 4) {
    // ------------------------------------------------ epilogue: thread = query row
    const int r = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int qi = m * 128 + r;
    const bool live = qi < p.S;
    const bool rot = p.rope_cos && live && in_range(p.status, (long long)qi * (D / 2), D / 2, p.rope_n);
    if (rot) rope_prefetch(p.rope_cos + (size_t)qi * (D / 2), p.rope_sin + (size_t)qi * (D / 2));
    if (dev::warp_wait(bar + kDBarAcc, 0, abort_flag, gst)) {
      tc_fence_after_sync();
      const int s_rank = qi / p.Sl, t = qi - s_rank * p.Sl;
      const int rr = rb / p.B, bb = rb - rr * p.B;
      const size_t row = (((size_t)(s_rank * p.B + bb) * p.Sl + t) * p.n_head + (rr * p.hp + j)) * D;
      const bool put = live && in_range(p.status, (long long)row, D, p.dq_n) &&
                       (!p.rope_cos || in_range(p.status, (long long)qi * (D / 2), D / 2, p.rope_n));
      // rotation pairs (i, i + D/2), 32 at a time
#pragma unroll
      for (int i0 = 0; i0 < D / 2; i0 += 32) {
        RopeRow angles;
        if (rot) rope_load(angles, p.rope_cos + (size_t)qi * (D / 2) + i0, p.rope_sin + (size_t)qi * (D / 2) + i0);
        uint32_t x[32], y[32];
        tmem_ld32(tmem + lane_base + i0, x);
        tmem_ld32(tmem + lane_base + D / 2 + i0, y);
        tmem_wait_ld();
        if (put) store_unrotated(p.dq + row + i0, p.dq + row + D / 2 + i0, x, y, p.scale, rot, angles);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kDSMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, D < 32 ? 32 : D);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_BWD_TIMEOUT);
}

// Which of the backward kernels a launch runs.
enum BwdPart { kBwdDkDv = 1, kBwdDq = 2, kBwdFused = 4, kBwdFinish = 8, kBwdDqDS = 16 };

// Causal (key tile, query tile) pairs of one head: n_kt (n_kt + 1) / 2.
inline long long n_tiles_pairs(const ulysses_problem &p) {
  const long long n = (p.S + 127) / 128;
  return n * (n + 1) / 2;
}

template <int D>
cudaError_t launch_d(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                     const void *v, const void *do_head, const float *nlse, const float *delta,
                     const void *ws, void *dq, void *dk, void *dv, float *dqacc, void *ds, uint32_t *status,
                     int parts, bool folded, cudaStream_t st, int head0, int head_n) {
  const int Pu = group_ranks(p), Cs = chunk_len(p), Sl = p.S / p.P;
  const int hp = p.n_head / Pu, kvp = kv_per_rank(p), PB = p.P * p.B;
  // head-layout maps [P*B][Cs][hp|kvp][D], or folded the sequence-sharded
  // [P*B][Sl][n_head|n_kv_head][D]; the delta / nlse rows [P*B*hp][Cs] (Ld apart)
  const int rows = folded ? Sl : Cs, qh = folded ? p.n_head : hp, kh = folded ? p.n_kv_head : kvp;
  if (folded && (ring_of(p) > 1 || Sl % 128 != 0)) return cudaErrorInvalidValue;
  CUtensorMap mK128, mV128, mL, mDl, mQ128, mdO128;
  if ((parts & kBwdDqDS) && !(parts & (kBwdDkDv | kBwdDq | kBwdFused))) {  // dQ from the dS store reads K only
    if (!make_act_map(enc, &mK128, k, D, kh, rows, PB, 128)) return cudaErrorInvalidValue;
  } else if (parts & (kBwdDkDv | kBwdDq | kBwdFused)) {  // the dQ finish step reads no tile
    const bool ok = make_act_map(enc, &mK128, k, D, kh, rows, PB, 128) &&
                    make_act_map(enc, &mV128, v, D, kh, rows, PB, 128) &&
                    make_row_map(enc, &mL, nlse, Cs, delta_ld(p), PB * hp, 128) &&
                    make_row_map(enc, &mDl, delta, Cs, delta_ld(p), PB * hp, 128) &&
                    make_act_map(enc, &mQ128, q, D, qh, rows, PB, 128) &&
                    make_act_map(enc, &mdO128, do_head, D, qh, rows, PB, 128);
    if (!ok) return cudaErrorInvalidValue;
  }
  BwdParams bp;
  bp.B = p.B;
  bp.S = p.S;
  bp.P = p.P;
  bp.Sl = p.S / p.P;
  bp.hp = hp;
  bp.kvp = kvp;
  bp.group = hp / kvp;
  bp.causal = p.causal;
  bp.n_head = p.n_head;
  bp.n_kv = p.n_kv_head;
  bp.Pu = Pu;
  bp.Cs = Cs;
  bp.folded = folded ? 1 : 0;
  bp.dq_n = (long long)p.B * p.S * p.n_head * D;
  bp.dkv_n = kv_replicas(p) > 1 ? (long long)p.P * p.B * Cs * D : (long long)p.B * p.S * p.n_kv_head * D;
  bp.qo_n = (long long)p.B * p.S * p.n_head * D;
  bp.Ld = delta_ld(p);
  bp.rows_n = (long long)PB * hp * bp.Ld;
  bp.Sp = (p.S + 127) / 128 * 128;
  bp.rope_n = (long long)p.S * (D / 2);
  // CTA units: (group member, batch, head), each over the full sequence.
  const int UB = Pu * p.B;
  // dK/dV CTAs of a kv-head stream the Q and dO of its q-heads; dQ CTAs of a
  // q-head stream its kv-head's K and V (shared by the group's q-heads).
  const long long n_t = (p.S + 127) / 128;
  // Budgets measured at the pages' sizing (16 MiB of K and V, or of Q and dO,
  // per head; DRAM bytes per launch, same kernel times): dK/dV 1.80 GB with
  // 48 MiB (3-head groups), 1.63 GB with 32 MiB (the algorithmic 1.61 GB); dQ
  // 1.72 GB with 48 MiB, 1.43 GB with 32 MiB, 1.36 GB with 16 MiB (algorithmic
  // 1.34 GB).  Half of the 129 MB L2 sits on each die, and the tiles of the
  // running groups share it with the outputs and the other operands.
  // A launch of the dK/dV or the dQ-from-dS kernel may cover a range of the
  // kv-heads (and their q-heads); the other kernels cover all of them.
  const int all_kv = UB * kvp;
  if (head_n < 0) head_n = all_kv;
  if (head0 < 0 || head_n <= 0 || head0 + head_n > all_kv ||
      ((parts & (kBwdDq | kBwdFused | kBwdFinish)) && (head0 != 0 || head_n != all_kv)))
    return cudaErrorInvalidValue;
  bp.head0 = head0;
  bp.head_n = head_n;
  bp.group_kv = l2_head_group((size_t)4 * p.S * D * bp.group, head_n, n_t * head_n, (size_t)32 << 20);
  bp.group_q = l2_head_group((size_t)4 * p.S * D / bp.group, head_n * bp.group, n_t * head_n * bp.group,
                             (size_t)16 << 20);
  bp.scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)D);
  bp.scale_log2 = bp.scale * kLog2e;
  bp.nlse = nlse;
  bp.delta = delta;
  bp.q = static_cast<const __nv_bfloat16 *>(q);
  bp.dout = static_cast<const __nv_bfloat16 *>(do_head);
  if (p.use_rope) {
    const WorkspaceLayout W = workspace_layout(p);
    bp.rope_cos = reinterpret_cast<const float *>(static_cast<const uint8_t *>(ws) + W.rope);
    bp.rope_sin = bp.rope_cos + (size_t)p.S * (D / 2);
  } else {
    bp.rope_cos = bp.rope_sin = nullptr;
  }
  bp.kv_rep = kv_replicas(p);
  bp.dq = static_cast<__nv_bfloat16 *>(dq);
  bp.dk = static_cast<__nv_bfloat16 *>(dk);
  bp.dv = static_cast<__nv_bfloat16 *>(dv);
  bp.status = status;
  bp.rope_key = rope_key(p);
  bp.ds = static_cast<__nv_bfloat16 *>(ds);
  bp.ds_pairs = p.causal ? n_tiles_pairs(p) : (long long)((p.S + 127) / 128) * ((p.S + 127) / 128);

  const long long kv_blocks = n_t * head_n;             // the dK/dV kernels' CTAs
  const long long q_blocks = n_t * head_n * bp.group;   // the dQ kernels' CTAs
  if (kv_blocks > 0x7fffffffll || q_blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (parts & kBwdDkDv) {
    e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)KVLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dkdv_kernel<D><<<(unsigned)kv_blocks, kThreadsKV, KVLayout<D>::kAlloc, st>>>(mK128, mV128, mQ128, mdO128,
                                                                                mL, mDl, bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (parts & kBwdDq) {
    e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dq_kernel<D><<<(unsigned)q_blocks, kThreadsQ, QLayout<D>::kAlloc, st>>>(mK128, mV128, bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (parts & kBwdDqDS) {
    if (!ds || (reinterpret_cast<uintptr_t>(ds) & 15)) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(dq_ds_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DSLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dq_ds_kernel<D><<<(unsigned)q_blocks, kThreadsDS, DSLayout<D>::kAlloc, st>>>(mK128, bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // the float dQ accumulator [Pu*B*hp*Sp][D]: the fused kernel adds [128 x 32] boxes into it
  const long long acc_rows = (long long)UB * hp * bp.Sp;
  if ((parts & (kBwdFused | kBwdFinish)) && acc_rows > 0x7fffffffll) return cudaErrorInvalidValue;  // int coords
  if (parts & kBwdFused) {
    CUtensorMap mAcc;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)acc_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 4};
    const cuuint32_t box[2] = {32, 128};  // 128-byte rows, swizzled like the staging areas
    const cuuint32_t estr[2] = {1, 1};
    if (!dqacc || enc.encode(&mAcc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dqacc, dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    // the fused kernel's CTAs also keep their heads' dQ accumulator rows in L2
    bp.group_kv = l2_head_group((size_t)4 * p.S * D * bp.group * 2, UB * kvp, n_t * UB * kvp);
    e = cudaFuncSetAttribute(dkdvq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dkdvq_kernel<D><<<(unsigned)kv_blocks, kThreadsF, FLayout<D>::kAlloc, st>>>(mK128, mV128, mQ128, mdO128, mL,
                                                                                  mDl, mAcc, bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (parts & kBwdFinish) {
    if (!dqacc) return cudaErrorInvalidValue;
    const long long tasks = (long long)p.B * p.S * p.n_head * (D / 8);  // (token, head, 4 rotation pairs)
    const long long grid = (tasks + 255) / 256;
    if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
    dq_finish_kernel<D><<<(unsigned)grid, 256, 0, st>>>(dqacc, bp);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_parts(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                         const void *v, const void *do_head, const float *nlse, const float *delta,
                         const void *ws, void *dq, void *dk, void *dv, float *dqacc, void *ds, uint32_t *status,
                         int parts, bool folded, cudaStream_t st, int head0 = 0, int head_n = -1) {
  if (p.head_dim == 128)
    return launch_d<128>(p, enc, q, k, v, do_head, nlse, delta, ws, dq, dk, dv, dqacc, ds, status, parts, folded, st,
                         head0, head_n);
  if (p.head_dim == 64)
    return launch_d<64>(p, enc, q, k, v, do_head, nlse, delta, ws, dq, dk, dv, dqacc, ds, status, parts, folded, st,
                        head0, head_n);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                                 const void *k, const void *v, const void *do_head, const float *nlse,
                                 const float *delta, const void *ws, void *dk_seq, void *dv_seq,
                                 uint32_t *status, cudaStream_t st, bool folded, void *ds, int head0,
                                 int head_n) {
  return launch_parts(p, enc, q, k, v, do_head, nlse, delta, ws, nullptr, dk_seq, dv_seq, nullptr, ds, status,
                      kBwdDkDv, folded, st, head0, head_n);
}

cudaError_t launch_attn_bwd_fused(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                                  const void *v, const void *do_head, const float *nlse, const float *delta,
                                  const void *ws, float *dq_acc, void *dk_seq, void *dv_seq, uint32_t *status,
                                  cudaStream_t st, bool folded) {
  return launch_parts(p, enc, q, k, v, do_head, nlse, delta, ws, nullptr, dk_seq, dv_seq, dq_acc, nullptr, status,
                      kBwdFused, folded, st);
}

cudaError_t launch_dq_from_ds(const ulysses_problem &p, const TmaEncoder &enc, const void *k, const void *ws,
                              const void *ds, void *dq_seq, uint32_t *status, cudaStream_t st, int head0,
                              int head_n) {
  // the K map and the parameters are those of the packed (head-layout) backward
  return launch_parts(p, enc, nullptr, k, nullptr, nullptr, nullptr, nullptr, ws, dq_seq, nullptr, nullptr, nullptr,
                      const_cast<void *>(ds), status, kBwdDqDS, false, st, head0, head_n);
}

cudaError_t launch_dq_finish(const ulysses_problem &p, const TmaEncoder &enc, const void *ws, float *dq_acc,
                             void *dq_seq, uint32_t *status, cudaStream_t st) {
  return launch_parts(p, enc, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, ws, dq_seq, nullptr, nullptr,
                      dq_acc, nullptr, status, kBwdFinish, false, st);
}

cudaError_t launch_attn_bwd_dq(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                               const void *k, const void *v, const void *do_head, const float *nlse,
                               const float *delta, const void *ws, void *dq_seq, uint32_t *status,
                               cudaStream_t st, bool folded) {
  return launch_parts(p, enc, q, k, v, do_head, nlse, delta, ws, dq_seq, nullptr, nullptr, nullptr, nullptr, status,
                      kBwdDq, folded, st);
}

}  // namespace ulysses
