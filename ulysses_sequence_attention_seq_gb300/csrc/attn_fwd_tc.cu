// attn_fwd_tc.cu -- bf16 attention forward on the 5th-generation tensor cores.
//
// What it computes ("Sequence Parallelism II: DeepSpeed Ulysses and All-to-All
// Attention", §2 fourth step, and §8: causal attention keeps its triangular
// work inside each head): for every virtual rank r, batch b and local head j
// of the head-sharded layout, O = softmax(scale * Q K^T [+ causal mask]) V over
// the full sequence, plus the row log-sum-exp.  Query head g = r*hp + j reads
// kv-head g / (n_head / n_kv_head), i.e. local kv index j / (hp / kvp).
//
// How: one CTA per pair of 128-query tiles (A = rows [256i, 256i+128),
// B = the next 128) of one head, 12 warps (warps 10-11 only complete the
// third warpgroup, which the per-warpgroup register split needs).
//   warp 8      TMA producer: both Q tiles and K_0 once, then ring entries
//               e = 0, 1, ... of a 2-entry ring, entry e holding V_e and
//               K_{e+1}: exactly what key tile e's two bursts below read, so
//               one barrier reports both (128 rows x D per tile, 128-byte
//               swizzle, 4-D tensor maps over [P*B][S][heads][D] so a tile
//               never crosses a sequence end).  Every K/V tile serves 256
//               query rows.
//   warp 9      MMA issuer (one thread), in the order
//                 S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | PV_A(1) ...
//               so the tensor core alternates between the two tiles while the
//               other tile's softmax runs.  Because S_X(j+1) is issued after
//               PV_X(j), the commit that reports S_X(j+1) also reports that
//               PV_X(j) has finished: the softmax can then rescale O_X
//               without any further barrier.  S_X(j+1) overwrites P_X(j) only
//               after PV_X(j) has read it (one issuer's MMAs run in order).
//               A thread with MMAs in flight stalls on its next shared-memory
//               access (such as a barrier wait, ~100 cycles even on a
//               completed phase) until they have been taken by the tensor
//               core, and each such stall leaves a gap in the pipe, so the
//               issuer waits once per burst, for P_X(j) alone: the softmax
//               warps whose burst opens key tile j wait for ring entry j
//               before publishing P, so that arrival vouches for the entry.
//   warps 0-3   softmax of tile A, warps 4-7 of tile B: thread i of a
//               warpgroup owns query row i = TMEM lane i.  It reads its score
//               row from TMEM, takes the row maximum (base-2 domain) on the
//               first key tile only and afterwards keeps that reference until
//               a tile's row sum of P passes 2^16, when it moves the reference
//               to the new maximum and rescales its TMEM accumulator row and
//               the row sum (so no maximum pass on most tiles), writes P (bf16, two keys per
//               32-bit column) over the first 64 columns of its S row, where
//               the PV MMA reads it as its A operand straight from TMEM, and at
//               the end divides by the row sum and stores O (bf16) and the LSE.
// TMEM: S_A, S_B (128 columns each; P_X in the first 64 of S_X), O_A, O_B (D
// columns each).  Keeping P out of shared memory leaves the shared-memory
// port, which a 128x128x16 MMA with both operands there saturates, to Q, K, V
// and the TMA writes.
// Causal tiles past the diagonal are skipped; only the diagonal tile and the
// ragged tail are masked.  CTAs are ordered longest-first.  Every wait is
// bounded (2 s); a timeout sets a status bit, the CTA drains its tensor-core
// work and copies in flight, frees TMEM and exits, and the other CTAs stop.
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

constexpr int BM = 128;        // query rows per tile (two tiles per CTA)
constexpr int BN = 128;        // keys per tile
constexpr int kThreads = 384;  // warpgroups 0-1 softmax, warpgroup 2: TMA, MMA, 2 idle warps
constexpr int kTmaWarp = 8, kMmaWarp = 9;
// Register split (launch: 384 threads x 168): warpgroup 2 drops to 64, the
// softmax warpgroups rise to 216: 128*64 + 256*216 = 63488 <= 384*168.  (With
// 72 for warpgroup 2, ptxas allocated the kernel with a 4-byte spill; with 64
// it has none.)
constexpr uint32_t kRegsProducer = 64, kRegsSoftmax = 216;
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= 384 * 168, "register split over budget");
constexpr int kSlots = 2;  // K/V ring entries: entry e holds V_e and K_{e+1}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128 * 128;    // 128 rows x 128 bytes (64 bf16)

template <int D>
struct Layout {
  static constexpr uint32_t kTile = 128u * D * 2;       // one 128-row tile of Q, K or V
  static constexpr uint32_t kEntry = 2 * kTile;          // V_e, then K_{e+1}
  static constexpr uint32_t kQ = 0;                      // Q_A, Q_B
  static constexpr uint32_t kK0 = kQ + 2 * kTile;        // K_0
  static constexpr uint32_t kKV = kK0 + kTile;           // ring of kSlots entries
  static constexpr uint32_t kBar = kKV + kSlots * kEntry;
  static constexpr uint32_t kAlloc = kBar + 256 + 1024;  // room to align the base to 1024
};
static_assert(Layout<128>::kAlloc <= 232448, "shared memory");

// Barrier slots (byte offsets inside the barrier block).
enum : uint32_t {
  kBarQFull = 0,
  kBarKVFull = 8,                         // [kSlots]
  kBarKVEmpty = kBarKVFull + 8 * kSlots,  // [kSlots]
  kBarSFull = kBarKVEmpty + 8 * kSlots,   // [2] A, B
  kBarPFull = kBarSFull + 16,             // [2] A, B (128 arrivals)
  kBarODone = kBarPFull + 16,             // [2] A, B
  kBarDrain = kBarODone + 16,
  kTmemSlot = kBarDrain + 8,
  kAbortSlot = kTmemSlot + 4
};
static_assert(kAbortSlot + 4 <= 256, "barrier block");

struct FwdParams {
  int B, S, P, hp, kvp, group, causal, n_pairs;
  // Folded addressing: the tensor maps cover the sequence-sharded buffers
  // [P][B][Sl][heads][D] and O is written in sequence layout [P][B][Sl][H]
  // (the two All-to-Alls become addressing).  Needs Sl % 128 == 0 so a tile
  // never straddles two ranks' shards.
  int folded, Sl, n_head, n_kv_head;
  int head_group;  // heads per CTA group (grouped_order)
  int kv_rep;      // > 1: replicated kv-heads, rank r reads kv-head r / kv_rep
  // Ulysses x ring hybrid: Pu ranks per ring position, Cs tokens per chunk;
  // the 128-row tile at global position pos of group member u lives in the
  // head-layout buffer of rank (pos / Cs) * Pu + u, row pos % Cs.  Plain
  // Ulysses: Pu = P, Cs = S.
  int Pu, Cs;
  float scale_log2;
  __nv_bfloat16 *o;  // [P][B][S][hp][D], or [P][B][Sl][H] when folded
  float *lse;        // [P][B][hp][S]
  long long o_n, lse_n;  // their elements (range checks of a checked build)
  uint32_t *status;
};

// TMA coordinates (head, row, rank*B+batch) of the 128-row tiles of one head,
// walked in position order.  The tile at global position pos sits in block
// c = pos / period at row pos % period: a block is a ring position's chunk
// (period Cs; plain Ulysses has one block, the whole sequence) in head
// layout, or, folded, a rank's sequence shard (period Sl).  Head `lh` of group
// member `r` (the rank, without a ring), batch `b`; `rep` > 1: a replicated
// kv-head (folded: rank r reads global kv-head r / rep).
struct TileWalk {
  int head, base, row, c, last, period, step;  // outer coordinate = c * step + base
  __device__ __forceinline__ TileWalk(const FwdParams &p, int r, int b, int lh, int heads_local, int pos,
                                      int rep = 1) {
    if (!p.folded) {
      head = lh, period = p.Cs, step = p.Pu * p.B, base = r * p.B + b;
    } else {
      head = rep > 1 ? r / rep : r * heads_local + lh, period = p.Sl, step = p.B, base = b;
    }
    // a tile starting past the sequence end stays in the last block, its rows
    // out of range (read as zeros)
    last = (p.S - 1) / period;
    c = (pos < p.S ? pos : p.S - 1) / period;
    row = pos - c * period;
  }
  __device__ __forceinline__ int outer() const { return c * step + base; }
  __device__ __forceinline__ void next() {  // the tile 128 positions on
    row += 128;
    if (row >= period && c < last) row -= period, ++c;
  }
};

// Slot and phase parity of ring entry e.
__device__ __forceinline__ uint32_t ring_slot(int e) { return (uint32_t)(e % kSlots); }
__device__ __forceinline__ uint32_t ring_parity(int e) { return (uint32_t)((e / kSlots) & 1); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using L = Layout<D>;
  constexpr int kChunks = D / 64;  // 128-byte swizzle chunks per row
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sQ = sb + L::kQ, sK0 = sb + L::kK0, sKV = sb + L::kKV;
  const uint32_t bar = sb + L::kBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBar + kAbortSlot);
  const volatile uint32_t *gst = p.status;
  // A CTA of this grid (or an earlier launch on this workspace) gave up on a
  // wait: do not start more work.
  if (*gst & (ULYSSES_STATUS_FWD_TIMEOUT | ULYSSES_STATUS_BWD_TIMEOUT)) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads_total = p.Pu * p.B * p.hp;
  const dev::HeadTile ht = dev::grouped_order((int)blockIdx.x, heads_total, p.n_pairs, p.head_group);
  const int qp = p.n_pairs - 1 - ht.rank;  // longest pairs first
  const int hid = ht.head;
  const int j = hid % p.hp;
  const int rb = hid / p.hp;  // r*B + b
  const int kl = j / p.group;
  const int n_kt = (p.S + BN - 1) / BN;
  const int nA = p.causal ? min(2 * qp + 1, n_kt) : n_kt;  // key tiles of query tile A
  const int nB = p.causal ? min(2 * qp + 2, n_kt) : n_kt;  // ... of query tile B (>= nA)

  if (threadIdx.x == 0) {
    mbar_init(bar + kBarQFull, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar + kBarKVFull + 8 * i, 1);
      mbar_init(bar + kBarKVEmpty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + kBarSFull + 8 * i, 1);
      mbar_init(bar + kBarPFull + 8 * i, 128);
      mbar_init(bar + kBarODone + 8 * i, 1);
    }
    mbar_init(bar + kBarDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kBar + kTmemSlot);

  if (warp >= 8) {
    regs_dec<kRegsProducer>();
    if (warp == kTmaWarp) {
      if (lane == 0) {
        // ---------------------------------------------------------- producer
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const int member = rb / p.B, bb = rb - member * p.B;
        // Q_A, Q_B and K_0 on one barrier
        mbar_arrive_expect_tx(bar + kBarQFull, 3 * L::kTile);
        TileWalk tq(p, member, bb, j, p.hp, qp * 2 * BM);
        for (int x = 0; x < 2; ++x, tq.next())
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(sQ + x * L::kTile + c * kChunkBytes, &tmQ, bar + kBarQFull, c * 64, tq.head, tq.row,
                        tq.outer());
        TileWalk tv(p, member, bb, kl, p.kvp, 0, p.kv_rep);  // key tile e (K_e, V_e)
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(sK0 + c * kChunkBytes, &tmK, bar + kBarQFull, c * 64, tv.head, tv.row, tv.outer());
        // entry e = V_e and (when tile B goes on) K_{e+1}: what key tile e's two bursts read
        int issued = -1;
        for (int e = 0; e < nB; ++e) {
          const uint32_t slot = ring_slot(e), full = bar + kBarKVFull + 8 * slot;
          if (!mbar_wait_bounded(bar + kBarKVEmpty + 8 * slot, ring_parity(e) ^ 1, abort_flag, gst)) break;
          const bool has_k = e + 1 < nB;
          mbar_arrive_expect_tx(full, (has_k ? 2u : 1u) * L::kTile);
          const uint32_t dst = sKV + slot * L::kEntry;
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(dst + c * kChunkBytes, &tmV, full, c * 64, tv.head, tv.row, tv.outer());
          tv.next();
          if (has_k)
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(dst + L::kTile + c * kChunkBytes, &tmK, full, c * 64, tv.head, tv.row, tv.outer());
          issued = e;
        }
        if (*abort_flag) {
          // Let the copies already in flight land before the CTA goes away.
          volatile int never = 0;
          mbar_wait_bounded(bar + kBarQFull, 0, &never, nullptr, 500000000ull);
          for (int e = issued - (kSlots - 1); e <= issued; ++e)
            if (e >= 0)
              mbar_wait_bounded(bar + kBarKVFull + 8 * ring_slot(e), ring_parity(e), &never, nullptr,
                                500000000ull);
        }
      }
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        // -------------------------------------------------------------- MMA
        constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
        constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);  // P (TMEM), V MN-major
        // S_x(t) = Q_x K_t^T (K_t has landed: the caller waited for it).
        auto issue_s = [&](int x, int t) {
          const uint32_t kt = t == 0 ? sK0 : sKV + ring_slot(t - 1) * L::kEntry + L::kTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + x * BN, smem_desc_sw128(sQ + x * L::kTile + koff, 16, 1024),
                        smem_desc_sw128(kt + koff, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar + kBarSFull + 8 * x);
        };
        // O_x += P_x(t) V_t (P_x(t) published and V_t landed: the caller waited).
        auto issue_pv = [&](int x, int t) {
          const uint32_t vt = sKV + ring_slot(t) * L::kEntry;
          // keys 16kk..16kk+15 of P_X are TMEM columns x*BN + 8kk ..
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t b = smem_desc_sw128(vt + kk * 16 * 128, kChunkBytes, 1024);
            mma_bf16_ts(tmem + 2 * BN + x * D, tmem + x * BN + kk * 8, b, idPV, (t > 0 || kk > 0) ? 1u : 0u);
          }
        };
        // Entry t is free once key tile t's two bursts have finished: its
        // commit follows tile B's burst.  (A commit at the head of a burst,
        // issued while the pipe is idle after the waits, was measured to delay
        // the burst's MMAs by ~90 cycles; at the tail it costs nothing.)
        auto release = [&](int e) { mma_commit(bar + kBarKVEmpty + 8 * ring_slot(e)); };
        bool ok = mbar_wait_bounded(bar + kBarQFull, 0, abort_flag, gst);
        if (ok && nA > 0) issue_s(0, 0);
        if (ok) issue_s(1, 0);
        for (int t = 0; ok && t < nB; ++t) {
          // tile A's burst: P_A(t) (whose arrival vouches for entry t)
          if (t < nA) {
            if (!(ok = mbar_wait_bounded(bar + kBarPFull, t & 1, abort_flag, gst))) break;
            tc_fence_after_sync();
            issue_pv(0, t);
            if (t == nA - 1)
              mma_commit(bar + kBarODone);
            else
              issue_s(0, t + 1);
          }
          // then tile B's: P_B(t) (vouching for entry t if A skipped it)
          if (!(ok = mbar_wait_bounded(bar + kBarPFull + 8, t & 1, abort_flag, gst))) break;
          tc_fence_after_sync();
          issue_pv(1, t);
          if (t == nB - 1)
            mma_commit(bar + kBarODone + 8);
          else
            issue_s(1, t + 1);
          release(t);
        }
        // All tensor-core work of this CTA is complete once this commit lands.
        mma_commit(bar + kBarDrain);
        volatile int never = 0;
        mbar_wait_bounded(bar + kBarDrain, 0, &never, nullptr);
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------ softmax warpgroups A, B
    const int x = warp >> 2;                 // 0: tile A, 1: tile B
    const int row = (warp & 3) * 32 + lane;  // query row in the tile == TMEM lane
    const int qpos = qp * 2 * BM + x * BM + row;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + x * BN;
    const uint32_t tO = tmem + lane_base + 2 * BN + x * D;
    const int n_mine = x ? nB : nA;
    const int own_entry_from = x ? nA : 0;  // key tiles whose first burst is this tile's
    const int diag = p.causal ? 2 * qp + x : -1;  // the key tile holding this tile's diagonal
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // running max (scaled, base 2) and row sum
    bool ok = true;
    for (int t = 0; t < n_mine; ++t) {
      if (!warp_wait(bar + kBarSFull + 8 * x, t & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(s[c]);
      const int kv0 = t * BN;
      if (t == diag || kv0 + BN > p.S) {
        // keys past this query row (causal) or past the sequence end
        const int lim = min(p.causal ? qpos - kv0 : BN - 1, p.S - 1 - kv0);
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
      // Row maximum of the raw scores: eight independent chains of
      // three-input maxima over 16 columns each.
      auto row_max = [&]() -> float {
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t *r = &s[i >> 1][(i & 1) * 16];
          float m = max3(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]));
#pragma unroll
          for (int e = 3; e < 15; e += 2) m = max3(m, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
          mx[i] = fmaxf(m, __uint_as_float(r[15]));
        }
        return max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      };
      // P = exp2(scale*log2(e)*s - m) into the first 64 columns of S (bf16,
      // two keys per column); returns the row's sum of P.
      auto exps = [&](float m) -> float {
        const float2 sl22 = make_float2(sl2, sl2), nb2 = make_float2(-m, -m);
        float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // keys [32c, 32c+32) -> P columns [16c, 16c+16) of this row
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 a =
                fma2(make_float2(__uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1])), sl22, nb2);
            const float2 pe = make_float2(ex2(a.x), ex2(a.y));
            rs[e & 1] = add2(rs[e & 1], pe);
            w[e] = pack_bf16x2(pe.x, pe.y);
          }
          tmem_st16(tS + c * 16, w);
        }
        return (rs[0].x + rs[1].x) + (rs[0].y + rs[1].y);
      };
      // The reference m_used only guards against overflow (the exponentials'
      // relative precision does not depend on it), so it is set from the row
      // maximum on the first tile and afterwards moved only when a tile's row
      // sum of P exceeds 2^16 (some score more than 9 above it): then that
      // tile's P is formed again against the new maximum and O and l are
      // rescaled.  P <= 2^16 keeps l and O at most 2^24 times |V|.
      float tsum = 0.f;
      bool set_ref = t == 0, need = true;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (set_ref) {
          // t == 0: m_used = -inf.  Otherwise the S_X(t) commit we waited on
          // also covers PV_X(t-1): O_X is final for tiles < t and no MMA
          // touches it until P_X(t) is published.
          const float ms = need ? fmaxf(row_max() * sl2, m_used) : m_used;
          if (t > 0) {
            const float alpha = ex2(m_used - ms);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float2 v = mul2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                      make_float2(alpha, alpha));
                r[e] = __float_as_uint(v.x);
                r[e + 1] = __float_as_uint(v.y);
              }
              tmem_st32(tO + c * 32, r);
            }
            tmem_wait_st();
            l *= alpha;
          }
          m_used = ms;
        }
        tsum = exps(m_used);
        if (set_ref) break;
        need = !(tsum <= 65536.0f);  // also true for inf
        if (!__any_sync(0xffffffffu, need)) break;
        set_ref = true;
      }
      l += tsum;
      tmem_wait_st();
      tc_fence_before_sync();
      // The issuer waits for this arrival alone before the burst PV_X(t)
      // S_X(t+1); when that burst is key tile t's first (tile A's, or B's once
      // A is done) the arrival also vouches for ring entry t having landed.
      if (t >= own_entry_from &&
          !warp_wait(bar + kBarKVFull + 8 * ring_slot(t), ring_parity(t), abort_flag, gst)) {
        ok = false;
        break;
      }
      mbar_arrive(bar + kBarPFull + 8 * x);
    }
    // --------------------------------------------------------------- epilogue
    if (ok) ok = warp_wait(bar + kBarODone + 8 * x, 0, abort_flag, gst);
    if (ok) {
      tc_fence_after_sync();
      const float inv = 1.0f / l;
      __nv_bfloat16 *orow;
      size_t ooff;
      if (!p.folded) {  // rank (qpos / Cs) * Pu + member, row qpos % Cs
        ooff = ((((size_t)(qpos / p.Cs) * p.Pu * p.B + rb) * p.Cs + qpos % p.Cs) * p.hp + j) * D;
      } else {  // token qpos of rank qpos/Sl, global head r*hp + j
        const int r = rb / p.B, b = rb - r * p.B, dst = qpos / p.Sl;
        ooff = (((size_t)(dst * p.B + b) * p.Sl + (qpos - dst * p.Sl)) * p.n_head + r * p.hp + j) * D;
      }
      orow = p.o + ooff;
      const bool store = qpos < p.S && in_range(p.status, (long long)ooff, D, p.o_n);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
        if (store) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
      }
      if (qpos < p.S) {
        const size_t hr = (size_t)(qpos / p.Cs) * p.Pu * p.B + rb;  // head-layout rank * B + b
        const size_t li = (hr * p.hp + j) * p.Cs + qpos % p.Cs;
        if (in_range(p.status, (long long)li, 1, p.lse_n))
          p.lse[li] = (m_used + log2f(l)) * 0.69314718055994530942f;
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
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_FWD_TIMEOUT);
}

template <int D>
cudaError_t launch_d(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                     const void *v, void *o, float *lse, uint32_t *status, bool folded, cudaStream_t st) {
  const int Pu = group_ranks(p), Cs = chunk_len(p);
  const int hp = p.n_head / Pu, kvp = kv_per_rank(p), PB = p.P * p.B, Sl = p.S / p.P;
  CUtensorMap mq, mk, mv;
  // head-sharded maps: [P*B][S][hp|kvp][D]; folded maps: [P*B][Sl][n_head|n_kv_head][D]
  const int rows = folded ? Sl : Cs;
  if (!make_act_map(enc, &mq, q, D, folded ? p.n_head : hp, rows, PB, 128) ||
      !make_act_map(enc, &mk, k, D, folded ? p.n_kv_head : kvp, rows, PB, 128) ||
      !make_act_map(enc, &mv, v, D, folded ? p.n_kv_head : kvp, rows, PB, 128))
    return cudaErrorInvalidValue;
  FwdParams fp;
  fp.B = p.B;
  fp.S = p.S;
  fp.P = p.P;
  fp.hp = hp;
  fp.kvp = kvp;
  fp.group = hp / kvp;
  fp.causal = p.causal;
  fp.n_pairs = (p.S + 2 * BM - 1) / (2 * BM);
  fp.folded = folded ? 1 : 0;
  fp.Sl = Sl;
  fp.n_head = p.n_head;
  fp.n_kv_head = p.n_kv_head;
  fp.kv_rep = kv_replicas(p);
  fp.Pu = Pu;
  fp.Cs = Cs;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)D);
  fp.scale_log2 = scale * 1.4426950408889634f;
  // a q-head's CTAs stream its kv-head's K and V; the group's q-heads share them
  const int units = Pu * p.B * hp;  // (group member, batch, local head): one full-sequence head each
  // 32 MiB: at the pages' sizing 3-head groups (48 MiB) moved 1.18 GB of DRAM
  // per launch, 2-head groups 1.06 GB (the algorithmic 1.08 GB), in the same
  // time (16 MiB, 1-head groups: 2 % slower).
  fp.head_group = l2_head_group((size_t)4 * p.S * D / fp.group, units, (long long)fp.n_pairs * units,
                                (size_t)32 << 20);
  fp.o = static_cast<__nv_bfloat16 *>(o);
  fp.lse = lse;
  fp.o_n = (long long)p.B * p.S * p.n_head * D;  // O in head or sequence layout: the same elements
  fp.lse_n = (long long)p.B * p.n_head * p.S;
  fp.status = status;
  const long long blocks = (long long)fp.n_pairs * units;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  attn_fwd_tc_kernel<D><<<(unsigned)blocks, kThreads, Layout<D>::kAlloc, st>>>(mq, mk, mv, fp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const ulysses_problem &p, const TmaEncoder &enc, const void *q,
                               const void *k, const void *v, void *o, float *lse, uint32_t *status,
                               bool folded, cudaStream_t st) {
  if (p.head_dim == 128) return launch_d<128>(p, enc, q, k, v, o, lse, status, folded, st);
  if (p.head_dim == 64) return launch_d<64>(p, enc, q, k, v, o, lse, status, folded, st);
  return cudaErrorInvalidValue;
}

}  // namespace ulysses
