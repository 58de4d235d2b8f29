// attn_fwd_tc.cu -- bf16 attention forward on the 5th-generation tensor cores.
//
// What it computes ("Sequence Parallelism II: DeepSpeed Ulysses and All-to-All
// Attention", §2 fourth step, and §8: causal attention keeps its triangular
// work inside each head): for every virtual rank r, batch b and local head j
// of the head-sharded layout, O = softmax(scale * Q K^T [+ causal mask]) V over
// the full sequence, plus the row log-sum-exp.  Query head g = r*hp + j reads
// kv-head g / (n_head / n_kv_head), i.e. local kv index j / (hp / kvp).
//
// How (one CTA per 128-query tile of one head, 6 warps):
//   warp 4      TMA producer: Q tile once, then K_t and V_t tiles into a
//               2-stage ring (128 rows x D, 128-byte swizzle, 4-D tensor maps
//               over [P*B][S][heads][D] so tiles never cross a sequence end).
//   warp 5      MMA issuer (one thread): S_t = Q K_t^T into one of two TMEM
//               score buffers, then O += P_{t-1} V_{t-1} into the TMEM output
//               accumulator, so the score MMA of tile t runs while the softmax
//               warps work on tile t-1.  Completion is signalled with
//               tcgen05.commit on mbarriers.
//   warps 0-3   softmax: thread i owns query row i = TMEM lane i.  It reads its
//               score row from TMEM, applies scale and mask, keeps a running
//               max in the base-2 domain and rescales the TMEM accumulator only
//               when the max grows by more than 2^8 (otherwise the stale max is
//               kept: every exponent stays <= 2^8, exact in fp32 and bf16), and
//               writes P (bf16) into one of two shared-memory buffers in the
//               swizzled K-major layout the next MMA reads.  At the end it
//               divides by the row sum and stores O (bf16) and the LSE.
// Causal tiles beyond the diagonal are skipped entirely; only the diagonal
// tile is masked.  CTAs are ordered longest-first (highest query tile first)
// so the triangular work balances across the 152 SMs.
// Every wait is bounded (a few seconds); a timeout sets a status bit, the CTA
// drains its outstanding tensor-core work, frees TMEM and exits.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace ulysses {
namespace {

using namespace sm100;

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;  // S buffers at columns 0 and 128, O at 256
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)

template <int D>
struct Layout {
  static constexpr uint32_t kTile = 128u * D * 2;  // one 128-row tile of Q, K or V
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTile;          // 2 stages
  static constexpr uint32_t kV = kK + 2 * kTile;      // 2 stages
  static constexpr uint32_t kP = kV + 2 * kTile;      // 2 buffers of 128x128 bf16
  static constexpr uint32_t kBar = kP + 2 * 2 * kChunkBytes;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;   // room to align the base to 1024
};

// Barrier slots (byte offsets inside the barrier block).
enum : uint32_t {
  kBarQFull = 0,
  kBarKFull = 8,     // [2]
  kBarKEmpty = 24,   // [2]
  kBarVFull = 40,    // [2]
  kBarVEmpty = 56,   // [2]
  kBarSFull = 72,    // [2]
  kBarPFull = 88,    // [2]
  kBarPVDone = 104,  // [2]
  kBarDrain = 120,
  kTmemSlot = 128,
  kAbortSlot = 132
};

struct FwdParams {
  int B, S, P, hp, kvp, group, causal, n_qt;
  float scale_log2;
  __nv_bfloat16 *o;  // [P][B][S][hp][D]
  float *lse;        // [P][B][hp][S]
  uint32_t *status;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const volatile uint32_t *gst) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, gst);
  return __all_sync(0xffffffffu, ok);
}

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
  const uint32_t sQ = sb + L::kQ, sK = sb + L::kK, sV = sb + L::kV, sP = sb + L::kP;
  const uint32_t bar = sb + L::kBar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBar + kAbortSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const volatile uint32_t *gst = p.status;
  // A CTA of this grid (or an earlier launch on this workspace) gave up on a
  // wait: do not start more work.
  if (*gst & (ULYSSES_STATUS_FWD_TIMEOUT | ULYSSES_STATUS_BWD_TIMEOUT)) return;
  const int heads_total = p.P * p.B * p.hp;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / heads_total);  // longest tiles first
  const int hid = (int)(blockIdx.x % heads_total);
  const int j = hid % p.hp;
  const int rb = hid / p.hp;  // r*B + b
  const int kl = j / p.group;
  const int n_kv = p.causal ? qt + 1 : (p.S + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(bar + kBarQFull, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + kBarKFull + 8 * i, 1);
      mbar_init(bar + kBarKEmpty + 8 * i, 1);
      mbar_init(bar + kBarVFull + 8 * i, 1);
      mbar_init(bar + kBarVEmpty + 8 * i, 1);
      mbar_init(bar + kBarSFull + 8 * i, 1);
      mbar_init(bar + kBarPFull + 8 * i, 128);
      mbar_init(bar + kBarPVDone + 8 * i, 1);
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

  if (warp == kTmaWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar + kBarQFull, L::kTile);
      for (int c = 0; c < kChunks; ++c)
        tma_load_4d(sQ + c * kChunkBytes, &tmQ, bar + kBarQFull, c * 64, j, qt * BM, rb);
      int issued_k = -1, issued_v = -1;
      for (int t = 0; t < n_kv; ++t) {
        const int st = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!mbar_wait_bounded(bar + kBarKEmpty + 8 * st, ph ^ 1, abort_flag, gst)) break;
        mbar_arrive_expect_tx(bar + kBarKFull + 8 * st, L::kTile);
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(sK + st * L::kTile + c * kChunkBytes, &tmK, bar + kBarKFull + 8 * st, c * 64,
                      kl, t * BN, rb);
        issued_k = t;
        if (!mbar_wait_bounded(bar + kBarVEmpty + 8 * st, ph ^ 1, abort_flag, gst)) break;
        mbar_arrive_expect_tx(bar + kBarVFull + 8 * st, L::kTile);
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(sV + st * L::kTile + c * kChunkBytes, &tmV, bar + kBarVFull + 8 * st, c * 64,
                      kl, t * BN, rb);
        issued_v = t;
      }
      if (*abort_flag) {
        // Let the copies already in flight land before the CTA goes away.
        volatile int never = 0;
        mbar_wait_bounded(bar + kBarQFull, 0, &never, nullptr, 500000000ull);
        for (int t = issued_k - 1; t <= issued_k; ++t)
          if (t >= 0) mbar_wait_bounded(bar + kBarKFull + 8 * (t & 1), (t >> 1) & 1, &never, nullptr, 500000000ull);
        for (int t = issued_v - 1; t <= issued_v; ++t)
          if (t >= 0) mbar_wait_bounded(bar + kBarVFull + 8 * (t & 1), (t >> 1) & 1, &never, nullptr, 500000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);  // P K-major, V MN-major
      auto issue_pv = [&](int i) -> bool {
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait_bounded(bar + kBarPFull + 8 * st, ph, abort_flag, gst)) return false;
        if (!mbar_wait_bounded(bar + kBarVFull + 8 * st, ph, abort_flag, gst)) return false;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(
              sP + st * 2 * kChunkBytes + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(sV + st * L::kTile + kk * 16 * 128, kChunkBytes, 1024);
          mma_bf16_ss(tmem + kColO, a, b, idPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar + kBarPVDone + 8 * st);
        mma_commit(bar + kBarVEmpty + 8 * st);
        return true;
      };
      bool ok = mbar_wait_bounded(bar + kBarQFull, 0, abort_flag, gst);
      for (int t = 0; ok && t < n_kv; ++t) {
        const int st = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!mbar_wait_bounded(bar + kBarKFull + 8 * st, ph, abort_flag, gst)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          const uint64_t a = smem_desc_sw128(sQ + koff, 16, 1024);
          const uint64_t b = smem_desc_sw128(sK + st * L::kTile + koff, 16, 1024);
          mma_bf16_ss(tmem + st * BN, a, b, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar + kBarSFull + 8 * st);
        mma_commit(bar + kBarKEmpty + 8 * st);
        if (t > 0) ok = issue_pv(t - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      // All tensor-core work of this CTA is complete once this commit lands.
      mma_commit(bar + kBarDrain);
      volatile int never = 0;
      mbar_wait_bounded(bar + kBarDrain, 0, &never, nullptr);
    }
  } else {
    // ---------------------------------------------------------- softmax warps
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const int qpos = qt * BM + row;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n_kv; ++t) {
      const int st = t & 1;
      if (!warp_wait(bar + kBarSFull + 8 * st, (t >> 1) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sr[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem + lane_base + st * BN + c * 32, sr[c]);
      tmem_wait_ld();
      float s[BN];
      const int kv0 = t * BN;
      const bool need_mask = (p.causal && t == qt) || (kv0 + BN > p.S);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        float x = __uint_as_float(sr[c >> 5][c & 31]) * p.scale_log2;
        if (need_mask) {
          const int kv = kv0 + c;
          if (kv >= p.S || (p.causal && kv > qpos)) x = -INFINITY;
        }
        s[c] = x;
        mx = fmaxf(mx, x);
      }
      // P buffer `st` is free once the PV MMA of tile t-2 has completed.
      if (t >= 2 && !warp_wait(bar + kBarPVDone + 8 * st, ((t - 2) >> 1) & 1, abort_flag, gst)) {
        ok = false;
        break;
      }
      const bool need = mx > m_used + 8.0f;  // first tile: m_used = -inf
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m_used - mx) : 1.0f;
        if (t >= 1) {
          // Rescale the accumulator row once the PV MMA of tile t-1 is done.
          if (!warp_wait(bar + kBarPVDone + 8 * ((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, gst)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + kColO + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(tmem + lane_base + kColO + c * 32, r);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_used = mx;
        }
      }
      uint32_t pk[BN / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = ex2(s[2 * c] - m_used), p1 = ex2(s[2 * c + 1] - m_used);
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += rs;
      // Row `row` of P into buffer st: two 64-key chunks, 8 swizzled 16-byte units each.
      const uint32_t prow = sP + st * 2 * kChunkBytes + row * 128;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int w = ch * 32 + u * 4;
          st_shared_v4(prow + ch * kChunkBytes + ((u ^ (row & 7)) << 4), pk[w], pk[w + 1], pk[w + 2],
                       pk[w + 3]);
        }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar + kBarPFull + 8 * st);
    }
    // --------------------------------------------------------------- epilogue
    if (ok) ok = warp_wait(bar + kBarPVDone + 8 * ((n_kv - 1) & 1), ((n_kv - 1) >> 1) & 1, abort_flag, gst);
    if (ok) {
      tc_fence_after_sync();
      const float inv = 1.0f / l;
      __nv_bfloat16 *orow = p.o + (((size_t)rb * p.S + qpos) * p.hp + j) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColO + c * 32, r);
        tmem_wait_ld();
        if (qpos < p.S) {
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
      if (qpos < p.S)
        p.lse[((size_t)rb * p.hp + j) * p.S + qpos] = (m_used + log2f(l)) * 0.69314718055994530942f;
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

bool make_map(const TmaEncoder &enc, CUtensorMap *m, const void *base, int D, int heads, int S,
              int PB) {
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)S, (cuuint64_t)PB};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2,
                                 (cuuint64_t)S * heads * D * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const ulysses_problem &p, const TmaEncoder &enc, const void *q, const void *k,
                     const void *v, void *o, float *lse, uint32_t *status, cudaStream_t st) {
  const int hp = p.n_head / p.P, kvp = p.n_kv_head / p.P;
  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, q, D, hp, p.S, p.P * p.B) || !make_map(enc, &mk, k, D, kvp, p.S, p.P * p.B) ||
      !make_map(enc, &mv, v, D, kvp, p.S, p.P * p.B))
    return cudaErrorInvalidValue;
  FwdParams fp;
  fp.B = p.B;
  fp.S = p.S;
  fp.P = p.P;
  fp.hp = hp;
  fp.kvp = kvp;
  fp.group = hp / kvp;
  fp.causal = p.causal;
  fp.n_qt = (p.S + BM - 1) / BM;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)D);
  fp.scale_log2 = scale * 1.4426950408889634f;
  fp.o = static_cast<__nv_bfloat16 *>(o);
  fp.lse = lse;
  fp.status = status;
  const long long blocks = (long long)fp.n_qt * p.P * p.B * hp;
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
                               cudaStream_t st) {
  if (p.head_dim == 128) return launch_d<128>(p, enc, q, k, v, o, lse, status, st);
  if (p.head_dim == 64) return launch_d<64>(p, enc, q, k, v, o, lse, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace ulysses
