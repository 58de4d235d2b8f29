// qkv_proj_tc.cu -- the QKV projection with the seq -> head All-to-All and
// RoPE fused into its epilogue, on the 5th-generation tensor cores.
//
// "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention", §2
// second and third steps: every rank applies the complete (replicated) q/k/v
// projections to its own tokens, then the All-to-All hands each rank its heads
// over the full sequence; "Comparing Ulysses and Megatron Sequence
// Parallelism", "A simple attention skeleton": q, k, v = x W^T, viewed as
// heads, RoPE on q and k, then the transpose.
//
// All P virtual ranks' tokens form one GEMM: X [M = P*B*Sl][H] (the
// sequence-sharded activations, rank-major) times W^T, W [N][H] with
// N = (n_head + 2 n_kv_head) * D (the three projection weights stacked, rows
// q, then k, then v, in the Linear layout [out][in]).  The epilogue adds the
// optional bias, rotates q and k pairs (i, i + D/2) by the token's global
// position in fp32 and writes each row of each head straight to its place in
// the head-sharded layout of the rank that owns the head (with replicated
// kv-heads, to every replica): the pack becomes the epilogue's addressing and
// the projection output never makes an HBM round trip.
//
// Persistent CTAs, one per SM, over 128 x 256 tiles (two heads at D = 128)
// in groups of 8 M-tiles per N-sweep (the group's W tiles stay in L2).
//   warp 8      TMA: X and W tiles of 64 columns of H (one 128-byte swizzle
//               row) through a 4-stage ring.
//   warp 9      MMA issuer: 128x256x16 tcgen05.mma, both operands K-major,
//               into one of two 256-column TMEM accumulators; every wait of
//               a burst of two stages (8 MMAs) is taken before it is issued.
//   warps 0-7   epilogue: warpgroup g owns columns [128g, 128g + 128) of a
//               tile, thread = token row = TMEM lane; it drains accumulator
//               t & 1 while the MMAs of the next tile fill the other.
// All waits are bounded; a timeout sets the forward-timeout status bit.
//
// The same kernel in its second mode is the output projection fused with the
// head -> seq All-to-All ([SP2] §2 fifth step: the inverse All-to-All restores
// [B, S/P, H], then every rank applies the complete output projection to its
// tokens; [CMP] skeleton: y = output_proj(y)).  The A operand is the attention
// output in head layout: the 64 input features of a K-block lie in one head,
// computed by rank head / hp, and a 128-token tile lies in one sequence shard
// (S/P a multiple of 128), so each A tile is one TMA box of that rank's
// head-sharded buffer at the tile's global positions -- the unpack becomes the
// load addressing.  The epilogue adds the bias and writes sequence-layout rows.
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

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr int kGroupM = 8;  // M-tiles per N-sweep
constexpr uint32_t kATile = BM * BK * 2;  // 16 KB
constexpr uint32_t kBTile = BN * BK * 2;  // 32 KB
constexpr uint32_t kStage = kATile + kBTile;
constexpr uint32_t kBarOff = kStages * kStage;
enum : uint32_t {
  kBFull = 0,       // [4]
  kBEmpty = 32,     // [4]
  kBAccFull = 64,   // [2]
  kBAccEmpty = 80,  // [2], 256 arrivals
  kBDrain = 96,
  kBTmem = 104,
  kBAbort = 108
};
constexpr uint32_t kAlloc = kBarOff + 128 + 1024;  // room to align the base to 1024

enum ProjMode { kQkvPack = 0, kOutUnpack = 1 };

struct ProjParams {
  int M, N, H;  // tokens (P*B*Sl), output features, input features
  int B, Sl, S, P, n_head, n_kv, hp, kvp, R;
  int n_mt, n_nt;
  const __nv_bfloat16 *bias;         // [N] or null
  const float *rope_cos, *rope_sin;  // [S][D/2] or null
  __nv_bfloat16 *q, *k, *v;          // head layout (QKV mode)
  __nv_bfloat16 *y;                  // [P][B][Sl][N] sequence layout (output mode)
  uint32_t *status;
  uint32_t rope_key;
  // elements of q / k / v (head layout) or y, and of each RoPE table (range
  // checks of a checked build; the bias has N)
  long long q_n, kv_n, y_n, rope_n;
};

__device__ __forceinline__ void tile_mn(const ProjParams &p, int t, int &m, int &n) {
  const int grp = t / (kGroupM * p.n_nt);
  const int first = grp * kGroupM;
  const int gm = min(kGroupM, p.n_mt - first);
  const int r = t - grp * kGroupM * p.n_nt;
  m = first + r % gm;
  n = r / gm;
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sb = raw + pad, bar = sb + kBarOff;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kBarOff + kBAbort);
  const volatile uint32_t *gst = p.status;
  if (*gst & (ULYSSES_STATUS_FWD_TIMEOUT | ULYSSES_STATUS_BWD_TIMEOUT)) return;
  if (p.rope_cos && p.status[1] != p.rope_key) {  // workspace prepared for another problem
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_ROPE_TABLE);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = p.n_mt * p.n_nt;
  const int n_k = p.H / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar + kBFull + 8 * i, 1);
      mbar_init(bar + kBEmpty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + kBAccFull + 8 * i, 1);
      mbar_init(bar + kBAccEmpty + 8 * i, 256);
    }
    mbar_init(bar + kBDrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_alloc(bar + kBTmem, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kBarOff + kBTmem);

  if (warp == kTmaWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW);
      long long it = 0, issued = -1;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        int m, n;
        tile_mn(p, t, m, n);
        for (int kb = 0; kb < n_k; ++kb, ++it) {
          const int st = (int)(it % kStages);
          if (!(ok = mbar_wait_bounded(bar + kBEmpty + 8 * st, (uint32_t)((it / kStages) & 1) ^ 1u, abort_flag, gst)))
            break;
          mbar_arrive_expect_tx(bar + kBFull + 8 * st, kStage);
          const uint32_t sA = sb + st * kStage;
          if (MODE == kQkvPack) {
            dev::tma_load_2d(sA, &tmX, bar + kBFull + 8 * st, kb * BK, m * BM);
          } else {
            // features [64kb, 64kb+64) are elements e0.. of head hd (rank hd / hp,
            // local head hd % hp); tokens m*128.. are positions pos0.. of (s, b)
            const int f0 = kb * BK, hd = f0 / D, e0 = f0 - hd * D;
            const int m0 = m * BM, sbk = m0 / p.Sl, pos0 = (sbk / p.B) * p.Sl + (m0 - sbk * p.Sl);
            tma_load_4d(sA, &tmX, bar + kBFull + 8 * st, e0, hd % p.hp, pos0, (hd / p.hp) * p.B + sbk % p.B);
          }
          dev::tma_load_2d(sA + kATile, &tmW, bar + kBFull + 8 * st, kb * BK, n * BN);
          issued = it;
        }
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA goes away
        volatile int never = 0;
        for (long long i = issued - (kStages - 1); i <= issued; ++i)
          if (i >= 0)
            mbar_wait_bounded(bar + kBFull + 8 * (int)(i % kStages), (uint32_t)((i / kStages) & 1), &never, nullptr,
                              500000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);  // X, W both K-major
      long long it = 0;
      int ti = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++ti) {
        const int acc = ti & 1;
        // the epilogue has drained this accumulator (tile ti - 2)
        if (!(ok = mbar_wait_bounded(bar + kBAccEmpty + 8 * acc, (uint32_t)((ti >> 1) & 1) ^ 1u, abort_flag, gst)))
          break;
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; ok && kb < n_k; kb += 2) {
          const int nb = min(2, n_k - kb);
          for (int q = 0; q < nb; ++q) {
            const long long i = it + q;
            if (!(ok = mbar_wait_bounded(bar + kBFull + 8 * (int)(i % kStages), (uint32_t)((i / kStages) & 1),
                                         abort_flag, gst)))
              break;
          }
          if (!ok) break;
          tc_fence_after_sync();
          for (int q = 0; q < nb; ++q, ++it) {
            const int st = (int)(it % kStages);
            const uint32_t sA = sb + st * kStage, sB = sA + kATile;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_bf16_ss(d, smem_desc_sw128(sA + kk * 32, 16, 1024), smem_desc_sw128(sB + kk * 32, 16, 1024), idesc,
                          (kb + q > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar + kBEmpty + 8 * st);
          }
        }
        if (ok) mma_commit(bar + kBAccFull + 8 * acc);
      }
      mma_commit(bar + kBDrain);
      volatile int never = 0;
      mbar_wait_bounded(bar + kBDrain, 0, &never, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int g = warp >> 2, w4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const int n_heads_out = p.n_head + 2 * p.n_kv;
    int ti = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++ti) {
      int m, n;
      tile_mn(p, t, m, n);
      const int acc = ti & 1;
      if (!warp_wait(bar + kBAccFull + 8 * acc, (uint32_t)((ti >> 1) & 1), abort_flag, gst)) break;
      tc_fence_after_sync();
      const int row = m * BM + w4 * 32 + lane;
      const bool live = row < p.M;
      if (MODE == kOutUnpack) {
        // plain sequence-layout rows: columns [128g, 128g+128) of the tile, + bias
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = n * BN + g * 128 + c * 32;
          if (col >= p.N) break;  // ragged feature tail: the same for the whole warp
          uint32_t xr[32];
          tmem_ld32(tmem + lane_base + acc * BN + g * 128 + c * 32, xr);
          tmem_wait_ld();
          reg_fence(xr);
          uint32_t wx[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a = __uint_as_float(xr[2 * e]), b2 = __uint_as_float(xr[2 * e + 1]);
            if (p.bias) {
              a += __bfloat162float(p.bias[col + 2 * e]);
              b2 += __bfloat162float(p.bias[col + 2 * e + 1]);
            }
            wx[e] = pack_bf16x2(a, b2);
          }
          if (live && in_range(p.status, (long long)row * p.N + col, 32, p.y_n) &&
              (!p.bias || in_range(p.status, col, 32, p.N))) {
            uint4 *o = reinterpret_cast<uint4 *>(p.y + (size_t)row * p.N + col);
#pragma unroll
            for (int v = 0; v < 4; ++v) o[v] = make_uint4(wx[4 * v], wx[4 * v + 1], wx[4 * v + 2], wx[4 * v + 3]);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(bar + kBAccEmpty + 8 * acc);
        continue;
      }
      const int rr = live ? row : 0;
      const int tt = rr % p.Sl, sbk = rr / p.Sl;  // row = (s*B + b)*Sl + t
      const int b = sbk % p.B, s = sbk / p.B;
      const int pos = s * p.Sl + tt;
#pragma unroll
      for (int hh = 0; hh < 128 / D; ++hh) {
        const int col0 = n * BN + g * 128 + hh * D;  // first output feature of this head
        const int hd = col0 / D;                     // head in [q heads | k heads | v heads]
        if (hd >= n_heads_out) break;                // ragged N tail: the same for the whole warp
        int kind, head;
        if (hd < p.n_head) {
          kind = 0;
          head = hd;
        } else if (hd < p.n_head + p.n_kv) {
          kind = 1;
          head = hd - p.n_head;
        } else {
          kind = 2;
          head = hd - p.n_head - p.n_kv;
        }
        const bool rope = p.rope_cos != nullptr && kind < 2;
        const uint32_t tcol = tmem + lane_base + acc * BN + g * 128 + hh * D;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          // elements i = 32c .. 32c+31 and their rotation partners i + D/2
          uint32_t xr[32], yr[32];
          tmem_ld32(tcol + c * 32, xr);
          tmem_ld32(tcol + D / 2 + c * 32, yr);
          tmem_wait_ld();
          reg_fence(xr);
          reg_fence(yr);
          float fx[32], fy[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            fx[e] = __uint_as_float(xr[e]);
            fy[e] = __uint_as_float(yr[e]);
          }
          if (p.bias && in_range(p.status, col0 + c * 32, D / 2 + 32, p.N)) {
            const __nv_bfloat16 *bx = p.bias + col0 + c * 32, *by = bx + D / 2;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              fx[e] += __bfloat162float(bx[e]);
              fy[e] += __bfloat162float(by[e]);
            }
          }
          if (rope && in_range(p.status, (long long)pos * (D / 2) + c * 32, 32, p.rope_n)) {
            // x' = x cos a - y sin a, y' = y cos a + x sin a, a = pos * theta_i
            const float *cs = p.rope_cos + (size_t)pos * (D / 2) + c * 32;
            const float *sn = p.rope_sin + (size_t)pos * (D / 2) + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 c4 = *reinterpret_cast<const float4 *>(cs + e);
              const float4 s4 = *reinterpret_cast<const float4 *>(sn + e);
              const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float x = fx[e + q], y = fy[e + q];
                fx[e + q] = x * cc[q] - y * ss[q];
                fy[e + q] = y * cc[q] + x * ss[q];
              }
            }
          }
          uint32_t wx[16], wy[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            wx[e] = pack_bf16x2(fx[2 * e], fx[2 * e + 1]);
            wy[e] = pack_bf16x2(fy[2 * e], fy[2 * e + 1]);
          }
          if (live) {
            // destination rank(s), local head and layout width of this head
            int d0, nd, j, width;
            __nv_bfloat16 *base;
            if (kind == 0) {
              d0 = head / p.hp, nd = 1, j = head % p.hp, width = p.hp, base = p.q;
            } else {
              base = kind == 1 ? p.k : p.v;
              if (p.R > 1)
                d0 = head * p.R, nd = p.R, j = 0, width = 1;
              else
                d0 = head / p.kvp, nd = 1, j = head % p.kvp, width = p.kvp;
            }
            for (int dd = 0; dd < nd; ++dd) {
              const long long off = ((((long long)(d0 + dd) * p.B + b) * p.S + pos) * width + j) * D + c * 32;
              if (!in_range(p.status, off, D / 2 + 32, kind == 0 ? p.q_n : p.kv_n)) continue;
              __nv_bfloat16 *dst = base + off;
              uint4 *ox = reinterpret_cast<uint4 *>(dst), *oy = reinterpret_cast<uint4 *>(dst + D / 2);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                ox[v] = make_uint4(wx[4 * v], wx[4 * v + 1], wx[4 * v + 2], wx[4 * v + 3]);
                oy[v] = make_uint4(wy[4 * v], wy[4 * v + 1], wy[4 * v + 2], wy[4 * v + 3]);
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(bar + kBAccEmpty + 8 * acc);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_FWD_TIMEOUT);
}

template <int D, int MODE>
cudaError_t launch_d(const ulysses_problem &p, const TmaEncoder &enc, const void *x, const void *w,
                     const void *bias, void *q, void *k, void *v, void *y, const void *ws, cudaStream_t st) {
  ProjParams pp;
  pp.H = MODE == kQkvPack ? p.hidden : p.n_head * D;
  pp.M = p.B * p.S;
  pp.N = MODE == kQkvPack ? (p.n_head + 2 * p.n_kv_head) * D : p.hidden;
  pp.B = p.B;
  pp.Sl = p.S / p.P;
  pp.S = p.S;
  pp.P = p.P;
  pp.n_head = p.n_head;
  pp.n_kv = p.n_kv_head;
  pp.hp = p.n_head / p.P;
  pp.kvp = kv_per_rank(p);
  pp.R = kv_replicas(p);
  pp.n_mt = (pp.M + BM - 1) / BM;
  pp.n_nt = (pp.N + BN - 1) / BN;
  pp.bias = static_cast<const __nv_bfloat16 *>(bias);
  const WorkspaceLayout L = workspace_layout(p);
  const uint8_t *wsb = static_cast<const uint8_t *>(ws);
  if (p.use_rope) {
    pp.rope_cos = reinterpret_cast<const float *>(wsb + L.rope);
    pp.rope_sin = pp.rope_cos + (size_t)p.S * (D / 2);
  } else {
    pp.rope_cos = pp.rope_sin = nullptr;
  }
  pp.q = static_cast<__nv_bfloat16 *>(q);
  pp.k = static_cast<__nv_bfloat16 *>(k);
  pp.v = static_cast<__nv_bfloat16 *>(v);
  pp.y = static_cast<__nv_bfloat16 *>(y);
  if (MODE == kOutUnpack) pp.rope_cos = pp.rope_sin = nullptr;  // no rotation on the output
  pp.status = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(wsb + L.status));
  pp.rope_key = rope_key(p);
  pp.q_n = (long long)p.B * p.S * p.n_head * D;
  pp.kv_n = (long long)p.P * p.B * p.S * pp.kvp * D;
  pp.y_n = (long long)pp.M * p.hidden;
  pp.rope_n = (long long)p.S * (D / 2);
  CUtensorMap mx, mw;
  const bool ok_x = MODE == kQkvPack ? make_mat_map(enc, &mx, x, pp.H, pp.M, BM)
                                     : make_act_map(enc, &mx, x, D, pp.hp, p.S, p.P * p.B, BM);
  if (!ok_x || !make_mat_map(enc, &mw, w, pp.H, pp.N, BN)) return cudaErrorInvalidValue;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)pp.n_mt * pp.n_nt;
  if (tiles > 0x7fffffffll) return cudaErrorInvalidValue;
  const int grid = (int)(tiles < sms ? tiles : sms);
  cudaError_t e =
      cudaFuncSetAttribute(qkv_proj_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAlloc);
  if (e != cudaSuccess) return e;
  qkv_proj_kernel<D, MODE><<<grid, kThreads, kAlloc, st>>>(mx, mw, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qkv_proj_pack(const ulysses_problem &p, const TmaEncoder &enc, const void *x, const void *w,
                                 const void *bias, void *q, void *k, void *v, const void *ws, cudaStream_t st) {
  if (p.head_dim == 128) return launch_d<128, kQkvPack>(p, enc, x, w, bias, q, k, v, nullptr, ws, st);
  if (p.head_dim == 64) return launch_d<64, kQkvPack>(p, enc, x, w, bias, q, k, v, nullptr, ws, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_out_proj_unpack(const ulysses_problem &p, const TmaEncoder &enc, const void *o_head,
                                   const void *w, const void *bias, void *y, const void *ws, cudaStream_t st) {
  if (p.head_dim == 128)
    return launch_d<128, kOutUnpack>(p, enc, o_head, w, bias, nullptr, nullptr, nullptr, y, ws, st);
  if (p.head_dim == 64)
    return launch_d<64, kOutUnpack>(p, enc, o_head, w, bias, nullptr, nullptr, nullptr, y, ws, st);
  return cudaErrorInvalidValue;
}

}  // namespace ulysses
