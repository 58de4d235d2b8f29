// attn_fwd_simt.cu -- fp32 attention forward on the CUDA cores.
//
// Per rank r, batch b and local head j (global head g = r*hp + j), every query
// row attends over the full sequence ("Sequence Parallelism II: DeepSpeed
// Ulysses and All-to-All Attention", §2 fourth step).  The fp32 workload asks
// for 1e-4 agreement, which the tf32 tensor-core path cannot give, so this
// kernel keeps every product and sum in fp32 FMA arithmetic with an online
// softmax (one thread per query row, K/V tiles staged in shared memory).
#include <math.h>
#include <stdint.h>

#include "check.cuh"
#include "internal.h"

namespace ulysses {
namespace {

constexpr int kRows = 128;  // query rows per block (one per thread)
constexpr int kKeys = 32;   // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(kRows) attn_fwd_simt_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    float *__restrict__ o, float *__restrict__ lse, int S, int hp, int kvp, int group, int causal,
    float scale_log2, uint32_t *status, long long qo_n, long long kv_n, long long lse_n) {
  __shared__ float Ks[kKeys][D];
  __shared__ float Vs[kKeys][D];
  const int n_qt = (S + kRows - 1) / kRows;
  const int qt = blockIdx.x % n_qt;
  const long long hid = blockIdx.x / n_qt;  // (r*B + b)*hp + j
  const int j = (int)(hid % hp);
  const long long rb = hid / hp;
  const int kl = j / group;
  const int i = qt * kRows + threadIdx.x;
  const bool live = i < S;

  float qr[D], acc[D];
  const long long qoff = ((rb * S + (live ? i : 0)) * hp + j) * D;
  const float *qrow = q + qoff;
  const bool get = live && in_range(status, qoff, D, qo_n);
#pragma unroll
  for (int e = 0; e < D; ++e) {
    qr[e] = get ? qrow[e] : 0.f;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int kend = causal ? min(S, qt * kRows + kRows) : S;
  const float *kbase = k + (rb * S * kvp + kl) * D;
  const float *vbase = v + (rb * S * kvp + kl) * D;
  for (int k0 = 0; k0 < kend; k0 += kKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeys * D; idx += kRows) {
      const int rr = idx / D, e = idx % D;
      const int kk = k0 + rr;
      const bool in = kk < S && in_range(status, (rb * S * kvp + kl) * D + (long long)kk * kvp * D + e, 1, kv_n);
      Ks[rr][e] = in ? kbase[(long long)kk * kvp * D + e] : 0.f;
      Vs[rr][e] = in ? vbase[(long long)kk * kvp * D + e] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    for (int rr = 0; rr < kKeys; ++rr) {
      const int kk = k0 + rr;
      if (kk >= S || (causal && kk > i)) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) dot = fmaf(qr[e], Ks[rr][e], dot);
      const float s = dot * scale_log2;
      if (s > m) {
        const float a = exp2f(m - s);
        l *= a;
#pragma unroll
        for (int e = 0; e < D; ++e) acc[e] *= a;
        m = s;
      }
      const float pe = exp2f(s - m);
      l += pe;
#pragma unroll
      for (int e = 0; e < D; ++e) acc[e] = fmaf(pe, Vs[rr][e], acc[e]);
    }
  }
  if (!live) return;
  const float inv = 1.f / l;
  const long long ooff = ((rb * S + i) * hp + j) * D;
  float *orow = o + ooff;
  if (in_range(status, ooff, D, qo_n)) {
#pragma unroll
    for (int e = 0; e < D; ++e) orow[e] = acc[e] * inv;
  }
  if (in_range(status, hid * S + i, 1, lse_n)) lse[hid * S + i] = (m + log2f(l)) * 0.69314718055994530942f;
}

}  // namespace

cudaError_t launch_attn_fwd_simt(const ulysses_problem &p, const float *q, const float *k,
                                 const float *v, float *o, float *lse, uint32_t *status, cudaStream_t st) {
  const long long qo_n = (long long)p.B * p.S * p.n_head * p.head_dim;
  const long long kv_n = (long long)p.P * p.B * p.S * kv_per_rank(p) * p.head_dim;
  const long long lse_n = (long long)p.B * p.n_head * p.S;
  const int hp = p.n_head / p.P, kvp = kv_per_rank(p), group = hp / kvp;
  const int n_qt = (p.S + kRows - 1) / kRows;
  const long long blocks = (long long)n_qt * p.P * p.B * hp;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
  const float scale_log2 = scale * 1.4426950408889634f;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  switch (p.head_dim) {
    case 32:
      attn_fwd_simt_kernel<32><<<(unsigned)blocks, kRows, 0, st>>>(q, k, v, o, lse, p.S, hp, kvp, group, p.causal, scale_log2,
                                                                  status, qo_n, kv_n, lse_n);
      break;
    case 64:
      attn_fwd_simt_kernel<64><<<(unsigned)blocks, kRows, 0, st>>>(q, k, v, o, lse, p.S, hp, kvp, group, p.causal, scale_log2,
                                                                  status, qo_n, kv_n, lse_n);
      break;
    case 128:
      attn_fwd_simt_kernel<128><<<(unsigned)blocks, kRows, 0, st>>>(q, k, v, o, lse, p.S, hp, kvp, group, p.causal, scale_log2,
                                                                  status, qo_n, kv_n, lse_n);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ulysses
