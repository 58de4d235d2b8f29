// permute.cu -- the All-to-All of the Ulysses method as on-device permutations.
//
// "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention", §3:
// every rank splits its local tensor into P pieces, keeps the one addressed to
// itself and sends the rest; afterwards every rank holds one piece from every
// rank.  With all P virtual ranks in one HBM this is a gather/scatter copy:
// the piece rank s sends to rank d is s's head slice [d*hp, (d+1)*hp) of every
// local token, and rank d stores it at sequence block s (§1: rank 0 goes from
// S0H0,S0H1,S0H2,S0H3 to S0H0,S1H0,S2H0,S3H0).
//
// One kernel serves both directions.  It walks the sequence-sharded index
// space (token row (s, b, t), destination rank d, local head j, 16-byte chunk
// c) and computes the head-sharded address of the same element; `to_head`
// selects which side is read.  For each (row, d) the hp*D elements of the
// piece are contiguous on both sides, so a warp moves contiguous 512-byte
// spans with 16-byte vector loads and stores.  RoPE ("Comparing Ulysses and
// Megatron Sequence Parallelism", skeleton: rope before the transpose) is
// fused: a thread owning chunk c of the first half also owns chunk c of the
// second half, so each rotation pair (i, i + D/2) is in one thread.
// In the Ulysses x ring hybrid ("Sequence Parallelism II", §4 and §8) the
// same All-to-All runs inside each ring position: source rank s sends to the
// Pu ranks (s / Pu)*Pu + d of its own ring position, which store the piece at
// row (s % Pu)*Sl + t of their Cs = Pu*Sl-token chunk.  Pu = P, Cs = S is
// plain Ulysses.
#include <cuda_bf16.h>
#include <stdint.h>

#include "check.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace ulysses {

namespace {

constexpr int kThreads = 256;
// A block of the permute kernel takes up to this many token rows per pass, so
// that jobs with few (head, chunk) units a row (few kv-heads, D = 64) still
// occupy its threads.
constexpr int kMaxRowsPerPass = 8;

struct PermJob {
  const void *src;  // read side
  void *dst;        // write side
  int heads;        // heads of this tensor
  int rope;         // 0: copy; +1: rotate by +angle; -1: rotate by -angle
  int rep;          // > 1: heads < P and every head goes to `rep` ranks (rank d gets head d / rep)
  long long src_n, dst_n;  // elements of each side (range checks of a checked build)
};

struct PermParams {
  PermJob job[3];
  int njobs;
  int P, B, Sl, D;
  int Pu, Cs;   // ranks of a ring position and its tokens (plain Ulysses: P, S)
  int to_head;  // 1: src is sequence-sharded (pack); 0: src is head-sharded (unpack)
  int nrow;     // token rows a block takes per pass (1 .. kMaxRowsPerPass)
  const float *rope_cos, *rope_sin;  // [S][D/2] each
  const uint32_t *rope_key_ptr;
  uint32_t rope_key;
  uint32_t *status;
  long long rope_n;  // floats in each of cos, sin
};

__device__ __forceinline__ void rotate(float &x, float &y, float c, float s, int dir) {
  // x' = x cos(a) - y sin(a), y' = y cos(a) + x sin(a), a = dir * angle.
  const float sn = dir > 0 ? s : -s;
  const float nx = x * c - y * sn;
  const float ny = y * c + x * sn;
  x = nx;
  y = ny;
}

template <typename T>
struct Chunk;

template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kVec = 8;
  static __device__ __forceinline__ void rope(uint4 &a, uint4 &b, const float *cs, const float *sn,
                                              int dir) {
    uint32_t *pa = reinterpret_cast<uint32_t *>(&a);
    uint32_t *pb = reinterpret_cast<uint32_t *>(&b);
    const float4 c0 = *reinterpret_cast<const float4 *>(cs);
    const float4 c1 = *reinterpret_cast<const float4 *>(cs + 4);
    const float4 s0 = *reinterpret_cast<const float4 *>(sn);
    const float4 s1 = *reinterpret_cast<const float4 *>(sn + 4);
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      __nv_bfloat162 xa = *reinterpret_cast<__nv_bfloat162 *>(&pa[w]);
      __nv_bfloat162 xb = *reinterpret_cast<__nv_bfloat162 *>(&pb[w]);
      float2 fa = __bfloat1622float2(xa), fb = __bfloat1622float2(xb);
      rotate(fa.x, fb.x, cc[2 * w], ss[2 * w], dir);
      rotate(fa.y, fb.y, cc[2 * w + 1], ss[2 * w + 1], dir);
      __nv_bfloat162 ra = __float22bfloat162_rn(fa), rb = __float22bfloat162_rn(fb);
      pa[w] = *reinterpret_cast<uint32_t *>(&ra);
      pb[w] = *reinterpret_cast<uint32_t *>(&rb);
    }
  }
};

template <>
struct Chunk<float> {
  static constexpr int kVec = 4;
  static __device__ __forceinline__ void rope(uint4 &a, uint4 &b, const float *cs, const float *sn,
                                              int dir) {
    float *fa = reinterpret_cast<float *>(&a);
    float *fb = reinterpret_cast<float *>(&b);
    const float4 c0 = *reinterpret_cast<const float4 *>(cs);
    const float4 s0 = *reinterpret_cast<const float4 *>(sn);
    const float cc[4] = {c0.x, c0.y, c0.z, c0.w};
    const float ss[4] = {s0.x, s0.y, s0.z, s0.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) rotate(fa[w], fb[w], cc[w], ss[w], dir);
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) permute_kernel(const PermParams p) {
  constexpr int V = Chunk<T>::kVec;
  const long long rows = (long long)p.P * p.B * p.Sl;
  bool any_rope = false;
#pragma unroll
  for (int q = 0; q < 3; ++q) any_rope |= (q < p.njobs && p.job[q].rope != 0);
  if (any_rope && *p.rope_key_ptr != p.rope_key) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, (uint32_t)ULYSSES_STATUS_ROPE_TABLE);
    return;
  }
  // per pass: each row's batch, global position, ring position and row in
  // that position's chunk, computed once by one thread each
  __shared__ int row_b[kMaxRowsPerPass], row_pos[kMaxRowsPerPass], row_rp[kMaxRowsPerPass],
      row_crow[kMaxRowsPerPass];
  const int nrow = p.nrow;
  for (long long row0 = (long long)blockIdx.x * nrow; row0 < rows; row0 += (long long)gridDim.x * nrow) {
    __syncthreads();  // the previous pass is done with the row table
    if ((int)threadIdx.x < nrow) {
      // row = (s*B + b)*Sl + t : token t of sequence shard s, batch b
      const long long row = row0 + threadIdx.x;
      const int t = (int)(row % p.Sl);
      const long long sb = row / p.Sl;
      const int s = (int)(sb / p.B);
      row_b[threadIdx.x] = (int)(sb % p.B);
      row_pos[threadIdx.x] = s * p.Sl + t;                         // global token position
      row_rp[threadIdx.x] = s / p.Pu;                              // ring position of the source rank
      row_crow[threadIdx.x] = s * p.Sl + t - (s / p.Pu) * p.Cs;    // row of the token in that position's chunk
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      if (q >= p.njobs) break;
      const PermJob J = p.job[q];
      const int hp = J.rep > 1 ? 1 : J.heads / p.Pu;
      // A unit is chunk c of both halves of a head (2 x 16 bytes), rotated or
      // not: two loads in flight per thread either way.  With replicated heads
      // the units run over the P destination ranks (one head each), so a head
      // of the token row is read once per replica.  A pass's nrow rows are
      // laid end to end: task i is unit i % units of row i / units.
      const int cph = p.D / (2 * V);
      const int run = hp * cph;                           // units per destination piece
      const int units = p.Pu * run;
      for (int task = threadIdx.x; task < nrow * units; task += kThreads) {
        const int rl = nrow == 1 ? 0 : task / units;
        const int u = task - rl * units;
        const long long row = row0 + rl;
        if (row >= rows) break;  // rows of a pass run in order: the rest are past the end too
        const int b = row_b[rl], pos = row_pos[rl], rp = row_rp[rl], crow = row_crow[rl];
        const long long seq_row = row * (long long)J.heads * p.D;
        const int d = u / run;  // the rank on the head side of this piece
        const int w = u - d * run;
        const int j = w / cph, c = w - j * cph;
        const long long head_off =
            (((long long)((rp * p.Pu + d) * p.B + b) * p.Cs + crow) * hp + j) * p.D + (long long)c * V;
        const int seq_head = J.rep > 1 ? d / J.rep : d * hp + j;
        const long long seq_off = seq_row + (long long)seq_head * p.D + (long long)c * V;
        const long long src_off = p.to_head ? seq_off : head_off;
        const long long dst_off = p.to_head ? head_off : seq_off;
        const T *src = static_cast<const T *>(J.src);
        T *dst = static_cast<T *>(J.dst);
        const int half = p.D / 2;
        const long long toff = (long long)pos * half + (long long)c * V;
        // a unit spans [off, off + D/2 + V) of each side
        if (!in_range(p.status, src_off, half + V, J.src_n) || !in_range(p.status, dst_off, half + V, J.dst_n) ||
            (J.rope && !in_range(p.status, toff, V, p.rope_n)))
          continue;
        uint4 x = __ldg(reinterpret_cast<const uint4 *>(src + src_off));
        uint4 y = __ldg(reinterpret_cast<const uint4 *>(src + src_off + half));
        if (J.rope) Chunk<T>::rope(x, y, p.rope_cos + toff, p.rope_sin + toff, J.rope);
        *reinterpret_cast<uint4 *>(dst + dst_off) = x;
        *reinterpret_cast<uint4 *>(dst + dst_off + half) = y;
      }
    }
  }
}

// The head -> seq direction with the copy engine.  One warp per block: for
// each token row of the sequence-sharded output it issues P bulk (TMA) loads
// of the hp*D-element pieces (one from every rank's head-sharded buffer) into
// a shared-memory stage and, once they have landed, one bulk store of the
// whole row.  A ring of kBulkStages stages keeps several rows in flight per
// block and many blocks share an SM, so the copy engine, not registers, holds
// the bytes in flight (about 6 TB/s on the pages' sizing).
constexpr int kBulkStages = 4;

template <typename T>
__global__ void __launch_bounds__(32) unpack_bulk_kernel(const PermParams p, uint32_t row_bytes) {
  using namespace sm100;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kBulkStages * row_bytes;  // one mbarrier per stage
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kBulkStages * row_bytes + 8 * kBulkStages);
  const int lane = threadIdx.x;
  const long long rows = (long long)p.P * p.B * p.Sl;
  const PermJob J = p.job[0];
  const int hp = J.heads / p.Pu;
  const uint32_t piece = row_bytes / p.Pu;  // hp * D elements
  const T *src = static_cast<const T *>(J.src);
  T *dst = static_cast<T *>(J.dst);
  if (lane == 0) {
    for (int i = 0; i < kBulkStages; ++i) mbar_init(bar0 + 8 * i, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  const long long n_mine = rows > blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto load_row = [&](long long k) {
    const long long row = blockIdx.x + k * gridDim.x;  // (d*B + b)*Sl + t of the output
    const int t = (int)(row % p.Sl);
    const long long db = row / p.Sl;
    const int d = (int)(db / p.B), b = (int)(db % p.B);
    const int rp = d / p.Pu, crow = (d - rp * p.Pu) * p.Sl + t;  // ring position, row in its chunk
    const uint32_t slot = (uint32_t)(k % kBulkStages);
    const uint32_t stage = sbase + slot * row_bytes, bar = bar0 + 8 * slot;
    if (lane == 0) mbar_arrive_expect_tx(bar, row_bytes);
    __syncwarp();
    // member r of the ring position holds heads [r*hp, (r+1)*hp) of the token
    for (int r = lane; r < p.Pu; r += 32) {
      const long long off = (((long long)((rp * p.Pu + r) * p.B + b) * p.Cs + crow) * hp) * p.D;
      // a skipped piece leaves the stage's transaction count short: that
      // stage's wait then times out and reports, as the check already has
      if (in_range(p.status, off, (long long)hp * p.D, J.src_n)) bulk_load(stage + r * piece, src + off, piece, bar);
    }
  };
  long long issued = -1, failed = n_mine;
  for (long long k = 0; k < kBulkStages - 1 && k < n_mine; ++k) load_row(issued = k);
  bool ok = true;
  for (long long k = 0; k < n_mine; ++k) {
    if (k + kBulkStages - 1 < n_mine) {
      if (lane == 0) bulk_wait_read_all();  // row k-1's store has left its stage
      __syncwarp();
      load_row(issued = k + kBulkStages - 1);
    }
    failed = k;
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * (uint32_t)(k % kBulkStages),
                                                   (uint32_t)((k / kBulkStages) & 1), abort_flag, p.status));
    if (!ok) break;
    failed = n_mine;
    if (lane == 0) {
      const long long row = blockIdx.x + k * gridDim.x;
      if (in_range(p.status, row * J.heads * p.D, (long long)J.heads * p.D, J.dst_n))
        bulk_store(dst + row * (long long)J.heads * p.D, sbase + (uint32_t)(k % kBulkStages) * row_bytes, row_bytes);
      bulk_commit();
    }
  }
  if (!ok) {
    // Let the loads already in flight land before the block goes away.
    volatile int never = 0;
    for (long long k = failed; k <= issued; ++k)
      mbar_wait_bounded(bar0 + 8 * (uint32_t)(k % kBulkStages), (uint32_t)((k / kBulkStages) & 1), &never,
                        nullptr, 200000000ull);
  }
  if (lane == 0) bulk_wait_all();
}

// cos/sin(p * base^(-2i/D)) in double precision, rounded to float.
__global__ void rope_table_kernel(float *cs, float *sn, int S, int D, double base, uint32_t *hdr,
                                  uint32_t key) {
  const int half = D / 2;
  const long long n = (long long)S * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(idx / half), i = (int)(idx % half);
    const double theta = pow(base, -2.0 * i / D);
    double sv, cv;
    sincos((double)pos * theta, &sv, &cv);
    cs[idx] = (float)cv;
    sn[idx] = (float)sv;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr[0] = 0u;   // status word
    hdr[1] = key;  // table key
  }
}

// dO: seq -> head, plus delta[d][b][j][pos] = sum_e dO * O (O read in head layout)
// and nlse = -lse * log2(e) at the same index (the exponent offset the backward
// kernels add to scale * s * log2(e)).  kFolded: O is read in sequence layout,
// at dO's own offset, and dO is not packed (the folded backward reads it in
// place); delta and nlse as above.
// One block per token row at a time (grid-stride over rows): the row's index
// arithmetic is done once, and its H*D/8 (head, 16-byte chunk) tasks are
// spread over the block's threads, D/8 consecutive lanes per head; bf16 only.
template <bool kFolded>
__global__ void __launch_bounds__(kThreads)
    pack_do_delta_kernel(const __nv_bfloat16 *__restrict__ dout, const __nv_bfloat16 *__restrict__ o,
                         const float *__restrict__ lse, __nv_bfloat16 *__restrict__ do_head,
                         float *__restrict__ delta, float *__restrict__ nlse, int P, int B,
                         int Sl, int H, int D, int Pu, int Cs, int Ld, uint32_t *status) {
  // elements of dO / O / dO in head layout, of the lse rows (Cs per row) and of
  // the delta / nlse rows (Ld >= Cs per row)
  const int hp = H / Pu;
  const long long act_n = (long long)P * B * Sl * H * D, rows_n = (long long)P * B * Sl * H,
                  ws_rows_n = (long long)P * B * hp * Ld;
  const int lanes = D / 8;  // 8 or 16: divides 32 and kThreads
  const int tasks = H * lanes;
  const long long rows = (long long)P * B * Sl;
  const int c = threadIdx.x % lanes;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    // row = (s*B + b)*Sl + t: token t of sequence shard s, batch b
    const int t = (int)(row % Sl);
    const long long sb = row / Sl;
    const int b = (int)(sb % B);
    const int s = (int)(sb / B);
    const int pos = s * Sl + t;
    const int rp = s / Pu;              // ring position; the token's row in its chunk:
    const int crow = pos - rp * Cs;
    // The trip count is uniform over the block, so the shuffles below see
    // every lane of every warp.
    for (int base = 0; base < tasks; base += kThreads) {
      const int task = base + (int)threadIdx.x;
      const bool live = task < tasks;
      const int g = task / lanes;       // head (global)
      const int d = rp * Pu + g / hp;   // the head-layout rank holding head g of the token
      const int j = g % hp;
      float acc = 0.f;
      const long long head_row = (((long long)(d * B + b) * Cs + crow) * hp + j) * D;
      const long long seq_off = (row * H + g) * D + c * 8;
      // the row's LSE is read before the products, so its load overlaps theirs
      const long long hrow = (long long)(d * B + b) * hp + j;
      const long long idx = hrow * Cs + crow, widx = hrow * Ld + crow;
      const bool writer =
          live && c == 0 && in_range(status, idx, 1, rows_n) && in_range(status, widx, 1, ws_rows_n);
      const float row_lse = writer ? __ldg(lse + idx) : 0.f;
      if (live && in_range(status, seq_off, 8, act_n) && in_range(status, head_row + c * 8, 8, act_n)) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(dout + seq_off));
        const uint4 y = __ldg(reinterpret_cast<const uint4 *>(o + (kFolded ? seq_off : head_row + c * 8)));
        if (!kFolded) *reinterpret_cast<uint4 *>(do_head + head_row + c * 8) = x;
        const __nv_bfloat162 *px = reinterpret_cast<const __nv_bfloat162 *>(&x);
        const __nv_bfloat162 *py = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          float2 a = __bfloat1622float2(px[w]), bb = __bfloat1622float2(py[w]);
          acc = fmaf(a.x, bb.x, acc);
          acc = fmaf(a.y, bb.y, acc);
        }
      }
      for (int off = lanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (writer) {
        delta[widx] = acc;
        nlse[widx] = -row_lse * 1.4426950408889634f;
      }
    }
  }
}

// A grid-stride kernel's grid: as many blocks as are resident at once on all
// SMs (the kernel's own occupancy at `threads` threads a block), so that none
// waits for a second wave, and no more blocks than work items.
template <typename Kernel>
int grid_for(Kernel kernel, int threads, long long rows) {
  int dev = 0, sms = 148, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  long long g = (long long)sms * per_sm;
  if (rows < g) g = rows;
  return (int)(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_rope_table(const ulysses_problem &p, void *ws, cudaStream_t st) {
  WorkspaceLayout L = workspace_layout(p);
  uint8_t *base = static_cast<uint8_t *>(ws);
  uint32_t *hdr = reinterpret_cast<uint32_t *>(base + L.status);
  if (!p.use_rope) {
    // no table: one thread clears the status word and writes the key (a kernel,
    // not a host copy, so nothing waits on the host and a captured graph holds
    // no pointer to host memory)
    rope_table_kernel<<<1, 32, 0, st>>>(nullptr, nullptr, 0, p.head_dim, 1.0, hdr, rope_key(p));
    return cudaGetLastError();
  }
  float *cs = reinterpret_cast<float *>(base + L.rope);
  float *sn = cs + (size_t)p.S * (p.head_dim / 2);
  long long n = (long long)p.S * (p.head_dim / 2);
  int grid = (int)((n + 255) / 256);
  if (grid > 4096) grid = 4096;
  rope_table_kernel<<<grid, 256, 0, st>>>(cs, sn, p.S, p.head_dim, (double)p.rope_base, hdr, rope_key(p));
  return cudaGetLastError();
}

__global__ void zero_kernel(float4 *p, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_zero(float *p, size_t n, cudaStream_t st) {
  const long long n4 = (long long)(n / 4);
  if (n % 4 || n4 == 0) return n4 == 0 && n == 0 ? cudaSuccess : cudaErrorInvalidValue;
  zero_kernel<<<grid_for(zero_kernel, 256, (n4 + 255) / 256), 256, 0, st>>>(reinterpret_cast<float4 *>(p), n4);
  return cudaGetLastError();
}

static PermParams base_params(const ulysses_problem &p, const void *ws, int to_head) {
  PermParams pp{};
  pp.P = p.P;
  pp.Pu = group_ranks(p);
  pp.Cs = chunk_len(p);
  pp.B = p.B;
  pp.Sl = p.S / p.P;
  pp.D = p.head_dim;
  pp.to_head = to_head;
  if (ws) {
    WorkspaceLayout L = workspace_layout(p);
    const uint8_t *base = static_cast<const uint8_t *>(ws);
    pp.status = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(base + L.status));
    pp.rope_key_ptr = pp.status + 1;
    pp.rope_key = rope_key(p);
    pp.rope_cos = reinterpret_cast<const float *>(base + L.rope);
    pp.rope_sin = pp.rope_cos + (size_t)p.S * (p.head_dim / 2);
    pp.rope_n = (long long)p.S * (p.head_dim / 2);
  }
  return pp;
}

template <typename T>
static cudaError_t launch_unpack_bulk(const ulysses_problem &p, const PermParams &pp, uint32_t row_bytes,
                                      cudaStream_t st) {
  const size_t smem = (size_t)kBulkStages * row_bytes + 8 * kBulkStages + 16;
  cudaError_t e = cudaFuncSetAttribute(unpack_bulk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, unpack_bulk_kernel<T>, 32, smem);
  per_sm = per_sm < 1 ? 1 : (per_sm > 32 ? 32 : per_sm);
  long long grid = (long long)sms * per_sm;
  const long long rows = (long long)p.B * p.S;
  if (grid > rows) grid = rows;
  unpack_bulk_kernel<T><<<(unsigned)grid, 32, smem, st>>>(pp, row_bytes);
  return cudaGetLastError();
}

static cudaError_t launch_perm(const ulysses_problem &p, const PermParams &pp, cudaStream_t st) {
  // A copy in the head -> seq direction whose output row fits a stage goes to
  // the copy engine; everything else (the pack with RoPE) to the thread kernel.
  const size_t row_bytes = (size_t)pp.job[0].heads * p.head_dim * elem_size(p);
  if (!pp.to_head && pp.njobs == 1 && pp.job[0].rope == 0 && row_bytes <= 48 * 1024) {
    if (p.dtype == ULYSSES_BF16) return launch_unpack_bulk<__nv_bfloat16>(p, pp, (uint32_t)row_bytes, st);
    return launch_unpack_bulk<float>(p, pp, (uint32_t)row_bytes, st);
  }
  const long long rows = (long long)p.B * p.S;
  // rows per pass: enough for the job with the fewest units a row to fill the block
  const int vec = p.dtype == ULYSSES_BF16 ? 8 : 4;
  int min_units = kThreads;
  for (int q = 0; q < pp.njobs; ++q) {
    const PermJob &J = pp.job[q];
    const int u = pp.Pu * (J.rep > 1 ? 1 : J.heads / pp.Pu) * (p.head_dim / (2 * vec));
    if (u < min_units) min_units = u;
  }
  PermParams pr = pp;
  const int fill = kThreads / min_units;
  pr.nrow = fill < 1 ? 1 : (fill > kMaxRowsPerPass ? kMaxRowsPerPass : fill);
  const long long passes = (rows + pr.nrow - 1) / pr.nrow;
  if (p.dtype == ULYSSES_BF16) {
    const int grid = grid_for(permute_kernel<__nv_bfloat16>, kThreads, passes);
    permute_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(pr);
  } else {
    const int grid = grid_for(permute_kernel<float>, kThreads, passes);
    permute_kernel<float><<<grid, kThreads, 0, st>>>(pr);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_qkv(const ulysses_problem &p, const void *q, const void *k, const void *v,
                            void *qh, void *kh, void *vh, void *ws, cudaStream_t st) {
  PermParams pp = base_params(p, ws, 1);
  const int r = p.use_rope ? 1 : 0;
  const int R = kv_replicas(p);
  // elements: the sequence-sharded tensor, and its head layout (P copies of
  // one kv-head's rows per rank with replicated kv-heads)
  const long long nq = (long long)p.B * p.S * p.n_head * p.head_dim;
  const long long nk = (long long)p.B * p.S * p.n_kv_head * p.head_dim;
  const long long nkh = (long long)p.P * p.B * chunk_len(p) * kv_per_rank(p) * p.head_dim;
  pp.job[0] = {q, qh, p.n_head, r, 1, nq, nq};
  pp.job[1] = {k, kh, p.n_kv_head, r, R, nk, nkh};
  pp.job[2] = {v, vh, p.n_kv_head, 0, R, nk, nkh};
  pp.njobs = 3;
  return launch_perm(p, pp, st);
}

cudaError_t launch_unpack(const ulysses_problem &p, const void *o_head, void *o_seq,
                          cudaStream_t st) {
  PermParams pp = base_params(p, nullptr, 0);
  const long long no = (long long)p.B * p.S * p.n_head * p.head_dim;
  pp.job[0] = {o_head, o_seq, p.n_head, 0, 1, no, no};
  pp.njobs = 1;
  return launch_perm(p, pp, st);
}

cudaError_t launch_pack_do_delta(const ulysses_problem &p, const void *do_seq, const void *o,
                                 const float *lse, void *do_head, float *delta, float *nlse,
                                 uint32_t *status, cudaStream_t st, bool folded) {
  auto kernel = folded ? pack_do_delta_kernel<true> : pack_do_delta_kernel<false>;
  const int grid = grid_for(kernel, kThreads, (long long)p.B * p.S);  // one token row per block at a time
  kernel<<<grid, kThreads, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(do_seq), static_cast<const __nv_bfloat16 *>(o),
      lse, static_cast<__nv_bfloat16 *>(do_head), delta, nlse, p.P, p.B, p.S / p.P, p.n_head,
      p.head_dim, group_ranks(p), chunk_len(p), delta_ld(p), status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Gradients of replicated kv-heads ("Sequence Parallelism II", §6: the
// gradients go back head -> seq): kv-head kv was handed to the R ranks
// kv*R .. kv*R+R-1 (of the token's ring position rp: ranks rp*Pu + kv*R + j),
// so its gradient is the sum of their partials, added in rank order:
//   dV_seq[d][b][t][kv][e] = sum_j dv_part[(rp*Pu + kv*R+j)*B + b][crow][e],
// crow = (d % Pu)*Sl + t the token's row in its ring position's chunk (plain
// Ulysses: rp = 0, Pu = P, crow = d*Sl + t)
// and dK the same, then scaled and rotated back by -angle(d*Sl+t) on the pairs
// (i, i+D/2).  One thread per (row, kv-head, 4 rotation pairs): float4 loads of
// both halves from each replica, two 8-byte bf16 stores per tensor.
namespace {

__global__ void __launch_bounds__(256) kv_reduce_kernel(const float *__restrict__ dkp, const float *__restrict__ dvp,
                                                        __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv,
                                                        int P, int B, int Sl, int n_kv, int D, int Pu, float scale,
                                                        const float *__restrict__ cs, const float *__restrict__ sn,
                                                        uint32_t *status) {
  const int R = Pu / n_kv, half = D / 2, q4 = half / 4;
  const int Cs = Pu * Sl;
  // elements of the float partials, of dK / dV in sequence layout, of cos / sin
  const long long part_n = (long long)P * B * Cs * D, seq_n = (long long)P * B * Sl * n_kv * D;
  const long long rope_n = (long long)P * Sl * half;
  const long long n = (long long)P * B * Sl * n_kv * q4;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < n; u += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(u % q4);
    long long rest = u / q4;
    const int kv = (int)(rest % n_kv);
    rest /= n_kv;
    const int t = (int)(rest % Sl);
    rest /= Sl;
    const int b = (int)(rest % B);
    const int d = (int)(rest / B);
    const int pos = d * Sl + t;
    const int rp = d / Pu, crow = (d - rp * Pu) * Sl + t;  // ring position, row in its chunk
    float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), ky = kx, vx = kx, vy = kx;
    const size_t o = (((size_t)(d * B + b) * Sl + t) * n_kv + kv) * D + (size_t)c * 4;
    if (!in_range(status, (long long)o, half + 4, seq_n) ||
        (cs && !in_range(status, (long long)pos * half + c * 4, 4, rope_n)))
      continue;
    bool whole = true;
    for (int j = 0; j < R; ++j)
      whole = whole && in_range(status, (((long long)(rp * Pu + kv * R + j) * B + b) * Cs + crow) * D + c * 4,
                                half + 4, part_n);
    if (!whole) continue;
    for (int j = 0; j < R; ++j) {
      const size_t off = (((size_t)(rp * Pu + kv * R + j) * B + b) * Cs + crow) * D + (size_t)c * 4;
      const float4 a = *reinterpret_cast<const float4 *>(dkp + off);
      const float4 a2 = *reinterpret_cast<const float4 *>(dkp + off + half);
      const float4 v1 = *reinterpret_cast<const float4 *>(dvp + off);
      const float4 v2 = *reinterpret_cast<const float4 *>(dvp + off + half);
      kx.x += a.x; kx.y += a.y; kx.z += a.z; kx.w += a.w;
      ky.x += a2.x; ky.y += a2.y; ky.z += a2.z; ky.w += a2.w;
      vx.x += v1.x; vx.y += v1.y; vx.z += v1.z; vx.w += v1.w;
      vy.x += v2.x; vy.y += v2.y; vy.z += v2.z; vy.w += v2.w;
    }
    float xs[4] = {kx.x * scale, kx.y * scale, kx.z * scale, kx.w * scale};
    float ys[4] = {ky.x * scale, ky.y * scale, ky.z * scale, ky.w * scale};
    if (cs) {
      const float4 c4 = *reinterpret_cast<const float4 *>(cs + (size_t)pos * half + c * 4);
      const float4 s4 = *reinterpret_cast<const float4 *>(sn + (size_t)pos * half + c * 4);
      const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // x' = x cos + y sin, y' = y cos - x sin
        const float x = xs[q], y = ys[q];
        xs[q] = x * cc[q] + y * ss[q];
        ys[q] = y * cc[q] - x * ss[q];
      }
    }
    const __nv_bfloat162 k0 = __floats2bfloat162_rn(xs[0], xs[1]), k1 = __floats2bfloat162_rn(xs[2], xs[3]);
    const __nv_bfloat162 k2 = __floats2bfloat162_rn(ys[0], ys[1]), k3 = __floats2bfloat162_rn(ys[2], ys[3]);
    const __nv_bfloat162 w0 = __floats2bfloat162_rn(vx.x, vx.y), w1 = __floats2bfloat162_rn(vx.z, vx.w);
    const __nv_bfloat162 w2 = __floats2bfloat162_rn(vy.x, vy.y), w3 = __floats2bfloat162_rn(vy.z, vy.w);
    *reinterpret_cast<uint2 *>(dk + o) = make_uint2(*reinterpret_cast<const uint32_t *>(&k0), *reinterpret_cast<const uint32_t *>(&k1));
    *reinterpret_cast<uint2 *>(dk + o + half) = make_uint2(*reinterpret_cast<const uint32_t *>(&k2), *reinterpret_cast<const uint32_t *>(&k3));
    *reinterpret_cast<uint2 *>(dv + o) = make_uint2(*reinterpret_cast<const uint32_t *>(&w0), *reinterpret_cast<const uint32_t *>(&w1));
    *reinterpret_cast<uint2 *>(dv + o + half) = make_uint2(*reinterpret_cast<const uint32_t *>(&w2), *reinterpret_cast<const uint32_t *>(&w3));
  }
}

}  // namespace

cudaError_t launch_kv_reduce(const ulysses_problem &p, const float *dk_part, const float *dv_part,
                             void *dk_seq, void *dv_seq, float scale, const void *ws, cudaStream_t st) {
  const float *cs = nullptr, *sn = nullptr;
  if (p.use_rope) {
    const WorkspaceLayout L = workspace_layout(p);
    cs = reinterpret_cast<const float *>(static_cast<const uint8_t *>(ws) + L.rope);
    sn = cs + (size_t)p.S * (p.head_dim / 2);
  }
  const long long n = (long long)p.B * p.S * p.n_kv_head * (p.head_dim / 8);
  const int grid = grid_for(kv_reduce_kernel, 256, n / 256 + 1);
  kv_reduce_kernel<<<grid, 256, 0, st>>>(dk_part, dv_part, static_cast<__nv_bfloat16 *>(dk_seq),
                                         static_cast<__nv_bfloat16 *>(dv_seq), p.P, p.B, p.S / p.P, p.n_kv_head,
                                         p.head_dim, group_ranks(p), scale, cs, sn,
                                         const_cast<uint32_t *>(static_cast<const uint32_t *>(ws)));
  return cudaGetLastError();
}

}  // namespace ulysses
