// Step-level scoring of many query tokens at once on the 5th-generation
// tensor cores (tcgen05 + TMEM).
//
// Evolve review of KVMem, "Strengths": recall is scheduled once per agent
// step (attention KL within a step is small), so all query tokens of a step
// are scored against the Mean-K index together.  Per KV head g, with the
// step's T tokens and the group's G heads as R = T*G query rows:
//   s[r, b]  = <q_r, kbar_b> / sqrt(d)                (bf16 operands, fp32 accumulation)
//   Gs[g, b] = sum_r softmax_b(s[r, :])[b]
// This is a dense R x n_blk x d contraction per head, evaluated twice:
//   pass 1  D = Q * Kbar^T  (M = 128 query rows, N = 256 blocks per MMA tile):
//           each epilogue thread owns one query row and keeps its running max
//           and sum of exponentials over its column range;
//   merge   per row: global max M_r and 1/Z_r;
//   pass 2  D = Kbar * Q^T  (M = 128 blocks, N = 256 query rows):
//           each epilogue thread owns one block and sums exp(s - M_r)/Z_r over
//           every query row, so Gs needs no cross-thread reduction.
// Operands are packed once per call into the no-swizzle K-major core-matrix
// layout (8 rows x 16 bytes per core matrix; core matrices adjacent in K are
// 128 B apart, 8-row groups d*16 B apart), so every tile is one contiguous
// 1-D bulk copy into shared memory.  Warp roles: warp 0 issues bulk copies,
// warp 1 owns TMEM and issues the MMAs, warps 2..5 drain TMEM (each warp can
// only read its quarter of the 128 TMEM lanes).  Every wait is bounded.
#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr int kEpiWarps = 16;   // epilogue: four warps per TMEM lane quarter, each taking a quarter of a tile's
                                // columns (pass 1) or rows (pass 2)
constexpr int kParts = kEpiWarps / 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA issuer, epilogue
constexpr int kRowsM = 128;     // MMA M
constexpr int kColsN = 256;     // MMA N
constexpr uint32_t kTmemCols = 512;

// ---------------------------------------------------------------- packing
// Index fp32 [S][h_kv][max_blocks][D] -> bf16 core-matrix layout [S*h_kv][blk_cap_pad/8][D/8][8][8].
template <int D>
__global__ void pack_index_kernel(const float* __restrict__ index, int64_t max_blocks, SessionArgs a, int h_kv,
                                  int64_t blk_cap_pad, uint16_t* __restrict__ out) {
  constexpr int KC = D / 8;  // core matrices per 8-row group
  const int sg = blockIdx.z;
  const int s = sg / h_kv;
  const int64_t groups = (a.n_blk[s] + 255) / 256 * 32;  // 8-row groups up to the padded tile end
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;  // (group, kc, rr) with rr fastest
  if (idx >= groups * KC * 8) return;
  const int rr = (int)(idx & 7);
  const int kc = (int)((idx >> 3) % KC);
  const int64_t grp = (idx >> 3) / KC;
  const int64_t row = grp * 8 + rr;
  uint4 w = make_uint4(0, 0, 0, 0);
  if (row < a.n_blk[s]) {
    const float4* src = reinterpret_cast<const float4*>(index + ((int64_t)sg * max_blocks + row) * D + kc * 8);
    const float4 x = __ldg(src), y = __ldg(src + 1);
    w = make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
  }
  *reinterpret_cast<uint4*>(out + ((int64_t)sg * blk_cap_pad + grp * 8) * D + (kc * 8 + rr) * 8) = w;
}

// Queries bf16 [S][n_q][h_q][D] -> rows r = t*G + hh of KV head g, same packed layout, rows_pad rows.
template <int D>
__global__ void pack_query_kernel(const uint16_t* __restrict__ q, int n_q, int h_q, int h_kv, int group,
                                  int rows_pad, uint16_t* __restrict__ out) {
  constexpr int KC = D / 8;
  const int sg = blockIdx.z;
  const int s = sg / h_kv, g = sg % h_kv;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows_pad / 8 * KC * 8) return;
  const int rr = idx & 7, kc = (idx >> 3) % KC, grp = (idx >> 3) / KC;
  const int row = grp * 8 + rr;
  uint4 w = make_uint4(0, 0, 0, 0);
  if (row < n_q * group) {
    const int t = row / group, hh = row % group;
    w = __ldg(reinterpret_cast<const uint4*>(q + (((int64_t)s * n_q + t) * h_q + g * group + hh) * D + kc * 8));
  }
  *reinterpret_cast<uint4*>(out + ((int64_t)sg * rows_pad + grp * 8) * D + (kc * 8 + rr) * 8) = w;
}

struct Bars {
  uint64_t a_full, b_full[2], b_empty[2], d_full[2], d_empty[2];
};

__device__ __forceinline__ void init_bars(Bars& b) {
  mbar_init(&b.a_full, 1);
  for (int i = 0; i < 2; ++i) {
    mbar_init(&b.b_full[i], 1);
    mbar_init(&b.b_empty[i], 1);
    mbar_init(&b.d_full[i], 1);
    mbar_init(&b.d_empty[i], kEpiWarps);
  }
  mbar_fence_init();
}

// ---------------------------------------------------------------- pass 1: row max / sum
// grid (rows_pad/128, n_ranges, S*h_kv).  Each CTA: 128 query rows x a range of 256-column tiles.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) step_rowstats_kernel(
    const uint16_t* __restrict__ qpk, const uint16_t* __restrict__ kpk, int rows_pad, int64_t blk_cap_pad,
    SessionArgs a, int h_kv, int tiles_per_range, float2* __restrict__ part, int n_ranges, float scale_log2,
    uint32_t* __restrict__ status) {
  constexpr uint32_t A_BYTES = kRowsM * D * 2, B_BYTES = kColsN * D * 2;
  constexpr uint32_t SBO = D / 8 * 128, LBO = 128;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t IDESC = idesc_bf16_f32(kRowsM, kColsN);
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* a_s = smem;
  unsigned char* b_s = smem + A_BYTES;  // 2 stages
  __shared__ Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float2 half_state[kParts][kRowsM];  // each column part's (max, sum) per row

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = blockIdx.z, s = sg / h_kv;
  const int n_blk = a.n_blk[s];
  const int n_tiles_all = (n_blk + kColsN - 1) / kColsN;
  const int j0 = blockIdx.y * tiles_per_range;
  const int nt = min(tiles_per_range, n_tiles_all - j0);
  const int row0 = blockIdx.x * kRowsM;
  if (nt <= 0) return;

  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    init_bars(bars);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // producer: the query tile once, then the index tiles through a 2-deep ring
    mbar_arrive_expect_tx(&bars.a_full, A_BYTES);
    bulk_g2s(a_s, qpk + ((int64_t)sg * rows_pad + row0) * D, A_BYTES, &bars.a_full);
    int j = 0;
    for (; j < nt && !abort_flag; ++j) {
      const int st = j & 1;
      if (j >= 2 && !mbar_wait(&bars.b_empty[st], ((j >> 1) - 1) & 1, status)) {
        abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(&bars.b_full[st], B_BYTES);
      bulk_g2s(b_s + st * B_BYTES, kpk + ((int64_t)sg * blk_cap_pad + (int64_t)(j0 + j) * kColsN) * D, B_BYTES,
               &bars.b_full[st]);
    }
    // drain: copies still in flight must land before the CTA can exit
    mbar_wait(&bars.a_full, 0, status);
    for (int i = max(0, j - 2); i < j; ++i) mbar_wait(&bars.b_full[i & 1], (i >> 1) & 1, status);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    int j = 0;
    if (!mbar_wait(&bars.a_full, 0, status)) abort_flag = 1;
    const uint32_t a_addr = smem_addr(a_s);
    for (; j < nt && !abort_flag; ++j) {
      const int st = j & 1;
      if (!mbar_wait(&bars.b_full[st], (j >> 1) & 1, status) ||
          (j >= 2 && !mbar_wait(&bars.d_empty[st], ((j >> 1) - 1) & 1, status))) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t b_addr = smem_addr(b_s + st * B_BYTES);
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk)
        mma_bf16(tmem + st * kColsN, smem_desc(a_addr + kk * 256, LBO, SBO), smem_desc(b_addr + kk * 256, LBO, SBO),
                 IDESC, kk > 0);
      mma_commit(&bars.d_full[st]);
      mma_commit(&bars.b_empty[st]);
    }
    if (j > 0) mbar_wait(&bars.d_full[(j - 1) & 1], ((j - 1) >> 1) & 1, status);  // last MMAs done
  } else if (warp >= 2) {
    // epilogue: one query row per thread, a part of each tile's columns per warp
    const int quarter = warp & 3, half = (warp - 2) >> 2;  // half: the column part
    float m = -INFINITY, z = 0.f;
    for (int j = 0; j < nt; ++j) {
      const int st = j & 1;
      if (__any_sync(0xffffffffu, abort_flag) || !mbar_wait_warp(&bars.d_full[st], (j >> 1) & 1, status)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int col0 = (j0 + j) * kColsN;
      const bool full = col0 + kColsN <= n_blk;  // no column past the history in this tile
#pragma unroll 1
      for (int cc = half * (kColsN / 32 / kParts); cc < (half + 1) * (kColsN / 32 / kParts); ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + st * kColsN + cc * 32, v);
        tmem_wait_ld();
        // raw scores; the log2-domain scale (positive) is applied to the maximum and inside each exponent's FMA
        float x[32];
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = (col0 + cc * 32 + i < n_blk) ? __uint_as_float(v[i]) : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(x[i], x[i + 8]), fmaxf(x[i + 16], x[i + 24]));
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) mx[i] = fmaxf(mx[i], mx[i + w]);
        const float mn = fmaxf(m, mx[0] * scale_log2);
        if (mn != -INFINITY) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i & 3] += fast_exp2(fmaf(x[i], scale_log2, -mn));
          z = z * fast_exp2(m - mn) + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
          m = mn;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.d_empty[st]);
    }
    half_state[half][quarter * 32 + lane] = make_float2(m, z);
  }
  tc_fence_before();
  __syncthreads();
  if (warp >= 2 && warp < 6) {  // the column parts of each row: (max, sum) combined in part order
    const int r = (warp & 3) * 32 + lane, row = row0 + r;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kParts; ++k) M = fmaxf(M, half_state[k][r].x);
    float z = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < kParts; ++k) {
        const float2 pk = half_state[k][r];
        z += pk.x == -INFINITY ? 0.f : pk.y * fast_exp2(pk.x - M);
      }
    }
    if (row < rows_pad) part[((int64_t)sg * n_ranges + blockIdx.y) * rows_pad + row] = make_float2(M, z);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Per query row: M = max over ranges and Z = sum z * 2^(m - M), stored as (M + log2 Z, 1/Z); padded rows get
// (+inf, 0).
__global__ void step_merge_kernel(const float2* __restrict__ part, int n_ranges, int rows_pad, int n_rows,
                                  float2* __restrict__ stats) {
  const int sg = blockIdx.y;
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= rows_pad) return;
  float2 r = make_float2(INFINITY, 0.f);
  if (row < n_rows) {
    float M = -INFINITY;
    for (int k = 0; k < n_ranges; ++k) M = fmaxf(M, part[((int64_t)sg * n_ranges + k) * rows_pad + row].x);
    float Z = 0.f;
    for (int k = 0; k < n_ranges; ++k) {
      const float2 p = part[((int64_t)sg * n_ranges + k) * rows_pad + row];
      if (p.x != -INFINITY) Z += p.y * exp2f(p.x - M);
    }
    // (M + log2 Z, 1/Z): pass 2 folds the normaliser into the exponent
    r = Z > 0.f ? make_float2(M + log2f(Z), 1.f / Z) : make_float2(INFINITY, 0.f);
  }
  stats[(int64_t)sg * rows_pad + row] = r;
}

// ---------------------------------------------------------------- pass 2: group scores
// grid (blk_cap tiles of 128 blocks, 1, S*h_kv).  Each CTA: 128 blocks x every query row.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) step_colsum_kernel(
    const uint16_t* __restrict__ qpk, const uint16_t* __restrict__ kpk, const float2* __restrict__ stats,
    int rows_pad, int64_t blk_cap_pad, SessionArgs a, int h_kv, int64_t max_blocks, float scale_log2,
    float* __restrict__ gs_out, uint32_t* __restrict__ status) {
  constexpr uint32_t A_BYTES = kRowsM * D * 2, B_BYTES = kColsN * D * 2;
  constexpr uint32_t SBO = D / 8 * 128, LBO = 128;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t IDESC = idesc_bf16_f32(kRowsM, kColsN);
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* a_s = smem;
  unsigned char* b_s = smem + A_BYTES;
  float* st_s = reinterpret_cast<float*>(smem + A_BYTES + 2 * B_BYTES);  // [rows_pad]: M + log2 Z per row
  __shared__ Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float half_acc[kParts][kRowsM];  // each part's partial group score per block

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = blockIdx.z, s = sg / h_kv;
  const int n_blk = a.n_blk[s];
  const int blk0 = blockIdx.x * kRowsM;
  if (blk0 >= n_blk) return;
  const int nchunk = rows_pad / kColsN;

  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    init_bars(bars);
  }
  for (int i = tid; i < rows_pad; i += kThreads) st_s[i] = stats[(int64_t)sg * rows_pad + i].x;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(&bars.a_full, A_BYTES);
    bulk_g2s(a_s, kpk + ((int64_t)sg * blk_cap_pad + blk0) * D, A_BYTES, &bars.a_full);
    int j = 0;
    for (; j < nchunk && !abort_flag; ++j) {
      const int st = j & 1;
      if (j >= 2 && !mbar_wait(&bars.b_empty[st], ((j >> 1) - 1) & 1, status)) {
        abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(&bars.b_full[st], B_BYTES);
      bulk_g2s(b_s + st * B_BYTES, qpk + ((int64_t)sg * rows_pad + (int64_t)j * kColsN) * D, B_BYTES,
               &bars.b_full[st]);
    }
    mbar_wait(&bars.a_full, 0, status);
    for (int i = max(0, j - 2); i < j; ++i) mbar_wait(&bars.b_full[i & 1], (i >> 1) & 1, status);
  } else if (warp == 1 && lane == 0) {
    int j = 0;
    if (!mbar_wait(&bars.a_full, 0, status)) abort_flag = 1;
    const uint32_t a_addr = smem_addr(a_s);
    for (; j < nchunk && !abort_flag; ++j) {
      const int st = j & 1;
      if (!mbar_wait(&bars.b_full[st], (j >> 1) & 1, status) ||
          (j >= 2 && !mbar_wait(&bars.d_empty[st], ((j >> 1) - 1) & 1, status))) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t b_addr = smem_addr(b_s + st * B_BYTES);
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk)
        mma_bf16(tmem + st * kColsN, smem_desc(a_addr + kk * 256, LBO, SBO), smem_desc(b_addr + kk * 256, LBO, SBO),
                 IDESC, kk > 0);
      mma_commit(&bars.d_full[st]);
      mma_commit(&bars.b_empty[st]);
    }
    if (j > 0) mbar_wait(&bars.d_full[(j - 1) & 1], ((j - 1) >> 1) & 1, status);
  } else if (warp >= 2) {
    // one block per thread, a part of each tile's query rows per warp
    const int quarter = warp & 3, half = (warp - 2) >> 2;  // half: the row part
    float acc = 0.f;
    for (int j = 0; j < nchunk; ++j) {
      const int st = j & 1;
      if (__any_sync(0xffffffffu, abort_flag) || !mbar_wait_warp(&bars.d_full[st], (j >> 1) & 1, status)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = half * (kColsN / 32 / kParts); cc < (half + 1) * (kColsN / 32 / kParts); ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + st * kColsN + cc * 32, v);
        tmem_wait_ld();
        const float* sr = st_s + j * kColsN + cc * 32;
        float a4[4] = {0.f, 0.f, 0.f, 0.f};  // p / Z = 2^(s c - (M + log2 Z)); short dependency chains
#pragma unroll
        for (int i = 0; i < 32; ++i)  // sr[i]: the same address in every lane (broadcast)
          a4[i & 3] += fast_exp2(fmaf(__uint_as_float(v[i]), scale_log2, -sr[i]));
        acc += (a4[0] + a4[1]) + (a4[2] + a4[3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.d_empty[st]);
    }
    half_acc[half][quarter * 32 + lane] = acc;
  }
  tc_fence_before();
  __syncthreads();
  if (warp >= 2 && warp < 6) {  // the parts of the query rows summed in part order
    const int r = (warp & 3) * 32 + lane, blk = blk0 + r;
    float g = 0.f;
#pragma unroll
    for (int k = 0; k < kParts; ++k) g += half_acc[k][r];
    if (blk < n_blk) gs_out[(int64_t)sg * max_blocks + blk] = g;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_step_d(const Ctx& c, const uint16_t* q, int n_q, const float* index, int n_sessions,
                          const SessionArgs& a, float* gs_out, cudaStream_t st) {
  const int G = c.group;
  const int n_rows = n_q * G;
  const int rows_pad = (n_rows + kColsN - 1) / kColsN * kColsN;
  const int64_t blk_cap_pad = c.step_blk_cap_pad;
  int max_blk = 0;
  for (int s = 0; s < n_sessions; ++s) max_blk = max(max_blk, a.n_blk[s]);
  if (max_blk == 0) return cudaSuccess;
  const int SG = n_sessions * c.p.h_kv;
  cudaError_t e;
  {
    const int64_t groups = (int64_t)(max_blk + 255) / 256 * 32;
    const int64_t n = groups * (D / 8) * 8;
    // the bf16 operand: the copy kept by the appends when it holds every scored block, else converted here
    // (which overwrites the copy: the caller then marks it stale)
    if (!shadow_ready(c, index, n_sessions, a))
      pack_index_kernel<D><<<dim3((unsigned)((n + 255) / 256), 1, SG), 256, 0, st>>>(index, c.p.max_blocks, a,
                                                                                      c.p.h_kv, blk_cap_pad,
                                                                                      c.step_kpk);
    const int nq = rows_pad / 8 * (D / 8) * 8;
    pack_query_kernel<D><<<dim3((nq + 255) / 256, 1, SG), 256, 0, st>>>(q, n_q, c.p.h_q, c.p.h_kv, G, rows_pad,
                                                                        c.step_qpk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int n_tiles = (max_blk + kColsN - 1) / kColsN;
  // spread pass 1 over about two waves of CTAs: ranges of column tiles per 128-row block
  const int row_blocks = rows_pad / kRowsM;
  int n_ranges = (2 * c.num_sms + row_blocks * SG - 1) / (row_blocks * SG);
  n_ranges = max(1, min(min(n_ranges, n_tiles), kStepMaxRanges));
  const int tiles_per_range = (n_tiles + n_ranges - 1) / n_ranges;
  n_ranges = (n_tiles + tiles_per_range - 1) / tiles_per_range;
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  const size_t smem1 = (size_t)kRowsM * D * 2 + 2 * (size_t)kColsN * D * 2;
  if ((e = ensure_smem(step_rowstats_kernel<D>, c.device, smem1)) != cudaSuccess) return e;
  step_rowstats_kernel<D><<<dim3(row_blocks, n_ranges, SG), kThreads, smem1, st>>>(
      c.step_qpk, c.step_kpk, rows_pad, blk_cap_pad, a, c.p.h_kv, tiles_per_range, c.step_part, n_ranges,
      scale_log2, c.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  step_merge_kernel<<<dim3((rows_pad + 127) / 128, SG), 128, 0, st>>>(c.step_part, n_ranges, rows_pad, n_rows,
                                                                       c.step_stats);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smem2 = smem1 + (size_t)rows_pad * sizeof(float2);
  if ((e = ensure_smem(step_colsum_kernel<D>, c.device, smem2)) != cudaSuccess) return e;
  step_colsum_kernel<D><<<dim3((max_blk + kRowsM - 1) / kRowsM, 1, SG), kThreads, smem2, st>>>(
      c.step_qpk, c.step_kpk, c.step_stats, rows_pad, blk_cap_pad, a, c.p.h_kv, c.p.max_blocks, scale_log2, gs_out,
      c.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step_scores(const Ctx& c, const uint16_t* q, int n_q, const float* index, int n_sessions,
                               const SessionArgs& a, float* gs_out, cudaStream_t st) {
  return c.p.d == 128 ? launch_step_d<128>(c, q, n_q, index, n_sessions, a, gs_out, st)
                      : launch_step_d<64>(c, q, n_q, index, n_sessions, a, gs_out, st);
}

}  // namespace kvm
