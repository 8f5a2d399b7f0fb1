// Step 2 — block scoring, per-head softmax summed over the GQA group, and
// top-k selection with forced sink / recent blocks.
//
// KVMEM reproduction README, "Core equation": s_b = <q, kbar_b>/sqrt(d), then
// the selected KV is concatenated within the block budget.  Same page,
// "2026-09-08 validation correction": the query is the normalised one and
// each query head gets its own softmax; heads are not averaged before it.
//
// Kernel A (score_tile_kernel), grid (tiles, h_kv, sessions):
//   streams a tile of index rows of one KV head through shared memory with
//   1-D bulk copies (4-stage mbarrier pipeline), computes the G scores of
//   each row with 8 lanes per row and shuffle reductions, then writes
//   e[b][h] = exp(s[b][h] - m_tile[h]) and the tile's (m_tile, sum e) per head.
// Kernel B (select_kernel), grid (C, h_kv, sessions), clusters of C CTAs:
//   each CTA owns 1/C of the blocks.  From the tiles' partials it forms the
//   softmax normalisers, Gs[b] = sum_h e[b][h] * exp(m_tile - M_h) / Z_h, and
//   then runs an exact 3-pass radix select (11/11/10 bits) over the
//   candidates, histograms merged through distributed shared memory, followed
//   by a cluster-wide stable compaction: ascending ids, equal scores resolved
//   toward the lower id.
#include <cooperative_groups.h>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace cg = cooperative_groups;

namespace kvm {
namespace {

constexpr int kScoreThreads = 256;  // 8 warps, 4 rows each per stage
constexpr int kStageRows = 32;
constexpr int kStages = 4;
constexpr int kSelectThreads = 512;
constexpr int kRadixBins = 2048;

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_tile_kernel(
    const uint16_t* __restrict__ q, const float* __restrict__ index, int64_t max_blocks, int h_kv, int h_q,
    SessionArgs a, int rows_per_tile, float* __restrict__ e_buf, float2* __restrict__ part, int64_t max_tiles,
    float* __restrict__ head_scores, uint32_t* __restrict__ status) {
  constexpr int NV = D / 32;  // float4 chunks per lane per row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* stage_buf = reinterpret_cast<float*>(smem_raw);                   // [kStages][32][D]
  float* s_tile = stage_buf + kStages * kStageRows * D;                    // [rows_per_tile][G]
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ float red[kScoreThreads / 32][G];
  __shared__ float tile_max[G];

  const int s = blockIdx.z, g = blockIdx.y, tile = blockIdx.x;
  const int64_t n_blk = a.n_blk[s];
  const int64_t r0 = (int64_t)tile * rows_per_tile;
  if (r0 >= n_blk) return;
  const int nrows = (int)(rows_per_tile < n_blk - r0 ? (int64_t)rows_per_tile : n_blk - r0);
  const int nstage = (nrows + kStageRows - 1) / kStageRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane & 7;                 // 8 lanes per row
  const int rsel = warp * 4 + (lane >> 3);  // row within a stage
  const float* src = index + (((int64_t)s * h_kv + g) * max_blocks + r0) * D;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int k) {
    const int rows = min(kStageRows, nrows - k * kStageRows);
    const uint32_t bytes = (uint32_t)(rows * D * 4);
    mbar_arrive_expect_tx(&full_bar[k % kStages], bytes);
    bulk_g2s(stage_buf + (k % kStages) * kStageRows * D, src + (int64_t)k * kStageRows * D, bytes,
             &full_bar[k % kStages]);
  };
  if (tid == 0)
    for (int k = 0; k < min(kStages, nstage); ++k) issue(k);

  // Query slice of this lane, scaled by 1/sqrt(d): dims 4*sub + 32*i + {0..3}.
  float qv[G][NV * 4];
  const float inv_sqrt_d = __frsqrt_rn((float)D);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint16_t* qh = q + ((int64_t)s * h_q + g * G + h) * D;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh + 4 * sub + 32 * i));
      qv[h][4 * i + 0] = bf16lo(w.x) * inv_sqrt_d;
      qv[h][4 * i + 1] = bf16hi(w.x) * inv_sqrt_d;
      qv[h][4 * i + 2] = bf16lo(w.y) * inv_sqrt_d;
      qv[h][4 * i + 3] = bf16hi(w.y) * inv_sqrt_d;
    }
  }
  float run_max = -INFINITY;  // lane (sub == h) tracks head h over its rows

  int k = 0;
  bool aborted = false;
  for (; k < nstage; ++k) {
    const bool ok = mbar_wait(&full_bar[k % kStages], (k / kStages) & 1, status);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const int rows = min(kStageRows, nrows - k * kStageRows);
    const bool valid_row = rsel < rows;  // all lanes compute (uniform shuffles); only valid rows store
    const float* row = stage_buf + (k % kStages) * kStageRows * D + (valid_row ? rsel : 0) * D;
    float dot[G];
#pragma unroll
    for (int h = 0; h < G; ++h) dot[h] = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(row + 4 * sub + 32 * i);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        dot[h] = fmaf(qv[h][4 * i + 0], v.x, dot[h]);
        dot[h] = fmaf(qv[h][4 * i + 1], v.y, dot[h]);
        dot[h] = fmaf(qv[h][4 * i + 2], v.z, dot[h]);
        dot[h] = fmaf(qv[h][4 * i + 3], v.w, dot[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], 1);
      dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], 2);
      dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], 4);
    }
    if (valid_row) {
      const int r = k * kStageRows + rsel;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (sub == h) {
          s_tile[r * G + h] = dot[h];
          run_max = fmaxf(run_max, dot[h]);
          if (head_scores) head_scores[((int64_t)s * h_q + g * G + h) * max_blocks + r0 + r] = dot[h];
        }
      }
    }
    __syncthreads();  // every warp is done with this stage buffer
    if (tid == 0 && k + kStages < nstage) issue(k + kStages);
  }
  if (aborted) {
    // drain the copies still in flight into this CTA's shared memory (bounded), then leave
    if (tid == 0)
      for (int j = k; j < min(k + kStages, nstage); ++j) mbar_wait(&full_bar[j % kStages], (j / kStages) & 1, status);
    __syncthreads();
    return;
  }

  // Tile max per head: lanes with the same `sub` hold partial maxima.
  float m = run_max;
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  if (lane < G) red[warp][lane] = m;
  __syncthreads();
  if (tid < G) {
    float mm = -INFINITY;
    for (int w = 0; w < kScoreThreads / 32; ++w) mm = fmaxf(mm, red[w][tid]);
    tile_max[tid] = mm;
  }
  __syncthreads();
  // e = exp(s - m_tile), written in place and to global in flat (row, head) order.
  float* e_dst = e_buf + (((int64_t)s * h_kv + g) * max_blocks + r0) * G;
  for (int i = tid; i < nrows * G; i += kScoreThreads) {
    const float e = expf(s_tile[i] - tile_max[i % G]);
    s_tile[i] = e;
    e_dst[i] = e;
  }
  __syncthreads();
  // Sum of e per head, fixed order: each warp owns heads h = warp, warp + 8, ...
  for (int h = warp; h < G; h += kScoreThreads / 32) {
    float z = 0.f;
    for (int r = lane; r < nrows; r += 32) z += s_tile[r * G + h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) part[((int64_t)s * h_q + g * G + h) * max_tiles + tile] = make_float2(tile_max[h], z);
  }
}

// Block-wide exclusive scan of one int per thread (kSelectThreads threads); returns the total via *total.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelectThreads / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[32 + lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[32 + warp - 1] : 0) + x - v;
  *total = scratch[32 + kSelectThreads / 32 - 1];
  __syncthreads();
  return before;
}

struct RadixResult {
  uint32_t digit;
  int krem;
};

template <int G>
__global__ void __launch_bounds__(kSelectThreads) select_kernel(
    const float* __restrict__ e_buf, const float2* __restrict__ part, int64_t max_tiles, int64_t max_blocks,
    int h_kv, int h_q, SessionArgs a, int rows_per_tile, int n_sink, int n_recent, int top_k, int budget,
    int slice_cap, int32_t* __restrict__ kept, float* __restrict__ group_scores, const float* __restrict__ gs_in) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int C = (int)cluster.num_blocks();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_raw);        // [slice_cap]
  float* coef = reinterpret_cast<float*>(key + slice_cap);       // [tiles in slice][G]
  __shared__ float s_M[G], s_invZ[G];
  __shared__ int hist[kRadixBins];
  __shared__ int tot[kRadixBins];
  __shared__ int scan_scratch[64];
  __shared__ RadixResult res;
  __shared__ int cta_count;

  const int s = blockIdx.z, g = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_blk = a.n_blk[s];
  const int sl = (n_blk + C - 1) / C;
  const int lo = min(n_blk, crank * sl), hi = min(n_blk, lo + sl);
  const int n_tiles = (n_blk + rows_per_tile - 1) / rows_per_tile;
  int32_t* kept_row = kept + ((int64_t)s * h_kv + g) * budget;

  if (gs_in != nullptr) {
    // group scores given (step-level scoring): keys straight from them
    const float* src = gs_in + ((int64_t)s * h_kv + g) * max_blocks;
    float* gs_dst = (group_scores && group_scores != gs_in) ? group_scores + ((int64_t)s * h_kv + g) * max_blocks
                                                              : nullptr;
    for (int b = lo + tid; b < hi; b += kSelectThreads) {
      const float gs = src[b];
      key[b - lo] = order_key(gs);
      if (gs_dst) gs_dst[b] = gs;
    }
    __syncthreads();
  } else {
  // 1. softmax normalisers of the group's heads (every CTA computes them the same way)
  if (warp < G) {
    const float2* p = part + ((int64_t)s * h_q + g * G + warp) * max_tiles;
    float M = -INFINITY;
    for (int t = lane; t < n_tiles; t += 32) M = fmaxf(M, p[t].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Z = 0.f;
    for (int t = lane; t < n_tiles; t += 32) Z += p[t].y * expf(p[t].x - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    if (lane == 0) {
      s_M[warp] = M;
      s_invZ[warp] = 1.f / Z;
    }
  }
  __syncthreads();
  // 2. per-tile coefficients exp(m_tile - M) / Z for the tiles overlapping this slice
  const int t0 = lo / rows_per_tile;
  const int nt = hi > lo ? (hi - 1) / rows_per_tile - t0 + 1 : 0;
  for (int i = tid; i < nt * G; i += kSelectThreads) {
    const int t = t0 + i / G, h = i % G;
    const float2 p = part[((int64_t)s * h_q + g * G + h) * max_tiles + t];
    coef[i] = expf(p.x - s_M[h]) * s_invZ[h];
  }
  __syncthreads();
  // 3. group scores of the slice
  const float* e_src = e_buf + ((int64_t)s * h_kv + g) * max_blocks * G;
  float* gs_dst = group_scores ? group_scores + ((int64_t)s * h_kv + g) * max_blocks : nullptr;
  for (int b = lo + tid; b < hi; b += kSelectThreads) {
    const float* cf = coef + (b / rows_per_tile - t0) * G;
    float gs = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) gs = fmaf(e_src[(int64_t)b * G + h], cf[h], gs);
    key[b - lo] = order_key(gs);
    if (gs_dst) gs_dst[b] = gs;
  }
  __syncthreads();
  }

  if (n_blk <= budget) {  // every block is kept (uniform across the cluster)
    for (int b = lo + tid; b < hi; b += kSelectThreads) kept_row[b] = b;
    if (crank == 0)
      for (int i = n_blk + tid; i < budget; i += kSelectThreads) kept_row[i] = -1;
    return;  // no distributed shared memory access on this path
  }
  const int cand_lo = n_sink, cand_hi = n_blk - n_recent;  // candidates [cand_lo, cand_hi)

  // 4. exact radix select of the top_k-th largest candidate key
  uint32_t prefix = 0, pmask = 0;
  int krem = top_k;
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < kRadixBins; i += kSelectThreads) hist[i] = 0;
    __syncthreads();
    const int clo = max(lo, cand_lo), chi = min(hi, cand_hi);
    for (int b = clo + tid; b < chi; b += kSelectThreads) {
      const uint32_t k = key[b - lo];
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (nb - 1)], 1);
    }
    cluster.sync();
    if (crank == 0) {
      // merged histogram; each thread owns 4 consecutive bins
      int local[4], sum = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bin = 4 * tid + j;
        int v = 0;
        if (bin < nb)
          for (int r = 0; r < C; ++r) v += cluster.map_shared_rank(hist, r)[bin];
        local[j] = v;
        sum += v;
      }
      // suffix sums over threads: count of keys in bins owned by higher threads
      // keys in bins owned by higher threads: an exclusive scan in reversed thread order
      int rev_total;
      tot[tid] = sum;
      __syncthreads();
      const int mine = tot[kSelectThreads - 1 - tid];
      const int excl = block_exclusive_scan(mine, scan_scratch, &rev_total);
      // thread tid' = kSelectThreads-1-tid owns `mine`; keys above tid' = excl
      tot[kSelectThreads - 1 - tid] = excl;
      __syncthreads();
      int above = tot[tid];
      for (int j = 3; j >= 0; --j) {
        const int bin = 4 * tid + j;
        if (bin < nb && local[j] > 0 && above < krem && krem <= above + local[j]) {
          res.digit = (uint32_t)bin;
          res.krem = krem - above;
        }
        above += local[j];
      }
    }
    cluster.sync();
    const RadixResult r = *cluster.map_shared_rank(&res, 0);
    prefix |= r.digit << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem = r.krem;
  }
  const uint32_t T = prefix;
  const int need_eq = krem;  // how many keys equal to T are taken (lowest ids first)

  // 5. stable compaction: each thread owns a contiguous run of the slice
  const int len = hi - lo;
  const int per = (len + kSelectThreads - 1) / kSelectThreads;
  const int u0 = lo + min(len, tid * per), u1 = lo + min(len, (tid + 1) * per);
  auto is_cand = [&](int b) { return b >= cand_lo && b < cand_hi; };
  int n_eq = 0;
  for (int b = u0; b < u1; ++b) n_eq += (is_cand(b) && key[b - lo] == T);
  int cta_eq;
  const int eq_off = block_exclusive_scan(n_eq, scan_scratch, &cta_eq);
  if (tid == 0) cta_count = cta_eq;
  cluster.sync();
  int eq_base = 0;
  for (int r = 0; r < crank; ++r) eq_base += *cluster.map_shared_rank(&cta_count, r);
  cluster.sync();  // everyone has read cta_count before it is reused
  int n_keep_local = 0, e_i = eq_base + eq_off;
  for (int b = u0; b < u1; ++b) {
    bool keep;
    if (!is_cand(b)) {
      keep = true;
    } else {
      const uint32_t k = key[b - lo];
      keep = k > T || (k == T && e_i < need_eq);
      e_i += (k == T);
    }
    n_keep_local += keep;
  }
  int cta_keep;
  const int keep_off = block_exclusive_scan(n_keep_local, scan_scratch, &cta_keep);
  if (tid == 0) cta_count = cta_keep;
  cluster.sync();
  int keep_base = 0;
  for (int r = 0; r < crank; ++r) keep_base += *cluster.map_shared_rank(&cta_count, r);
  int pos = keep_base + keep_off;
  e_i = eq_base + eq_off;
  for (int b = u0; b < u1; ++b) {
    bool keep;
    if (!is_cand(b)) {
      keep = true;
    } else {
      const uint32_t k = key[b - lo];
      keep = k > T || (k == T && e_i < need_eq);
      e_i += (k == T);
    }
    if (keep) kept_row[pos++] = b;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

template <int G>
cudaError_t launch_select(const Ctx& c, int n_sessions, const SessionArgs& a, int rpt, int max_blk, int32_t* kept,
                          float* group_scores, const float* gs_in, cudaStream_t st) {
  int C = (max_blk + 4095) / 4096;
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  const int slice_cap = (max_blk + C - 1) / C;
  const int tiles_cap = slice_cap / rpt + 2;
  const size_t smem_b = (size_t)slice_cap * 4 + (size_t)tiles_cap * G * 4;
  auto kb = select_kernel<G>;
  cudaError_t e;
  if ((e = ensure_smem(kb, c.device, smem_b)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, c.p.h_kv, n_sessions);
  cfg.blockDim = dim3(kSelectThreads);
  cfg.dynamicSmemBytes = smem_b;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kb, (const float*)c.e_buf, (const float2*)c.part, c.max_tiles, c.p.max_blocks,
                            c.p.h_kv, c.p.h_q, a, rpt, c.p.n_sink, c.p.n_recent, c.p.top_k, c.budget, slice_cap,
                            kept, group_scores, gs_in);
}

template <int D, int G>
cudaError_t launch_g(const Ctx& c, const uint16_t* q, const float* index, int n_sessions, const SessionArgs& a,
                     int32_t* kept, float* group_scores, float* head_scores, cudaStream_t st) {
  int max_blk = 0;
  int64_t rows = 0;
  for (int s = 0; s < n_sessions; ++s) {
    max_blk = max(max_blk, a.n_blk[s]);
    rows += (int64_t)a.n_blk[s] * c.p.h_kv;
  }
  if (max_blk == 0) {
    // nothing to score: every kept list is empty
    return cudaMemsetAsync(kept, 0xFF, sizeof(int32_t) * (size_t)n_sessions * c.p.h_kv * c.budget, st);
  }
  // rows per score tile: about 512 tiles over the call, 32..1024 rows each
  int64_t want = rows / 512;
  int rpt = kStageRows;
  while (rpt < want && rpt < 1024) rpt <<= 1;
  const int tiles = (max_blk + rpt - 1) / rpt;
  const size_t smem_a = (size_t)kStages * kStageRows * D * 4 + (size_t)rpt * G * 4;
  auto ka = score_tile_kernel<D, G>;
  cudaError_t e = ensure_smem(ka, c.device, smem_a);
  if (e != cudaSuccess) return e;
  ka<<<dim3(tiles, c.p.h_kv, n_sessions), kScoreThreads, smem_a, st>>>(
      q, index, c.p.max_blocks, c.p.h_kv, c.p.h_q, a, rpt, c.e_buf, c.part, c.max_tiles, head_scores, c.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  return launch_select<G>(c, n_sessions, a, rpt, max_blk, kept, group_scores, nullptr, st);
}

template <int D>
cudaError_t launch_d(const Ctx& c, const uint16_t* q, const float* index, int n_sessions, const SessionArgs& a,
                     int32_t* kept, float* gs, float* hs, cudaStream_t st) {
  switch (c.group) {
    case 1: return launch_g<D, 1>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 2: return launch_g<D, 2>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 3: return launch_g<D, 3>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 4: return launch_g<D, 4>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 5: return launch_g<D, 5>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 6: return launch_g<D, 6>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 7: return launch_g<D, 7>(c, q, index, n_sessions, a, kept, gs, hs, st);
    case 8: return launch_g<D, 8>(c, q, index, n_sessions, a, kept, gs, hs, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_select_given(const Ctx& c, const float* gs, int n_sessions, const SessionArgs& a, int32_t* kept,
                                float* group_scores_out, cudaStream_t st) {
  int max_blk = 0;
  for (int s = 0; s < n_sessions; ++s) max_blk = max(max_blk, a.n_blk[s]);
  if (max_blk == 0)
    return cudaMemsetAsync(kept, 0xFF, sizeof(int32_t) * (size_t)n_sessions * c.p.h_kv * c.budget, st);
  switch (c.group) {
    case 1: return launch_select<1>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 2: return launch_select<2>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 3: return launch_select<3>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 4: return launch_select<4>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 5: return launch_select<5>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 6: return launch_select<6>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 7: return launch_select<7>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
    case 8: return launch_select<8>(c, n_sessions, a, kStageRows, max_blk, kept, group_scores_out, gs, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_score_select(const Ctx& c, const uint16_t* q, int n_q, const float* index, int n_sessions,
                                const SessionArgs& a, int32_t* kept, float* group_scores, float* head_scores,
                                cudaStream_t st) {
  if (n_q != 1) {
    float* gs = group_scores ? group_scores : c.step_gs;
    cudaError_t e = launch_step_scores(c, q, n_q, index, n_sessions, a, gs, st);
    if (e != cudaSuccess) return e;
    return launch_select_given(c, gs, n_sessions, a, kept, group_scores, st);
  }
  return c.p.d == 128 ? launch_d<128>(c, q, index, n_sessions, a, kept, group_scores, head_scores, st)
                      : launch_d<64>(c, q, index, n_sessions, a, kept, group_scores, head_scores, st);
}

}  // namespace kvm
