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
//   1-D bulk copies (5-stage mbarrier pipeline; one warp polls, one CTA
//   barrier per stage), computes the G scores of
//   each row with 8 lanes per row and shuffle reductions, then writes
//   e[b][h] = exp(s[b][h] - m_tile[h]) and the tile's (m_tile, sum e) per head.
// Kernel B (select_kernel), grid (C, h_kv, sessions), clusters of C CTAs:
//   each CTA owns 1/C of the blocks.  From the tiles' partials it forms the
//   softmax normalisers, Gs[b] = sum_h e[b][h] * exp(m_tile - M_h) / Z_h, and
//   then runs an exact 3-pass radix select (11/11/10 bits) over the
//   candidates: per pass each CTA builds its slice's histogram with
//   shared-memory atomics, one cluster barrier, and every CTA pulls the C
//   histograms through distributed shared memory (16-byte loads, 4 bins each)
//   and scans the merged counts itself (double-buffered histograms, so one
//   barrier a pass).
//   A stable compaction follows (one exchange of per-CTA tie / kept counts):
//   ascending ids, equal scores resolved toward the lower id.
#include <cooperative_groups.h>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace cg = cooperative_groups;

namespace kvm {
namespace {

constexpr int kScoreThreads = 256;  // 8 warps, 4 rows each per stage
constexpr int kStageRows = 32;
constexpr int kStages = 5;
constexpr int kSelectThreads = 512;
constexpr int kRadixBins = 2048;

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_tile_kernel(
    const uint16_t* __restrict__ q, const float* __restrict__ index, int64_t max_blocks, int h_kv, int h_q,
    SessionArgs a, int rows_per_tile, float* __restrict__ e_buf, float2* __restrict__ part, int64_t max_tiles,
    float* __restrict__ head_scores, uint32_t* __restrict__ status, int q_heads, int avg_group) {
  // q_heads: query heads per session in q.  avg_group > 0 (with G == 1): the withdrawn scoring, one score row
  // per KV head from the unweighted mean of its avg_group query heads (taken in fp32).
  constexpr int NV = D / 32;  // float4 chunks per lane per row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* stage_buf = reinterpret_cast<float*>(smem_raw);                   // [kStages][32][D]
  float* s_tile = stage_buf + kStages * kStageRows * D;                    // [rows_per_tile][G]
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ float red[kScoreThreads / 32][G];
  __shared__ float tile_max[G];

  griddep_wait();
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
  if (G == 1 && avg_group > 0) {
#pragma unroll
    for (int j = 0; j < NV * 4; ++j) qv[0][j] = 0.f;
    for (int h = 0; h < avg_group; ++h) {
      const uint16_t* qh = q + ((int64_t)s * q_heads + g * avg_group + h) * D;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh + 4 * sub + 32 * i));
        qv[0][4 * i + 0] += bf16lo(w.x);
        qv[0][4 * i + 1] += bf16hi(w.x);
        qv[0][4 * i + 2] += bf16lo(w.y);
        qv[0][4 * i + 3] += bf16hi(w.y);
      }
    }
#pragma unroll
    for (int j = 0; j < NV * 4; ++j) qv[0][j] = qv[0][j] / (float)avg_group * inv_sqrt_d;
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint16_t* qh = q + ((int64_t)s * q_heads + g * G + h) * D;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh + 4 * sub + 32 * i));
        qv[h][4 * i + 0] = bf16lo(w.x) * inv_sqrt_d;
        qv[h][4 * i + 1] = bf16hi(w.x) * inv_sqrt_d;
        qv[h][4 * i + 2] = bf16lo(w.y) * inv_sqrt_d;
        qv[h][4 * i + 3] = bf16hi(w.y) * inv_sqrt_d;
      }
    }
  }
  float run_max = -INFINITY;  // lane (sub == h) tracks head h over its rows

  int k = 0;
  bool aborted = false;
  for (; k < nstage; ++k) {
    // warp 0 alone polls the stage's barrier; the CTA barrier then releases everyone, and (being past every
    // warp's work on stage k - 1) lets thread 0 refill that stage
    bool ok = true;
    if (warp == 0) ok = mbar_wait(&full_bar[k % kStages], (k / kStages) & 1, status);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid == 0 && k >= 1 && k - 1 + kStages < nstage) issue(k - 1 + kStages);
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
  }
  if (aborted) {
    // drain the copies still in flight into this CTA's shared memory (bounded), then leave: stages k .. issued-1
    const int issued = min(k == 0 ? kStages : k - 1 + kStages, nstage);
    if (tid == 0)
      for (int j = k; j < issued; ++j) mbar_wait(&full_bar[j % kStages], (j / kStages) & 1, status);
    __syncthreads();
    return;
  }
  __syncthreads();  // every warp is done with the last stage (s_tile complete)
  griddep_launch_dependents();  // the selection may be scheduled while this epilogue runs

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

struct RadixResult {
  uint32_t digit;
  int krem;
};

// Block-wide exclusive scan of one int per thread for NT threads; returns the total via *total.
template <int NT>
__device__ int block_exclusive_scan_n(int v, int* scratch, int* total) {
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
    int w = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[32 + lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[32 + warp - 1] : 0) + x - v;
  *total = scratch[32 + NT / 32 - 1];
  __syncthreads();
  return before;
}

template <int G>
__global__ void __launch_bounds__(kSelectThreads) select_kernel(
    const float* __restrict__ e_buf, const float2* __restrict__ part, int64_t max_tiles, int64_t max_blocks,
    int h_kv, int h_q, SessionArgs a, int rows_per_tile, int n_sink, int n_recent, int top_k, int budget,
    int slice_cap, int32_t* __restrict__ kept, float* __restrict__ group_scores, const float* __restrict__ gs_in) {
  constexpr int NT = kSelectThreads;
  griddep_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int C = (int)cluster.num_blocks();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_raw);        // [slice_cap]
  float* coef = reinterpret_cast<float*>(key + slice_cap);       // [tiles in slice][G]
  __shared__ float s_M[G], s_invZ[G];
  __shared__ __align__(16) int hist[2][kRadixBins];  // double-buffered: pass p builds hist[p & 1] while others may read the other
  __shared__ int scan_scratch[64];
  __shared__ RadixResult res;
  __shared__ int cnt[2];               // this CTA's (equal to T, kept otherwise) counts, read by higher ranks
  __shared__ int sums[NT];             // per-thread merged bin counts, then the counts above each thread

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
    for (int b = lo + tid; b < hi; b += NT) {
      const float gs = src[b];
      key[b - lo] = order_key(gs);
      if (gs_dst) gs_dst[b] = gs;
    }
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
    for (int i = tid; i < nt * G; i += NT) {
      const int t = t0 + i / G, h = i % G;
      const float2 p = part[((int64_t)s * h_q + g * G + h) * max_tiles + t];
      coef[i] = expf(p.x - s_M[h]) * s_invZ[h];
    }
    __syncthreads();
    // 3. group scores of the slice
    const float* e_src = e_buf + ((int64_t)s * h_kv + g) * max_blocks * G;
    float* gs_dst = group_scores ? group_scores + ((int64_t)s * h_kv + g) * max_blocks : nullptr;
#pragma unroll 4
    for (int b = lo + tid; b < hi; b += NT) {
      const float* cf = coef + (b / rows_per_tile - t0) * G;
      float gs = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) gs = fmaf(e_src[(int64_t)b * G + h], cf[h], gs);
      key[b - lo] = order_key(gs);
      if (gs_dst) gs_dst[b] = gs;
    }
  }
  __syncthreads();

  if (n_blk <= budget) {  // every block is kept (uniform across the cluster)
    for (int b = lo + tid; b < hi; b += NT) kept_row[b] = b;
    if (crank == 0)
      for (int i = n_blk + tid; i < budget; i += NT) kept_row[i] = -1;
    return;  // no distributed shared memory access on this path
  }
  const int cand_lo = n_sink, cand_hi = n_blk - n_recent;  // candidates [cand_lo, cand_hi)
  const int len = hi - lo;
  const int n_iter = (len + NT - 1) / NT;

  // 4. exact radix select of the top_k-th largest candidate key (11 + 11 + 10 bits).  Each CTA builds the
  //    histogram of its slice; after one cluster barrier every CTA pulls all C histograms (independent
  //    loads) and scans the merged counts itself, so all CTAs reach the same digit without a second barrier.
  uint32_t prefix = 0, pmask = 0;
  int krem = top_k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    int* h = hist[pass & 1];
    for (int i = tid; i < kRadixBins; i += NT) h[i] = 0;
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < n_iter; ++j) {
      const int b = lo + tid + j * NT;
      int d = -1;
      if (b < hi && b >= cand_lo && b < cand_hi) {
        const uint32_t k = key[b - lo];
        if ((k & pmask) == prefix) d = (int)((k >> shift) & (uint32_t)(nb - 1));
      }
      if (d >= 0) atomicAdd(&h[d], 1);
    }
    cluster.sync();  // every slice's histogram is complete (and the previous pass's pulls are done)
    // merged counts of this thread's 4 bins (one 16-byte remote load per rank), then keys in bins owned by
    // higher threads (reversed scan)
    int local[4] = {0, 0, 0, 0}, sum = 0;
    if (4 * tid < nb) {
      int4 parts[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < C) parts[r] = *reinterpret_cast<const int4*>(cluster.map_shared_rank(h, r) + 4 * tid);
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < C) {
          local[0] += parts[r].x;
          local[1] += parts[r].y;
          local[2] += parts[r].z;
          local[3] += parts[r].w;
        }
      sum = local[0] + local[1] + local[2] + local[3];
    }
    const int rev = NT - 1 - tid;
    sums[tid] = sum;
    __syncthreads();
    int total;
    const int excl_rev = block_exclusive_scan_n<NT>(sums[rev], scan_scratch, &total);
    sums[rev] = excl_rev;  // keys in bins owned by threads above `rev`
    __syncthreads();
    int above = sums[tid];
#pragma unroll
    for (int jb = 3; jb >= 0; --jb) {
      const int bin = 4 * tid + jb;
      if (bin < nb && local[jb] > 0 && above < krem && krem <= above + local[jb]) {
        res.digit = (uint32_t)bin;
        res.krem = krem - above;
      }
      above += local[jb];
    }
    __syncthreads();
    prefix |= res.digit << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem = res.krem;
    __syncthreads();  // res and sums are rewritten by the next pass
  }
  const uint32_t T = prefix;
  const int need_eq = krem;  // how many keys equal to T are taken (lowest ids first, over the whole cluster)
  griddep_launch_dependents();  // the view kernel may be scheduled while the compaction runs

  // 5. stable compaction.  Warp w owns slice positions [w * 32 * n_iter, (w + 1) * 32 * n_iter), lane-interleaved
  //    (conflict-free shared-memory reads); block order is kept within and across warps and CTAs.
  auto is_cand = [&](int b) { return b >= cand_lo && b < cand_hi; };
  const int wbase = lo + warp * 32 * n_iter;
  int eq_w = 0, gt_w = 0, nc_w = 0;
  for (int j = 0; j < n_iter; ++j) {
    const int b = wbase + j * 32 + lane;
    bool eq = false, gt = false, nc = false;
    if (b < hi) {
      if (!is_cand(b)) {
        nc = true;
      } else {
        const uint32_t k = key[b - lo];
        eq = k == T;
        gt = k > T;
      }
    }
    eq_w += __popc(__ballot_sync(0xffffffffu, eq));
    gt_w += __popc(__ballot_sync(0xffffffffu, gt));
    nc_w += __popc(__ballot_sync(0xffffffffu, nc));
  }
  int eq_cta, other_cta;
  const int eq_before = block_exclusive_scan_n<NT>(lane == 0 ? eq_w : 0, scan_scratch, &eq_cta);
  block_exclusive_scan_n<NT>(lane == 0 ? gt_w + nc_w : 0, scan_scratch, &other_cta);
  if (tid == 0) {
    cnt[0] = eq_cta;
    cnt[1] = other_cta;
  }
  cluster.sync();
  // counts of the lower ranks: ties before this CTA, and kept blocks before it
  int eq_base = 0, keep_base = 0;
  for (int r = 0; r < crank; ++r) {
    const int* rc = cluster.map_shared_rank(cnt, r);
    const int e_r = rc[0], o_r = rc[1];
    const int taken = max(0, min(e_r, need_eq - eq_base));
    keep_base += o_r + taken;
    eq_base += e_r;
  }
  // per warp: ties before the warp (within the cluster) and kept blocks before the warp
  const int eq_warp0 = eq_base + __shfl_sync(0xffffffffu, eq_before, 0);
  int keep_w = 0;
  {
    int eq_run = eq_warp0;
    for (int j = 0; j < n_iter; ++j) {
      const int b = wbase + j * 32 + lane;
      bool keep = false, eq = false;
      if (b < hi) {
        if (!is_cand(b)) {
          keep = true;
        } else {
          const uint32_t k = key[b - lo];
          eq = k == T;
          keep = k > T;
        }
      }
      const unsigned eqm = __ballot_sync(0xffffffffu, eq);
      if (eq) keep = eq_run + __popc(eqm & ((1u << lane) - 1)) < need_eq;
      eq_run += __popc(eqm);
      keep_w += __popc(__ballot_sync(0xffffffffu, keep));
    }
  }
  int keep_cta;
  const int keep_before = block_exclusive_scan_n<NT>(lane == 0 ? keep_w : 0, scan_scratch, &keep_cta);
  int pos = keep_base + __shfl_sync(0xffffffffu, keep_before, 0);
  {
    int eq_run = eq_warp0;
    for (int j = 0; j < n_iter; ++j) {
      const int b = wbase + j * 32 + lane;
      bool keep = false, eq = false;
      if (b < hi) {
        if (!is_cand(b)) {
          keep = true;
        } else {
          const uint32_t k = key[b - lo];
          eq = k == T;
          keep = k > T;
        }
      }
      const unsigned eqm = __ballot_sync(0xffffffffu, eq);
      if (eq) keep = eq_run + __popc(eqm & ((1u << lane) - 1)) < need_eq;
      eq_run += __popc(eqm);
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) kept_row[pos + __popc(km & ((1u << lane) - 1))] = b;
      pos += __popc(km);
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

template <int G>
cudaError_t launch_select(const Ctx& c, int n_sessions, const SessionArgs& a, int rpt, int max_blk, int32_t* kept,
                          float* group_scores, const float* gs_in, cudaStream_t st, int part_heads = -1) {
  if (part_heads < 0) part_heads = c.p.h_q;  // score rows per session in the tile partials
  int C = (max_blk + 4095) / 4096;
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  const int slice_cap = (max_blk + C - 1) / C;
  const int tiles_cap = slice_cap / rpt + 2;
  const size_t smem_b = (size_t)slice_cap * 4 + (size_t)tiles_cap * G * 4;
  auto kb = select_kernel<G>;
  cudaError_t e;
  if ((e = ensure_smem(kb, c.device, smem_b)) != cudaSuccess) return e;
  return launch_pdl(kb, dim3(C, c.p.h_kv, n_sessions), dim3(kSelectThreads), smem_b, st, C, (const float*)c.e_buf,
                    (const float2*)c.part, c.max_tiles, c.p.max_blocks, c.p.h_kv, part_heads, a, rpt, c.p.n_sink,
                    c.p.n_recent, c.p.top_k, c.budget, slice_cap, kept, group_scores, gs_in);
}

// Rows per score tile: one wave of two CTAs per SM over the call (a multiple of 32 rows, 32..4096).
int rows_per_tile(const Ctx& c, int n_sessions, int max_blk) {
  const int64_t units = (int64_t)c.p.h_kv * n_sessions;
  const int64_t sms = c.num_sms > 0 ? c.num_sms : 1;
  const int64_t tiles_per_head = (2 * sms + units - 1) / units;
  int64_t rpt64 = (max_blk + tiles_per_head - 1) / tiles_per_head;
  rpt64 = (rpt64 + kStageRows - 1) / kStageRows * kStageRows;
  return (int)(rpt64 < kStageRows ? kStageRows : (rpt64 > 4096 ? 4096 : rpt64));
}

// The withdrawn scoring (a control): one softmax per KV head over the scores of the group's averaged query.
template <int D>
cudaError_t launch_withdrawn(const Ctx& c, const uint16_t* q, const float* index, int n_sessions, const SessionArgs& a,
                             int32_t* kept, float* group_scores, cudaStream_t st) {
  int max_blk = 0;
  for (int s = 0; s < n_sessions; ++s) max_blk = max(max_blk, a.n_blk[s]);
  if (max_blk == 0) return cudaMemsetAsync(kept, 0xFF, sizeof(int32_t) * (size_t)n_sessions * c.p.h_kv * c.budget, st);
  const int rpt = rows_per_tile(c, n_sessions, max_blk);
  const int tiles = (max_blk + rpt - 1) / rpt;
  const size_t smem_a = (size_t)kStages * kStageRows * D * 4 + (size_t)rpt * 4;
  auto ka = score_tile_kernel<D, 1>;
  cudaError_t e = ensure_smem(ka, c.device, smem_a);
  if (e != cudaSuccess) return e;
  // partial rows are indexed per KV head here (h_kv score rows per session)
  if ((e = launch_pdl(ka, dim3(tiles, c.p.h_kv, n_sessions), dim3(kScoreThreads), smem_a, st, 1, q, index,
                      c.p.max_blocks, c.p.h_kv, c.p.h_kv, a, rpt, c.e_buf, c.part, c.max_tiles, (float*)nullptr,
                      c.status, c.p.h_q, c.group)) != cudaSuccess)
    return e;
  return launch_select<1>(c, n_sessions, a, rpt, max_blk, kept, group_scores, nullptr, st, c.p.h_kv);
}

// The recent-only control: the last min(n_blk, budget) blocks, ascending, -1 padded.
__global__ void recent_only_kernel(int32_t* __restrict__ kept, int h_kv, int budget, SessionArgs a) {
  griddep_wait();
  const int g = blockIdx.x, s = blockIdx.y;
  const int n_keep = a.n_keep[s], n_blk = a.n_blk[s];
  int32_t* row = kept + ((int64_t)s * h_kv + g) * budget;
  for (int i = threadIdx.x; i < budget; i += blockDim.x) row[i] = i < n_keep ? n_blk - n_keep + i : -1;
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
  (void)rows;
  const int rpt = rows_per_tile(c, n_sessions, max_blk);
  const int tiles = (max_blk + rpt - 1) / rpt;
  const size_t smem_a = (size_t)kStages * kStageRows * D * 4 + (size_t)rpt * G * 4;
  auto ka = score_tile_kernel<D, G>;
  cudaError_t e = ensure_smem(ka, c.device, smem_a);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(ka, dim3(tiles, c.p.h_kv, n_sessions), dim3(kScoreThreads), smem_a, st, 1, q, index,
                      c.p.max_blocks, c.p.h_kv, c.p.h_q, a, rpt, c.e_buf, c.part, c.max_tiles, head_scores,
                      c.status, c.p.h_q, 0)) != cudaSuccess)
    return e;

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

cudaError_t launch_select_control(const Ctx& c, int control, const uint16_t* q, const float* index, int n_sessions,
                                  const SessionArgs& a, int32_t* kept, float* group_scores, cudaStream_t st) {
  if (control == KVM_CONTROL_RECENT_ONLY)
    return launch_pdl(recent_only_kernel, dim3(c.p.h_kv, n_sessions), dim3(256), 0, st, 1, kept, c.p.h_kv, c.budget, a);
  return c.p.d == 128 ? launch_withdrawn<128>(c, q, index, n_sessions, a, kept, group_scores, st)
                      : launch_withdrawn<64>(c, q, index, n_sessions, a, kept, group_scores, st);
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
