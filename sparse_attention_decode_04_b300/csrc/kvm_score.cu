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
//   Before waiting for the preceding kernel it prefetches the rows of its first
//   stages into L2.
// Kernel B (select_kernel), grid (C, h_kv, sessions), clusters of C CTAs:
//   each CTA owns 1/C of the blocks.  From the tiles' partials it forms the
//   softmax normalisers, Gs[b] = sum_h e[b][h] * exp(m_tile - M_h) / Z_h (the
//   exponentials are loaded into registers before the normalisers are formed,
//   so the two L2 round trips overlap), and builds the first radix histogram as
//   it goes.
//   Exact radix select over the candidates' order keys, 12 + 12 + 8 bits: per
//   pass one cluster barrier, then a single warp locates the boundary bin over
//   the merged counts with two rounds of distributed-shared-memory loads (64
//   super-bin sums from every CTA, then the bins of the one super-bin that
//   holds the boundary).  The passes stop as soon as the boundary bin holds
//   exactly the keys still to take (all of them are kept), and after the second
//   pass a boundary bin of at most 32 keys is settled without a third pass: its
//   keys travel with the compaction's count exchange and every CTA ranks them.
//   A stable compaction follows: each CTA pushes its counts (and boundary keys)
//   into the other CTAs before one last cluster barrier, so no CTA reads
//   another's shared memory after it.  Ids come out ascending; equal scores
//   resolve toward the lower id.
#include <cooperative_groups.h>

#include <algorithm>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace cg = cooperative_groups;

namespace kvm {
namespace {

// Moves [src, src + bytes) into L2 (no completion to wait for); src and bytes multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

constexpr int kScoreThreads = 256;  // 8 warps, 4 rows each per stage
constexpr int kStageRows = 32;
constexpr int kStages = 5;
constexpr int kSelectThreads = 512;

// The query slice a lane holds for its row's dot products (LPR lanes per row), scaled by 1/sqrt(d): dims
// 4*sub + 4*LPR*i + {0..3} of each of the G query heads of KV head g.  avg_group > 0 (with G == 1): the withdrawn scoring's single row, the
// unweighted mean of the group's avg_group query heads (taken in fp32).
template <int D, int G, int LPR>
__device__ __forceinline__ void load_query(float (&qv)[G][D / LPR], const uint16_t* __restrict__ q, int s, int g,
                                           int q_heads, int avg_group, int sub) {
  constexpr int NV = D / (4 * LPR);  // float4 chunks per lane per row
  const float inv_sqrt_d = __frsqrt_rn((float)D);
  if (G == 1 && avg_group > 0) {
#pragma unroll
    for (int j = 0; j < NV * 4; ++j) qv[0][j] = 0.f;
    for (int h = 0; h < avg_group; ++h) {
      const uint16_t* qh = q + ((int64_t)s * q_heads + g * avg_group + h) * D;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh + 4 * sub + 4 * LPR * i));
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
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh + 4 * sub + 4 * LPR * i));
        qv[h][4 * i + 0] = bf16lo(w.x) * inv_sqrt_d;
        qv[h][4 * i + 1] = bf16hi(w.x) * inv_sqrt_d;
        qv[h][4 * i + 2] = bf16lo(w.y) * inv_sqrt_d;
        qv[h][4 * i + 3] = bf16hi(w.y) * inv_sqrt_d;
      }
    }
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_tile_kernel(
    const uint16_t* __restrict__ q, const float* __restrict__ index, int64_t max_blocks, int h_kv, int h_q,
    SessionArgs a, int rows_per_tile, float* __restrict__ e_buf, int64_t e_stride, float2* __restrict__ part,
    int64_t max_tiles, float* __restrict__ head_scores, uint32_t* __restrict__ status, int q_heads, int avg_group) {
  // q_heads: query heads per session in q.  avg_group > 0 (with G == 1): the withdrawn scoring, one score row
  // per KV head from the unweighted mean of its avg_group query heads (taken in fp32).
  constexpr int NV = D / 32;  // float4 chunks per lane per row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* stage_buf = reinterpret_cast<float*>(smem_raw);                   // [kStages][32][D]
  float* s_tile = stage_buf + kStages * kStageRows * D;                    // [rows_per_tile][G]
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ float red[kScoreThreads / 32][G];
  __shared__ float tile_max[G];

  // While the preceding kernel finishes, warm L2 with the rows of this tile's first stages.  A prefetch only
  // moves lines into L2, the point of coherence, so rows written before the wait below completes (an index
  // append earlier in the stream) are still what the stage loads read.
  if (threadIdx.x == 0) {
    const int64_t nb = a.n_blk[blockIdx.z], rr0 = (int64_t)blockIdx.x * rows_per_tile;
    if (rr0 < nb) {
      const int64_t cap = kStages * kStageRows < rows_per_tile ? kStages * kStageRows : rows_per_tile;
      const int64_t pr = cap < nb - rr0 ? cap : nb - rr0;
      prefetch_l2(index + (((int64_t)blockIdx.z * h_kv + blockIdx.y) * max_blocks + rr0) * D,
                  (uint32_t)(pr * D * 4));
    }
  }
  griddep_wait();
  const int s = blockIdx.z, g = blockIdx.y, tile = blockIdx.x;
  const int64_t n_blk = a.n_blk[s];
  const int64_t r0 = (int64_t)tile * rows_per_tile;
  if (r0 >= n_blk) return;
  const int nrows = (int)(rows_per_tile < n_blk - r0 ? (int64_t)rows_per_tile : n_blk - r0);
  const int nstage = (nrows + kStageRows - 1) / kStageRows;
  KVM_DEBUG_CHECK(r0 + nrows <= max_blocks && r0 + nrows <= e_stride && tile < max_tiles, status);
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

  float qv[G][NV * 4];
  load_query<D, G, 8>(qv, q, s, g, q_heads, avg_group, sub);
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
  // e = exp(s - m_tile), written in place and to global head-major ([head][block]: the selection reads one
  // head of 32 consecutive blocks per warp-wide load).
  float* e_dst = e_buf + ((int64_t)s * h_kv + g) * G * e_stride + r0;
  for (int i = tid; i < nrows * G; i += kScoreThreads) {
    const int h = i / nrows, r = i - h * nrows;
    const float e = expf(s_tile[r * G + h] - tile_max[h]);
    s_tile[r * G + h] = e;
    e_dst[(int64_t)h * e_stride + r] = e;
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

// Digits of the order keys: pass 0 takes bits 31..20 (sign, exponent, 3 mantissa bits), pass 1 bits 19..8,
// pass 2 bits 7..0.  A pass's histogram is merged across the cluster in two small steps: per-CTA sums of 64
// super-bins (each nb/64 bins) are pulled first, then the bins of the one super-bin that holds the boundary.
constexpr int kSelBins = 4096;
constexpr int kSelSup = 64;
constexpr int kMaxCluster = 8;  // CTAs per cluster at most

__device__ __forceinline__ int sel_shift(int pass) { return pass == 0 ? 20 : (pass == 1 ? 8 : 0); }
__device__ __forceinline__ int sel_bins(int pass) { return pass == 2 ? 256 : kSelBins; }

struct SelResult {
  uint32_t digit;  // boundary bin of the pass
  int krem;        // keys still to take inside the boundary bin
  int count;       // keys in the boundary bin (cluster-wide)
};

// Split cluster barrier: every CTA arrives when it starts and waits before its first store into another CTA's
// shared memory, so that no CTA is written before it runs.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Warp 0: finds, over the cluster's merged counts, the bin holding the krem-th largest key of this pass.
// sup_all[r] holds CTA r's super-bin sums (pushed into every CTA before the pass's cluster barrier); hist is this
// CTA's histogram buffer, and the same offsets are read in every CTA of the cluster.
__device__ __forceinline__ SelResult sel_boundary(cg::cluster_group& cluster, int C, const int (*sup_all)[kSelSup],
                                                  const int* hist, int nb, int krem) {
  const int lane = threadIdx.x & 31;
  // 1. super-bins 2*lane and 2*lane + 1, summed over the cluster (local loads)
  int c0 = 0, c1 = 0;
#pragma unroll
  for (int r = 0; r < kMaxCluster; ++r)
    if (r < C) {
      const int2 v = *reinterpret_cast<const int2*>(sup_all[r] + 2 * lane);
      c0 += v.x;
      c1 += v.y;
    }
  // keys above each of this lane's super-bins: inclusive suffix sum over the higher lanes
  int suf = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += y;
  }
  const int above1 = suf - c0 - c1, above0 = above1 + c1;
  const bool in1 = above1 < krem && krem <= above1 + c1, in0 = above0 < krem && krem <= above0 + c0;
  const unsigned hit = __ballot_sync(0xffffffffu, in0 || in1);
  const int src = hit ? __ffs(hit) - 1 : 0;  // exactly one lane holds the boundary super-bin
  const int sb = __shfl_sync(0xffffffffu, in1 ? 2 * lane + 1 : 2 * lane, src);
  const int sabove = __shfl_sync(0xffffffffu, in1 ? above1 : above0, src);
  // 2. the bins of that super-bin (nb / 64 of them, two per lane), summed over the cluster
  const int bw = nb / kSelSup;
  int b0 = 0, b1 = 0;
  if (2 * lane < bw) {
    int2 v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < C) v[r] = *reinterpret_cast<const int2*>(cluster.map_shared_rank(hist, r) + sb * bw + 2 * lane);
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < C) {
        b0 += v[r].x;
        b1 += v[r].y;
      }
  }
  int suf2 = b0 + b1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, suf2, o);
    if (lane + o < 32) suf2 += y;
  }
  const int a1 = sabove + suf2 - b0 - b1, a0 = a1 + b1;
  const bool j1 = b1 > 0 && a1 < krem && krem <= a1 + b1, j0 = b0 > 0 && a0 < krem && krem <= a0 + b0;
  const unsigned hit2 = __ballot_sync(0xffffffffu, j0 || j1);
  const int src2 = hit2 ? __ffs(hit2) - 1 : 0;
  SelResult r;
  r.digit = (uint32_t)__shfl_sync(0xffffffffu, sb * bw + (j1 ? 2 * lane + 1 : 2 * lane), src2);
  r.krem = krem - __shfl_sync(0xffffffffu, j1 ? a1 : a0, src2);
  r.count = __shfl_sync(0xffffffffu, j1 ? b1 : b0, src2);
  return r;
}

constexpr int kSelTilesPerLane = 10;  // tile partials a normaliser lane holds: up to 320 tiles per head
constexpr int kSelPre = 2;            // 4-block groups of exponentials a thread loads before the normalisers
constexpr int kSelList = 32;          // boundary keys resolved by an exchanged list instead of a third pass
constexpr int kSelSlice = 2048;       // blocks per CTA of the selection cluster (up to kMaxCluster CTAs)

// Shared-memory state of the radix select and the compaction (one per CTA).
struct SelShared {
  static constexpr int NW = kSelectThreads / 32;
  int hist[2][kSelBins];  // pass p builds hist[p & 1]; the other may still be read remotely
  int sup_all[2][kMaxCluster][kSelSup];  // pass p: every CTA's super-bin sums, pushed by their owners
  int warp_cnt[NW][2];               // per warp: blocks kept for sure, keys equal to the boundary key
  int warp_taken[NW];                // per warp: boundary-list keys taken (list mode)
  int cnts[kMaxCluster][2];          // pushed by the lower-ranked CTAs of the cluster: the same, per CTA
  uint2 blist[kMaxCluster][kSelList];  // list mode: each CTA's boundary-bin keys (key, block), pushed to all
  int blist_n[kMaxCluster];
  int taken_cnt[kMaxCluster];        // list mode: keys of each CTA's list that are taken
  int own_taken[kSelList];           // list mode: this CTA's taken blocks
  uint2 flat[kSelList];              // list mode: the cluster's boundary keys in one row
  uint32_t tmask[kSelectThreads];    // list mode: per thread, which of its slice positions are taken
  int own_n, own_taken_n;
  SelResult res;
};

// Clears what the selection accumulates into; the caller synchronises the CTA before the keys' histogram.
__device__ __forceinline__ void sel_init(SelShared& S) {
  const int tid = threadIdx.x;
  for (int i = tid; i < kSelBins; i += kSelectThreads) S.hist[0][i] = 0;
  if (tid < kMaxCluster) S.taken_cnt[tid] = 0;
  if (tid < SelShared::NW) S.warp_taken[tid] = 0;
  if (tid == 0) S.own_n = S.own_taken_n = 0;
  S.tmask[tid] = 0;
}

// The order keys of the slice's blocks [lo, hi) are in key[0 .. hi - lo), and S.hist[0] holds the pass-0
// histogram of this CTA's candidates.  Finds the top_k-th largest candidate key over the cluster and writes the
// kept blocks (candidates above it, the forced sink / recent blocks, ties resolved toward the lower block) to
// kept_row in ascending block order.
__device__ void sel_radix_compact(cg::cluster_group& cluster, SelShared& S, const uint32_t* key, int lo, int hi,
                                  int cand_lo, int cand_hi, int top_k, int budget, int32_t* kept_row,
                                  uint32_t* status) {
  constexpr int NT = kSelectThreads, NW = SelShared::NW;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int crank = (int)cluster.block_rank();
  const int C = (int)cluster.num_blocks();
  const int n_iter = (hi - lo + NT - 1) / NT;
  auto is_cand = [&](int b) { return b >= cand_lo && b < cand_hi; };

  // ---- radix select of the top_k-th largest candidate key.  After pass p the boundary is the bin `prefix`
  //      of the key's bits above `sh`.  The passes stop early when the boundary bin holds exactly the keys
  //      still to take (all of them are kept), or, after the second pass, when it holds at most kSelList
  //      keys: those are then exchanged as a list and ranked exactly in the compaction.
  cluster_wait();  // paired with the arrival at the kernel's start: every CTA of the cluster is running
  uint32_t prefix = 0;
  int sh = 32, krem = top_k, bcount = 0;
  bool resolved = top_k == 0;  // no candidate is taken: the boundary lies above every key
  bool list_mode = false;
#pragma unroll 1
  for (int pass = 0; pass < 3 && !resolved; ++pass) {
    const int shift = sel_shift(pass), nb = sel_bins(pass);
    int* h = S.hist[pass & 1];
    if (pass > 0) {
      // histogram of this pass's digit over the candidates inside the boundary bin (h was cleared below)
      for (int j = 0; j < n_iter; ++j) {
        const int b = lo + tid + j * NT;
        if (b < hi && is_cand(b)) {
          const uint32_t k = key[b - lo];
          if ((k >> sh) == prefix) atomicAdd(&h[(k >> shift) & (uint32_t)(nb - 1)], 1);
        }
      }
    }
    __syncthreads();  // this CTA's histogram is complete
    // per-CTA super-bin sums (nb / 64 bins each): 4096 bins, 8 per thread, then over 8 consecutive lanes; or
    // 256 bins, 4 per thread in the first 64 threads
    static_assert(kSelBins == 8 * NT && kSelSup * 8 == NT, "super-bin sums assume 512 threads and 4096 bins");
    // each sum is pushed into every CTA of the cluster (itself included): thread 8 * sbin + j stores super-bin
    // sbin into CTAs j, j + 8, so the boundary search reads all of them locally after the barrier
    if (nb == kSelBins) {
      const int4 u = reinterpret_cast<const int4*>(h)[2 * tid], w = reinterpret_cast<const int4*>(h)[2 * tid + 1];
      int v = u.x + u.y + u.z + u.w + w.x + w.y + w.z + w.w;
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      for (int r = lane & 7; r < C; r += 8)
        cluster.map_shared_rank(&S.sup_all[pass & 1][0][0], r)[crank * kSelSup + (tid >> 3)] = v;
    } else if (tid < kSelSup) {
      const int4 u = reinterpret_cast<const int4*>(h)[tid];
      const int v = u.x + u.y + u.z + u.w;
      for (int r = 0; r < C; ++r) cluster.map_shared_rank(&S.sup_all[pass & 1][0][0], r)[crank * kSelSup + tid] = v;
    }
    cluster.sync();
    // the other buffer (read remotely in the previous pass, finished by every CTA before this barrier) is
    // cleared for the next pass
    if (pass < 2) {
      int4* nh = reinterpret_cast<int4*>(S.hist[(pass + 1) & 1]);
      nh[2 * tid] = make_int4(0, 0, 0, 0);
      nh[2 * tid + 1] = make_int4(0, 0, 0, 0);
    }
    if (warp == 0) {
      const SelResult r = sel_boundary(cluster, C, S.sup_all[pass & 1], h, nb, krem);
      if (lane == 0) S.res = r;
    }
    __syncthreads();
    const SelResult r = S.res;
    prefix = sh == 32 ? r.digit : ((prefix << (sh - shift)) | r.digit);
    sh = shift;
    krem = r.krem;
    bcount = r.count;
    list_mode = pass == 1 && bcount != krem && bcount <= kSelList;
    resolved = bcount == krem || sh == 0 || list_mode;
    __syncthreads();  // S.res is rewritten by the next pass
  }
  griddep_launch_dependents();  // the view kernel may be scheduled while the compaction runs

  // ---- compaction.  A candidate is kept if its bits above sh exceed the boundary prefix, or equal it and
  //      either the whole boundary bin is taken, or (list mode) it ranks among the first krem of the
  //      exchanged boundary list by (key, lower block first), or (sh == 0, equal keys) it is among the first
  //      krem of the cluster's equal keys in block order.  Thread t owns the consecutive slice positions
  //      [t * per, (t + 1) * per), so block order runs across threads, warps and CTAs; the positions of its
  //      kept blocks come from scans of the per-thread counts.
  const bool all_eq = top_k == 0 ? false : bcount == krem;
  const bool tie_mode = !all_eq && !list_mode && top_k > 0;
  // 0 = dropped, 1 = kept, 2 = equal to the boundary key (tie mode), 3 = in the boundary list (list mode)
  auto classify = [&](int b) -> int {
    if (!is_cand(b)) return 1;
    if (top_k == 0) return 0;
    const uint32_t kp = key[b - lo] >> sh;
    if (kp > prefix) return 1;
    if (kp < prefix) return 0;
    return all_eq ? 1 : (list_mode ? 3 : 2);
  };
  const int per = (hi - lo + NT - 1) / NT;
  const int p0 = min(hi, lo + tid * per), p1 = min(hi, p0 + per);
  const bool cache = per <= 16;  // the classes of the thread's positions kept in one register, 2 bits each
  uint32_t cls = 0;
  int keep_t = 0, eq_t = 0;
  for (int b = p0; b < p1; ++b) {
    const int cl = classify(b);
    if (cache) cls |= (uint32_t)cl << (2 * (b - p0));
    keep_t += cl == 1;
    eq_t += cl == 2;
    if (cl == 3) {  // at most kSelList keys over the cluster
      const int i = atomicAdd(&S.own_n, 1);
      if (i < kSelList) S.own_taken[i] = b;  // scratch until the list is ranked
    }
  }
  // inclusive scans over the warp's threads
  int keep_inc = keep_t, eq_inc = eq_t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, keep_inc, o), z = __shfl_up_sync(0xffffffffu, eq_inc, o);
    if (lane >= o) {
      keep_inc += y;
      eq_inc += z;
    }
  }
  if (lane == 31) {
    S.warp_cnt[warp][0] = keep_inc;
    S.warp_cnt[warp][1] = eq_inc;
  }
  __syncthreads();
  if (tid == 0) {
    int kc = 0, ec = 0;
    for (int w2 = 0; w2 < NW; ++w2) {
      kc += S.warp_cnt[w2][0];
      ec += S.warp_cnt[w2][1];
    }
    // pushed into every higher-ranked CTA: after the barrier each CTA reads only its own shared memory, so no
    // CTA needs to wait for another before it exits
    for (int r = crank + 1; r < C; ++r) {
      int* dst = cluster.map_shared_rank(&S.cnts[0][0], r) + 2 * crank;
      dst[0] = kc;
      dst[1] = ec;
    }
  }
  if (list_mode) {
    // this CTA's boundary keys, pushed into every CTA of the cluster (itself included)
    const int n_own = min(S.own_n, kSelList);
    for (int i = tid; i < C * kSelList; i += NT) {
      const int r = i / kSelList, k = i - r * kSelList;
      if (k < n_own) {
        const int b = S.own_taken[k];
        cluster.map_shared_rank(&S.blist[0][0], r)[crank * kSelList + k] = make_uint2(key[b - lo], (uint32_t)b);
      }
      if (k == 0) cluster.map_shared_rank(S.blist_n, r)[crank] = n_own;
    }
  }
  cluster.sync();
  if (list_mode) {
    // rank every listed key by (key descending, block ascending); the first krem are taken
    if (warp == 0) {
      uint2 e = make_uint2(0u, 0xFFFFFFFFu);
      int src = -1, seen = 0;
      for (int r = 0; r < C; ++r) {
        const int n = S.blist_n[r];
        if (lane >= seen && lane < seen + n) {
          e = S.blist[r][lane - seen];
          src = r;
        }
        seen += n;
      }
      S.flat[lane] = e;  // the listed keys in one row, read back as broadcasts
      __syncwarp();
      int rank = 0;
#pragma unroll
      for (int o = 0; o < kSelList; ++o) {
        const uint2 f = S.flat[o];
        rank += (o < seen && (f.x > e.x || (f.x == e.x && f.y < e.y))) ? 1 : 0;
      }
      const bool take = src >= 0 && rank < krem;
      if (take) {
        atomicAdd(&S.taken_cnt[src], 1);
        if (src == crank) {
          const int off = (int)e.y - lo;
          S.own_taken[atomicAdd(&S.own_taken_n, 1)] = (int)e.y;
          atomicAdd(&S.warp_taken[off / per / 32], 1);
          if (per <= 32) atomicOr(&S.tmask[off / per], 1u << (off % per));
        }
      }
    }
    __syncthreads();
  }
  // listed blocks of this thread that are taken (a bit per position where a thread holds at most 32), and the
  // same over the warp's threads before it
  int list_t = 0, list_excl = 0;
  const uint32_t tmask = list_mode && per <= 32 ? S.tmask[tid] : 0u;
  if (list_mode) {
    if (per <= 32) {
      list_t = __popc(tmask);
    } else {
      const int nt = S.own_taken_n;
      for (int i = 0; i < nt; ++i) {
        const int b = S.own_taken[i];
        list_t += (b >= p0 && b < p1) ? 1 : 0;
      }
    }
    int inc = list_t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    list_excl = inc - list_t;
  }
  // blocks kept before this thread (cluster-wide, in block order), and equal keys before it
  int keep_base = 0, eq_base = 0;
  for (int r = 0; r < crank; ++r) {
    const int taken = tie_mode ? max(0, min(S.cnts[r][1], krem - eq_base)) : (list_mode ? S.taken_cnt[r] : 0);
    keep_base += S.cnts[r][0] + taken;
    eq_base += S.cnts[r][1];
  }
  for (int w2 = 0; w2 < warp; ++w2) {
    const int taken =
        tie_mode ? max(0, min(S.warp_cnt[w2][1], krem - eq_base)) : (list_mode ? S.warp_taken[w2] : 0);
    keep_base += S.warp_cnt[w2][0] + taken;
    eq_base += S.warp_cnt[w2][1];
  }
  {
    const int eq_excl = eq_inc - eq_t;
    const int taken = tie_mode ? max(0, min(eq_excl, krem - eq_base)) : list_excl;
    keep_base += keep_inc - keep_t + taken;
    eq_base += eq_excl;
  }
  int pos = keep_base, eq_run = eq_base;
  for (int b = p0; b < p1; ++b) {
    const int cl = cache ? (int)((cls >> (2 * (b - p0))) & 3u) : classify(b);
    bool kp = cl == 1;
    if (cl == 2) kp = eq_run++ < krem;
    if (cl == 3) {
      if (per <= 32) {
        kp = (tmask >> (b - p0)) & 1u;
      } else {
        const int nt = S.own_taken_n;
        for (int i = 0; i < nt; ++i) kp |= S.own_taken[i] == b;
      }
    }
    if (kp) {
      KVM_DEBUG_CHECK(pos < budget, status);
      if (pos < budget) kept_row[pos] = b;  // never past the row, whatever the keys hold
      ++pos;
    }
  }
}

template <int G>
__global__ void __launch_bounds__(kSelectThreads, 1) select_kernel(
    const float* __restrict__ e_buf, int64_t e_stride, const float2* __restrict__ part, int64_t max_tiles,
    int64_t max_blocks, int h_kv, int h_q, SessionArgs a, int rows_per_tile, int n_sink, int n_recent, int top_k,
    int budget, int slice_cap, int32_t* __restrict__ kept, float* __restrict__ group_scores,
    const float* __restrict__ gs_in, uint32_t* __restrict__ status) {
  constexpr int NT = kSelectThreads;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_raw);        // [slice_cap]
  float* coef = reinterpret_cast<float*>(key + slice_cap);       // [tiles in slice][G]
  __shared__ __align__(16) SelShared S;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  sel_init(S);
  cluster_arrive_relaxed();  // paired with the wait before the first store into another CTA's shared memory
  griddep_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int C = (int)cluster.num_blocks();
  const int s = blockIdx.z, g = blockIdx.y;
  const int n_blk = a.n_blk[s];
  const int sl = ((n_blk + C - 1) / C + 3) & ~3;  // slices start on 16-byte boundaries of the exponentials
  const int lo = min(n_blk, crank * sl), hi = min(n_blk, lo + sl);
  const int len = hi - lo;
  const int n_iter = (len + NT - 1) / NT;
  KVM_DEBUG_CHECK(len <= slice_cap && hi <= max_blocks, status);
  int32_t* kept_row = kept + ((int64_t)s * h_kv + g) * budget;
  const bool select_all = n_blk <= budget;  // uniform across the cluster
  const int cand_lo = n_sink, cand_hi = n_blk - n_recent;  // candidates [cand_lo, cand_hi)
  auto is_cand = [&](int b) { return b >= cand_lo && b < cand_hi; };
  float* gs_dst = group_scores ? group_scores + ((int64_t)s * h_kv + g) * max_blocks : nullptr;

  // ---- 1. group scores of the slice as order keys, and the pass-0 histogram of the candidates
  // (plain shared-memory atomics measured faster here than aggregating equal digits within the warp first)
  auto put_key = [&](bool valid, int b, float gsv) {
    const uint32_t k = order_key(gsv);
    if (valid) {
      key[b - lo] = k;
      if (gs_dst && gs_dst != gs_in) gs_dst[b] = gsv;
      if (!select_all && is_cand(b)) atomicAdd(&S.hist[0][k >> 20], 1);
    }
  };
  if (gs_in != nullptr) {
    // group scores given (step-level scoring): keys straight from them
    const float* src = gs_in + ((int64_t)s * h_kv + g) * max_blocks;
    __syncthreads();  // hist[0] cleared
    for (int j = 0; j < n_iter; ++j) {
      const int b = lo + tid + j * NT;
      put_key(b < hi, b, b < hi ? src[b] : 0.f);
    }
  } else {
    // The slice's exponentials (G rows of the head-major scratch, just written by the score kernel and still in
    // L2) go straight into registers, four blocks per 16-byte load; the first kSelPre groups of each thread are
    // requested before the normalisers are formed, so their latency hides behind that step.  Slices start at a
    // multiple of 4 blocks and the scratch rows are padded to a multiple of 4, so every load is aligned and
    // stays inside its row; lanes past the slice's end are masked when the keys are formed.
    const float* e_src = e_buf + ((int64_t)s * h_kv + g) * G * e_stride + lo;
    const int n_tiles = (n_blk + rows_per_tile - 1) / rows_per_tile;
    const int t0 = lo / rows_per_tile;
    const int nt = hi > lo ? (hi - 1) / rows_per_tile - t0 + 1 : 0;
    const int n_grp = (len + 3) >> 2;
    KVM_DEBUG_CHECK(lo + 4 * (int64_t)n_grp <= e_stride, status);
    auto load_group = [&](int q4, float4 (&e4)[G]) {
#pragma unroll
      for (int h = 0; h < G; ++h) e4[h] = __ldcg(reinterpret_cast<const float4*>(e_src + (int64_t)h * e_stride) + q4);
    };
    float4 ev[kSelPre][G];
#pragma unroll
    for (int j = 0; j < kSelPre; ++j)
      if (tid + j * NT < n_grp) load_group(tid + j * NT, ev[j]);
    // softmax normaliser of query head `warp` (< G): M = the largest tile maximum, Z = the tile sums rescaled
    // to M; then the slice's per-tile coefficients exp(m_tile - M) / Z.  Each lane holds its tiles' partials.
    if (warp < G) {
      const float2* p = part + ((int64_t)s * h_q + g * G + warp) * max_tiles;
      float2 pt[kSelTilesPerLane];
#pragma unroll
      for (int i = 0; i < kSelTilesPerLane; ++i) {
        const int t = lane + 32 * i;
        pt[i] = t < n_tiles ? __ldcg(p + t) : make_float2(-INFINITY, 0.f);
      }
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < kSelTilesPerLane; ++i) M = fmaxf(M, pt[i].x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float Z = 0.f;
#pragma unroll
      for (int i = 0; i < kSelTilesPerLane; ++i)
        if (lane + 32 * i < n_tiles) Z += pt[i].y * expf(pt[i].x - M);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
      const float invZ = 1.f / Z;
#pragma unroll
      for (int i = 0; i < kSelTilesPerLane; ++i) {
        const int t = lane + 32 * i;
        if (t >= t0 && t < t0 + nt) coef[(t - t0) * G + warp] = expf(pt[i].x - M) * invZ;
      }
    }
    __syncthreads();  // coefficients ready, hist[0] cleared
    // the four blocks of a group lie in one tile (tiles are multiples of 32 rows, groups start at multiples of 4)
    auto put_group = [&](int q4, const float4 (&e4)[G]) {
      const int b0 = lo + 4 * q4;
      const float* cf = coef + (b0 / rows_per_tile - t0) * G;
      float g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float c = cf[h];
        g0 = fmaf(e4[h].x, c, g0);
        g1 = fmaf(e4[h].y, c, g1);
        g2 = fmaf(e4[h].z, c, g2);
        g3 = fmaf(e4[h].w, c, g3);
      }
      put_key(b0 < hi, b0, g0);
      put_key(b0 + 1 < hi, b0 + 1, g1);
      put_key(b0 + 2 < hi, b0 + 2, g2);
      put_key(b0 + 3 < hi, b0 + 3, g3);
    };
#pragma unroll
    for (int j = 0; j < kSelPre; ++j)
      if (tid + j * NT < n_grp) put_group(tid + j * NT, ev[j]);
    for (int q4 = tid + kSelPre * NT; q4 < n_grp; q4 += NT) {
      float4 e4[G];
      load_group(q4, e4);
      put_group(q4, e4);
    }
  }

  if (select_all) {  // every block is kept
    for (int b = lo + tid; b < hi; b += NT) kept_row[b] = b;
    if (crank == 0)
      for (int i = n_blk + tid; i < budget; i += NT) kept_row[i] = -1;
    cluster_wait();  // completes the start barrier; no distributed shared memory access on this path
    return;
  }
  sel_radix_compact(cluster, S, key, lo, hi, cand_lo, cand_hi, top_k, budget, kept_row, status);
}

template <int G>
cudaError_t launch_select(const Ctx& c, int n_sessions, const SessionArgs& a, int rpt, int max_blk, int32_t* kept,
                          float* group_scores, const float* gs_in, cudaStream_t st, int part_heads = -1) {
  if (part_heads < 0) part_heads = c.p.h_q;  // score rows per session in the tile partials
  // slices of about kSelSlice blocks, as many CTAs as one per SM allows across the call's (session, KV head)
  // units, at most kMaxCluster per unit
  const int units = n_sessions * c.p.h_kv;
  int C = std::min((max_blk + kSelSlice - 1) / kSelSlice, std::max(1, (c.num_sms > 0 ? c.num_sms : 1) / units));
  C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
  if (gs_in == nullptr && (max_blk + rpt - 1) / rpt > 32 * kSelTilesPerLane) return cudaErrorInvalidValue;
  const int slice_cap = ((max_blk + C - 1) / C + 3) & ~3;  // as the kernel's slices: multiples of 4 blocks
  const int tiles_cap = slice_cap / rpt + 2;
  auto kb = select_kernel<G>;
  cudaError_t e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kb)) != cudaSuccess) return e;
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device)) != cudaSuccess) return e;
  const size_t smem_b = (size_t)slice_cap * 4 + (gs_in ? 0 : (size_t)tiles_cap * G * 4);
  if (smem_b + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
  if ((e = ensure_smem(kb, c.device, smem_b)) != cudaSuccess) return e;
  return launch_pdl(kb, dim3(C, c.p.h_kv, n_sessions), dim3(kSelectThreads), smem_b, st, C, (const float*)c.e_buf,
                    c.e_stride, (const float2*)c.part, c.max_tiles, c.p.max_blocks, c.p.h_kv, part_heads, a, rpt,
                    c.p.n_sink, c.p.n_recent, c.p.top_k, c.budget, slice_cap, kept, group_scores, gs_in, c.status);
}

// Rows per score tile (a multiple of 32, 32..4096): whole waves of two CTAs per SM, as many waves as keep tiles
// near 900 rows (one wave for a 1M-token session's 8 heads, two for 8 sessions of 256K tokens), never more
// tiles than fill the waves.
int rows_per_tile(const Ctx& c, int n_sessions, int max_blk) {
  const int64_t units = (int64_t)c.p.h_kv * n_sessions;
  const int64_t slots = 2 * (int64_t)(c.num_sms > 0 ? c.num_sms : 1);
  const int64_t rows = units * max_blk;
  const int64_t waves = std::min<int64_t>(4, std::max<int64_t>(1, (rows + slots * 448) / (slots * 896)));
  const int64_t tiles_per_head = std::max<int64_t>(1, slots * waves / units);
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
                      c.p.max_blocks, c.p.h_kv, c.p.h_kv, a, rpt, c.e_buf, c.e_stride, c.part, c.max_tiles,
                      (float*)nullptr,
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
                      c.p.max_blocks, c.p.h_kv, c.p.h_q, a, rpt, c.e_buf, c.e_stride, c.part, c.max_tiles, head_scores,
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
