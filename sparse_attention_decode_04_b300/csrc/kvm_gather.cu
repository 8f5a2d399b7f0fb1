// Page tiers beyond the bf16 HBM pool: FP8 E4M3 pages (quantised KV) and
// pages resident in pinned host memory.
//
// KVMEM reproduction README, "Background and main changes": overflowed
// history is kept as paged KV across GPU memory, host memory and NVMe, and the
// deployment runs in NVFP4.  The pages fix no precision for the paged KV; the
// quantised variant here stores FP8 E4M3 codes with one fp32 scale per
// (page, KV head), for K and for V (value = code * scale).
//
//   quantize_pages   bf16 pages -> codes + scales: scale = amax / 448 (fp32),
//                    code = E4M3(x / scale), nearest even, saturating.
//   index_append_q   Mean-K index over the dequantised keys (fp32, token order).
//   gather_view      kept blocks -> K / V view, re-RoPE'd keys at view
//                    positions, for a bf16 source anywhere in the address space
//                    (HBM, or mapped pinned host memory read over the link) or
//                    an FP8 source dequantised on the fly.
//
// gather_view: one warp per (session, KV head, kept slot).  A lane takes one
// token row and one pair of 8-element chunks (elements i and i + d/2 rotate
// together), so each load and store instruction of the warp covers whole
// 128-byte (bf16) or 64-byte (fp8) row segments.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr int kGatherWarps = 4;

// ---------------------------------------------------------------- quantisation
// One warp per (listed page, KV head); lane = token row.
template <int D>
__global__ void __launch_bounds__(128) quantize_pages_kernel(const uint16_t* __restrict__ pool, int64_t n_pages,
                                                             const int32_t* __restrict__ pages, int64_t n_list,
                                                             int h_kv, uint8_t* __restrict__ pool8,
                                                             float* __restrict__ scales, uint32_t* __restrict__ status) {
  griddep_wait();
  const int64_t item = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= n_list * h_kv) return;
  const int64_t li = item / h_kv;
  const int g = (int)(item % h_kv);
  const int32_t page = pages[li];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) atomicOr(status, KVM_DEV_BAD_PAGE);
    return;
  }
  const int64_t base = ((int64_t)page * h_kv + g) * 32 + lane;  // this lane's row
  const uint4* src = reinterpret_cast<const uint4*>(pool + base * D);
  uint4 w[D / 8];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    w[c] = __ldg(src + c);
    const uint32_t u[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(u[k])), fabsf(bf16hi(u[k]))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint4* dst = reinterpret_cast<uint4*>(pool8 + base * D);
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {  // 16 codes per store
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 a = w[2 * c + (k >> 1)];
      const uint32_t u0 = (k & 1) ? a.z : a.x, u1 = (k & 1) ? a.w : a.y;
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(bf16lo(u0), scale), __fdiv_rn(bf16hi(u0), scale)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(bf16lo(u1), scale), __fdiv_rn(bf16hi(u1), scale)), __NV_SATFINITE, __NV_E4M3);
      q[k] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    dst[c] = make_uint4(q[0], q[1], q[2], q[3]);
  }
  if (lane == 0) scales[(int64_t)page * h_kv + g] = scale;
}

// Two E4M3 codes (low byte first) -> their exact values times `scale` (one fp32 rounding each).
__device__ __forceinline__ float2 dequant2(uint32_t codes16, float scale) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(codes16 & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return make_float2(f.x * scale, f.y * scale);
}

// ---------------------------------------------------------------- Mean-K index over quantised keys
// One warp per (session, KV head, block touched by the append); lane l owns d/32 consecutive dimensions.
template <int D>
__global__ void __launch_bounds__(128) index_append_q_kernel(const uint8_t* __restrict__ k8,
                                                             const float* __restrict__ kscale, int64_t n_pages,
                                                             const int32_t* __restrict__ bt, int64_t max_blocks,
                                                             int h_kv, SessionArgs a, float* __restrict__ index,
                                                             uint32_t* __restrict__ status) {
  constexpr int PER = D / 32;  // codes per lane: 4 (d 128) or 2 (d 64)
  griddep_wait();
  const int s = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bi = (int64_t)blockIdx.x * 4 + warp;
  if (bi >= a.count[s]) return;
  const int64_t b = a.aux[s] + bi;
  const int64_t present = a.n_tok[s] - b * kBlock;
  const int nv = present >= kBlock ? kBlock : (int)present;
  const int32_t page = bt[(int64_t)s * max_blocks + b];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) atomicOr(status, KVM_DEV_BAD_PAGE);
    return;
  }
  const float scale = __ldg(kscale + (int64_t)page * h_kv + g);
  const uint8_t* src = k8 + ((int64_t)page * h_kv + g) * (int64_t)(kBlock * D) + lane * PER;
  uint32_t w[kBlock];
#pragma unroll
  for (int t = 0; t < kBlock; ++t) {
    if (t < nv) {
      if constexpr (PER == 4) w[t] = __ldg(reinterpret_cast<const uint32_t*>(src + t * D));
      else w[t] = __ldg(reinterpret_cast<const uint16_t*>(src + t * D));
    } else {
      w[t] = 0u;
    }
  }
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
  for (int t = 0; t < kBlock; ++t) {
    if (t < nv) {
      const float2 v0 = dequant2(w[t], scale);
      acc[0] += v0.x;
      acc[1] += v0.y;
      if constexpr (PER == 4) {
        const float2 v1 = dequant2(w[t] >> 16, scale);
        acc[2] += v1.x;
        acc[3] += v1.y;
      }
    }
  }
  float* dst = index + (((int64_t)s * h_kv + g) * max_blocks + b) * D + lane * PER;
  const float n = (float)nv;
  if constexpr (PER == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] / n, acc[1] / n, acc[2] / n, acc[3] / n);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0] / n, acc[1] / n);
  }
}

// ---------------------------------------------------------------- view gather
struct GatherArgs {
  const void* k_src;        // bf16 [n_pages][h_kv][32][d], or E4M3 codes of the same shape
  const void* v_src;
  const float* k_scale;     // [n_pages][h_kv] (E4M3 source only)
  const float* v_scale;
  int64_t n_pages;
  const int32_t* bt;        // [S][max_blocks]
  int64_t max_blocks;
  const int32_t* kept;      // [S][h_kv][budget]
  uint16_t* k_view;         // [S][h_kv][32 * budget][d]
  uint16_t* v_view;
  int32_t* view_len;        // [S][h_kv]
  const float2* rope_base;  // [budget + 1][d/2] cos/sin of 32 * slot * theta_i (hi and lo parts)
  const float2* rope_base_lo;
  const float2* rope_off;   // [32][d/2] cos/sin of r * theta_i
  const float2* rope_off_lo;
  int h_kv, budget;
  uint32_t* status;
};

// Eight elements of one token row starting at element e0: bf16 bits or codes -> fp32 values.
template <int D, bool Q8>
__device__ __forceinline__ void load8(const void* src, int64_t row, int e0, float scale, float (&x)[8],
                                      uint4& raw) {
  if constexpr (Q8) {
    const uint2 c = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(src) + row * D + e0);
    const uint32_t u[2] = {c.x, c.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 a = dequant2(u[k], scale), b = dequant2(u[k] >> 16, scale);
      x[4 * k] = a.x;
      x[4 * k + 1] = a.y;
      x[4 * k + 2] = b.x;
      x[4 * k + 3] = b.y;
    }
    raw = make_uint4(0, 0, 0, 0);
  } else {
    raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(src) + row * D + e0);
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = bf16lo(u[k]);
      x[2 * k + 1] = bf16hi(u[k]);
    }
  }
}

template <int D, bool Q8>
__global__ void __launch_bounds__(kGatherWarps * 32) gather_view_kernel(const GatherArgs ga, const SessionArgs a) {
  constexpr int CP = D / 16;      // chunk pairs per row (8 elements each, paired with the chunk d/2 further)
  constexpr int RPI = 32 / CP;    // rows per warp iteration
  griddep_wait();
  const int s = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = blockIdx.x * kGatherWarps + warp;
  const int sg = s * ga.h_kv + g;
  const int n_keep = a.n_keep[s];
  const int32_t* kept = ga.kept + (int64_t)sg * ga.budget;
  if (slot == 0 && lane == 0) {
    // view length: every kept block is full except the history's last block when it is partial
    int L = kBlock * n_keep;
    const int rem = (int)(a.n_tok[s] % kBlock);
    if (n_keep > 0 && rem != 0 && kept[n_keep - 1] == a.n_blk[s] - 1) L -= kBlock - rem;
    ga.view_len[sg] = L;
  }
  if (slot >= n_keep) return;
  const int32_t b = kept[slot];
  if (b < 0 || b >= a.n_blk[s] || (slot > 0 && kept[slot - 1] >= b)) {
    if (lane == 0) atomicOr(ga.status, KVM_DEV_BAD_BLOCK);
    return;
  }
  const int32_t page = ga.bt[(int64_t)s * ga.max_blocks + b];
  if (page < 0 || page >= ga.n_pages) {
    if (lane == 0) atomicOr(ga.status, KVM_DEV_BAD_PAGE);
    return;
  }
  const int64_t rem_tok = a.n_tok[s] - (int64_t)b * kBlock;
  const int valid = rem_tok >= kBlock ? kBlock : (int)rem_tok;
  const int64_t prow = ((int64_t)page * ga.h_kv + g) * kBlock;  // first source row of this page and head
  const float ks = Q8 ? __ldg(ga.k_scale + (int64_t)page * ga.h_kv + g) : 1.f;
  const float vs = Q8 ? __ldg(ga.v_scale + (int64_t)page * ga.h_kv + g) : 1.f;
  const int cp = lane % CP, rsub = lane / CP;
  const int e1 = 8 * cp, e2 = D / 2 + 8 * cp;  // this lane's element chunks
  // the base angle of every row of this slot (position 32 * slot + r) and this lane's 8 pairs
  float2 bh[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) bh[e] = __ldg(ga.rope_base + (int64_t)slot * (D / 2) + e1 + e);
  uint16_t* kv = ga.k_view + ((int64_t)sg * kBlock * ga.budget + (int64_t)slot * kBlock) * D;
  uint16_t* vv = ga.v_view + ((int64_t)sg * kBlock * ga.budget + (int64_t)slot * kBlock) * D;
#pragma unroll 2
  for (int it = 0; it < kBlock / RPI; ++it) {
    const int r = it * RPI + rsub;
    if (r >= valid) continue;
    float x1[8], x2[8], y1[8], y2[8];
    uint4 raw1, raw2;
    load8<D, Q8>(ga.k_src, prow + r, e1, ks, x1, raw1);
    load8<D, Q8>(ga.k_src, prow + r, e2, ks, x2, raw2);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 o = __ldg(ga.rope_off + r * (D / 2) + e1 + e);
      float cs, sn;
      rope_cs(bh[e], o.x, o.y, cs, sn);
      y1[e] = fmaf(x1[e], cs, -x2[e] * sn);
      y2[e] = fmaf(x2[e], cs, x1[e] * sn);
      // a rotation that cancels is redone in float-float from the hi/lo tables (within one bf16 ulp)
      if (fminf(fabsf(y1[e]), fabsf(y2[e])) < 0x1p-13f * (fabsf(x1[e]) + fabsf(x2[e]))) {
        const float2 bl = __ldg(ga.rope_base_lo + (int64_t)slot * (D / 2) + e1 + e);
        const float2 ol = __ldg(ga.rope_off_lo + r * (D / 2) + e1 + e);
        rotate_exact(x1[e], x2[e], make_float4(bh[e].x, bl.x, bh[e].y, bl.y), make_float4(o.x, ol.x, o.y, ol.y),
                     y1[e], y2[e]);
      }
    }
    uint4 k1, k2;
    k1.x = pack_bf16x2(y1[0], y1[1]);
    k1.y = pack_bf16x2(y1[2], y1[3]);
    k1.z = pack_bf16x2(y1[4], y1[5]);
    k1.w = pack_bf16x2(y1[6], y1[7]);
    k2.x = pack_bf16x2(y2[0], y2[1]);
    k2.y = pack_bf16x2(y2[2], y2[3]);
    k2.z = pack_bf16x2(y2[4], y2[5]);
    k2.w = pack_bf16x2(y2[6], y2[7]);
    *reinterpret_cast<uint4*>(kv + (int64_t)r * D + e1) = k1;
    *reinterpret_cast<uint4*>(kv + (int64_t)r * D + e2) = k2;
    uint4 v1, v2;
    if constexpr (Q8) {
      float z1[8], z2[8];
      load8<D, Q8>(ga.v_src, prow + r, e1, vs, z1, v1);
      load8<D, Q8>(ga.v_src, prow + r, e2, vs, z2, v2);
      v1 = make_uint4(pack_bf16x2(z1[0], z1[1]), pack_bf16x2(z1[2], z1[3]), pack_bf16x2(z1[4], z1[5]),
                      pack_bf16x2(z1[6], z1[7]));
      v2 = make_uint4(pack_bf16x2(z2[0], z2[1]), pack_bf16x2(z2[2], z2[3]), pack_bf16x2(z2[4], z2[5]),
                      pack_bf16x2(z2[6], z2[7]));
    } else {  // bit copy
      v1 = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(ga.v_src) + (prow + r) * D + e1);
      v2 = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(ga.v_src) + (prow + r) * D + e2);
    }
    *reinterpret_cast<uint4*>(vv + (int64_t)r * D + e1) = v1;
    *reinterpret_cast<uint4*>(vv + (int64_t)r * D + e2) = v2;
  }
}

}  // namespace

cudaError_t launch_quantize_pages(const Ctx& c, const uint16_t* pool, int64_t n_pages, const int32_t* pages,
                                  int64_t n_list, uint8_t* pool8, float* scales, cudaStream_t st) {
  if (n_list <= 0) return cudaSuccess;
  const int64_t items = n_list * c.p.h_kv;
  const dim3 grid((unsigned)((items + 3) / 4));
  return c.p.d == 128 ? launch_pdl(quantize_pages_kernel<128>, grid, dim3(128), 0, st, 1, pool, n_pages, pages, n_list,
                                   c.p.h_kv, pool8, scales, c.status)
                      : launch_pdl(quantize_pages_kernel<64>, grid, dim3(128), 0, st, 1, pool, n_pages, pages, n_list,
                                   c.p.h_kv, pool8, scales, c.status);
}

cudaError_t launch_index_append_q(const Ctx& c, const uint8_t* k8, const float* kscale, int64_t n_pages,
                                  const int32_t* bt, int n_sessions, const SessionArgs& a, int max_count,
                                  float* index, cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  const dim3 grid((max_count + 3) / 4, c.p.h_kv, n_sessions);
  return c.p.d == 128 ? launch_pdl(index_append_q_kernel<128>, grid, dim3(128), 0, st, 1, k8, kscale, n_pages, bt,
                                   c.p.max_blocks, c.p.h_kv, a, index, c.status)
                      : launch_pdl(index_append_q_kernel<64>, grid, dim3(128), 0, st, 1, k8, kscale, n_pages, bt,
                                   c.p.max_blocks, c.p.h_kv, a, index, c.status);
}

cudaError_t launch_gather_view(const Ctx& c, bool fp8, const void* k_src, const void* v_src, const float* k_scale,
                               const float* v_scale, int64_t n_pages, const int32_t* bt, int n_sessions,
                               const SessionArgs& a, const int32_t* kept, uint16_t* k_view, uint16_t* v_view,
                               int32_t* view_len, cudaStream_t st) {
  GatherArgs ga;
  ga.k_src = k_src;
  ga.v_src = v_src;
  ga.k_scale = k_scale;
  ga.v_scale = v_scale;
  ga.n_pages = n_pages;
  ga.bt = bt;
  ga.max_blocks = c.p.max_blocks;
  ga.kept = kept;
  ga.k_view = k_view;
  ga.v_view = v_view;
  ga.view_len = view_len;
  ga.rope_base = reinterpret_cast<const float2*>(c.rope_base);
  ga.rope_base_lo = reinterpret_cast<const float2*>(c.rope_base_lo);
  ga.rope_off = reinterpret_cast<const float2*>(c.rope_off);
  ga.rope_off_lo = reinterpret_cast<const float2*>(c.rope_off_lo);
  ga.h_kv = c.p.h_kv;
  ga.budget = c.budget;
  ga.status = c.status;
  int max_keep = 1;  // at least one warp per head writes the view length
  for (int s = 0; s < n_sessions; ++s) max_keep = max(max_keep, a.n_keep[s]);
  const dim3 grid((max_keep + kGatherWarps - 1) / kGatherWarps, c.p.h_kv, n_sessions);
  const dim3 block(kGatherWarps * 32);
  if (c.p.d == 128)
    return fp8 ? launch_pdl(gather_view_kernel<128, true>, grid, block, 0, st, 1, ga, a)
               : launch_pdl(gather_view_kernel<128, false>, grid, block, 0, st, 1, ga, a);
  return fp8 ? launch_pdl(gather_view_kernel<64, true>, grid, block, 0, st, 1, ga, a)
             : launch_pdl(gather_view_kernel<64, false>, grid, block, 0, st, 1, ga, a);
}

}  // namespace kvm
