// Attention-mass diagnostic: how much of each query head's full attention falls in each history block.
//
// KVMEM reproduction README, "Background and main changes": a few blocks hold most of the attention (the top
// 8 of about 103 blocks held 66.5% of it).  For one decode query per session, with the query at position
// N = n_tok and each key at its history position t:
//   mass[g][b] = sum_{h in g} sum_{t in b} softmax_t(<RoPE(q_h, N), RoPE(k_t, t)>/sqrt(d))
// Rotary attention depends on N - t only, so each score is <RoPE(q_h, N - t), k_t> with the pre-RoPE key;
// cos/sin of (N - t) theta_i come from the context's fp64-filled tables of 32 a theta_i and r theta_i,
// composed in fp32.
//
//   mass_tile_kernel      one CTA per 32 blocks (1024 tokens) of a (session, KV head): a warp walks its
//                         blocks token by token, each lane holding two rotation pairs of the query heads
//                         and of the key (coalesced 4-byte loads), the dot products reduced across the warp;
//                         per tile: the maximum score m and e[b][h] = sum_{t in b} 2^(s - m) per head.
//   mass_finalize_kernel  one CTA per (session, KV head): per head the global maximum and normaliser from
//                         the tile partials, then mass[b] = sum_h e[b][h] 2^(m_tile - M_h) / Z_h.
// The tile partials use the scoring scratch of the context (same layouts as the single-query scoring).
#include "kvm_device.cuh"
#include "kvm_mass.h"

namespace kvm {
namespace {

constexpr int kMassWarps = 8;
constexpr int kTileBlocks = 32;  // blocks per tile (the scratch's tile size)

__global__ void mass_table_kernel(float2* base, float2* base_lo, int row0, int row1, int d, double rope_theta) {
  const int half = d / 2;
  const int64_t n = (int64_t)(row1 - row0) * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = row0 + idx / half;
    const int i = (int)(idx % half);
    double sn, cs;
    sincos(32.0 * (double)row * pow(rope_theta, -2.0 * i / d), &sn, &cs);
    const float ch = (float)cs, sh = (float)sn;
    base[row * half + i] = make_float2(ch, sh);
    base_lo[row * half + i] = make_float2((float)(cs - (double)ch), (float)(sn - (double)sh));
  }
}

// grid (tiles of 32 blocks, h_kv, S); lane l owns rotation pairs (2l, 2l + d/2) and (2l + 1, 2l + 1 + d/2)
// (d = 128) or (l, l + d/2) (d = 64).
template <int D, int G>
__global__ void __launch_bounds__(kMassWarps * 32) mass_tile_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k_pool, int64_t n_pages,
    const int32_t* __restrict__ bt, int64_t max_blocks, int h_kv, int h_q, SessionArgs a,
    const float2* __restrict__ rope_base, const float2* __restrict__ rope_off, float q_scale,
    float* __restrict__ e_buf, float2* __restrict__ part, int64_t max_tiles, uint32_t* __restrict__ status) {
  constexpr int PL = D / 64;  // rotation pairs per lane
  griddep_wait();
  const int s = blockIdx.z, g = blockIdx.y, tile = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blk = a.n_blk[s];
  const int64_t N = a.n_tok[s];
  const int b0 = tile * kTileBlocks;
  if (b0 >= n_blk) return;
  __shared__ float2 blk_ms[kTileBlocks][G];  // per block and head: (block max, sum of 2^(s - block max))
  __shared__ float tile_m[G];

  // this lane's query pairs, pre-scaled to the log2 domain
  float q1[G][PL], q2[G][PL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint16_t* qh = q + ((int64_t)s * h_q + g * G + h) * D;
#pragma unroll
    for (int p = 0; p < PL; ++p) {
      const int i = PL * lane + p;
      q1[h][p] = __uint_as_float((uint32_t)qh[i] << 16) * q_scale;
      q2[h][p] = __uint_as_float((uint32_t)qh[i + D / 2] << 16) * q_scale;
    }
  }
  for (int bi = warp; bi < kTileBlocks; bi += kMassWarps) {
    const int b = b0 + bi;
    float sc[G];  // lane t: token t's scores
#pragma unroll
    for (int h = 0; h < G; ++h) sc[h] = -INFINITY;
    if (b < n_blk) {
      const int32_t page = bt[(int64_t)s * max_blocks + b];
      if (page < 0 || page >= n_pages) {
        if (lane == 0) atomicOr(status, KVM_DEV_BAD_PAGE);
      } else {
        const uint16_t* kb = k_pool + ((int64_t)page * h_kv + g) * (int64_t)(kBlock * D);
        const int64_t rem = N - (int64_t)b * kBlock;
        const int nv = rem >= kBlock ? kBlock : (int)rem;
        for (int t = 0; t < nv; ++t) {
          const int64_t delta = N - ((int64_t)b * kBlock + t);  // >= 1
          float k1[PL], k2[PL];
          if constexpr (PL == 2) {
            const uint32_t w1 = __ldg(reinterpret_cast<const uint32_t*>(kb + t * D + 2 * lane));
            const uint32_t w2 = __ldg(reinterpret_cast<const uint32_t*>(kb + t * D + D / 2 + 2 * lane));
            k1[0] = bf16lo(w1);
            k1[1] = bf16hi(w1);
            k2[0] = bf16lo(w2);
            k2[1] = bf16hi(w2);
          } else {
            k1[0] = __uint_as_float((uint32_t)__ldg(kb + t * D + lane) << 16);
            k2[0] = __uint_as_float((uint32_t)__ldg(kb + t * D + D / 2 + lane) << 16);
          }
          float part_h[G];
#pragma unroll
          for (int h = 0; h < G; ++h) part_h[h] = 0.f;
#pragma unroll
          for (int p = 0; p < PL; ++p) {
            const int i = PL * lane + p;
            const float2 bb = __ldg(rope_base + (delta >> 5) * (D / 2) + i);
            const float2 oo = __ldg(rope_off + (delta & 31) * (D / 2) + i);
            float cs, sn;
            rope_cs(bb, oo.x, oo.y, cs, sn);
            const float dd = k1[p] * cs + k2[p] * sn;  // <R(delta) q, k> = q1 (k1 c + k2 s) + q2 (k2 c - k1 s)
            const float ee = k2[p] * cs - k1[p] * sn;
#pragma unroll
            for (int h = 0; h < G; ++h) part_h[h] = fmaf(q1[h][p], dd, fmaf(q2[h][p], ee, part_h[h]));
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) part_h[h] += __shfl_xor_sync(0xffffffffu, part_h[h], o);
            if (lane == t) sc[h] = part_h[h];
          }
        }
      }
    }
    // block maximum and sum per head (lanes past the block's tokens hold -inf)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float m = sc[h];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float e = m == -INFINITY ? 0.f : fast_exp2(sc[h] - m);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      if (lane == 0) blk_ms[bi][h] = make_float2(m, e);
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY;
    for (int bi = 0; bi < kTileBlocks; ++bi) m = fmaxf(m, blk_ms[bi][threadIdx.x].x);
    tile_m[threadIdx.x] = m;
  }
  __syncthreads();
  // e[b][h] relative to the tile maximum; the tile's (max, sum) per head
  if (threadIdx.x < kTileBlocks * G) {
    const int bi = threadIdx.x / G, h = threadIdx.x % G, b = b0 + bi;
    const float2 ms = blk_ms[bi][h];
    const float e = ms.x == -INFINITY ? 0.f : ms.y * fast_exp2(ms.x - tile_m[h]);
    if (b < n_blk) e_buf[(((int64_t)s * h_kv + g) * max_blocks + b) * G + h] = e;
    blk_ms[bi][h].y = e;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float z = 0.f;
    for (int bi = 0; bi < kTileBlocks; ++bi) z += blk_ms[bi][threadIdx.x].y;
    part[((int64_t)s * h_q + g * G + threadIdx.x) * max_tiles + tile] = make_float2(tile_m[threadIdx.x], z);
  }
}

// grid (h_kv, S), 1024 threads; dynamic shared memory: [n_tiles][G] factors.
template <int G>
__global__ void __launch_bounds__(1024) mass_finalize_kernel(const float* __restrict__ e_buf,
                                                             const float2* __restrict__ part, int64_t max_tiles,
                                                             int64_t max_blocks, int h_kv, int h_q, SessionArgs a,
                                                             float* __restrict__ mass) {
  griddep_wait();
  extern __shared__ float fac[];  // [n_tiles][G]: 2^(m_tile - M_h) / Z_h
  __shared__ float red[32];
  __shared__ float s_M, s_Z;
  const int g = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_blk = a.n_blk[s];
  const int n_tiles = (n_blk + kTileBlocks - 1) / kTileBlocks;
  for (int h = 0; h < G; ++h) {
    const float2* p = part + ((int64_t)s * h_q + g * G + h) * max_tiles;
    float m = -INFINITY;
    for (int t = tid; t < n_tiles; t += blockDim.x) m = fmaxf(m, p[t].x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      float v = lane < (int)(blockDim.x >> 5) ? red[lane] : -INFINITY;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) s_M = v;
    }
    __syncthreads();
    const float M = s_M;
    float z = 0.f;
    for (int t = tid; t < n_tiles; t += blockDim.x) z += p[t].x == -INFINITY ? 0.f : p[t].y * exp2f(p[t].x - M);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    __syncthreads();
    if (lane == 0) red[warp] = z;
    __syncthreads();
    if (warp == 0) {
      float v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_Z = v;
    }
    __syncthreads();
    const float inv = s_Z > 0.f ? 1.f / s_Z : 0.f;
    for (int t = tid; t < n_tiles; t += blockDim.x)
      fac[t * G + h] = p[t].x == -INFINITY ? 0.f : exp2f(p[t].x - M) * inv;
    __syncthreads();
  }
  const float* e = e_buf + ((int64_t)s * h_kv + g) * max_blocks * G;
  for (int b = tid; b < n_blk; b += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) acc = fmaf(e[(int64_t)b * G + h], fac[(b / kTileBlocks) * G + h], acc);
    mass[((int64_t)s * h_kv + g) * max_blocks + b] = acc;
  }
}

template <int D, int G>
cudaError_t launch_dg(const Ctx& c, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages, const int32_t* bt,
                      int n_sessions, const SessionArgs& a, float* mass, cudaStream_t st) {
  int max_blk = 0;
  for (int s = 0; s < n_sessions; ++s) max_blk = max(max_blk, a.n_blk[s]);
  if (max_blk == 0) return cudaSuccess;
  const int tiles = (max_blk + kTileBlocks - 1) / kTileBlocks;
  cudaError_t e = launch_pdl(mass_tile_kernel<D, G>, dim3(tiles, c.p.h_kv, n_sessions), dim3(kMassWarps * 32), 0,
                             st, 1, q, k_pool, n_pages, bt, c.p.max_blocks, c.p.h_kv, c.p.h_q, a,
                             reinterpret_cast<const float2*>(c.rope_base), reinterpret_cast<const float2*>(c.rope_off),
                             (float)(1.4426950408889634 / sqrt((double)D)), c.e_buf, c.part, c.max_tiles, c.status);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)tiles * G * sizeof(float);
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device)) != cudaSuccess) return e;
  if (smem > (size_t)optin) return cudaErrorInvalidConfiguration;  // the caller checks this bound up front
  if ((e = ensure_smem(mass_finalize_kernel<G>, c.device, smem)) != cudaSuccess) return e;
  return launch_pdl(mass_finalize_kernel<G>, dim3(c.p.h_kv, n_sessions), dim3(1024), smem, st, 1,
                    (const float*)c.e_buf, (const float2*)c.part, c.max_tiles, c.p.max_blocks, c.p.h_kv, c.p.h_q, a,
                    mass);
}

template <int D>
cudaError_t launch_d(const Ctx& c, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages, const int32_t* bt,
                     int n_sessions, const SessionArgs& a, float* mass, cudaStream_t st) {
  switch (c.group) {
    case 1: return launch_dg<D, 1>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 2: return launch_dg<D, 2>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 3: return launch_dg<D, 3>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 4: return launch_dg<D, 4>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 5: return launch_dg<D, 5>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 6: return launch_dg<D, 6>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 7: return launch_dg<D, 7>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
    case 8: return launch_dg<D, 8>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_mass_tables(const Ctx& c, cudaStream_t st) {
  const int row0 = c.budget + 1, row1 = (int)(c.p.max_blocks + 1);
  if (row1 <= row0) return cudaSuccess;
  mass_table_kernel<<<256, 256, 0, st>>>(reinterpret_cast<float2*>(c.rope_base),
                                         reinterpret_cast<float2*>(c.rope_base_lo), row0, row1, c.p.d,
                                         (double)c.p.rope_theta);
  return cudaGetLastError();
}

cudaError_t launch_attention_mass(const Ctx& c, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages,
                                  const int32_t* bt, int n_sessions, const SessionArgs& a, float* mass,
                                  cudaStream_t st) {
  return c.p.d == 128 ? launch_d<128>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st)
                      : launch_d<64>(c, q, k_pool, n_pages, bt, n_sessions, a, mass, st);
}

}  // namespace kvm
