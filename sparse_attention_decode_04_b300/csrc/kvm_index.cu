// Step 1 — Mean-K index append.
//
// KVMEM reproduction README, "Core equation" (index vector kbar_b per block);
// Evolve review of KVMem, "Summary" (a position-independent Mean-K index over
// 32-token blocks).  kbar_b is the mean of the block's pre-RoPE keys,
// accumulated in fp32.  A context that scores many query tokens at once
// (max_queries > 1) also gets each written row rounded to bf16 (nearest
// even) in the tensor cores' core-matrix order, the operand layout of the
// step scoring, so that scoring need not convert the whole index each call.
//
// One warp per (session, KV head, block touched by the append).  Lane l owns
// d/32 consecutive dimensions; every load instruction reads one contiguous
// 2*d-byte key row, and all rows of the block are in flight at once.  A partial
// last block is averaged over the tokens present.  Rows are independent, so
// re-running an append over the same tokens rewrites the same values.
#include <type_traits>

#include "kvm_device.cuh"
#include "kvm_internal.h"
#include "kvm_layers.h"

namespace kvm {
namespace {

constexpr int kWarps = 4;

// One warp: the index row of block a.aux[s] + bi of session s, KV head g (and its bf16 copy when shadow is set).
template <int D>
__device__ __forceinline__ void append_block(const uint16_t* __restrict__ k_pool, int64_t n_pages,
                                             const int32_t* __restrict__ bt, int64_t max_blocks, int h_kv,
                                             const SessionArgs& a, float* __restrict__ index,
                                             uint16_t* __restrict__ shadow, int64_t shadow_rows,
                                             uint32_t* __restrict__ status, int s, int g, int64_t bi) {
  constexpr int PER = D / 32;  // dims per lane
  const int lane = threadIdx.x & 31;
  if (bi >= a.count[s]) return;
  const int64_t b = a.aux[s] + bi;                         // block id
  KVM_DEBUG_CHECK(b < max_blocks, status);
  const int64_t present = a.n_tok[s] - b * kBlock;          // tokens of this block present so far
  const int nv = present >= kBlock ? kBlock : (int)present;
  const int32_t page = bt[(int64_t)s * max_blocks + b];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) atomicOr(status, KVM_DEV_BAD_PAGE);
    return;
  }
  const uint16_t* src = k_pool + ((int64_t)page * h_kv + g) * (int64_t)(kBlock * D) + lane * PER;
  // all rows of the block are loaded before any is summed (one memory round trip), then added in token
  // order, so the result does not depend on how the history was split into appends
  using Vec = typename std::conditional<PER == 4, uint2, uint32_t>::type;
  Vec w[kBlock];
#pragma unroll
  for (int t = 0; t < kBlock; ++t) {
    if (t < nv) {
      w[t] = __ldg(reinterpret_cast<const Vec*>(src + t * D));
    } else {
      if constexpr (PER == 4) w[t] = make_uint2(0u, 0u); else w[t] = 0u;
    }
  }
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
  for (int t = 0; t < kBlock; ++t) {
    if (t < nv) {
      if constexpr (PER == 4) {
        acc[0] += bf16lo(w[t].x);
        acc[1] += bf16hi(w[t].x);
        acc[2] += bf16lo(w[t].y);
        acc[3] += bf16hi(w[t].y);
      } else {
        acc[0] += bf16lo(w[t]);
        acc[1] += bf16hi(w[t]);
      }
    }
  }
  float* dst = index + (((int64_t)s * h_kv + g) * max_blocks + b) * D + lane * PER;
  const float n = (float)nv;  // 32 for full blocks: the division is then exact
  float m[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) m[i] = acc[i] / n;
  if constexpr (PER == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(m[0], m[1], m[2], m[3]);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(m[0], m[1]);
  }
  if (shadow) {
    // element (b, c) at ((b / 8) * (D / 8) + c / 8) * 64 + (b % 8) * 8 + c % 8 of this head's rows
    const int c = lane * PER;
    uint16_t* sdst = shadow + ((int64_t)s * h_kv + g) * shadow_rows * D + ((b >> 3) * (D / 8) + (c >> 3)) * 64 +
                     (b & 7) * 8 + (c & 7);
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(sdst) = make_uint2(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]));
    } else {
      *reinterpret_cast<uint32_t*>(sdst) = pack_bf16x2(m[0], m[1]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) index_append_kernel(const uint16_t* __restrict__ k_pool,
                                                                   int64_t n_pages,
                                                                   const int32_t* __restrict__ bt,
                                                                   int64_t max_blocks, int h_kv, SessionArgs a,
                                                                   float* __restrict__ index,
                                                                   uint16_t* __restrict__ shadow,
                                                                   int64_t shadow_rows, uint32_t* __restrict__ status) {
  griddep_wait();
  append_block<D>(k_pool, n_pages, bt, max_blocks, h_kv, a, index, shadow, shadow_rows, status, blockIdx.z,
                  blockIdx.y, (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5));
}

// The same appends for several layers in one launch: grid z runs over (layer, session), layer-major.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) index_append_layers_kernel(const AppendLayers layers, int n_sessions,
                                                                          int64_t n_pages,
                                                                          const int32_t* __restrict__ bt,
                                                                          int64_t max_blocks, int h_kv, SessionArgs a,
                                                                          uint32_t* __restrict__ status) {
  griddep_wait();
  const int layer = blockIdx.z / n_sessions, s = blockIdx.z % n_sessions;
  append_block<D>(layers.k_pool[layer], n_pages, bt, max_blocks, h_kv, a, layers.index[layer], nullptr, 0, status,
                  s, blockIdx.y, (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5));
}

}  // namespace

cudaError_t launch_index_append_layers(const Ctx& c, const AppendLayers& layers, int n_layers, int64_t n_pages,
                                       const int32_t* bt, int n_sessions, const SessionArgs& a, int max_count,
                                       cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  dim3 grid((max_count + kWarps - 1) / kWarps, c.p.h_kv, n_layers * n_sessions);
  return c.p.d == 128 ? launch_pdl(index_append_layers_kernel<128>, grid, dim3(kWarps * 32), 0, st, 1, layers,
                                    n_sessions, n_pages, bt, c.p.max_blocks, c.p.h_kv, a, c.status)
                       : launch_pdl(index_append_layers_kernel<64>, grid, dim3(kWarps * 32), 0, st, 1, layers,
                                    n_sessions, n_pages, bt, c.p.max_blocks, c.p.h_kv, a, c.status);
}

cudaError_t launch_index_append(const Ctx& c, const uint16_t* k_pool, int64_t n_pages, const int32_t* bt,
                                int n_sessions, const SessionArgs& a, int max_count, float* index, uint16_t* shadow,
                                cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  dim3 grid((max_count + kWarps - 1) / kWarps, c.p.h_kv, n_sessions);
  return c.p.d == 128 ? launch_pdl(index_append_kernel<128>, grid, dim3(kWarps * 32), 0, st, 1, k_pool, n_pages, bt,
                                    c.p.max_blocks, c.p.h_kv, a, index, shadow, c.step_blk_cap_pad, c.status)
                       : launch_pdl(index_append_kernel<64>, grid, dim3(kWarps * 32), 0, st, 1, k_pool, n_pages, bt,
                                    c.p.max_blocks, c.p.h_kv, a, index, shadow, c.step_blk_cap_pad, c.status);
}

}  // namespace kvm
