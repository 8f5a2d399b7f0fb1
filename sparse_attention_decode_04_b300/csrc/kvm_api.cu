// C ABI of the KVMem decode hot path: context, validation, launches.
// Every entry point checks its arguments on the host before anything is
// enqueued; the kernels only ever see sizes the checks accepted.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <new>
#include <utility>

#include "kvm.h"
#include "kvm_batch.h"
#include "kvm_diag.h"
#include "kvm_internal.h"
#include "kvm_layers.h"
#include "kvm_mass.h"

using kvm::Ctx;
using kvm::SessionArgs;

struct kvm_ctx {
  Ctx c;
};

namespace {

thread_local char g_err[512] = "";

kvm_status fail(kvm_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

kvm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Largest block capacity the cluster select keeps in shared memory (8 CTAs,
// 40960 fp32 keys each).
constexpr int64_t kMaxBlocksLimit = 8 * 40960;

kvm_status check_ctx(const kvm_ctx* ctx) {
  if (!ctx) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != ctx->c.device)
    return fail(KVM_ERR_INVALID_ARG, "current device %d is not the context's device %d", dev, ctx->c.device);
  return KVM_OK;
}

kvm_status check_sessions(const Ctx& c, int32_t n_sessions) {
  if (n_sessions < 0 || n_sessions > c.p.max_sessions)
    return fail(KVM_ERR_SHAPE, "n_sessions=%d outside [0, %d]", n_sessions, c.p.max_sessions);
  return KVM_OK;
}

// Fills n_tok / n_blk / n_keep / seg_base from host history lengths.
kvm_status history_args(const Ctx& c, const int64_t* n_tok, int32_t n_sessions, SessionArgs* a) {
  memset(a, 0, sizeof(*a));
  if (n_sessions > 0 && !n_tok) return fail(KVM_ERR_INVALID_ARG, "n_tok is NULL");
  int64_t base = 0;
  for (int s = 0; s < n_sessions; ++s) {
    if (n_tok[s] < 0) return fail(KVM_ERR_INVALID_ARG, "n_tok[%d]=%lld is negative", s, (long long)n_tok[s]);
    const int64_t nb = (n_tok[s] + kvm::kBlock - 1) / kvm::kBlock;
    if (nb > c.p.max_blocks)
      return fail(KVM_ERR_SHAPE, "session %d: %lld blocks exceed max_blocks=%lld", s, (long long)nb,
                  (long long)c.p.max_blocks);
    a->n_tok[s] = n_tok[s];
    a->n_blk[s] = (int32_t)nb;
    a->n_keep[s] = (int32_t)(nb < c.budget ? nb : c.budget);
    a->seg_base[s] = base;
    base += (int64_t)c.p.h_kv * a->n_keep[s];
  }
  a->seg_base[n_sessions] = base;
  return KVM_OK;
}

// First block and block count of each session's append, from host token ranges.
kvm_status append_args(const Ctx& c, int32_t n_sessions, const int64_t* tok_begin, const int64_t* n_tok,
                       SessionArgs* a, int* max_count) {
  memset(a, 0, sizeof(*a));
  *max_count = 0;
  for (int i = 0; i < n_sessions; ++i) {
    if (tok_begin[i] < 0 || n_tok[i] < 0)
      return fail(KVM_ERR_INVALID_ARG, "session %d: negative tok_begin or n_tok", i);
    const int64_t end = tok_begin[i] + n_tok[i];
    if ((end + kvm::kBlock - 1) / kvm::kBlock > c.p.max_blocks)
      return fail(KVM_ERR_SHAPE, "session %d: token %lld beyond max_blocks", i, (long long)end);
    const int64_t b0 = tok_begin[i] / kvm::kBlock;
    const int64_t b1 = n_tok[i] ? (end + kvm::kBlock - 1) / kvm::kBlock : b0;
    a->n_tok[i] = end;  // tokens present after the append
    a->aux[i] = b0;     // first block touched
    a->count[i] = (int32_t)(b1 - b0);
    if (a->count[i] > *max_count) *max_count = a->count[i];
  }
  return KVM_OK;
}

}  // namespace

void kvm::set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

cudaError_t kvm::ensure_smem_impl(const void* kernel, int device, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> limit;
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = limit[{kernel, device}];
  if (cur >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

extern "C" {

int32_t kvm_debug_checks(void) {
#ifdef KVM_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

const char* kvm_status_string(kvm_status s) {
  switch (s) {
    case KVM_OK: return "KVM_OK";
    case KVM_ERR_INVALID_ARG: return "KVM_ERR_INVALID_ARG";
    case KVM_ERR_SHAPE: return "KVM_ERR_SHAPE";
    case KVM_ERR_BUDGET: return "KVM_ERR_BUDGET";
    case KVM_ERR_CUDA: return "KVM_ERR_CUDA";
    case KVM_ERR_TIMEOUT: return "KVM_ERR_TIMEOUT";
    case KVM_ERR_DEVICE: return "KVM_ERR_DEVICE";
  }
  return "KVM_ERR_UNKNOWN";
}

const char* kvm_last_error(void) { return g_err; }

kvm_status kvm_create(const kvm_params* p, kvm_ctx** out) {
  if (!p || !out) return fail(KVM_ERR_INVALID_ARG, "params or out is NULL");
  *out = nullptr;
  if (p->d != 64 && p->d != 128) return fail(KVM_ERR_SHAPE, "d=%d: only 64 and 128 are built", p->d);
  if (p->h_q <= 0 || p->h_kv <= 0 || p->h_q % p->h_kv != 0)
    return fail(KVM_ERR_SHAPE, "h_q=%d must be a positive multiple of h_kv=%d", p->h_q, p->h_kv);
  if (p->h_q / p->h_kv > kvm::kMaxGroup)
    return fail(KVM_ERR_SHAPE, "GQA group %d exceeds %d", p->h_q / p->h_kv, kvm::kMaxGroup);
  if (p->n_sink < 0 || p->n_recent < 0 || p->top_k < 0)
    return fail(KVM_ERR_BUDGET, "n_sink, n_recent and top_k must be >= 0");
  const int64_t budget = (int64_t)p->n_sink + p->n_recent + p->top_k;
  if (budget < 1 || budget > (1 << 20)) return fail(KVM_ERR_BUDGET, "budget %lld outside [1, 2^20]", (long long)budget);
  if (!(p->rope_theta > 1.0f)) return fail(KVM_ERR_INVALID_ARG, "rope_theta must be > 1");
  if (p->max_blocks < 1 || p->max_blocks > kMaxBlocksLimit)
    return fail(KVM_ERR_SHAPE, "max_blocks=%lld outside [1, %lld]", (long long)p->max_blocks,
                (long long)kMaxBlocksLimit);
  if (p->max_sessions < 1 || p->max_sessions > kvm::kMaxSessionsHost)
    return fail(KVM_ERR_SHAPE, "max_sessions=%d outside [1, %d]", p->max_sessions, kvm::kMaxSessionsHost);
  if (p->max_queries < 1) return fail(KVM_ERR_SHAPE, "max_queries must be >= 1");
  if ((int64_t)p->max_queries * (p->h_q / (p->h_kv > 0 ? p->h_kv : 1)) > 8192)
    return fail(KVM_ERR_SHAPE, "max_queries * group must be <= 8192");

  kvm_ctx* ctx = new (std::nothrow) kvm_ctx();
  if (!ctx) return fail(KVM_ERR_CUDA, "host allocation failed");
  Ctx& c = ctx->c;
  c.p = *p;
  c.group = p->h_q / p->h_kv;
  c.budget = (int)budget;
  cudaError_t e = cudaGetDevice(&c.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, c.device);
  if (e != cudaSuccess) {
    delete ctx;
    return cuda_fail(e, "device query");
  }
  c.view_ctas = c.num_sms;
  c.max_tiles = (p->max_blocks + 31) / 32;
  const size_t S = (size_t)p->max_sessions;
  c.e_stride = (p->max_blocks + 3) & ~(int64_t)3;
  const size_t sz_e = S * p->h_kv * (size_t)c.e_stride * c.group * sizeof(float);
  const size_t sz_part = S * p->h_q * (size_t)c.max_tiles * sizeof(float2);
  const size_t sz_rec =
      ((size_t)c.view_ctas + S * p->h_kv) * (kvm::kViewWarps + 1) * c.group * (4 + p->d) * sizeof(float);
  const size_t sz_cnt = S * p->h_kv * sizeof(uint32_t);
  // base rows cover view slots and, for the attention-mass diagnostic, every history block position
  const size_t sz_base = (size_t)((budget > p->max_blocks ? budget : p->max_blocks) + 1) * (p->d / 2) * sizeof(float2);
  const size_t sz_off = (size_t)32 * (p->d / 2) * sizeof(float2);
  constexpr int kBufs = 9;
  void* ptrs[kBufs] = {};
  const size_t sizes[kBufs] = {sz_e, sz_part, sz_rec, sz_base, sz_off, 256, sz_base, sz_off, sz_cnt};
  for (int i = 0; i < kBufs && e == cudaSuccess; ++i) e = cudaMalloc(&ptrs[i], sizes[i]);
  if (e != cudaSuccess) {
    for (void* q : ptrs)
      if (q) cudaFree(q);
    delete ctx;
    return cuda_fail(e, "cudaMalloc of context scratch");
  }
  c.e_buf = (float*)ptrs[0];
  c.part = (float2*)ptrs[1];
  c.rec = (float*)ptrs[2];
  c.rope_base = (float*)ptrs[3];
  c.rope_off = (float*)ptrs[4];
  c.status = (uint32_t*)ptrs[5];
  c.rope_base_lo = (float*)ptrs[6];
  c.rope_off_lo = (float*)ptrs[7];
  c.seg_count = (uint32_t*)ptrs[8];
  for (size_t s : sizes) c.bytes += s;
  if (p->max_queries > 1) {
    c.step_blk_cap_pad = (p->max_blocks + 255) / 256 * 256;
    c.step_rows_cap_pad = (int)(((int64_t)p->max_queries * c.group + 255) / 256 * 256);
    const size_t SG = S * p->h_kv;
    c.attn_units_cap = 8 * c.num_sms;
    const size_t sz[8] = {SG * c.step_blk_cap_pad * p->d * 2,
                          SG * c.step_rows_cap_pad * p->d * 2,
                          SG * kvm::kStepMaxRanges * c.step_rows_cap_pad * sizeof(float2),
                          SG * c.step_rows_cap_pad * sizeof(float2),
                          SG * p->max_blocks * sizeof(float),
                          2 * SG * c.step_rows_cap_pad * p->d * 2,
                          (size_t)c.attn_units_cap * 128 * (p->d + 2) * sizeof(float),
                          (size_t)c.attn_units_cap * sizeof(uint32_t)};
    void* q5[8] = {};
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaMalloc(&q5[i], sz[i]);
    c.step_kpk = (uint16_t*)q5[0];
    c.step_qpk = (uint16_t*)q5[1];
    c.step_part = (float2*)q5[2];
    c.step_stats = (float2*)q5[3];
    c.step_gs = (float*)q5[4];
    c.attn_q = (uint16_t*)q5[5];
    c.attn_part = (float*)q5[6];
    c.attn_cnt = (uint32_t*)q5[7];
    if (e == cudaSuccess) e = cudaMemset(c.attn_cnt, 0, sz[7]);
    if (e == cudaSuccess) e = cudaMemset(c.step_kpk, 0, sz[0]);  // rows no append wrote read as zeros
    for (size_t b : sz) c.bytes += b;
    if (e != cudaSuccess) {
      kvm_destroy(ctx);
      return cuda_fail(e, "cudaMalloc of step-scoring scratch");
    }
  }
  e = cudaMemset(c.status, 0, 256);
  if (e == cudaSuccess) e = cudaMemset(c.seg_count, 0, sz_cnt);
  if (e == cudaSuccess) e = kvm::launch_rope_tables(c, 0);
  if (e == cudaSuccess) e = kvm::launch_mass_tables(c, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    kvm_destroy(ctx);
    return cuda_fail(e, "context initialisation");
  }
  *out = ctx;
  return KVM_OK;
}

kvm_status kvm_destroy(kvm_ctx* ctx) {
  if (!ctx) return KVM_OK;
  Ctx& c = ctx->c;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != c.device) cudaSetDevice(c.device);
  cudaError_t e = cudaDeviceSynchronize();
  void* ptrs[17] = {c.e_buf,       c.part,     c.rec,       c.rope_base,  c.rope_off, c.status,
                    c.rope_base_lo, c.rope_off_lo, c.step_kpk, c.step_qpk, c.step_part, c.step_stats,
                    c.step_gs,      c.seg_count, c.attn_q,   c.attn_part, c.attn_cnt};
  for (void* q : ptrs)
    if (q) cudaFree(q);
  if (prev >= 0 && prev != c.device) cudaSetDevice(prev);
  delete ctx;
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_destroy");
}

size_t kvm_scratch_bytes(const kvm_ctx* ctx) { return ctx ? ctx->c.bytes : 0; }

kvm_status kvm_set_wait_limit(kvm_ctx* ctx, int64_t wait_ns, int32_t stall_first_wait) {
  if (!ctx) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
  if (wait_ns < 1000 || wait_ns > 2000000000ll)
    return fail(KVM_ERR_INVALID_ARG, "wait_ns=%lld outside [1000, 2e9]", (long long)wait_ns);
  if (stall_first_wait != 0 && stall_first_wait != 1)
    return fail(KVM_ERR_INVALID_ARG, "stall_first_wait must be 0 or 1");
  ctx->c.wait_ns = (uint64_t)wait_ns;
  ctx->c.stall_first_wait = stall_first_wait;
  return KVM_OK;
}

kvm_status kvm_index_append(kvm_ctx* ctx, const uint16_t* k_pool, int64_t n_pages, const int32_t* block_table,
                            int32_t n_sessions, const int64_t* tok_begin, const int64_t* n_tok, float* index,
                            void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!k_pool || !block_table || !tok_begin || !n_tok || !index)
    return fail(KVM_ERR_INVALID_ARG, "kvm_index_append: NULL pointer argument");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(k_pool, 16) || !aligned(index, 16))
    return fail(KVM_ERR_INVALID_ARG, "k_pool and index must be 16-byte aligned");
  SessionArgs a;
  int max_count = 0;
  if ((s = append_args(c, n_sessions, tok_begin, n_tok, &a, &max_count)) != KVM_OK) return s;
  // the bf16 copy (contexts that score many queries at once): it follows one index; an append to another index
  // restarts it, and a session's copy counts as complete up to the last block of a run of appends from block 0
  Ctx& cm = ctx->c;
  uint16_t* shadow = cm.step_kpk;
  if (shadow) {
    if (cm.shadow_of != index) {
      cm.shadow_of = index;
      for (int64_t& nb : cm.shadow_blocks) nb = 0;
    }
    for (int i = 0; i < n_sessions; ++i) {
      const int64_t b0 = tok_begin[i] / kvm::kBlock, b1 = (tok_begin[i] + n_tok[i] + kvm::kBlock - 1) / kvm::kBlock;
      if (n_tok[i] > 0 && b0 <= cm.shadow_blocks[i] && b1 > cm.shadow_blocks[i]) cm.shadow_blocks[i] = b1;
    }
  }
  cudaError_t e = kvm::launch_index_append(c, k_pool, n_pages, block_table, n_sessions, a, max_count, index, shadow,
                                           (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_index_append launch");
}

kvm_status kvm_index_append_layers(kvm_ctx* ctx, int32_t n_layers, const uint16_t* const* k_pools,
                                   int64_t n_pages, const int32_t* block_table, int32_t n_sessions,
                                   const int64_t* tok_begin, const int64_t* n_tok, float* const* indexes,
                                   void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_layers < 1 || n_layers > kvm::kMaxAppendLayers)
    return fail(KVM_ERR_INVALID_ARG, "n_layers=%d must be in [1, %d]", n_layers, kvm::kMaxAppendLayers);
  if (!k_pools || !indexes || !block_table || !tok_begin || !n_tok)
    return fail(KVM_ERR_INVALID_ARG, "kvm_index_append_layers: NULL pointer argument");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  kvm::AppendLayers layers;
  memset(&layers, 0, sizeof(layers));
  for (int i = 0; i < n_layers; ++i) {
    if (!k_pools[i] || !indexes[i])
      return fail(KVM_ERR_INVALID_ARG, "kvm_index_append_layers: layer %d has a NULL pointer", i);
    if (!aligned(k_pools[i], 16) || !aligned(indexes[i], 16))
      return fail(KVM_ERR_INVALID_ARG, "layer %d: k_pool and index must be 16-byte aligned", i);
    layers.k_pool[i] = k_pools[i];
    layers.index[i] = indexes[i];
  }
  if (n_sessions == 0) return KVM_OK;
  SessionArgs a;
  int max_count = 0;
  if ((s = append_args(c, n_sessions, tok_begin, n_tok, &a, &max_count)) != KVM_OK) return s;
  // the bf16 copy follows single-layer appends only: an index it mirrors is about to change without it
  Ctx& cm = ctx->c;
  for (int i = 0; i < n_layers; ++i)
    if (cm.step_kpk && indexes[i] == cm.shadow_of) {
      cm.shadow_of = nullptr;
      for (int64_t& nb : cm.shadow_blocks) nb = 0;
    }
  cudaError_t e = kvm::launch_index_append_layers(c, layers, n_layers, n_pages, block_table, n_sessions, a,
                                                  max_count, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_index_append_layers launch");
}

kvm_status kvm_index_append_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales, int64_t n_pages,
                                const int32_t* block_table, int32_t n_sessions, const int64_t* tok_begin,
                                const int64_t* n_tok, float* index, void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!k_pool8 || !k_scales || !block_table || !tok_begin || !n_tok || !index)
    return fail(KVM_ERR_INVALID_ARG, "kvm_index_append_fp8: NULL pointer argument");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(k_pool8, 16) || !aligned(index, 16) || !aligned(k_scales, 4))
    return fail(KVM_ERR_INVALID_ARG, "k_pool8 and index must be 16-byte aligned, k_scales 4-byte aligned");
  SessionArgs a;
  int max_count = 0;
  if ((s = append_args(c, n_sessions, tok_begin, n_tok, &a, &max_count)) != KVM_OK) return s;
  if (ctx->c.shadow_of == index) ctx->c.shadow_of = nullptr;  // the bf16 copy does not follow this append
  cudaError_t e = kvm::launch_index_append_q(c, k_pool8, k_scales, n_pages, block_table, n_sessions, a, max_count,
                                             index, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_index_append_fp8 launch");
}

kvm_status kvm_quantize_pages(kvm_ctx* ctx, const uint16_t* pool, int64_t n_pages, const int32_t* pages,
                              int64_t n_list, uint8_t* pool8, float* scales, void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if (n_list < 0) return fail(KVM_ERR_INVALID_ARG, "n_list=%lld is negative", (long long)n_list);
  if (n_list == 0) return KVM_OK;
  if (!pool || !pages || !pool8 || !scales) return fail(KVM_ERR_INVALID_ARG, "kvm_quantize_pages: NULL pointer");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(pool, 16) || !aligned(pool8, 16) || !aligned(pages, 4) || !aligned(scales, 4))
    return fail(KVM_ERR_INVALID_ARG, "pool and pool8 must be 16-byte aligned, pages and scales 4-byte aligned");
  cudaError_t e = kvm::launch_quantize_pages(c, pool, n_pages, pages, n_list, pool8, scales, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_quantize_pages launch");
}

static kvm_status gather_call(kvm_ctx* ctx, bool fp8, const void* k_src, const void* v_src, const float* k_scales,
                              const float* v_scales, int64_t n_pages, const int32_t* block_table,
                              const int64_t* n_tok, int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view,
                              uint16_t* v_view, int32_t* view_len, void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!k_src || !v_src || !block_table || !kept_ids || !k_view || !v_view || !view_len ||
      (fp8 && (!k_scales || !v_scales)))
    return fail(KVM_ERR_INVALID_ARG, "NULL pool, scales, block_table, kept_ids or view output");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(k_view, 16) || !aligned(v_view, 16) ||
      !aligned(view_len, 4) || !aligned(kept_ids, 4) || !aligned(k_scales, 4) || !aligned(v_scales, 4))
    return fail(KVM_ERR_INVALID_ARG, "pools and views must be 16-byte aligned");
  SessionArgs a;
  if ((s = history_args(c, n_tok, n_sessions, &a)) != KVM_OK) return s;
  cudaError_t e = kvm::launch_gather_view(c, fp8, k_src, v_src, k_scales, v_scales, n_pages, block_table, n_sessions,
                                          a, kept_ids, k_view, v_view, view_len, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "gather kernel launch");
}

kvm_status kvm_materialize_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales, const uint8_t* v_pool8,
                               const float* v_scales, int64_t n_pages, const int32_t* block_table,
                               const int64_t* n_tok, int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view,
                               uint16_t* v_view, int32_t* view_len, void* stream) {
  return gather_call(ctx, true, k_pool8, v_pool8, k_scales, v_scales, n_pages, block_table, n_tok, n_sessions,
                     kept_ids, k_view, v_view, view_len, stream);
}

kvm_status kvm_materialize_host(kvm_ctx* ctx, const uint16_t* k_pool_host, const uint16_t* v_pool_host,
                                int64_t n_pages, const int32_t* block_table, const int64_t* n_tok,
                                int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view, uint16_t* v_view,
                                int32_t* view_len, void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  // the pools must be pinned host memory mapped into the device address space; the kernel reads them through
  // their device-side address
  const void* dev[2] = {nullptr, nullptr};
  const uint16_t* host[2] = {k_pool_host, v_pool_host};
  for (int i = 0; i < 2; ++i) {
    if (!host[i]) return fail(KVM_ERR_INVALID_ARG, "kvm_materialize_host: NULL pool");
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, host[i]);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
      cudaGetLastError();
      return fail(KVM_ERR_INVALID_ARG, "kvm_materialize_host: %s pool is not mapped pinned host memory",
                  i ? "V" : "K");
    }
    dev[i] = attr.devicePointer;
  }
  return gather_call(ctx, false, dev[0], dev[1], nullptr, nullptr, n_pages, block_table, n_tok, n_sessions, kept_ids,
                     k_view, v_view, view_len, stream);
}

kvm_status kvm_score_select(kvm_ctx* ctx, const uint16_t* q, int32_t n_q, const float* index, const int64_t* n_tok,
                            int32_t n_sessions, int32_t* kept_ids, float* group_scores, float* head_scores,
                            void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!q || !index || !kept_ids) return fail(KVM_ERR_INVALID_ARG, "kvm_score_select: NULL pointer argument");
  if (n_q < 1 || n_q > c.p.max_queries)
    return fail(KVM_ERR_SHAPE, "n_q=%d outside [1, max_queries=%d]", n_q, c.p.max_queries);
  if (n_q > 1 && head_scores) return fail(KVM_ERR_INVALID_ARG, "head_scores is only written for n_q == 1");
  if (n_q > 1 && !ctx->c.step_kpk)
    return fail(KVM_ERR_SHAPE, "n_q > 1 needs a context created with max_queries > 1");
  if (!aligned(q, 16) || !aligned(index, 16) || !aligned(kept_ids, 4) || !aligned(group_scores, 4) ||
      !aligned(head_scores, 4))
    return fail(KVM_ERR_INVALID_ARG, "q and index must be 16-byte aligned, outputs 4-byte aligned");
  SessionArgs a;
  if ((s = history_args(c, n_tok, n_sessions, &a)) != KVM_OK) return s;
  const bool converts = n_q > 1 && !kvm::shadow_ready(c, index, n_sessions, a);
  cudaError_t e = kvm::launch_score_select(c, q, n_q, index, n_sessions, a, kept_ids, group_scores, head_scores,
                                           (cudaStream_t)stream);
  if (converts) ctx->c.shadow_of = nullptr;  // the conversion overwrote the appends' bf16 copy
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_score_select launch");
}

kvm_status kvm_select_control(kvm_ctx* ctx, int32_t control, const uint16_t* q, const float* index,
                              const int64_t* n_tok, int32_t n_sessions, int32_t* kept_ids, float* group_scores,
                              void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if (control != KVM_CONTROL_RECENT_ONLY && control != KVM_CONTROL_WITHDRAWN_AVERAGE)
    return fail(KVM_ERR_INVALID_ARG, "unknown selection control %d", control);
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!kept_ids) return fail(KVM_ERR_INVALID_ARG, "kvm_select_control: kept_ids is NULL");
  if (control == KVM_CONTROL_WITHDRAWN_AVERAGE) {
    if (!q || !index) return fail(KVM_ERR_INVALID_ARG, "kvm_select_control: NULL q or index");
    if (!aligned(q, 16) || !aligned(index, 16) || !aligned(group_scores, 4))
      return fail(KVM_ERR_INVALID_ARG, "q and index must be 16-byte aligned, outputs 4-byte aligned");
  }
  if (!aligned(kept_ids, 4)) return fail(KVM_ERR_INVALID_ARG, "kept_ids must be 4-byte aligned");
  SessionArgs a;
  if ((s = history_args(c, n_tok, n_sessions, &a)) != KVM_OK) return s;
  cudaError_t e = kvm::launch_select_control(c, control, q, index, n_sessions, a, kept_ids,
                                             control == KVM_CONTROL_WITHDRAWN_AVERAGE ? group_scores : nullptr,
                                             (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_select_control launch");
}

static kvm_status view_call(kvm_ctx* ctx, int mode, const uint16_t* k_src, const uint16_t* v_src, int64_t n_pages,
                            const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions,
                            const int32_t* kept_ids, const uint16_t* q, uint16_t* k_view, uint16_t* v_view,
                            int32_t* view_len, float* out, void* stream, const float* k_scales = nullptr,
                            const float* v_scales = nullptr) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!k_src || !v_src || !view_len) return fail(KVM_ERR_INVALID_ARG, "NULL K/V source or view_len");
  if (mode != 1 && (!block_table || !kept_ids || !k_view || !v_view))
    return fail(KVM_ERR_INVALID_ARG, "NULL block_table, kept_ids or view output");
  if (mode != 0 && (!q || !out)) return fail(KVM_ERR_INVALID_ARG, "NULL q or out");
  if (mode != 1 && n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(k_view, 16) || !aligned(v_view, 16) ||
      !aligned(q, 16) || !aligned(out, 16) || !aligned(view_len, 4) || !aligned(kept_ids, 4))
    return fail(KVM_ERR_INVALID_ARG, "K/V/q/out buffers must be 16-byte aligned");
  if (mode == 3 && (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4)))
    return fail(KVM_ERR_INVALID_ARG, "FP8 pages need 4-byte aligned K and V scale arrays");
  SessionArgs a;
  if (mode == 1) {
    // the view lengths live on the device: walk every slot of each view, skip the empty ones
    memset(&a, 0, sizeof(a));
    int64_t base = 0;
    for (int i = 0; i < n_sessions; ++i) {
      a.n_keep[i] = c.budget;
      a.n_blk[i] = c.budget;
      a.n_tok[i] = (int64_t)c.budget * kvm::kBlock;
      a.seg_base[i] = base;
      base += (int64_t)c.p.h_kv * c.budget;
    }
    a.seg_base[n_sessions] = base;
  } else if ((s = history_args(c, n_tok, n_sessions, &a)) != KVM_OK) {
    return s;
  }
  cudaError_t e = kvm::launch_view(c, mode, k_src, v_src, n_pages, block_table, n_sessions, a, kept_ids, q, k_view,
                                   v_view, view_len, out, (cudaStream_t)stream, k_scales, v_scales);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "view kernel launch");
}

kvm_status kvm_materialize_attn_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales, const uint8_t* v_pool8,
                                    const float* v_scales, int64_t n_pages, const int32_t* block_table,
                                    const int64_t* n_tok, int32_t n_sessions, const int32_t* kept_ids,
                                    const uint16_t* q, uint16_t* k_view, uint16_t* v_view, int32_t* view_len,
                                    float* out, void* stream) {
  return view_call(ctx, 3, reinterpret_cast<const uint16_t*>(k_pool8), reinterpret_cast<const uint16_t*>(v_pool8),
                   n_pages, block_table, n_tok, n_sessions, kept_ids, q, k_view, v_view, view_len, out, stream,
                   k_scales, v_scales);
}

kvm_status kvm_materialize(kvm_ctx* ctx, const uint16_t* k_pool, const uint16_t* v_pool, int64_t n_pages,
                           const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions,
                           const int32_t* kept_ids, uint16_t* k_view, uint16_t* v_view, int32_t* view_len,
                           void* stream) {
  return view_call(ctx, 0, k_pool, v_pool, n_pages, block_table, n_tok, n_sessions, kept_ids, nullptr, k_view,
                   v_view, view_len, nullptr, stream);
}

kvm_status kvm_decode_attn(kvm_ctx* ctx, const uint16_t* q, const uint16_t* k_view, const uint16_t* v_view,
                           const int32_t* view_len, int32_t n_sessions, float* out, void* stream) {
  return view_call(ctx, 1, k_view, v_view, 0, nullptr, nullptr, n_sessions, nullptr, q, nullptr, nullptr,
                   const_cast<int32_t*>(view_len), out, stream);
}

kvm_status kvm_materialize_attn(kvm_ctx* ctx, const uint16_t* k_pool, const uint16_t* v_pool, int64_t n_pages,
                                const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions,
                                const int32_t* kept_ids, const uint16_t* q, uint16_t* k_view, uint16_t* v_view,
                                int32_t* view_len, float* out, void* stream) {
  return view_call(ctx, 2, k_pool, v_pool, n_pages, block_table, n_tok, n_sessions, kept_ids, q, k_view, v_view,
                   view_len, out, stream);
}

kvm_status kvm_step_attn(kvm_ctx* ctx, const uint16_t* q, int32_t n_q, const uint16_t* k_view,
                         const uint16_t* v_view, const int32_t* view_len, int32_t n_sessions, float* out,
                         void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!q || !k_view || !v_view || !view_len || !out)
    return fail(KVM_ERR_INVALID_ARG, "kvm_step_attn: NULL pointer argument");
  if (n_q < 1 || n_q > c.p.max_queries)
    return fail(KVM_ERR_SHAPE, "n_q=%d outside [1, max_queries=%d]", n_q, c.p.max_queries);
  if (!c.attn_q) return fail(KVM_ERR_SHAPE, "kvm_step_attn needs a context created with max_queries > 1");
  if ((int64_t)n_q > (int64_t)kvm::kBlock * c.budget)
    return fail(KVM_ERR_SHAPE, "n_q=%d exceeds the view capacity %d", n_q, kvm::kBlock * c.budget);
  if (!aligned(q, 16) || !aligned(k_view, 16) || !aligned(v_view, 16) || !aligned(out, 16) || !aligned(view_len, 4))
    return fail(KVM_ERR_INVALID_ARG, "q, k_view, v_view and out must be 16-byte aligned");
  cudaError_t e = kvm::launch_step_attn(c, q, n_q, k_view, v_view, view_len, n_sessions, out, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_step_attn launch");
}

kvm_status kvm_attention_mass(kvm_ctx* ctx, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages,
                              const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions, float* mass,
                              void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  const Ctx& c = ctx->c;
  if ((s = check_sessions(c, n_sessions)) != KVM_OK) return s;
  if (n_sessions == 0) return KVM_OK;
  if (!q || !k_pool || !block_table || !mass) return fail(KVM_ERR_INVALID_ARG, "kvm_attention_mass: NULL pointer");
  if (n_pages < 1) return fail(KVM_ERR_INVALID_ARG, "n_pages=%lld must be >= 1", (long long)n_pages);
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(mass, 4) || !aligned(block_table, 4))
    return fail(KVM_ERR_INVALID_ARG, "q and k_pool must be 16-byte aligned, mass and block_table 4-byte aligned");
  SessionArgs a;
  if ((s = history_args(c, n_tok, n_sessions, &a)) != KVM_OK) return s;
  // the finalising kernel stages one fp32 factor per (32-block tile, query head of the group) in shared memory
  int max_blk = 0, optin = 0;
  for (int i = 0; i < n_sessions; ++i) max_blk = a.n_blk[i] > max_blk ? a.n_blk[i] : max_blk;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
  if (e != cudaSuccess) return cuda_fail(e, "kvm_attention_mass");
  const size_t fac_bytes = (size_t)((max_blk + 31) / 32) * c.group * sizeof(float);
  if (fac_bytes > (size_t)optin)
    return fail(KVM_ERR_SHAPE,
                "kvm_attention_mass: %d blocks x group %d need %zu bytes of per-tile factors in shared memory; "
                "the device allows %d (at most %lld blocks for this group)",
                max_blk, c.group, fac_bytes, optin, (long long)optin / (long long)(c.group * sizeof(float)) * 32);
  e = kvm::launch_attention_mass(c, q, k_pool, n_pages, block_table, n_sessions, a, mass, (cudaStream_t)stream);
  return e == cudaSuccess ? KVM_OK : cuda_fail(e, "kvm_attention_mass launch");
}

kvm_status kvm_device_status(kvm_ctx* ctx, uint32_t* out, int32_t clear, void* stream) {
  kvm_status s = check_ctx(ctx);
  if (s != KVM_OK) return s;
  if (!out) return fail(KVM_ERR_INVALID_ARG, "out is NULL");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemcpy(out, ctx->c.status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(ctx->c.status, 0, sizeof(uint32_t));
  // a stopped view kernel may have left segment arrival counters behind: clearing restarts them
  if (e == cudaSuccess && clear && *out != 0)
    e = cudaMemset(ctx->c.seg_count, 0, sizeof(uint32_t) * ctx->c.p.max_sessions * ctx->c.p.h_kv);
  if (e == cudaSuccess && clear && *out != 0 && ctx->c.attn_cnt)
    e = cudaMemset(ctx->c.attn_cnt, 0, sizeof(uint32_t) * ctx->c.attn_units_cap);
  if (e != cudaSuccess) return cuda_fail(e, "kvm_device_status");
  if (*out == 0) return KVM_OK;
  if (*out & KVM_DEV_TIMEOUT) return fail(KVM_ERR_TIMEOUT, "a device-side wait timed out (status 0x%x)", *out);
  return fail(KVM_ERR_DEVICE, "device status 0x%x (bad page, block id or view length)", *out);
}

}  // extern "C"
