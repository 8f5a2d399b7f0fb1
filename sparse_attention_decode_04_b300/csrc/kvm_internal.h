// Internal interface between the C-ABI layer (kvm_api.cu) and the kernel
// files: the context object and the per-step launch functions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvm.h"

namespace kvm {

constexpr int kBlock = 32;            // tokens per block / page
constexpr int kMaxGroup = 8;          // query heads per KV head
constexpr int kMaxSessionsHost = 64;  // sessions per call (kernel-parameter arrays)
constexpr int kViewWarps = 2;         // attention warps (attention-record slots) per view-kernel CTA

// Per-session values passed by value to the kernels (they size the grids, so
// they live on the host; passing them as kernel parameters keeps every call
// capturable in a CUDA graph).
struct SessionArgs {
  int64_t n_tok[kMaxSessionsHost];   // history tokens
  int64_t aux[kMaxSessionsHost];     // call-specific (first block of an append, ...)
  int32_t n_blk[kMaxSessionsHost];   // ceil(n_tok / 32)
  int32_t n_keep[kMaxSessionsHost];  // kept blocks per KV head
  int32_t count[kMaxSessionsHost];   // call-specific (blocks touched by an append, ...)
  int64_t seg_base[kMaxSessionsHost + 1];  // flat offset of session s's first kept block over all heads
};

struct Ctx {
  kvm_params p;
  int device = 0;
  int num_sms = 0;
  int group = 1;        // h_q / h_kv
  int budget = 0;       // n_sink + n_recent + top_k
  int view_ctas = 0;    // persistent CTAs of the view kernels
  size_t bytes = 0;     // device bytes allocated
  // scratch (device)
  float* e_buf = nullptr;      // [S][h_kv][group][e_stride] exp(s - tile max) (score kernels)
  int64_t e_stride = 0;        // max_blocks rounded up to a multiple of 4 (16-byte rows for bulk copies)
  float2* part = nullptr;      // [S][h_q][max_tiles] (tile max, tile sum) in log2 domain
  float* rec = nullptr;        // [view_ctas + S*h_kv][kViewWarps + 1][group][4 + d] attention partials
  uint32_t* seg_count = nullptr;  // [S*h_kv] CTAs of a view call done with each segment (0 between calls)
  float* rope_base = nullptr;  // [budget + 1][d/2][2] cos/sin of 32*slot*theta_i
  float* rope_off = nullptr;   // [32][d/2][2] cos/sin of r*theta_i
  float* rope_base_lo = nullptr;  // [budget + 1][d/2][2] what the fp32 rounding of rope_base dropped
  float* rope_off_lo = nullptr;   // [32][d/2][2] the same for rope_off (read on the cancellation fallback)
  uint32_t* status = nullptr;  // device status word
  uint64_t wait_ns = 2000000000ull;  // wall-clock limit of the view kernel's pipeline waits
  int stall_first_wait = 0;          // the view kernel's first rotation wait is on a barrier nothing completes
  int64_t max_tiles = 0;
  // step-level (multi-query) scoring scratch, allocated when max_queries > 1
  int64_t step_blk_cap_pad = 0;  // max_blocks rounded up to 256
  int step_rows_cap_pad = 0;     // max_queries * group rounded up to 256
  uint16_t* step_kpk = nullptr;  // packed bf16 index [S*h_kv][step_blk_cap_pad][d] (core-matrix order): the
                                 // bf16 copy that kvm_index_append keeps of the index it writes
  const float* shadow_of = nullptr;            // the index the bf16 copy mirrors
  int64_t shadow_blocks[kMaxSessionsHost] = {};  // per session: leading blocks the copy holds (written by appends)
  uint16_t* step_qpk = nullptr;  // packed bf16 query rows [S*h_kv][step_rows_cap_pad][d]
  float2* step_part = nullptr;   // row (max, sum) per column range [S*h_kv][kStepMaxRanges][rows]
  float2* step_stats = nullptr;  // row (max + log2 sum, 1/sum) [S*h_kv][rows]
  float* step_gs = nullptr;      // group scores when the caller does not ask for them [S][h_kv][max_blocks]
  // step attention over the view (multi-query), allocated when max_queries > 1
  uint16_t* attn_q = nullptr;     // rotated, scaled query rows, bf16 part then residual: [2][S*h_kv][rows][d]
  int attn_units_cap = 0;         // (row tile, view chunk) units a split step-attention call may use
  float* attn_part = nullptr;     // per unit: unnormalised O [128][d], then (max, sum) [128][2]
  uint32_t* attn_cnt = nullptr;   // per (KV head, row tile): chunks done (0 between calls)
};

constexpr int kStepMaxRanges = 64;

// kvm_index.cu
// (shadow: the context's bf16 copy of the index in the step scoring's core-matrix order, or null)
cudaError_t launch_index_append(const Ctx& c, const uint16_t* k_pool, int64_t n_pages, const int32_t* bt,
                                int n_sessions, const SessionArgs& a, int max_count, float* index, uint16_t* shadow,
                                cudaStream_t st);

// kvm_score.cu
cudaError_t launch_score_select(const Ctx& c, const uint16_t* q, int n_q, const float* index, int n_sessions,
                                const SessionArgs& a, int32_t* kept, float* group_scores, float* head_scores,
                                cudaStream_t st);

// kvm_score.cu: the selection controls (recent-only; withdrawn head-averaged scoring)
cudaError_t launch_select_control(const Ctx& c, int control, const uint16_t* q, const float* index, int n_sessions,
                                  const SessionArgs& a, int32_t* kept, float* group_scores, cudaStream_t st);

// The context's bf16 copy of the index holds every block the call scores (appended to this very index).
inline bool shadow_ready(const Ctx& c, const float* index, int n_sessions, const SessionArgs& a) {
  if (!c.step_kpk || index != c.shadow_of) return false;
  for (int s = 0; s < n_sessions; ++s)
    if (a.n_blk[s] > c.shadow_blocks[s]) return false;
  return true;
}

// kvm_step_score.cu: step-level scores of n_q > 1 query tokens (tcgen05) into gs_out [S][h_kv][max_blocks]
cudaError_t launch_step_scores(const Ctx& c, const uint16_t* q, int n_q, const float* index, int n_sessions,
                               const SessionArgs& a, float* gs_out, cudaStream_t st);
// kvm_score.cu: the cluster top-k on given group scores
cudaError_t launch_select_given(const Ctx& c, const float* gs, int n_sessions, const SessionArgs& a, int32_t* kept,
                                float* group_scores_out, cudaStream_t st);

// kvm_step_attn.cu: attention of n_q step tokens over the view (tcgen05); out [S][n_q][h_q][d] fp32
cudaError_t launch_step_attn(const Ctx& c, const uint16_t* q, int n_q, const uint16_t* k_view, const uint16_t* v_view,
                             const int32_t* view_len, int n_sessions, float* out, cudaStream_t st);

// kvm_gather.cu: quantised (FP8 E4M3) pages and the gather of views from quantised or host-resident pages
cudaError_t launch_quantize_pages(const Ctx& c, const uint16_t* pool, int64_t n_pages, const int32_t* pages,
                                  int64_t n_list, uint8_t* pool8, float* scales, cudaStream_t st);
cudaError_t launch_index_append_q(const Ctx& c, const uint8_t* k8, const float* kscale, int64_t n_pages,
                                  const int32_t* bt, int n_sessions, const SessionArgs& a, int max_count,
                                  float* index, cudaStream_t st);
cudaError_t launch_gather_view(const Ctx& c, bool fp8, const void* k_src, const void* v_src, const float* k_scale,
                               const float* v_scale, int64_t n_pages, const int32_t* bt, int n_sessions,
                               const SessionArgs& a, const int32_t* kept, uint16_t* k_view, uint16_t* v_view,
                               int32_t* view_len, cudaStream_t st);

// kvm_view.cu — mode: 0 materialise, 1 attend over a view, 2 fused, 3 fused from FP8 pages (k_src / v_src are
// then the code pools, with their per-(page, KV head) scales)
cudaError_t launch_view(const Ctx& c, int mode, const uint16_t* k_src, const uint16_t* v_src, int64_t n_pages,
                        const int32_t* bt, int n_sessions, const SessionArgs& a, const int32_t* kept,
                        const uint16_t* q, uint16_t* k_view, uint16_t* v_view, int32_t* view_len, float* out,
                        cudaStream_t st, const float* k_scale = nullptr, const float* v_scale = nullptr);

cudaError_t launch_rope_tables(const Ctx& c, cudaStream_t st);
// kvm_view.cu: a 4-D tensor map whose 64-row boxes are the tensor cores' no-swizzle core-matrix layout
cudaError_t make_core_matrix_map(CUtensorMap* m, const void* base, uint64_t rows, int d);

// Sets the message kvm_last_error() returns on this thread (kvm_api.cu).
void set_last_error(const char* msg);

// Launches `kernel` on `st` with programmatic stream serialisation (the kernel must call griddep_wait()
// before touching its predecessor's data; see kvm_device.cuh), and an optional cluster of `cluster_x` CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on `device`.
// The limit only ever grows, and each (kernel, device) pair is configured once
// per size, so steady-state calls (and calls under CUDA-graph capture) make no
// attribute calls.  Defined in kvm_api.cu.
cudaError_t ensure_smem_impl(const void* kernel, int device, size_t bytes);
template <typename F>
cudaError_t ensure_smem(F* kernel, int device, size_t bytes) {
  return ensure_smem_impl(reinterpret_cast<const void*>(kernel), device, bytes);
}

}  // namespace kvm
