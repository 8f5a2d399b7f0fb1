/*
 * kvm.h — C ABI of the KVMem decode hot path on one B300 (sm_103a).
 *
 * KVMem keeps a long agent history as paged KV and, for each decode step,
 * selects the history blocks relevant to the current query and materialises
 * them into a bounded execution view (KVMEM reproduction README, "Background
 * and main changes"; Evolve review of KVMem, "Summary").  Per layer and KV
 * head the path is:
 *   1. kvm_index_append   Mean-K index: the mean of each 32-token block's
 *                         pre-RoPE keys, accumulated in fp32.
 *   2. kvm_score_select   s_b = <q, kbar_b>/sqrt(d) per query head; softmax over
 *                         blocks per head; probabilities summed over each GQA
 *                         group; sink + recent blocks forced, top-k of the rest.
 *   3. kvm_materialize    kept blocks gathered in original order into a
 *                         contiguous bf16 view; keys re-rotated (RoPE) at view
 *                         positions 0..L-1, values copied bit for bit.
 *   4. kvm_decode_attn    single-token attention over the view.
 *   kvm_materialize_attn  3 + 4 in one pass (the view is written once and never
 *                         re-read from HBM).
 *   kvm_step_attn         attention of a whole step's query tokens over the
 *                         view (tensor cores), after a multi-query selection.
 * Page tiers beyond the bf16 HBM pool:
 *   kvm_quantize_pages, kvm_index_append_fp8, kvm_materialize_fp8,
 *   kvm_materialize_attn_fp8
 *                         FP8 E4M3 pages (one fp32 scale per page and KV head),
 *                         dequantised inside the index and the gather (the
 *                         last fused with attention).
 *   kvm_materialize_host  the gather from a pool in mapped pinned host memory.
 *
 * Conventions shared by every call
 * --------------------------------
 * - bf16 tensors are passed as uint16_t bit patterns.  fp32 is float.
 * - Unless a parameter says "host", every pointer is DEVICE memory owned by the
 *   caller (for example a PyTorch tensor); the library never frees it.  K/V
 *   pools, views, queries, the index and attention outputs must be 16-byte
 *   aligned; int32 arrays 4-byte aligned (KVM_ERR_INVALID_ARG otherwise).
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call only enqueues work on it and returns; nothing
 *   synchronises the host except kvm_create, kvm_destroy and kvm_device_status.
 * - Block size is fixed: 32 tokens per block, one block per physical page.
 * - One context serves one device (the device current at kvm_create) and one
 *   head geometry.  kvm_score_select, kvm_materialize, kvm_decode_attn,
 *   kvm_materialize_attn and kvm_step_attn on one context must not run
 *   concurrently on different streams: they share the context's scratch
 *   buffers.  The index appends, kvm_quantize_pages and the gathers of
 *   kvm_materialize_fp8 / kvm_materialize_host use no scratch.
 *   kvm_index_append uses no scratch (only the status word, which it updates
 *   atomically), so appends may run on another stream alongside them, e.g.
 *   every layer's append at the start of a decode step.
 * - Layouts (all row-major, innermost last):
 *     pool (K or V) of one layer   [n_pages][h_kv][32][d]            bf16 (a page = 32 tokens, all KV heads)
 *     block_table                  [n_sessions][max_blocks]          int32: block -> page
 *     index of one layer           [n_sessions][h_kv][max_blocks][d] fp32
 *     q (one decode token)         [n_sessions][h_q][d]              bf16, post-q-norm, pre-RoPE
 *     q (step of n_q tokens)       [n_sessions][n_q][h_q][d]         bf16
 *     kept_ids                     [n_sessions][h_kv][budget]        int32 ascending, -1 padded
 *     k_view, v_view               [n_sessions][h_kv][32*budget][d]  bf16
 *     view_len                     [n_sessions][h_kv]                int32 tokens in the view
 *     out                          [n_sessions][h_q][d]              fp32
 *   where budget = n_sink + n_recent + top_k blocks and query head h belongs
 *   to KV head h / (h_q / h_kv).
 * - History length n_tok is given per session on the host; n_blk =
 *   ceil(n_tok / 32).  A partial last block is averaged over the tokens
 *   present, and only those tokens enter the view.
 * - Errors: each call validates its arguments on the host and returns a
 *   kvm_status without launching anything when they are wrong;
 *   kvm_last_error() then describes the problem (thread-local).  Data errors
 *   only the device can see (a page id outside the pool, a kept id outside
 *   the history) skip the access and set a bit in the context's device status
 *   word, read with kvm_device_status().  No kernel traps.
 */
#ifndef KVM_H_
#define KVM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVM_OK = 0,
  KVM_ERR_INVALID_ARG = 1, /* null pointer, negative size, unsupported value          */
  KVM_ERR_SHAPE = 2,       /* size beyond the context's capacity or unsupported d      */
  KVM_ERR_BUDGET = 3,      /* budget fields inconsistent (negative, top_k < 0, ...)    */
  KVM_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed              */
  KVM_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (status word bit)     */
  KVM_ERR_DEVICE = 6       /* the device status word reports a data error              */
} kvm_status;

/* Bits of the device status word. */
#define KVM_DEV_BAD_PAGE 0x1u    /* block_table entry outside [0, n_pages)          */
#define KVM_DEV_BAD_BLOCK 0x2u   /* kept id outside [0, n_blk) or not above the entry before it (slot skipped) */
#define KVM_DEV_TIMEOUT 0x4u     /* a pipeline wait exceeded its iteration limit    */
#define KVM_DEV_BAD_VIEW 0x8u    /* kvm_step_attn: view_len outside [n_q, 32*budget] */
#define KVM_DEV_DEBUG_CHECK 0x10u /* debug build only: an index check inside a kernel failed */

typedef struct kvm_ctx kvm_ctx; /* opaque */

typedef struct {
  int32_t h_q;          /* query heads                                                 */
  int32_t h_kv;         /* KV heads; h_q % h_kv == 0, group h_q / h_kv in [1, 8]        */
  int32_t d;            /* head dimension: 64 or 128                                   */
  int32_t n_sink;       /* leading blocks always kept                                  */
  int32_t n_recent;     /* trailing blocks always kept                                 */
  int32_t top_k;        /* further blocks kept by group score                         */
  float rope_theta;     /* RoPE base (rotate-half pairing, full head dimension)        */
  int64_t max_blocks;   /* block capacity per session (block-table row, index rows)    */
  int32_t max_sessions; /* sessions per call, 1..64                                    */
  int32_t max_queries;  /* query tokens per session in one kvm_score_select or kvm_step_attn, >= 1 */
} kvm_params;

/* Human-readable name of a status code (static storage). */
const char* kvm_status_string(kvm_status s);

/* Message describing the last error returned on this thread (static, thread-local). */
const char* kvm_last_error(void);

/* 1 in the debug build of the library (libkvm_debug.so: kernels check the indices they compute, before the
 * accesses that use them, and set KVM_DEV_DEBUG_CHECK in the status word when one is out of range; nothing
 * traps), 0 in the release build.  Results are identical in both builds. */
int32_t kvm_debug_checks(void);

/*
 * Creates a context on the current CUDA device: validates `p`, allocates the
 * scratch buffers (score, softmax and attention partials; RoPE tables, filled
 * in fp64 by a kernel) and the device status word.  Synchronises the device.
 * *out receives the context; free it with kvm_destroy.
 */
kvm_status kvm_create(const kvm_params* p, kvm_ctx** out);

/* Frees everything kvm_create allocated (synchronises the device first). NULL is accepted. */
kvm_status kvm_destroy(kvm_ctx* ctx);

/* Device bytes the context allocated (scratch + tables); 0 for NULL. */
size_t kvm_scratch_bytes(const kvm_ctx* ctx);

/*
 * Index append (step 1).  KVMEM reproduction README, "Core equation" (index
 * vector kbar_b); Evolve review, "Summary" (position-independent Mean-K index
 * over 32-token blocks).
 *
 * For each session s, tokens [tok_begin[s], tok_begin[s] + n_tok[s]) have
 * already been written into the pool (pre-RoPE, post-k-norm keys).  Every
 * block those tokens touch is recomputed from the pool:
 *   index[s][g][b][:] = fp32 mean of the keys of block b present so far.
 * Rows of other blocks are not touched.
 *   k_pool       [n_pages][h_kv][32][d] bf16 (this layer)
 *   block_table  [n_sessions][max_blocks] int32
 *   tok_begin    host int64[n_sessions]
 *   n_tok        host int64[n_sessions] (0 = nothing to do for that session)
 *   index        [n_sessions][h_kv][max_blocks][d] fp32, updated in place
 * With max_queries > 1 the context also keeps a bf16 copy (nearest even) of
 * the rows it writes, for the multi-query scoring; the copy follows the index
 * pointer of the latest append (an append to another index starts it over).
 */
kvm_status kvm_index_append(kvm_ctx* ctx, const uint16_t* k_pool, int64_t n_pages,
                            const int32_t* block_table, int32_t n_sessions,
                            const int64_t* tok_begin, const int64_t* n_tok, float* index,
                            void* stream);

/*
 * Score and select (step 2).  KVMEM reproduction README, "Core equation"
 * (s_b = <q, kbar_b>/sqrt d, selection within the block budget) and
 * "2026-09-08 validation correction" (normalised query; softmax per query
 * head, not over heads averaged first).
 *
 * For each session and KV head g:
 *   s[h][b]  = <q_h, index[g][b]>/sqrt(d) for the group's query heads h
 *   Gs[g][b] = sum_{h in g} softmax_b(s[h][:])[b]          (one query)
 *   Gs[g][b] = sum_t sum_{h in g} softmax_b(s_t[h][:])[b]   (n_q > 1 query tokens)
 * The softmax runs over all n_blk blocks.  Kept = blocks [0, n_sink) and the
 * last n_recent blocks, plus the top_k remaining blocks by Gs (equal scores:
 * the lower id first); if n_blk <= budget every block is kept.
 *   q            [n_sessions][n_q][h_q][d] bf16, post-q-norm, pre-RoPE
 *   n_q          query tokens per session, 1..max_queries
 *   index        [n_sessions][h_kv][max_blocks][d] fp32
 *   n_tok        host int64[n_sessions] history length (n_blk = ceil(n_tok/32) <= max_blocks)
 *   kept_ids     [n_sessions][h_kv][budget] int32 out: ascending ids, -1 after n_keep
 *   group_scores [n_sessions][h_kv][max_blocks] fp32 out, or NULL
 *   head_scores  [n_sessions][h_q][max_blocks] fp32 out (raw s, n_q == 1 only), or NULL
 * n_q > 1 multiplies bf16 operands on the tensor cores: the index rows rounded
 * to bf16 come from the context's copy when `index` is the one last appended
 * to through this context and every scored block was written by those
 * appends; otherwise the call converts `index` itself (and the copy is then
 * dropped until the next append).  An index changed by other means since its
 * last kvm_index_append must be appended again (or converted) before an
 * n_q > 1 call, as the copy would not see the change.
 */
kvm_status kvm_score_select(kvm_ctx* ctx, const uint16_t* q, int32_t n_q, const float* index,
                            const int64_t* n_tok, int32_t n_sessions, int32_t* kept_ids,
                            float* group_scores, float* head_scores, void* stream);

/*
 * Materialise (step 3).  KVMEM reproduction README, "Core equation"
 * (selected KV concatenated; address space and execution window kept apart);
 * Evolve review, "Summary" / "Scope & Claims" (blocks restored with
 * position-consistent re-RoPE into a bounded view).
 *
 * View slot j of (s, g) holds the j-th token of the kept blocks, in block
 * order.  v_view[s][g][j] is a bit copy of the value; k_view[s][g][j] is the
 * key rotated at position j (rotate-half pairing: dimension i with i + d/2,
 * angle j * theta^(-2i/d)) and rounded to bf16, nearest even.  Slots past
 * view_len are not written.
 *   k_pool, v_pool [n_pages][h_kv][32][d] bf16 (this layer)
 *   block_table    [n_sessions][max_blocks] int32
 *   n_tok          host int64[n_sessions]
 *   kept_ids       [n_sessions][h_kv][budget] int32 (as written by kvm_score_select)
 *   k_view, v_view [n_sessions][h_kv][32*budget][d] bf16 out
 *   view_len       [n_sessions][h_kv] int32 out
 */
kvm_status kvm_materialize(kvm_ctx* ctx, const uint16_t* k_pool, const uint16_t* v_pool,
                           int64_t n_pages, const int32_t* block_table, const int64_t* n_tok,
                           int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view,
                           uint16_t* v_view, int32_t* view_len, void* stream);

/*
 * Decode attention over a view (step 4).  KVMEM reproduction README, "Local
 * reproduction" (the view replaces full attention) and "2026-09-08
 * validation correction" (RoPE applied to the query).
 *   out[s][h] = sum_j softmax_j(<RoPE(q_h, L), k_view[g][j]>/sqrt(d)) v_view[g][j]
 * with L = view_len[s][g] (the query sits at the slot after the view).  An
 * empty view gives zeros.
 *   q         [n_sessions][h_q][d] bf16, post-q-norm, pre-RoPE
 *   k_view, v_view, view_len as written by kvm_materialize
 *   out       [n_sessions][h_q][d] fp32
 */
kvm_status kvm_decode_attn(kvm_ctx* ctx, const uint16_t* q, const uint16_t* k_view,
                           const uint16_t* v_view, const int32_t* view_len, int32_t n_sessions,
                           float* out, void* stream);

/*
 * Steps 3 and 4 fused: the same outputs as kvm_materialize followed by
 * kvm_decode_attn, reading each kept page once.
 */
kvm_status kvm_materialize_attn(kvm_ctx* ctx, const uint16_t* k_pool, const uint16_t* v_pool,
                                int64_t n_pages, const int32_t* block_table, const int64_t* n_tok,
                                int32_t n_sessions, const int32_t* kept_ids, const uint16_t* q,
                                uint16_t* k_view, uint16_t* v_view, int32_t* view_len, float* out,
                                void* stream);

/*
 * Attention of a step's n_q query tokens over the view, on the tensor cores.
 * Evolve review of KVMem, "Strengths" (recall once per agent step) and KVMEM
 * reproduction README, "Local reproduction" (the view replaces full
 * attention).  The step's tokens are the history's last n_q tokens, so they
 * sit in the view's last slots: token t is at view position
 * p_t = L - n_q + t (L = view_len[s][g]) and attends the slots j <= p_t:
 *   out[s][t][h] = sum_{j<=p_t} softmax_j(<RoPE(q[s][t][h], p_t), k_view[g][j]>/sqrt(d)) v_view[g][j]
 * Products are fp32-accurate (each bf16 MMA operand that is not already bf16
 * -- the rotated query and the probabilities -- is split into a bf16 part
 * and its bf16 residual); accumulation is fp32.
 *   q          [n_sessions][n_q][h_q][d] bf16, post-q-norm, pre-RoPE
 *   k_view, v_view, view_len as written by kvm_materialize ([n_sessions][h_kv]
 *              [32*budget][d] bf16, read in place in 64-token tiles; slots
 *              at or past view_len may hold anything: they never contribute)
 *   out        [n_sessions][n_q][h_q][d] fp32 (16-byte aligned)
 * Needs a context created with max_queries > 1 (it owns the packed query
 * rows and the partial-state scratch) and 1 <= n_q <= max_queries,
 * n_q <= 32*budget (KVM_ERR_SHAPE otherwise).  A view_len outside
 * [n_q, 32*budget] sets KVM_DEV_BAD_VIEW; that head's outputs are then
 * undefined.
 */
kvm_status kvm_step_attn(kvm_ctx* ctx, const uint16_t* q, int32_t n_q, const uint16_t* k_view,
                         const uint16_t* v_view, const int32_t* view_len, int32_t n_sessions, float* out,
                         void* stream);

/*
 * Quantised KV pages.  KVMEM reproduction README, "Background and main
 * changes" (paged KV kept beyond GPU memory; the deployment runs in NVFP4).
 * The pages give no precision for the paged KV; this variant stores each
 * (page, KV head) of K and of V as FP8 E4M3 codes (OCP format: bias 7, no
 * infinities, largest finite 448) with one fp32 scale, value = code * scale:
 *   scale = amax / 448 (fp32 division; amax over the page's 32 x d values as
 *           stored; a page of zeros gets scale 1)
 *   code  = E4M3(x / scale): fp32 division, nearest even, magnitudes past 448
 *           saturate.
 *   pool8   [n_pages][h_kv][32][d] uint8 codes (16-byte aligned)
 *   scales  [n_pages][h_kv] fp32
 *
 * kvm_quantize_pages: quantises the listed pages (every KV head) of a bf16
 * pool [n_pages][h_kv][32][d] into pool8 / scales.  pages is a device int32
 * array of n_list page ids; an id outside [0, n_pages) sets KVM_DEV_BAD_PAGE.
 */
kvm_status kvm_quantize_pages(kvm_ctx* ctx, const uint16_t* pool, int64_t n_pages, const int32_t* pages,
                              int64_t n_list, uint8_t* pool8, float* scales, void* stream);

/*
 * kvm_index_append as above, over quantised keys: each block's mean of the
 * dequantised keys (code * scale, fp32), accumulated in fp32 in token order.
 */
kvm_status kvm_index_append_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales, int64_t n_pages,
                                const int32_t* block_table, int32_t n_sessions, const int64_t* tok_begin,
                                const int64_t* n_tok, float* index, void* stream);

/*
 * kvm_materialize from quantised pages: view slot j holds the j-th kept token;
 * k_view is the dequantised key rotated at position j and rounded to bf16
 * (nearest even), v_view the dequantised value rounded to bf16 (nearest
 * even).  Arguments, layouts and errors otherwise as kvm_materialize; the
 * view then feeds kvm_decode_attn or kvm_step_attn unchanged.
 */
kvm_status kvm_materialize_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales, const uint8_t* v_pool8,
                               const float* v_scales, int64_t n_pages, const int32_t* block_table,
                               const int64_t* n_tok, int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view,
                               uint16_t* v_view, int32_t* view_len, void* stream);

/*
 * kvm_materialize_attn from quantised pages: the same outputs as
 * kvm_materialize_fp8 followed by kvm_decode_attn, in one pass that reads
 * each kept code page once (the bf16 view is written and never read back).
 * Arguments as kvm_materialize_fp8, plus q and out as in kvm_decode_attn.
 */
kvm_status kvm_materialize_attn_fp8(kvm_ctx* ctx, const uint8_t* k_pool8, const float* k_scales,
                                    const uint8_t* v_pool8, const float* v_scales, int64_t n_pages,
                                    const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions,
                                    const int32_t* kept_ids, const uint16_t* q, uint16_t* k_view,
                                    uint16_t* v_view, int32_t* view_len, float* out, void* stream);

/*
 * Host tier.  KVMEM reproduction README, "Background and main changes" and
 * Evolve review, "Summary" (history paged across GPU and host memory).  The
 * same outputs as kvm_materialize, with the K/V pools resident in host memory:
 * k_pool_host / v_pool_host must be pinned and mapped into the device address
 * space (cudaHostAlloc with cudaHostAllocMapped, or cudaHostRegister with
 * cudaHostRegisterMapped), else KVM_ERR_INVALID_ARG.  Only the kept pages'
 * rows cross the host link, read by the gather kernel directly (no staging
 * copy); block_table, kept_ids and the view stay in device memory.
 */
kvm_status kvm_materialize_host(kvm_ctx* ctx, const uint16_t* k_pool_host, const uint16_t* v_pool_host,
                                int64_t n_pages, const int32_t* block_table, const int64_t* n_tok,
                                int32_t n_sessions, const int32_t* kept_ids, uint16_t* k_view, uint16_t* v_view,
                                int32_t* view_len, void* stream);

/*
 * Selection controls (the comparisons the pages report next to the method).
 * KVMEM reproduction README, "Local reproduction" (a recent-only control at
 * the same block budget) and "2026-09-08 validation correction" (the
 * withdrawn scoring averaged the GQA query heads before the softmax).
 *   KVM_CONTROL_RECENT_ONLY       kept = the last min(n_blk, budget) blocks of
 *                                 each history, ascending; q, index and
 *                                 group_scores are not used (may be NULL).
 *   KVM_CONTROL_WITHDRAWN_AVERAGE per KV head g: q_bar = mean of the group's
 *                                 query heads (unweighted, not re-normalised),
 *                                 s[b] = <q_bar, index[g][b]>/sqrt(d),
 *                                 Gs[g][b] = softmax_b(s)[b]; then the same
 *                                 sink / recent / top_k selection as
 *                                 kvm_score_select.
 * Arguments and layouts are those of kvm_score_select with one query token
 * (n_q = 1); group_scores (nullable) receives the control's Gs.
 */
#define KVM_CONTROL_RECENT_ONLY 1
#define KVM_CONTROL_WITHDRAWN_AVERAGE 2
kvm_status kvm_select_control(kvm_ctx* ctx, int32_t control, const uint16_t* q, const float* index,
                              const int64_t* n_tok, int32_t n_sessions, int32_t* kept_ids, float* group_scores,
                              void* stream);

/*
 * Reads (and optionally clears) the device status word after synchronising
 * `stream`.  *out receives the KVM_DEV_* bits.  Returns KVM_OK when the word
 * is zero, KVM_ERR_DEVICE or KVM_ERR_TIMEOUT otherwise.  A timed-out view
 * call leaves its attention outputs unwritten; clearing a non-zero word also
 * resets the context's per-call merge state, so the context can be reused.
 */
kvm_status kvm_device_status(kvm_ctx* ctx, uint32_t* out, int32_t clear, void* stream);

/*
 * Allocation-free score and select for one decode query.  The method has no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory, for example a runtime whose memory pool owns every device byte, or
 * code that must not synchronise the device (cudaMalloc and cudaFree may), and
 * so cannot create a context with kvm_create.
 *
 * It computes exactly what kvm_score_select computes for n_q = 1 (same
 * kernels, same results), taking the head geometry and budget from `p`
 * (max_sessions and max_queries are ignored; the index rows and block-table
 * rows have max_blocks entries).  Arguments and layouts are those of
 * kvm_score_select; there is no head_scores output.
 *
 * Scratch: one fixed array of KVM_NOALLOC_SCRATCH_BYTES in device global memory,
 * which every GPU that loads this library holds until the process exits.  It
 * must fit n_sessions * (h_q * ceil(max_blocks/32) * 8 + h_kv * max_blocks *
 * (h_q/h_kv) * 4) bytes plus 512; larger calls return KVM_ERR_SHAPE and launch
 * nothing (one session of 40/8 heads fits 32,768 blocks).  The first call on
 * each device looks up the array's device address with that device current;
 * make that first call before any stream capture (outside capture every call
 * looks the address up again, so a reset device or another context is
 * followed; during capture the address last seen on the device is used).
 * Every call reuses the same array and leaves its contents behind, so calls
 * whose work overlaps on the GPU (different streams, or other threads) race
 * and must be serialised by the caller.  No device memory is allocated or
 * freed.  Argument errors are returned at once (kvm_last_error()); errors only
 * the device sees (a bounded wait that gave up: the kept ids of that call are
 * then undefined) set bits in a status word inside the array, which stays set
 * across calls until kvm_noalloc_status clears it.
 */
#define KVM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
kvm_status kvm_score_select_noalloc(const kvm_params* p, const uint16_t* q, const float* index,
                                   const int64_t* n_tok, int32_t n_sessions, int32_t* kept_ids,
                                   float* group_scores, void* stream);

/*
 * Reads (and optionally clears) the status word of kvm_score_select_noalloc on
 * the current device after synchronising `stream`: *out receives the KVM_DEV_*
 * bits set by any allocation-free call since the word was last cleared.
 * Returns KVM_OK when it is zero, KVM_ERR_TIMEOUT or KVM_ERR_DEVICE otherwise.
 * Allocates nothing; like the calls it reports on, it has no counterpart in the
 * method.
 */
kvm_status kvm_noalloc_status(uint32_t* out, int32_t clear, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVM_H_ */
