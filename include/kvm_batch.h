/*
 * kvm_batch.h — calls over several layers at once (C ABI, same conventions as kvm.h).
 */
#ifndef KVM_BATCH_H_
#define KVM_BATCH_H_

#include "kvm.h"

#ifdef __cplusplus
extern "C" {
#endif

#define KVM_MAX_APPEND_LAYERS 64

/*
 * kvm_index_append for n_layers layers in one launch.  KVMEM reproduction README, "Core equation" (index vector
 * kbar_b); Evolve review, "Summary" (Mean-K index over 32-token blocks).  The layers share the sessions, the
 * block table, the token ranges and the pool geometry; layer i reads k_pools[i] and updates indexes[i] exactly as
 * kvm_index_append(ctx, k_pools[i], n_pages, block_table, n_sessions, tok_begin, n_tok, indexes[i], stream)
 * would, bit for bit.  It serves a decode step whose new tokens have their keys for every layer when the step
 * starts: one launch instead of one per layer.
 *   n_layers     1 .. KVM_MAX_APPEND_LAYERS
 *   k_pools      host array of n_layers device pointers, each [n_pages][h_kv][32][d] bf16, 16-byte aligned
 *   indexes      host array of n_layers device pointers, each [n_sessions][h_kv][max_blocks][d] fp32,
 *                16-byte aligned, updated in place (distinct layers must not share an index)
 *   the rest     as kvm_index_append
 * The context's bf16 copy of an index (max_queries > 1) is not written: when one of the indexes is the one the
 * copy follows, the call drops the copy, and the next n_q > 1 kvm_score_select on it converts the index itself.
 * The host arrays are read before the call returns.
 * Errors: KVM_ERR_INVALID_ARG (NULL or unaligned pointer, n_layers out of range), KVM_ERR_SHAPE (a token range
 * beyond max_blocks), KVM_ERR_CUDA (launch); bad block-table entries set KVM_DEV_BAD_PAGE in the status word.
 */
kvm_status kvm_index_append_layers(kvm_ctx* ctx, int32_t n_layers, const uint16_t* const* k_pools,
                                   int64_t n_pages, const int32_t* block_table, int32_t n_sessions,
                                   const int64_t* tok_begin, const int64_t* n_tok, float* const* indexes,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVM_BATCH_H_ */
