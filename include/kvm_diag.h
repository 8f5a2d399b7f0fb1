/*
 * kvm_diag.h — diagnostics of the KVMem decode path (C ABI, same conventions as kvm.h).
 */
#ifndef KVM_DIAG_H_
#define KVM_DIAG_H_

#include "kvm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Full-attention mass per history block.  KVMEM reproduction README,
 * "Background and main changes": a few blocks hold most of the attention (the
 * top 8 of about 103 blocks held 66.5% of it).  For one decode query per
 * session, with the query at position N = n_tok[s] and each key at its
 * history position t (exact attention over the whole history, no selection):
 *   mass[s][g][b] = sum_{h in g} sum_{t in b} softmax_t(<RoPE(q_h, N), RoPE(k_t, t)>/sqrt(d))
 * so sum_b mass[s][g][b] = h_q / h_kv.  The share held by the k largest blocks
 * is a host-side sort of that row.
 *   q           [n_sessions][h_q][d] bf16, post-q-norm, pre-RoPE
 *   k_pool      [n_pages][h_kv][32][d] bf16 (this layer), block_table as in kvm.h
 *   n_tok       host int64[n_sessions]
 *   mass        [n_sessions][h_kv][max_blocks] fp32 out (entries past n_blk not written)
 * Uses the context's scoring scratch: not concurrent with kvm_score_select on
 * the same context.  A page id outside [0, n_pages) sets KVM_DEV_BAD_PAGE.
 */
kvm_status kvm_attention_mass(kvm_ctx* ctx, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages,
                              const int32_t* block_table, const int64_t* n_tok, int32_t n_sessions, float* mass,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVM_DIAG_H_ */
