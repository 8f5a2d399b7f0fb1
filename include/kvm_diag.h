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

/*
 * Failure-path testing of the view calls (kvm_materialize, kvm_decode_attn,
 * kvm_materialize_attn).  Their pipeline waits are bounded: a wait that gives
 * up sets KVM_DEV_TIMEOUT, the kernel waits (with the full limit) for its
 * copies in flight and returns without writing the outputs of the
 * (session, KV head) units it had a share in; kvm_device_status with clear
 * then also resets the per-call merge counters, so the context stays usable.
 *   wait_ns           wall-clock limit of each pipeline wait, in [1000, 2e9]
 *                     nanoseconds (2e9 by default; the waits for copies in
 *                     flight always keep 2e9)
 *   stall_first_wait  1: the first rotation wait of the first CTA is on a
 *                     barrier that nothing completes, so that wait (and the
 *                     waits on its stages) run out after wait_ns; 0: normal
 * The pages define no such control; it exists so that tests can exercise the
 * timeout path without faulting or hanging the GPU.
 */
kvm_status kvm_set_wait_limit(kvm_ctx* ctx, int64_t wait_ns, int32_t stall_first_wait);

#ifdef __cplusplus
}
#endif

#endif /* KVM_DIAG_H_ */
