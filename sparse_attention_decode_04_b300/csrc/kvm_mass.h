// Internal interface of the attention-mass diagnostic (kvm_mass.cu) for the C-ABI layer.
#pragma once

#include "kvm_internal.h"

namespace kvm {

// Fills the rows [budget + 1, max_blocks] of the RoPE base tables (cos/sin of 32 * row * theta_i, hi and lo),
// which only the diagnostic reads: every history position, not only view positions.
cudaError_t launch_mass_tables(const Ctx& c, cudaStream_t st);

// Per (session, KV head): the full-attention mass of every history block, summed over the group's query heads.
cudaError_t launch_attention_mass(const Ctx& c, const uint16_t* q, const uint16_t* k_pool, int64_t n_pages,
                                  const int32_t* bt, int n_sessions, const SessionArgs& a, float* mass,
                                  cudaStream_t st);

}  // namespace kvm
