// Calls that take several layers at once (internal side).
#pragma once

#include "kvm_internal.h"

namespace kvm {

constexpr int kMaxAppendLayers = 64;  // layers per kvm_index_append_layers call (kernel-parameter arrays)

// The layers' key pools and indexes, passed by value to the kernel.
struct AppendLayers {
  const uint16_t* k_pool[kMaxAppendLayers];
  float* index[kMaxAppendLayers];
};

// kvm_index.cu: the appends of n_layers layers (same sessions and token ranges) in one launch.
cudaError_t launch_index_append_layers(const Ctx& c, const AppendLayers& layers, int n_layers, int64_t n_pages,
                                       const int32_t* bt, int n_sessions, const SessionArgs& a, int max_count,
                                       cudaStream_t st);

}  // namespace kvm
