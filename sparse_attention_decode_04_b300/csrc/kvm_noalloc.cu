// Allocation-free score + select for a single decode query.
//
// Some callers cannot call cudaMalloc at all: code running inside an
// allocator-less runtime (an inference server whose memory pool owns every
// device byte, an embedded host that forbids allocation after start-up) or
// code that must not synchronise the device, which cudaMalloc/cudaFree may do.
// kvm_create allocates its scratch, so those callers cannot use
// kvm_score_select.  This entry point takes the head geometry directly and
// keeps its scratch (per-tile exponentials and softmax partials, and a status
// word) in one fixed array in device global memory that lives as long as the
// library stays loaded on each GPU.
//
// The kernels are the same ones kvm_score_select launches for one query; only
// where their scratch lives differs.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "kvm.h"
#include "kvm_internal.h"

namespace {

// Scratch shared by every call on a device: status word, tile partials, exponentials.
constexpr size_t kNoAllocScratchBytes = KVM_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

kvm_status na_fail(kvm_status s, const char* fmt, ...) {
  char msg[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  kvm::set_last_error(msg);  // readable through kvm_last_error()
  return s;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of the scratch array (its name is only a host-side stand-in).  Outside stream capture it is
// looked up again on every call, with the call's device current, so a reloaded module (after a device reset,
// or under another context) is always followed; during capture, when the runtime may not be asked, the
// address last seen on that device is used.
constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

cudaError_t scratch_address(int device, cudaStream_t st, unsigned char** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return e;
    g_addr[device] = p;
  } else if (!g_addr[device]) {
    return cudaErrorStreamCaptureUnsupported;  // the first call on a device must come before any capture
  }
  *out = static_cast<unsigned char*>(g_addr[device]);
  return cudaSuccess;
}

}  // namespace

extern "C" kvm_status kvm_score_select_noalloc(const kvm_params* p, const uint16_t* q, const float* index,
                                               const int64_t* n_tok, int32_t n_sessions, int32_t* kept_ids,
                                               float* group_scores, void* stream) {
  if (!p) return na_fail(KVM_ERR_INVALID_ARG, "params is NULL");
  if (p->d != 64 && p->d != 128) return na_fail(KVM_ERR_SHAPE, "d=%d: only 64 and 128 are built", p->d);
  if (p->h_q <= 0 || p->h_kv <= 0 || p->h_q % p->h_kv != 0 || p->h_q / p->h_kv > kvm::kMaxGroup)
    return na_fail(KVM_ERR_SHAPE, "h_q=%d, h_kv=%d: need h_q a multiple of h_kv with group <= %d", p->h_q, p->h_kv,
                   kvm::kMaxGroup);
  if (p->n_sink < 0 || p->n_recent < 0 || p->top_k < 0)
    return na_fail(KVM_ERR_BUDGET, "n_sink, n_recent and top_k must be >= 0");
  const int64_t budget = (int64_t)p->n_sink + p->n_recent + p->top_k;
  if (budget < 1 || budget > (1 << 20)) return na_fail(KVM_ERR_BUDGET, "budget %lld outside [1, 2^20]", (long long)budget);
  if (p->max_blocks < 1 || p->max_blocks > 8 * 40960)
    return na_fail(KVM_ERR_SHAPE, "max_blocks=%lld outside [1, %d]", (long long)p->max_blocks, 8 * 40960);
  if (n_sessions < 0 || n_sessions > kvm::kMaxSessionsHost)
    return na_fail(KVM_ERR_SHAPE, "n_sessions=%d outside [0, %d]", n_sessions, kvm::kMaxSessionsHost);
  if (n_sessions == 0) return KVM_OK;
  if (!q || !index || !kept_ids || !n_tok) return na_fail(KVM_ERR_INVALID_ARG, "NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(index)) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(kept_ids) % 4 != 0 || reinterpret_cast<uintptr_t>(group_scores) % 4 != 0)
    return na_fail(KVM_ERR_INVALID_ARG, "q and index must be 16-byte aligned, outputs 4-byte aligned");

  kvm::Ctx c;
  c.p = *p;
  c.p.max_sessions = n_sessions;
  c.p.max_queries = 1;
  c.group = p->h_q / p->h_kv;
  c.budget = (int)budget;
  c.max_tiles = (p->max_blocks + 31) / 32;

  // scratch layout: status word | tile partials [S][h_q][max_tiles] | exponentials [S][h_kv][G][e_stride]
  const size_t off_part = 256;
  const size_t sz_part = (size_t)n_sessions * p->h_q * (size_t)c.max_tiles * sizeof(float2);
  const size_t off_e = align256(off_part + sz_part);
  c.e_stride = (p->max_blocks + 3) & ~(int64_t)3;
  const size_t sz_e = (size_t)n_sessions * p->h_kv * (size_t)c.e_stride * c.group * sizeof(float);
  if (off_e + sz_e > kNoAllocScratchBytes)
    return na_fail(KVM_ERR_SHAPE,
                   "scratch for %d session(s) x %lld blocks needs %zu bytes; this entry point holds at most %zu",
                   n_sessions, (long long)p->max_blocks, off_e + sz_e, kNoAllocScratchBytes);

  kvm::SessionArgs a;
  memset(&a, 0, sizeof(a));
  int64_t base = 0;
  for (int s = 0; s < n_sessions; ++s) {
    if (n_tok[s] < 0) return na_fail(KVM_ERR_INVALID_ARG, "n_tok[%d] is negative", s);
    const int64_t nb = (n_tok[s] + kvm::kBlock - 1) / kvm::kBlock;
    if (nb > p->max_blocks) return na_fail(KVM_ERR_SHAPE, "session %d: %lld blocks exceed max_blocks", s, (long long)nb);
    a.n_tok[s] = n_tok[s];
    a.n_blk[s] = (int32_t)nb;
    a.n_keep[s] = (int32_t)(nb < budget ? nb : budget);
    a.seg_base[s] = base;
    base += (int64_t)p->h_kv * a.n_keep[s];
  }
  a.seg_base[n_sessions] = base;

  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaGetDevice(&c.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, c.device);
  unsigned char* scratch = nullptr;
  if (e == cudaSuccess) e = scratch_address(c.device, st, &scratch);
  if (e != cudaSuccess)
    return na_fail(KVM_ERR_CUDA, "scratch address: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  // the status word (first bytes of the array) collects device-side errors until kvm_noalloc_status clears it
  c.status = reinterpret_cast<uint32_t*>(scratch);
  c.part = reinterpret_cast<float2*>(scratch + off_part);
  c.e_buf = reinterpret_cast<float*>(scratch + off_e);

  e = kvm::launch_score_select(c, q, 1, index, n_sessions, a, kept_ids, group_scores, nullptr, st);
  if (e != cudaSuccess)
    return na_fail(KVM_ERR_CUDA, "kvm_score_select_noalloc launch: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  return KVM_OK;
}

extern "C" kvm_status kvm_noalloc_status(uint32_t* out, int32_t clear, void* stream) {
  if (!out) return na_fail(KVM_ERR_INVALID_ARG, "out is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  int device = 0;
  unsigned char* scratch = nullptr;
  cudaError_t e = cudaGetDevice(&device);
  if (e == cudaSuccess) e = scratch_address(device, st, &scratch);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(scratch, 0, sizeof(uint32_t));
  if (e != cudaSuccess)
    return na_fail(KVM_ERR_CUDA, "kvm_noalloc_status: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  if (*out == 0) return KVM_OK;
  if (*out & KVM_DEV_TIMEOUT) return na_fail(KVM_ERR_TIMEOUT, "a device-side wait timed out (status 0x%x)", *out);
  return na_fail(KVM_ERR_DEVICE, "device status 0x%x", *out);
}
