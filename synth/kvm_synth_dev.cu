// Device copy of the seeded input generator (kvm_synth.c), used to fill large
// paged K/V pools directly in HBM.  Same definition: Philox4x32-10 counters
// (Salmon et al., SC'11), Box-Muller normals, the topic-mixture key recipe and
// round-to-nearest-even bf16, all in fp64 with multiply-add contraction off
// (built with -fmad=false), so the bits match the host generator's (up to the
// last-place behaviour of the fp64 log/sin/cos, which only matters when a
// value lands within ~1e-16 of a bf16 rounding boundary).  Holds none of the
// method's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint32_t TAG_TOPIC = 1, TAG_KEY_NOISE = 2, TAG_VALUE = 3;

__device__ void philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1, uint32_t o[4]) {
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  o[0] = c0; o[1] = c1; o[2] = c2; o[3] = c3;
}

__device__ __forceinline__ double u01(uint32_t x) { return ((double)x + 0.5) * 0x1p-32; }

__device__ void normal_row(uint32_t seed, uint32_t tag, uint32_t item, uint32_t lh, uint32_t session, int n, double* z) {
  for (int j = 0; j < n / 4; ++j) {
    uint32_t o[4];
    philox((uint32_t)j, item, lh, session, seed, tag, o);
    const double r1 = sqrt(-2.0 * log(u01(o[0]))), a1 = 6.283185307179586 * u01(o[1]);
    const double r2 = sqrt(-2.0 * log(u01(o[2]))), a2 = 6.283185307179586 * u01(o[3]);
    z[4 * j + 0] = r1 * cos(a1);
    z[4 * j + 1] = r1 * sin(a1);
    z[4 * j + 2] = r2 * cos(a2);
    z[4 * j + 3] = r2 * sin(a2);
  }
}

__device__ uint16_t bf16_rne(double x) {
  if (x != x) return 0x7FC0;
  int e;
  frexp(x, &e);
  int q = e - 8;
  if (q < -133) q = -133;
  const double r = rint(ldexp(x, -q));
  const float f = (float)ldexp(r, q);
  return (uint16_t)(__float_as_uint(f) >> 16);
}

// One thread per (KV head, block): writes the block's tokens in [t0, t1).
template <int D>
__global__ void kv_pages_kernel(uint32_t seed, int session, int layer, int h_kv, int64_t t0, int64_t t1,
                                double eps_scale, const int32_t* page_of_block, int64_t n_pages, uint16_t* k_pool,
                                uint16_t* v_pool, int* bad) {
  const int64_t b0 = t0 / 32, nb = (t1 + 31) / 32 - b0;
  const int64_t gid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (gid >= nb * h_kv) return;
  const int h = (int)(gid % h_kv);
  const int64_t b = b0 + gid / h_kv;
  const int64_t page = page_of_block[b];
  if (page < 0 || page >= n_pages) {
    atomicOr(bad, 1);
    return;
  }
  const uint32_t lh = ((uint32_t)layer << 16) | (uint32_t)h;
  double mu[D], x[D];
  normal_row(seed, TAG_TOPIC, (uint32_t)b, lh, (uint32_t)session, D, mu);
  const int64_t ta = b * 32 > t0 ? b * 32 : t0, tb = b * 32 + 32 < t1 ? b * 32 + 32 : t1;
  for (int64_t t = ta; t < tb; ++t) {
    uint16_t* krow = k_pool + ((page * h_kv + h) * 32 + (t - b * 32)) * D;
    uint16_t* vrow = v_pool + ((page * h_kv + h) * 32 + (t - b * 32)) * D;
    normal_row(seed, TAG_KEY_NOISE, (uint32_t)t, lh, (uint32_t)session, D, x);
    double ss = 0.0;
    for (int k = 0; k < D; ++k) {
      x[k] = 0.5 * mu[k] + eps_scale * x[k];
      ss += x[k] * x[k];
    }
    const double inv = 1.0 / sqrt(ss / (double)D + 1e-6);
    for (int k = 0; k < D; k += 4) {
      const uint64_t w = (uint64_t)bf16_rne(x[k] * inv) | ((uint64_t)bf16_rne(x[k + 1] * inv) << 16) |
                         ((uint64_t)bf16_rne(x[k + 2] * inv) << 32) | ((uint64_t)bf16_rne(x[k + 3] * inv) << 48);
      *reinterpret_cast<uint64_t*>(krow + k) = w;
    }
    normal_row(seed, TAG_VALUE, (uint32_t)t, lh, (uint32_t)session, D, x);
    for (int k = 0; k < D; k += 4) {
      const uint64_t w = (uint64_t)bf16_rne(x[k]) | ((uint64_t)bf16_rne(x[k + 1]) << 16) |
                         ((uint64_t)bf16_rne(x[k + 2]) << 32) | ((uint64_t)bf16_rne(x[k + 3]) << 48);
      *reinterpret_cast<uint64_t*>(vrow + k) = w;
    }
  }
}

}  // namespace

// Fills tokens [t0, t1) of one session and layer into device pools laid out
// [n_pages][h_kv][32][d]; page_of_block is a device int32 array.  Returns a
// cudaError_t value (0 = success); *bad_dev (device int) gets 1 for a page
// outside [0, n_pages).
extern "C" int synth_dev_kv_pages(uint32_t seed, int session, int layer, int h_kv, int d, int64_t t0, int64_t t1,
                                  double eps_scale, const int32_t* page_of_block, int64_t n_pages, uint16_t* k_pool,
                                  uint16_t* v_pool, int* bad_dev, void* stream) {
  if (t1 <= t0) return 0;
  const int64_t nb = (t1 + 31) / 32 - t0 / 32;
  const int64_t n = nb * h_kv;
  const int threads = 64;
  const unsigned blocks = (unsigned)((n + threads - 1) / threads);
  cudaStream_t st = (cudaStream_t)stream;
  if (d == 128)
    kv_pages_kernel<128><<<blocks, threads, 0, st>>>(seed, session, layer, h_kv, t0, t1, eps_scale, page_of_block,
                                                      n_pages, k_pool, v_pool, bad_dev);
  else if (d == 64)
    kv_pages_kernel<64><<<blocks, threads, 0, st>>>(seed, session, layer, h_kv, t0, t1, eps_scale, page_of_block,
                                                     n_pages, k_pool, v_pool, bad_dev);
  else
    return (int)cudaErrorInvalidValue;
  return (int)cudaGetLastError();
}
