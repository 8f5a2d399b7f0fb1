/*
 * Seeded synthetic inputs for the KVMem decode hot path (host side).
 *
 * This file generates INPUTS only: paged bf16 keys/values, queries, planted
 * block sets and block tables.  It holds none of the method's arithmetic
 * (no index means, no scores, no selection, no RoPE, no attention), so both
 * the CUDA path and the CPU oracle can be fed from it.
 *
 * Random numbers: Philox4x32-10, the counter-based generator of Salmon,
 * Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 * (SC'11), Sec. 4.  Every draw is addressed by a 128-bit counter
 *   (j, item, (layer << 16) | head, session)
 * under the 64-bit key (seed, tag), so any block of any layer can be
 * regenerated alone.  Normals come from the Box-Muller transform
 * (Box & Muller 1958), two normals per pair of uniforms, in fp64.
 *
 * Workload recipe (the topic-mixture keys of the KVMem synthetic configs):
 *   mu_b  = 0.5 * z           z ~ N(0, I)  per (session, layer, kv head, block)
 *   x_t   = mu_b + eps * z'   z' ~ N(0, I) per token        (eps = 1 normally)
 *   k_t   = bf16_rne( x_t / sqrt(mean(x_t^2) + 1e-6) )
 *   v_t   = bf16_rne( z'' )   z'' ~ N(0, I)
 *   q_h   = bf16_rne( rms( rms(sum_{b in P_g} mu_b) + sqrt(qvar) * z''' ) )
 * with g = h / (h_q / h_kv) the KV head of query head h and P_g the planted
 * blocks of that KV head.
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared -ffp-contract=off (see synth/__init__.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  TAG_TOPIC = 1,     /* mu_b of a block            */
  TAG_KEY_NOISE = 2, /* per-token key noise         */
  TAG_VALUE = 3,     /* per-token value             */
  TAG_QUERY = 4,     /* per-(query token, head) noise */
  TAG_PLANT = 5,     /* planted block draws         */
  TAG_PERM = 6       /* block-table permutation     */
};

/* ---- Philox4x32-10 (Salmon et al. SC'11) ------------------------------- */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u; /* Weyl key schedule */
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline double u01(uint32_t x) { return ((double)x + 0.5) * 0x1p-32; }

/* n standard normals (n % 4 == 0) for the row addressed by (tag, item, lh, session). */
static void normal_row(uint32_t seed, uint32_t tag, uint32_t item, uint32_t lh, uint32_t session,
                       int n, double* z) {
  const uint32_t key[2] = {seed, tag};
  for (int j = 0; j < n / 4; ++j) {
    const uint32_t ctr[4] = {(uint32_t)j, item, lh, session};
    uint32_t o[4];
    synth_philox4x32_10(ctr, key, o);
    const double r1 = sqrt(-2.0 * log(u01(o[0]))), a1 = 6.283185307179586 * u01(o[1]);
    const double r2 = sqrt(-2.0 * log(u01(o[2]))), a2 = 6.283185307179586 * u01(o[3]);
    z[4 * j + 0] = r1 * cos(a1);
    z[4 * j + 1] = r1 * sin(a1);
    z[4 * j + 2] = r2 * cos(a2);
    z[4 * j + 3] = r2 * sin(a2);
  }
}

/* bf16 with round-to-nearest-even, directly from fp64 (no fp32 double rounding). */
uint16_t synth_bf16_rne(double x) {
  if (x != x) return 0x7FC0;
  int e;
  (void)frexp(x, &e); /* |x| = m * 2^e, m in [0.5, 1) */
  int q = e - 8;      /* 8 significant bits */
  if (q < -133) q = -133; /* bf16 subnormal spacing */
  const double r = nearbyint(ldexp(x, -q)); /* default rounding mode: to nearest even */
  const float f = (float)ldexp(r, q);       /* exact: r fits in 8 bits */
  uint32_t b;
  memcpy(&b, &f, 4);
  return (uint16_t)(b >> 16);
}

static void rms_normalise(double* x, int d) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss / (double)d + 1e-6);
  for (int i = 0; i < d; ++i) x[i] *= inv;
}

static inline uint32_t lh_of(int layer, int head) { return ((uint32_t)layer << 16) | (uint32_t)head; }

/* mu_b = 0.5 * N(0, I) for the listed blocks: out[n][d] (fp64). */
void synth_topics(uint32_t seed, int session, int layer, int head, int d, const int64_t* blocks,
                  int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) {
    normal_row(seed, TAG_TOPIC, (uint32_t)blocks[i], lh_of(layer, head), (uint32_t)session, d,
               out + i * d);
    for (int k = 0; k < d; ++k) out[i * d + k] *= 0.5;
  }
}

/*
 * Keys and values of tokens [t0, t1) of one session and layer, KV heads
 * [h_lo, h_hi), written straight into a paged pool laid out
 * [n_pages][h_kv][32][d] (bf16 bits).
 * page_of_block[b] is the physical page of logical block b.
 */
int synth_kv_pages(uint32_t seed, int session, int layer, int h_kv, int d, int64_t t0, int64_t t1,
                   double eps_scale, const int32_t* page_of_block, int64_t n_pages, uint16_t* k_pool,
                   uint16_t* v_pool, int n_threads, int h_lo, int h_hi) {
  if (d % 4 != 0 || d > 1024 || t0 < 0 || t1 < t0 || h_lo < 0 || h_hi > h_kv || h_lo > h_hi) return 1;
  const int64_t b0 = t0 / 32, b1 = (t1 + 31) / 32;
  const int64_t nb = b1 - b0;
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 4) collapse(2) reduction(| : bad)
#endif
  for (int h = h_lo; h < h_hi; ++h) {
    for (int64_t bi = 0; bi < nb; ++bi) {
      double mu[1024], x[1024];
      const int64_t b = b0 + bi;
      const int64_t page = page_of_block[b];
      if (page < 0 || page >= n_pages) { bad = 1; continue; }
      normal_row(seed, TAG_TOPIC, (uint32_t)b, lh_of(layer, h), (uint32_t)session, d, mu);
      const int64_t ta = (b * 32 > t0) ? b * 32 : t0;
      const int64_t tb = (b * 32 + 32 < t1) ? b * 32 + 32 : t1;
      for (int64_t t = ta; t < tb; ++t) {
        uint16_t* krow = k_pool + (((int64_t)page * h_kv + h) * 32 + (t - b * 32)) * d;
        uint16_t* vrow = v_pool + (((int64_t)page * h_kv + h) * 32 + (t - b * 32)) * d;
        normal_row(seed, TAG_KEY_NOISE, (uint32_t)t, lh_of(layer, h), (uint32_t)session, d, x);
        for (int k = 0; k < d; ++k) x[k] = 0.5 * mu[k] + eps_scale * x[k];
        rms_normalise(x, d);
        for (int k = 0; k < d; ++k) krow[k] = synth_bf16_rne(x[k]);
        normal_row(seed, TAG_VALUE, (uint32_t)t, lh_of(layer, h), (uint32_t)session, d, x);
        for (int k = 0; k < d; ++k) vrow[k] = synth_bf16_rne(x[k]);
      }
    }
  }
  return bad ? 2 : 0;
}

/*
 * n_planted distinct blocks drawn uniformly from [lo, hi) for one KV head,
 * returned in ascending order.
 */
int synth_planted(uint32_t seed, int session, int layer, int head, int64_t lo, int64_t hi,
                  int n_planted, int64_t* out) {
  if (hi - lo < n_planted || n_planted < 0) return 1;
  const uint32_t key[2] = {seed, TAG_PLANT};
  int have = 0;
  for (uint32_t j = 0; have < n_planted; ++j) {
    const uint32_t ctr[4] = {j, 0u, lh_of(layer, head), (uint32_t)session};
    uint32_t o[4];
    synth_philox4x32_10(ctr, key, o);
    for (int w = 0; w < 4 && have < n_planted; ++w) {
      const int64_t c = lo + (int64_t)(((uint64_t)o[w] * (uint64_t)(hi - lo)) >> 32);
      int dup = 0;
      for (int i = 0; i < have; ++i) dup |= (out[i] == c);
      if (!dup) out[have++] = c;
    }
  }
  for (int i = 1; i < have; ++i) { /* insertion sort, n is small */
    int64_t v = out[i];
    int k = i - 1;
    while (k >= 0 && out[k] > v) { out[k + 1] = out[k]; --k; }
    out[k + 1] = v;
  }
  return 0;
}

/*
 * Queries for one session and layer: out[n_q][h_q][d] bf16 bits.
 * planted[h_kv][n_planted] are the planted blocks of each KV head.
 */
int synth_queries(uint32_t seed, int session, int layer, int h_q, int h_kv, int d, int n_q,
                  const int64_t* planted, int n_planted, double q_noise_var, uint16_t* out) {
  if (d % 4 != 0 || d > 1024 || h_kv <= 0 || h_q % h_kv != 0) return 1;
  const int group = h_q / h_kv;
  const double sd = sqrt(q_noise_var);
  for (int g = 0; g < h_kv; ++g) {
    double u[1024], mu[1024], w[1024];
    for (int k = 0; k < d; ++k) u[k] = 0.0;
    for (int i = 0; i < n_planted; ++i) {
      synth_topics(seed, session, layer, g, d, planted + (int64_t)g * n_planted + i, 1, mu);
      for (int k = 0; k < d; ++k) u[k] += mu[k];
    }
    rms_normalise(u, d);
    for (int t = 0; t < n_q; ++t) {
      for (int hh = 0; hh < group; ++hh) {
        const int h = g * group + hh;
        normal_row(seed, TAG_QUERY, (uint32_t)t, lh_of(layer, h), (uint32_t)session, d, w);
        for (int k = 0; k < d; ++k) w[k] = u[k] + sd * w[k];
        rms_normalise(w, d);
        uint16_t* row = out + ((int64_t)t * h_q + h) * d;
        for (int k = 0; k < d; ++k) row[k] = synth_bf16_rne(w[k]);
      }
    }
  }
  return 0;
}

/* Uniform random permutation of [0, n) (Fisher-Yates), keyed by (seed, stream). */
int synth_permutation(uint32_t seed, uint32_t stream, int64_t n, int32_t* out) {
  if (n < 0 || n > 0x7FFFFFFF) return 1;
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  const uint32_t key[2] = {seed, TAG_PERM};
  for (int64_t i = n - 1; i > 0; --i) {
    const uint32_t ctr[4] = {(uint32_t)i, 0u, 0u, stream};
    uint32_t o[4];
    synth_philox4x32_10(ctr, key, o);
    const int64_t j = (int64_t)(((uint64_t)o[0] * (uint64_t)(i + 1)) >> 32);
    const int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
  return 0;
}
