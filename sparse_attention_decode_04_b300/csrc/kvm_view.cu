// Steps 3 and 4 — materialise the execution view (gather + re-RoPE) and
// single-token decode attention over it, separately or fused.
//
// KVMEM reproduction README, "Core equation": the selected KV is concatenated
// within the block budget; the address space and the execution window stay
// apart.  Evolve review of KVMem, "Summary" and "Scope & Claims": selected
// blocks are restored with position-consistent re-RoPE into a bounded view.
// KVMEM reproduction README, "Local reproduction": the view replaces full
// attention; "2026-09-08 validation correction": RoPE is applied to the query.
//
// Design (one kernel, three modes):
//   mode 0  materialise: pages -> rotated K view + copied V view
//   mode 1  attend:      view  -> attention partials
//   mode 2  fused:       pages -> views + attention partials (each page read once)
// The work is the flat list of kept blocks over (session, KV head); a
// persistent grid of P CTAs (one per SM) takes contiguous equal shares of it,
// so every SM streams the same number of pages.  Warp-specialised CTA:
//   producer warp  - resolves kept id -> page through the block table (32 blocks
//                    at a time, one per lane), then lane 0 issues 1-D bulk copies
//                    (K page + V page) into an NSTAGE-deep shared-memory ring,
//                    each stage completing on its own mbarrier;
//   consumer warps - CP = d/16 warps; warp w owns 32/CP tokens of each page and
//                    each token is split over CP lanes (dims [8c, 8c+8) and
//                    [d/2+8c, d/2+8c+8): the rotate-half pairs).  They rotate K
//                    at view position 32*i + r (cos/sin composed from a per-slot
//                    base table and a per-offset table, both filled in fp64),
//                    round to bf16 and store; copy V; dot the rounded keys with
//                    the rotated query (fp32, log2 domain); keep a per-warp
//                    online softmax; accumulate V (lane owns d/32 dims).
// At a segment boundary (new session/KV head) or the end of its share, the CTA
// merges its warps' states and writes one partial record (m, l, acc[d]) per
// query head at index cta + segment, which is unique.  A combine kernel merges
// the records of each (session, query head) with the log-sum-exp rule.
// Every mbarrier wait is bounded; a timeout sets KVM_DEV_TIMEOUT, the CTA
// drains its copies in flight and returns.
#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct ViewParams {
  const uint16_t* k_src;
  const uint16_t* v_src;
  int64_t n_pages;
  const int32_t* bt;
  int64_t max_blocks;
  const int32_t* kept;
  const uint16_t* q;
  uint16_t* k_view;
  uint16_t* v_view;
  int32_t* view_len;
  float* rec;
  const float2* rope_base;  // [budget + 1][d/2]
  const float2* rope_off;   // [32][d/2]
  const float4* rope_base_hl;  // hi/lo copies, read only on the cancellation fallback
  const float4* rope_off_hl;
  float* out;
  uint32_t* status;
  int64_t total;  // kept blocks over all (session, KV head)
  int budget;
  int h_kv;
  int h_q;
  int n_sessions;
  int P;  // CTAs
  float q_scale;  // log2(e) / sqrt(d)
};

template <int D>
struct Geo {
  static constexpr int CP = D / 16;       // lanes per token (chunk pairs)
  static constexpr int NCW = CP;          // consumer warps
  static constexpr int TPW = 32 / CP;     // tokens per consumer warp
  static constexpr int NCT = NCW * 32;    // consumer threads
  static constexpr int NT = NCT + 32;     // + producer warp
  static constexpr int PVD = D / 32;      // dims per lane in P.V
  static constexpr int NSTAGE = 8;
  static constexpr uint32_t PAGE = 32u * D * 2u;  // bytes of one K (or V) page
};

__device__ __forceinline__ int64_t cta_begin(int c, int64_t total, int P) { return (int64_t)c * total / P; }
// CTA whose share contains flat block f (shares are [floor(cT/P), floor((c+1)T/P))).
__device__ __forceinline__ int cta_of(int64_t f, int64_t total, int P) {
  return (int)(((f + 1) * (int64_t)P - 1) / total);
}

// Position of flat block f: session, KV head, index within the head's kept list.
struct Cursor {
  int s, g, i;
};
__device__ __forceinline__ Cursor locate(int64_t f, const SessionArgs& a, int n_sessions, int h_kv) {
  int s = 0;
  while (s + 1 < n_sessions && a.seg_base[s + 1] <= f) ++s;
  const int64_t local = f - a.seg_base[s];
  const int nk = a.n_keep[s];
  return Cursor{s, (int)(local / nk), (int)(local % nk)};
}
__device__ __forceinline__ void advance(Cursor& c, const SessionArgs& a, int n_sessions, int h_kv) {
  if (c.s >= n_sessions) return;
  if (++c.i < a.n_keep[c.s]) return;
  c.i = 0;
  if (++c.g < h_kv) return;
  c.g = 0;
  do {
    ++c.s;
  } while (c.s < n_sessions && a.n_keep[c.s] == 0);
}

// Tokens of kept block `id` present in session s's history.
__device__ __forceinline__ int block_tokens(int64_t id, const SessionArgs& a, int s) {
  const int tail = (int)(a.n_tok[s] & 31);
  return (id == a.n_blk[s] - 1 && tail) ? tail : 32;
}

// Float-float (unevaluated hi + lo) arithmetic, Dekker / Knuth error-free transformations.
struct ff {
  float h, l;
};
__device__ __forceinline__ ff two_prod(float a, float b) {
  const float p = a * b;
  return ff{p, fmaf(a, b, -p)};
}
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b, bb = s - a;
  return ff{s, (a - (s - bb)) + (b - bb)};
}
// x*y - u*v for hi/lo operands, to ~2^-44 of the operand magnitudes.
__device__ __forceinline__ ff ff_dot2(ff x, ff y, ff u, ff v) {
  const ff p = two_prod(x.h, y.h), q = two_prod(u.h, v.h);
  const ff s = two_sum(p.h, -q.h);
  const float lo = s.l + (p.l - q.l) + (fmaf(x.h, y.l, x.l * y.h) - fmaf(u.h, v.l, u.l * v.h));
  return two_sum(s.h, lo);
}
// Rotation of one (x1, x2) pair by the angle whose cos/sin are composed from the hi/lo base and offset
// tables; the result hi + lo is within ~2^-44 (|x1| + |x2|) of the exact rotation.
__device__ __forceinline__ void rotate_exact(float x1, float x2, float4 b, float4 o, float& y1, float& y2) {
  const ff cb{b.x, b.y}, sb{b.z, b.w}, co{o.x, o.y}, so{o.z, o.w};
  const ff c = ff_dot2(cb, co, sb, so);                 // cos(A + B)
  const ff s = ff_dot2(sb, co, ff{-cb.h, -cb.l}, so);   // sin(A + B) = sb co + cb so
  const ff r1 = ff_dot2(ff{x1, 0.f}, c, ff{x2, 0.f}, s);
  const ff r2 = ff_dot2(ff{x2, 0.f}, c, ff{-x1, 0.f}, s);
  y1 = r1.h + r1.l;
  y2 = r2.h + r2.l;
}

__device__ __forceinline__ void rope_cs(const float2 b, const float2 o, float& c, float& s) {
  // cos/sin of (base + offset) angle from cos/sin of each (angle addition)
  c = fmaf(b.x, o.x, -b.y * o.y);
  s = fmaf(b.y, o.x, b.x * o.y);
}

template <int D, int G, int MODE>
__global__ void __launch_bounds__(Geo<D>::NT, 1) view_kernel(const ViewParams vp, const SessionArgs a) {
  using Q = Geo<D>;
  constexpr int CP = Q::CP, NCW = Q::NCW, TPW = Q::TPW, NCT = Q::NCT, PVD = Q::PVD, NS = Q::NSTAGE;
  constexpr bool kWrite = MODE != 1;  // writes the view
  constexpr bool kAttend = MODE != 0;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint16_t* kbuf = reinterpret_cast<uint16_t*>(smem_raw);         // [NS][32][D]
  uint16_t* vbuf = kbuf + NS * 32 * D;                            // [NS][32][D]
  float* mscr = reinterpret_cast<float*>(vbuf + NS * 32 * D);     // [NCW][G][2 + D]
  float* pbuf = mscr + NCW * G * (2 + D);                         // [NCW][TPW][8]
  __shared__ __align__(8) uint64_t full_bar[NS];
  __shared__ __align__(8) uint64_t empty_bar[NS];
  __shared__ int meta[NS];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t fa = cta_begin(c, vp.total, vp.P), fb = cta_begin(c + 1, vp.total, vp.P);
  if (fa >= fb) return;

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NCW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer warp
    Cursor cur = locate(fa, a, vp.n_sessions, vp.h_kv);
    int64_t k = 0;
    int prev_id = -1;
    for (int64_t f0 = fa; f0 < fb; f0 += 32) {
      // lane j resolves flat block f0 + j
      Cursor cj = cur;
      if (f0 + lane < fb)
        for (int j = 0; j < lane; ++j) advance(cj, a, vp.n_sessions, vp.h_kv);
      int valid = 0;
      int64_t src_off = 0;
      int id = -1;
      if (f0 + lane < fb) {
        const int q = cj.s * vp.h_kv + cj.g;
        if (MODE == 1) {
          const int L = min(vp.view_len[q], 32 * vp.budget);
          valid = max(0, min(32, L - 32 * cj.i));
          src_off = ((int64_t)q * vp.budget * 32 + (int64_t)cj.i * 32) * D;
        } else {
          id = vp.kept[(int64_t)q * vp.budget + cj.i];
          if (id >= 0 && id < a.n_blk[cj.s]) {
            const int32_t page = vp.bt[(int64_t)cj.s * vp.max_blocks + id];
            if (page >= 0 && page < vp.n_pages) {
              valid = block_tokens(id, a, cj.s);
              src_off = (((int64_t)page * vp.h_kv + cj.g) * 32) * D;
            } else {
              atomicOr(vp.status, KVM_DEV_BAD_PAGE);
            }
          } else {
            atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
          }
        }
      }
      const int nb = (int)(fb - f0 < 32 ? fb - f0 : 32);
      for (int j = 0; j < nb; ++j) {
        int vj = __shfl_sync(0xffffffffu, valid, j);
        const int64_t oj = __shfl_sync(0xffffffffu, src_off, j);
        const int idj = __shfl_sync(0xffffffffu, id, j);
        const int ij = __shfl_sync(0xffffffffu, cj.i, j);
        if (MODE != 1 && vj > 0) {  // kept ids must ascend within a list
          if (ij > 0 && idj <= prev_id) {
            vj = 0;
            if (lane == 0) atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
          }
        }
        if (MODE != 1) prev_id = vj > 0 ? idj : prev_id;
        if (lane == 0) {
          const int st = (int)(k % NS);
          bool ok = true;
          if (k >= NS) ok = mbar_wait(&empty_bar[st], (uint32_t)((k / NS - 1) & 1), vp.status);
          if (!ok || abort_flag) {
            abort_flag = 1;
          } else {
            meta[st] = vj;
            if (vj > 0) {
              mbar_arrive_expect_tx(&full_bar[st], 2 * Q::PAGE);
              bulk_g2s(kbuf + st * 32 * D, vp.k_src + oj, Q::PAGE, &full_bar[st]);
              bulk_g2s(vbuf + st * 32 * D, vp.v_src + oj, Q::PAGE, &full_bar[st]);
            } else {
              mbar_arrive(&full_bar[st]);
            }
          }
        }
        ++k;
        if (__shfl_sync(0xffffffffu, (int)abort_flag, 0)) break;
      }
      if (__shfl_sync(0xffffffffu, (int)abort_flag, 0)) break;
      // the warp advances its cursor by 32 blocks
      for (int j = 0; j < nb; ++j) advance(cur, a, vp.n_sessions, vp.h_kv);
    }
    if (lane == 0 && abort_flag) {
      // drain: the last phase issued on each stage may still have copies in flight
      const int64_t k_issued = k;
      for (int64_t j = (k_issued > NS ? k_issued - NS : (int64_t)0); j < k_issued; ++j)
        mbar_wait(&full_bar[j % NS], (uint32_t)((j / NS) & 1), vp.status);
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    const int tw = lane / CP;             // token within the warp
    const int cp = lane % CP;             // chunk pair
    const int r = warp * TPW + tw;        // token row within the page
    float2 off[8];                        // cos/sin of r * theta_i for this lane's 8 frequencies
#pragma unroll
    for (int u = 0; u < 8; ++u) off[u] = vp.rope_off[r * (D / 2) + 8 * cp + u];

    float qr[G][16];  // rotated, scaled query slice: [0..8) first half, [8..16) second half
    float m[G], lsum[G], acc[G][PVD];
    Cursor cur = locate(fa, a, vp.n_sessions, vp.h_kv);
    int seg_q = -1;
    const int64_t n = fb - fa;

    auto flush = [&](int q) {
      // per-warp l: sum over the warp's tokens
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float l = lsum[hh];
#pragma unroll
        for (int o = CP; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        float* w = mscr + (warp * G + hh) * (2 + D);
        if (lane == 0) {
          w[0] = m[hh];
          w[1] = l;
        }
#pragma unroll
        for (int d = 0; d < PVD; ++d) w[2 + lane * PVD + d] = acc[hh][d];
      }
      named_sync(1, NCT);
      float* rec = vp.rec + (int64_t)(c + q) * G * (2 + D);
      for (int idx = tid; idx < G * D; idx += NCT) {
        const int hh = idx / D, dim = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, mscr[(w * G + hh) * (2 + D)]);
        float av = 0.f, lv = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < NCW; ++w) {
            const float* ws = mscr + (w * G + hh) * (2 + D);
            const float sc = fast_exp2(ws[0] - M);
            av = fmaf(ws[2 + dim], sc, av);
            lv = fmaf(ws[1], sc, lv);
          }
        }
        rec[hh * (2 + D) + 2 + dim] = av;
        if (dim == 0) {
          rec[hh * (2 + D)] = M;
          rec[hh * (2 + D) + 1] = lv;
        }
      }
      named_sync(1, NCT);
    };

    auto begin_segment = [&](const Cursor& cs) {
      const int q = cs.s * vp.h_kv + cs.g;
      const int nk = a.n_keep[cs.s];
      int L;
      if (MODE == 1) {
        L = vp.view_len[q];
        if (L < 0 || L > 32 * vp.budget) {  // caller-supplied: clamp so the RoPE table read stays in range
          if (tid == 0) atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
          L = L < 0 ? 0 : 32 * vp.budget;
        }
      } else {
        const int last = vp.kept[(int64_t)q * vp.budget + nk - 1];
        L = 32 * (nk - 1) + ((last >= 0 && last < a.n_blk[cs.s]) ? block_tokens(last, a, cs.s) : 32);
        if (cs.i == 0 && tid == 0) vp.view_len[q] = L;
      }
      if (kAttend) {
        // RoPE(q, L): cos/sin of L*theta_i composed from slot L/32 and offset L%32
        const float2* bb = vp.rope_base + (int64_t)(L >> 5) * (D / 2) + 8 * cp;
        const float2* oo = vp.rope_off + (L & 31) * (D / 2) + 8 * cp;
        float cs_[8], sn_[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rope_cs(bb[u], oo[u], cs_[u], sn_[u]);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const uint16_t* qh = vp.q + ((int64_t)cs.s * vp.h_q + cs.g * G + hh) * D;
          const uint4 w1 = *reinterpret_cast<const uint4*>(qh + 8 * cp);
          const uint4 w2 = *reinterpret_cast<const uint4*>(qh + D / 2 + 8 * cp);
          const uint32_t a1[4] = {w1.x, w1.y, w1.z, w1.w}, a2[4] = {w2.x, w2.y, w2.z, w2.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int v = 2 * u + e;
              const float x1 = e ? bf16hi(a1[u]) : bf16lo(a1[u]);
              const float x2 = e ? bf16hi(a2[u]) : bf16lo(a2[u]);
              qr[hh][v] = (x1 * cs_[v] - x2 * sn_[v]) * vp.q_scale;
              qr[hh][8 + v] = (x2 * cs_[v] + x1 * sn_[v]) * vp.q_scale;
            }
          }
          m[hh] = -INFINITY;
          lsum[hh] = 0.f;
#pragma unroll
          for (int d = 0; d < PVD; ++d) acc[hh][d] = 0.f;
        }
      }
      return q;
    };

    bool aborted = false;
    for (int64_t k = 0; k < n; ++k) {
      const int st = (int)(k % NS);
      const bool ok = mbar_wait(&full_bar[st], (uint32_t)((k / NS) & 1), vp.status);
      int bad;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(bad)
          : "r"((uint32_t)ok), "r"(NCT)
          : "memory");
      if (bad) {
        aborted = true;
        abort_flag = 1;
        break;
      }
      if (cur.i == 0 || seg_q < 0) {
        if (kAttend && seg_q >= 0) flush(seg_q);  // a share with only skipped blocks leaves a neutral record
        seg_q = begin_segment(cur);
      }
      const int valid = meta[st];
      if (valid > 0) {
        const uint16_t* kp = kbuf + st * 32 * D + r * D;
        const uint16_t* vpg = vbuf + st * 32 * D + r * D;
        const uint4 k1 = *reinterpret_cast<const uint4*>(kp + 8 * cp);
        const uint4 k2 = *reinterpret_cast<const uint4*>(kp + D / 2 + 8 * cp);
        float y1[8], y2[8];
        const uint32_t ka[4] = {k1.x, k1.y, k1.z, k1.w}, kb[4] = {k2.x, k2.y, k2.z, k2.w};
        if (kWrite) {
          const int64_t j = (int64_t)cur.i * 32 + r;  // view position
          const float2* bb = vp.rope_base + (int64_t)cur.i * (D / 2) + 8 * cp;
          uint32_t o1[4], o2[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float f1[2], f2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int v = 2 * u + e;
              float cs_, sn_;
              rope_cs(bb[v], off[v], cs_, sn_);
              const float x1 = e ? bf16hi(ka[u]) : bf16lo(ka[u]);
              const float x2 = e ? bf16hi(kb[u]) : bf16lo(kb[u]);
              f1[e] = fmaf(x1, cs_, -x2 * sn_);
              f2[e] = fmaf(x2, cs_, x1 * sn_);
              // fp32 tables put |error| <= 3e-7 (|x1| + |x2|) on f; that stays below one bf16 ulp of the
              // result unless the rotation cancels (|f| < ~8e-5 (|x1| + |x2|)).  Those pairs are redone in
              // float-float from hi/lo tables, so the stored key is always within one ulp of the exact rotation.
              const float tau = 0x1p-12f * (fabsf(x1) + fabsf(x2));
              if (fminf(fabsf(f1[e]), fabsf(f2[e])) < tau) {
                rotate_exact(x1, x2, vp.rope_base_hl[(int64_t)cur.i * (D / 2) + 8 * cp + v],
                             vp.rope_off_hl[r * (D / 2) + 8 * cp + v], f1[e], f2[e]);
              }
            }
            o1[u] = pack_bf16x2(f1[0], f1[1]);
            o2[u] = pack_bf16x2(f2[0], f2[1]);
            y1[2 * u] = bf16lo(o1[u]);
            y1[2 * u + 1] = bf16hi(o1[u]);
            y2[2 * u] = bf16lo(o2[u]);
            y2[2 * u + 1] = bf16hi(o2[u]);
          }
          if (r < valid) {
            const int q = seg_q;
            uint16_t* kd = vp.k_view + ((int64_t)q * vp.budget * 32 + j) * D;
            uint16_t* vd = vp.v_view + ((int64_t)q * vp.budget * 32 + j) * D;
            *reinterpret_cast<uint4*>(kd + 8 * cp) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            *reinterpret_cast<uint4*>(kd + D / 2 + 8 * cp) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
            *reinterpret_cast<uint4*>(vd + 8 * cp) = *reinterpret_cast<const uint4*>(vpg + 8 * cp);
            *reinterpret_cast<uint4*>(vd + D / 2 + 8 * cp) = *reinterpret_cast<const uint4*>(vpg + D / 2 + 8 * cp);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            y1[2 * u] = bf16lo(ka[u]);
            y1[2 * u + 1] = bf16hi(ka[u]);
            y2[2 * u] = bf16lo(kb[u]);
            y2[2 * u + 1] = bf16hi(kb[u]);
          }
        }
        if (kAttend) {
          float sc[G];
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float d0 = 0.f;
#pragma unroll
            for (int v = 0; v < 8; ++v) d0 = fmaf(qr[hh][v], y1[v], d0);
#pragma unroll
            for (int v = 0; v < 8; ++v) d0 = fmaf(qr[hh][8 + v], y2[v], d0);
#pragma unroll
            for (int o = 1; o < CP; o <<= 1) d0 += __shfl_xor_sync(0xffffffffu, d0, o);
            sc[hh] = r < valid ? d0 : -INFINITY;
          }
          float* pw = pbuf + warp * TPW * 8;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float bm = sc[hh];
#pragma unroll
            for (int o = CP; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            const float mn = fmaxf(m[hh], bm);
            float corr = 1.f, p = 0.f;
            if (mn != -INFINITY) {
              corr = fast_exp2(m[hh] - mn);  // 0 when m was -inf
              p = fast_exp2(sc[hh] - mn);    // 0 for rows past `valid`
            }
            m[hh] = mn;
            lsum[hh] = fmaf(lsum[hh], corr, p);
#pragma unroll
            for (int d = 0; d < PVD; ++d) acc[hh][d] *= corr;
            if (cp == 0) pw[tw * 8 + hh] = p;
          }
          __syncwarp();
          // P.V over the warp's tokens: lane owns dims [PVD*lane, PVD*lane + PVD)
#pragma unroll
          for (int t = 0; t < TPW; ++t) {
            if (warp * TPW + t >= valid) break;  // rows past the tail may hold any bits
            const uint16_t* vrow = vbuf + st * 32 * D + (warp * TPW + t) * D + PVD * lane;
            float vv[PVD];
            if constexpr (PVD == 4) {
              const uint2 w = *reinterpret_cast<const uint2*>(vrow);
              vv[0] = bf16lo(w.x);
              vv[1] = bf16hi(w.x);
              vv[2] = bf16lo(w.y);
              vv[3] = bf16hi(w.y);
            } else {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
              vv[0] = bf16lo(w);
              vv[1] = bf16hi(w);
            }
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              const float p = pw[t * 8 + hh];
#pragma unroll
              for (int d = 0; d < PVD; ++d) acc[hh][d] = fmaf(p, vv[d], acc[hh][d]);
            }
          }
          __syncwarp();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
      advance(cur, a, vp.n_sessions, vp.h_kv);
    }
    if (!aborted && kAttend && seg_q >= 0) flush(seg_q);
  }
  __syncthreads();
}

// Merges the partial records of each (session, query head) and writes out;
// also writes view_len = 0 for empty kept lists.
template <int D, int G>
__global__ void combine_kernel(const ViewParams vp, const SessionArgs a, int attend) {
  const int s = blockIdx.x / vp.h_q, h = blockIdx.x % vp.h_q;
  const int g = h / G, hh = h % G;
  const int q = s * vp.h_kv + g;
  const int nk = a.n_keep[s];
  if (nk == 0) {
    if (attend)
      for (int dim = threadIdx.x; dim < D; dim += blockDim.x) vp.out[((int64_t)s * vp.h_q + h) * D + dim] = 0.f;
    if (hh == 0 && threadIdx.x == 0 && vp.view_len) vp.view_len[q] = 0;
    return;
  }
  if (!attend) return;
  const int64_t start = a.seg_base[s] + (int64_t)g * nk, end = start + nk - 1;
  const int c0 = cta_of(start, vp.total, vp.P), c1 = cta_of(end, vp.total, vp.P);
  // CTAs between c0 and c1 with an empty share wrote no record: skip them
  auto empty = [&](int c) { return cta_begin(c, vp.total, vp.P) >= cta_begin(c + 1, vp.total, vp.P); };
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c)
    if (!empty(c)) M = fmaxf(M, vp.rec[((int64_t)(c + q) * G + hh) * (2 + D)]);
  for (int dim = threadIdx.x; dim < D; dim += blockDim.x) {
    float av = 0.f, lv = 0.f;
    if (M != -INFINITY) {
      for (int c = c0; c <= c1; ++c) {
        if (empty(c)) continue;
        const float* rc = vp.rec + ((int64_t)(c + q) * G + hh) * (2 + D);
        const float sc = exp2f(rc[0] - M);
        av = fmaf(rc[2 + dim], sc, av);
        lv = fmaf(rc[1], sc, lv);
      }
    }
    vp.out[((int64_t)s * vp.h_q + h) * D + dim] = lv > 0.f ? av / lv : 0.f;
  }
}

template <int D, int G>
cudaError_t launch_dg(const Ctx& c, int mode, const ViewParams& vp, const SessionArgs& a, cudaStream_t st) {
  using Q = Geo<D>;
  const size_t smem = (size_t)Q::NSTAGE * 2 * Q::PAGE + (size_t)Q::NCW * G * (2 + D) * 4 +
                      (size_t)Q::NCW * Q::TPW * 8 * 4;
  cudaError_t e = cudaSuccess;
  if (vp.total > 0) {
    void (*kern)(const ViewParams, const SessionArgs) =
        mode == 0 ? view_kernel<D, G, 0> : (mode == 1 ? view_kernel<D, G, 1> : view_kernel<D, G, 2>);
    if ((e = ensure_smem(kern, c.device, smem)) != cudaSuccess) return e;
    kern<<<vp.P, Q::NT, smem, st>>>(vp, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  combine_kernel<D, G><<<vp.n_sessions * vp.h_q, D, 0, st>>>(vp, a, mode != 0);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Ctx& c, int mode, const ViewParams& vp, const SessionArgs& a, cudaStream_t st) {
  switch (c.group) {
    case 1: return launch_dg<D, 1>(c, mode, vp, a, st);
    case 2: return launch_dg<D, 2>(c, mode, vp, a, st);
    case 3: return launch_dg<D, 3>(c, mode, vp, a, st);
    case 4: return launch_dg<D, 4>(c, mode, vp, a, st);
    case 5: return launch_dg<D, 5>(c, mode, vp, a, st);
    case 6: return launch_dg<D, 6>(c, mode, vp, a, st);
    case 7: return launch_dg<D, 7>(c, mode, vp, a, st);
    case 8: return launch_dg<D, 8>(c, mode, vp, a, st);
  }
  return cudaErrorInvalidValue;
}

// RoPE tables computed in fp64: base[slot][i] = (cos, sin)(32*slot*theta_i), off[r][i] = (cos, sin)(r*theta_i),
// theta_i = rope_theta^(-2i/d); stored as fp32 and as fp32 hi/lo pairs (value = hi + lo to ~2^-48).
__device__ __forceinline__ float4 hilo(double c, double s) {
  const float ch = (float)c, sh = (float)s;
  return make_float4(ch, (float)(c - (double)ch), sh, (float)(s - (double)sh));
}
__global__ void rope_table_kernel(float2* base, int n_slots, float2* off, float4* base_hl, float4* off_hl, int d,
                                  double rope_theta) {
  const int half = d / 2;
  const int64_t n = (int64_t)(n_slots + 32) * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = idx / half;
    const int i = (int)(idx % half);
    const double inv_freq = pow(rope_theta, -2.0 * i / d);
    double sn, cs;
    if (row < n_slots) {
      sincos(32.0 * (double)row * inv_freq, &sn, &cs);
      base[row * half + i] = make_float2((float)cs, (float)sn);
      base_hl[row * half + i] = hilo(cs, sn);
    } else {
      sincos((double)(row - n_slots) * inv_freq, &sn, &cs);
      off[(row - n_slots) * half + i] = make_float2((float)cs, (float)sn);
      off_hl[(row - n_slots) * half + i] = hilo(cs, sn);
    }
  }
}

}  // namespace

cudaError_t launch_view(const Ctx& c, int mode, const uint16_t* k_src, const uint16_t* v_src, int64_t n_pages,
                        const int32_t* bt, int n_sessions, const SessionArgs& a, const int32_t* kept,
                        const uint16_t* q, uint16_t* k_view, uint16_t* v_view, int32_t* view_len, float* out,
                        cudaStream_t st) {
  ViewParams vp;
  vp.k_src = k_src;
  vp.v_src = v_src;
  vp.n_pages = n_pages;
  vp.bt = bt;
  vp.max_blocks = c.p.max_blocks;
  vp.kept = kept;
  vp.q = q;
  vp.k_view = k_view;
  vp.v_view = v_view;
  vp.view_len = view_len;
  vp.rec = c.rec;
  vp.rope_base = reinterpret_cast<const float2*>(c.rope_base);
  vp.rope_off = reinterpret_cast<const float2*>(c.rope_off);
  vp.rope_base_hl = c.rope_base_hl;
  vp.rope_off_hl = c.rope_off_hl;
  vp.out = out;
  vp.status = c.status;
  vp.total = a.seg_base[n_sessions];
  vp.budget = c.budget;
  vp.h_kv = c.p.h_kv;
  vp.h_q = c.p.h_q;
  vp.n_sessions = n_sessions;
  vp.P = c.view_ctas;
  vp.q_scale = (float)(1.4426950408889634 / sqrt((double)c.p.d));
  return c.p.d == 128 ? launch_d<128>(c, mode, vp, a, st) : launch_d<64>(c, mode, vp, a, st);
}

cudaError_t launch_rope_tables(const Ctx& c, cudaStream_t st) {
  rope_table_kernel<<<256, 256, 0, st>>>(reinterpret_cast<float2*>(c.rope_base), c.budget + 1,
                                         reinterpret_cast<float2*>(c.rope_off),
                                         c.rope_base_hl, c.rope_off_hl, c.p.d, (double)c.p.rope_theta);
  return cudaGetLastError();
}

}  // namespace kvm
