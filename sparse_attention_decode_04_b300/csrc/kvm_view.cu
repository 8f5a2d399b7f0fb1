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
// One kernel, three modes:
//   mode 0  materialise: pages -> rotated K view + copied V view
//   mode 1  attend:      view  -> attention partials
//   mode 2  fused:       pages -> views + attention partials (each page read once)
// Work: the flat list of kept blocks over (session, KV head).  A persistent grid
// of one CTA per SM takes equal contiguous shares, so every SM streams the same
// number of pages.  Inside a CTA, eight warps each own one shared-memory stage
// (a K page and a V page) and take every eighth block of the share; warps never
// wait on one another.  Per block, a warp:
//   - receives the K and V pages by TMA tiled loads (64-column boxes) with the
//     128-byte swizzle, so the ldmatrix reads below are free of bank conflicts;
//   - rotates K in place at view positions 32*i + r (cos/sin composed in fp32
//     from a per-slot and a per-offset table, both filled in fp64; pairs whose
//     rotation cancels are redone in float-float), rounds to bf16, and writes
//     the rotated K and the untouched V to the view with TMA tiled stores;
//   - computes the scores with mma.sync (m16n8k16, bf16 -> fp32): A rows 0..7
//     hold the rotated, scaled query heads rounded to bf16 and rows 8..15 their
//     bf16 residuals, so one MMA gives both halves and their sum is an
//     fp32-accurate score;
//   - keeps an online softmax per head in the log2 domain (the running maximum
//     is raised only when it grows by more than 8, so rescaling is rare);
//   - accumulates P.V with mma.sync, P split the same way into bf16 + residual.
// The next block's K page is fetched as soon as the scores are done, its V page
// as soon as P.V is done, so the copies overlap the rest of the block's work.
// Each warp writes one partial record (max, sum, output) per segment (session,
// KV head) of its CTA's share — a neutral record for a segment it had no block
// of — at index ((cta + segment) * 8 + warp), which is unique.  The combine
// kernel merges the records of each (session, query head).
// Every mbarrier wait is bounded; a timeout sets KVM_DEV_TIMEOUT and the warp
// drains its copies and stops.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr int kWarps = kViewWarps;

struct ViewParams {
  const int32_t* bt;
  int64_t max_blocks;
  int64_t n_pages;
  const int32_t* kept;
  const uint16_t* q;
  uint16_t* k_view;
  uint16_t* v_view;
  int32_t* view_len;
  float* rec;
  const float2* rope_base;     // [budget + 1][d/2]
  const float2* rope_off;      // [32][d/2]
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
  static constexpr int BOXES = D / 64;          // 64-column (128-byte) boxes per page row
  static constexpr uint32_t BOX = 32 * 128;     // bytes of one box (32 rows)
  static constexpr uint32_t PAGE = 32 * D * 2;  // bytes of one K (or V) page
  static constexpr int CPR = D / 16;            // rotation items (chunk pairs) per row
  static constexpr int RPP = 32 / CPR;          // rows per rotation pass
  static constexpr int PASSES = CPR;            // rotation passes per page
  static constexpr int KS = D / 16;             // MMA k-steps over the head dimension
  static constexpr int NO = D / 8;              // output n-tiles
};

__device__ __forceinline__ int64_t cta_begin(int c, int64_t total, int P) { return (int64_t)c * total / P; }
// CTA whose share contains flat block f (shares are [floor(cT/P), floor((c+1)T/P))).
__device__ __forceinline__ int cta_of(int64_t f, int64_t total, int P) {
  return (int)(((f + 1) * (int64_t)P - 1) / total);
}

struct Cursor {
  int s, g, i;
};
__device__ __forceinline__ Cursor locate(int64_t f, const SessionArgs& a, int n_sessions) {
  int s = 0;
  while (s + 1 < n_sessions && a.seg_base[s + 1] <= f) ++s;
  const int64_t local = f - a.seg_base[s];
  const int nk = a.n_keep[s];
  return Cursor{s, (int)(local / nk), (int)(local % nk)};
}

// Tokens of kept block `id` present in session s's history.
__device__ __forceinline__ int block_tokens(int64_t id, const SessionArgs& a, int s) {
  const int tail = (int)(a.n_tok[s] & 31);
  return (id == a.n_blk[s] - 1 && tail) ? tail : 32;
}

// Byte offset of logical 16-byte chunk k of row r inside a 128-byte-swizzled page.
__device__ __forceinline__ uint32_t chunk_off(int r, int k) {
  return (uint32_t)((k >> 3) * (32 * 128) + r * 128 + (((k & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void rope_cs(const float2 b, const float c, const float s, float& co, float& sn) {
  // cos/sin of (base + offset) from cos/sin of each (angle addition)
  co = fmaf(b.x, c, -b.y * s);
  sn = fmaf(b.y, c, b.x * s);
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
// Rotation of (x1, x2) by the angle whose cos/sin are composed from hi/lo base and offset tables;
// the result is within ~2^-44 (|x1| + |x2|) of the exact rotation.
__device__ __forceinline__ void rotate_exact(float x1, float x2, float4 b, float4 o, float& y1, float& y2) {
  const ff cb{b.x, b.y}, sb{b.z, b.w}, co{o.x, o.y}, so{o.z, o.w};
  const ff c = ff_dot2(cb, co, sb, so);
  const ff s = ff_dot2(sb, co, ff{-cb.h, -cb.l}, so);
  const ff r1 = ff_dot2(ff{x1, 0.f}, c, ff{x2, 0.f}, s);
  const ff r2 = ff_dot2(ff{x2, 0.f}, c, ff{-x1, 0.f}, s);
  y1 = r1.h + r1.l;
  y2 = r2.h + r2.l;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// hi = bf16(x), lo = bf16(x - hi) for two values, each pair packed.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  lo = pack_bf16x2(x0 - bf16lo(hi), x1 - bf16hi(hi));
}

struct BlockMeta {
  int q;      // segment = s * h_kv + g
  int s;
  int i;      // index in the segment's kept list (view slot)
  int valid;  // tokens present (0: skipped)
  int ysrc;   // source tile row
};

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kWarps * 32, 1)
    view_kernel(const __grid_constant__ CUtensorMap tm_ksrc, const __grid_constant__ CUtensorMap tm_vsrc,
                const __grid_constant__ CUtensorMap tm_kdst, const __grid_constant__ CUtensorMap tm_vdst,
                const ViewParams vp, const SessionArgs a) {
  using Q = Geo<D>;
  constexpr bool kWrite = MODE != 1;
  constexpr bool kAttend = MODE != 0;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned stages: [warp][K page | V page]; then the offset table [32][4][CPR] float4
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  float4* off_s = reinterpret_cast<float4*>(smem + kWarps * 2 * Q::PAGE);
  __shared__ __align__(8) uint64_t full_k[kWarps], full_v[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t fa = cta_begin(c, vp.total, vp.P), fb = cta_begin(c + 1, vp.total, vp.P);
  if (fa >= fb) return;
  const int Lcap = 32 * vp.budget;

  if (kWrite) {
    for (int idx = tid; idx < 32 * 4 * Q::CPR; idx += kWarps * 32) {
      const int r = idx / (4 * Q::CPR), u = (idx / Q::CPR) % 4, cc = idx % Q::CPR;
      const float2 o0 = vp.rope_off[r * (D / 2) + 8 * cc + 2 * u];
      const float2 o1 = vp.rope_off[r * (D / 2) + 8 * cc + 2 * u + 1];
      off_s[idx] = make_float4(o0.x, o0.y, o1.x, o1.y);
    }
  }
  if (lane == 0) {
    mbar_init(&full_k[warp], 1);
    mbar_init(&full_v[warp], 1);
    mbar_fence_init();
  }
  __syncthreads();

  unsigned char* kbuf = smem + warp * 2 * Q::PAGE;
  unsigned char* vbuf = kbuf + Q::PAGE;
  const uint32_t kaddr = smem_addr(kbuf), vaddr = smem_addr(vbuf);
  const Cursor firstc = locate(fa, a, vp.n_sessions), lastc = locate(fb - 1, a, vp.n_sessions);
  const int seg_first = firstc.s * vp.h_kv + firstc.g;
  const int seg_last = lastc.s * vp.h_kv + lastc.g;

  // ------------------------------------------------------------ per-block metadata, 32 blocks at a time
  // lane l describes this warp's block number jb + l: flat index fa + warp + 8 * (jb + l)
  const int64_t nblk_w = (fb - fa - warp + kWarps - 1) / kWarps;  // blocks this warp processes (may be <= 0)
  auto resolve = [&](int64_t jb) -> BlockMeta {
    BlockMeta m{-1, 0, 0, 0, 0};
    const int64_t j = jb + lane;
    if (j >= nblk_w) return m;
    const int64_t f = fa + warp + (int64_t)kWarps * j;
    const Cursor cu = locate(f, a, vp.n_sessions);
    m.q = cu.s * vp.h_kv + cu.g;
    m.s = cu.s;
    m.i = cu.i;
    if (MODE == 1) {
      int L = vp.view_len[m.q];
      L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
      m.valid = max(0, min(32, L - 32 * cu.i));
      m.ysrc = m.q * Lcap + 32 * cu.i;
    } else {
      const int id = vp.kept[(int64_t)m.q * vp.budget + cu.i];
      const int prev = cu.i > 0 ? vp.kept[(int64_t)m.q * vp.budget + cu.i - 1] : -1;
      if (id >= 0 && id < a.n_blk[cu.s] && id > prev) {  // kept ids ascend within a list
        const int32_t page = vp.bt[(int64_t)cu.s * vp.max_blocks + id];
        if (page >= 0 && page < vp.n_pages) {
          m.valid = block_tokens(id, a, cu.s);
          m.ysrc = (int)(((int64_t)page * vp.h_kv + cu.g) * 32);
        } else {
          atomicOr(vp.status, KVM_DEV_BAD_PAGE);
        }
      } else {
        atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
      }
    }
    return m;
  };
  auto bcast = [&](const BlockMeta& m, int src) {
    BlockMeta r;
    r.q = __shfl_sync(0xffffffffu, m.q, src);
    r.s = __shfl_sync(0xffffffffu, m.s, src);
    r.i = __shfl_sync(0xffffffffu, m.i, src);
    r.valid = __shfl_sync(0xffffffffu, m.valid, src);
    r.ysrc = __shfl_sync(0xffffffffu, m.ysrc, src);
    return r;
  };
  auto issue_k = [&](const BlockMeta& m) {
    if (lane == 0) {
      if (m.valid > 0) {
        mbar_arrive_expect_tx(&full_k[warp], Q::PAGE);
#pragma unroll
        for (int b = 0; b < Q::BOXES; ++b) tma_load_2d(kbuf + b * Q::BOX, &tm_ksrc, 64 * b, m.ysrc, &full_k[warp]);
      } else {
        mbar_arrive(&full_k[warp]);
      }
    }
  };
  auto issue_v = [&](const BlockMeta& m) {
    if (lane == 0) {
      if (m.valid > 0) {
        mbar_arrive_expect_tx(&full_v[warp], Q::PAGE);
#pragma unroll
        for (int b = 0; b < Q::BOXES; ++b) tma_load_2d(vbuf + b * Q::BOX, &tm_vsrc, 64 * b, m.ysrc, &full_v[warp]);
      } else {
        mbar_arrive(&full_v[warp]);
      }
    }
  };

  // ------------------------------------------------------------ attention state of this warp
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group (query head) and column pair
  uint32_t qa[Q::KS][4];                     // query A fragments: rows 0..7 bf16 hi, rows 8..15 bf16 residual
  float o[Q::NO][4];                         // output accumulators: [0..1] hi part, [2..3] residual part
  float m_run = -INFINITY, l_run = 0.f;      // head gq, log2 domain; l is this thread's partial sum
  int seg = -1, last_written = seg_first - 1;

  auto write_record = [&](int sq, bool neutral) {
    if (!kAttend) return;
    float l = neutral ? 0.f : l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (gq >= G) return;
    float* rec = vp.rec + (((int64_t)(c + sq) * kWarps + warp) * G + gq) * (2 + D);
    if (tq == 0) {
      rec[0] = neutral ? -INFINITY : m_run;
      rec[1] = l;
    }
#pragma unroll
    for (int n = 0; n < Q::NO; ++n) {
      rec[2 + 8 * n + 2 * tq] = neutral ? 0.f : o[n][0] + o[n][2];
      rec[2 + 8 * n + 2 * tq + 1] = neutral ? 0.f : o[n][1] + o[n][3];
    }
  };
  auto neutral_upto = [&](int sq_end) {  // neutral records for segments (last_written, sq_end)
    for (int sq = last_written + 1; sq < sq_end; ++sq) write_record(sq, true);
    if (sq_end - 1 > last_written) last_written = sq_end - 1;
  };

  auto begin_segment = [&](const BlockMeta& m) {
    const int nk = a.n_keep[m.s];
    int L;
    if (MODE == 1) {
      L = vp.view_len[m.q];
      if (L < 0 || L > Lcap) {  // caller-supplied: clamp so the table reads stay in range
        if (lane == 0) atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
        L = L < 0 ? 0 : Lcap;
      }
    } else {
      const int last = vp.kept[(int64_t)m.q * vp.budget + nk - 1];
      L = 32 * (nk - 1) + ((last >= 0 && last < a.n_blk[m.s]) ? block_tokens(last, a, m.s) : 32);
      if (m.i == 0 && lane == 0) vp.view_len[m.q] = L;
    }
    if (!kAttend) return;
    // RoPE(q, L) for this thread's fragment elements: head gq, dims 16kk + 2tq + {0,1,8,9} (kk < KS/2),
    // each paired with the same dim + d/2, which sits in k-step kk + KS/2 at the same place
    const int g = m.q % vp.h_kv;
    const float2* bb = vp.rope_base + (int64_t)(L >> 5) * (D / 2);
    const float2* oo = vp.rope_off + (L & 31) * (D / 2);
    const uint16_t* qh = vp.q + ((int64_t)m.s * vp.h_q + g * G + (gq < G ? gq : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < Q::KS / 2; ++kk) {
      float y1[4], y2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int dim = 16 * kk + 2 * tq + (e & 1) + 8 * (e >> 1);
        const float x1 = __uint_as_float((uint32_t)qh[dim] << 16);
        const float x2 = __uint_as_float((uint32_t)qh[dim + D / 2] << 16);
        const float2 o2 = oo[dim];
        float cs, sn;
        rope_cs(bb[dim], o2.x, o2.y, cs, sn);
        y1[e] = gq < G ? (x1 * cs - x2 * sn) * vp.q_scale : 0.f;
        y2[e] = gq < G ? (x2 * cs + x1 * sn) * vp.q_scale : 0.f;
      }
      split2(y1[0], y1[1], qa[kk][0], qa[kk][1]);
      split2(y1[2], y1[3], qa[kk][2], qa[kk][3]);
      split2(y2[0], y2[1], qa[kk + Q::KS / 2][0], qa[kk + Q::KS / 2][1]);
      split2(y2[2], y2[3], qa[kk + Q::KS / 2][2], qa[kk + Q::KS / 2][3]);
    }
#pragma unroll
    for (int n = 0; n < Q::NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m_run = -INFINITY;
    l_run = 0.f;
  };

  // ------------------------------------------------------------ main loop over this warp's blocks
  BlockMeta batch = resolve(0);
  BlockMeta cur = bcast(batch, 0);
  if (nblk_w > 0) {
    issue_k(cur);
    issue_v(cur);
  }
  bool aborted = false;
  for (int64_t j = 0; j < nblk_w; ++j) {
    const uint32_t phase = (uint32_t)(j & 1);
    // metadata of the next block (the batch is refilled every 32 blocks)
    BlockMeta nxt{-1, 0, 0, 0, 0};
    if (j + 1 < nblk_w) {
      if (((j + 1) & 31) == 0) batch = resolve(j + 1);
      nxt = bcast(batch, (int)((j + 1) & 31));
    }
    if (cur.q != seg) {
      if (seg >= 0) {
        write_record(seg, false);
        last_written = seg;
      }
      neutral_upto(cur.q);
      seg = cur.q;
      begin_segment(cur);
    }
    const int valid = cur.valid;
    const int64_t ydst = (int64_t)cur.q * Lcap + 32 * cur.i;

    // ---- K: wait, rotate in place, store (the abort decision is made by the whole warp)
    if (__any_sync(0xffffffffu, !mbar_wait(&full_k[warp], phase, vp.status))) {
      aborted = true;
      break;
    }
    if (valid > 0 && kWrite) {
      const int cc = lane % Q::CPR;
      float2 bb[8];
      {
        const float4* bp = reinterpret_cast<const float4*>(vp.rope_base + (int64_t)cur.i * (D / 2) + 8 * cc);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 t = __ldg(bp + u);
          bb[2 * u] = make_float2(t.x, t.y);
          bb[2 * u + 1] = make_float2(t.z, t.w);
        }
      }
#pragma unroll 2
      for (int pass = 0; pass < Q::PASSES; ++pass) {
        const int r = lane / Q::CPR + Q::RPP * pass;
        const uint32_t a1 = kaddr + chunk_off(r, cc), a2 = kaddr + chunk_off(r, cc + D / 16);
        const uint4 w1 = lds128(a1), w2 = lds128(a2);
        const uint32_t xa[4] = {w1.x, w1.y, w1.z, w1.w}, xb[4] = {w2.x, w2.y, w2.z, w2.w};
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 ofs = off_s[(r * 4 + u) * Q::CPR + cc];
          float f1[2], f2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int v = 2 * u + e;
            float cs, sn;
            rope_cs(bb[v], e ? ofs.z : ofs.x, e ? ofs.w : ofs.y, cs, sn);
            const float x1 = e ? bf16hi(xa[u]) : bf16lo(xa[u]);
            const float x2 = e ? bf16hi(xb[u]) : bf16lo(xb[u]);
            f1[e] = fmaf(x1, cs, -x2 * sn);
            f2[e] = fmaf(x2, cs, x1 * sn);
            // fp32 tables put |error| <= 3e-7 (|x1| + |x2|) on f, below one bf16 ulp of the result unless
            // the rotation cancels; those pairs are redone in float-float so every stored key is within
            // one ulp of the exact rotation.
            const float tau = 0x1p-12f * (fabsf(x1) + fabsf(x2));
            if (fminf(fabsf(f1[e]), fabsf(f2[e])) < tau)
              rotate_exact(x1, x2, vp.rope_base_hl[(int64_t)cur.i * (D / 2) + 8 * cc + v],
                           vp.rope_off_hl[r * (D / 2) + 8 * cc + v], f1[e], f2[e]);
          }
          oa[u] = pack_bf16x2(f1[0], f1[1]);
          ob[u] = pack_bf16x2(f2[0], f2[1]);
        }
        sts128(a1, make_uint4(oa[0], oa[1], oa[2], oa[3]));
        sts128(a2, make_uint4(ob[0], ob[1], ob[2], ob[3]));
        if (valid < 32 && r < valid) {  // partial block: plain stores of the rows present
          uint16_t* kd = vp.k_view + (ydst + r) * D;
          *reinterpret_cast<uint4*>(kd + 8 * cc) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
          *reinterpret_cast<uint4*>(kd + D / 2 + 8 * cc) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (valid == 32 && lane == 0) {
#pragma unroll
        for (int b = 0; b < Q::BOXES; ++b) tma_store_2d(&tm_kdst, 64 * b, (int)ydst, kbuf + b * Q::BOX);
        bulk_commit();
      }
    }

    // ---- scores S = q . K^T for the block's 32 tokens (4 n-tiles of 8)
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
    if (kAttend && valid > 0) {
#pragma unroll
      for (int kk = 0; kk < Q::KS; ++kk) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int tok = 16 * np + (lane & 7) + 8 * (lane >> 4);
          const int chk = 2 * kk + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kaddr + chunk_off(tok, chk), b0, b1, b2, b3);
          mma_16816(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_16816(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
    }
    // the K page is no longer needed: once its store has read it, fetch the next block's K
    __syncwarp();
    if (lane == 0) {
      bulk_wait_read_all();
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (j + 1 < nblk_w) issue_k(nxt);

    // ---- V: wait, store, P.V
    if (__any_sync(0xffffffffu, !mbar_wait(&full_v[warp], phase, vp.status))) {
      aborted = true;
      break;
    }
    if (valid > 0 && kWrite) {
      if (valid == 32) {
        if (lane == 0) {
#pragma unroll
          for (int b = 0; b < Q::BOXES; ++b) tma_store_2d(&tm_vdst, 64 * b, (int)ydst, vbuf + b * Q::BOX);
          bulk_commit();
        }
      } else {
        const int cc = lane % Q::CPR;
#pragma unroll 1
        for (int pass = 0; pass < Q::PASSES; ++pass) {
          const int r = lane / Q::CPR + Q::RPP * pass;
          if (r < valid) {
            uint16_t* vd = vp.v_view + (ydst + r) * D;
            *reinterpret_cast<uint4*>(vd + 8 * cc) = lds128(vaddr + chunk_off(r, cc));
            *reinterpret_cast<uint4*>(vd + D / 2 + 8 * cc) = lds128(vaddr + chunk_off(r, cc + D / 16));
          }
        }
      }
    }
    if (kAttend && valid > 0) {
      if (valid < 32) {  // rows past the tail may hold any bits: zero them before P.V
        __syncwarp();
        const int cc = lane % Q::CPR;
#pragma unroll 1
        for (int pass = 0; pass < Q::PASSES; ++pass) {
          const int r = lane / Q::CPR + Q::RPP * pass;
          if (r >= valid) {
            sts128(vaddr + chunk_off(r, cc), make_uint4(0, 0, 0, 0));
            sts128(vaddr + chunk_off(r, cc + D / 16), make_uint4(0, 0, 0, 0));
          }
        }
        __syncwarp();
      }
      // online softmax for head gq over this block
      float s[8], bm = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = 8 * n + 2 * tq + e;
          const float v = sc[n][e] + sc[n][2 + e];
          s[2 * n + e] = tok < valid ? v : -INFINITY;
          bm = fmaxf(bm, s[2 * n + e]);
        }
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      if (bm > m_run + 8.f) {  // raise the reference only when it grows by more than 8 (a factor 256)
        const float corr = fast_exp2(m_run - bm);  // 0 when m_run was -inf
        l_run *= corr;
#pragma unroll
        for (int n = 0; n < Q::NO; ++n) {
          o[n][0] *= corr;
          o[n][1] *= corr;
          o[n][2] *= corr;
          o[n][3] *= corr;
        }
        m_run = bm;
      }
      uint32_t ph[4], pl[4];  // P for n-tiles 0..3: bf16 hi and residual, packed pairs
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float p0 = fast_exp2(s[2 * n] - m_run), p1 = fast_exp2(s[2 * n + 1] - m_run);
        l_run += p0 + p1;
        split2(p0, p1, ph[n], pl[n]);
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int np = 0; np < Q::NO / 2; ++np) {
          const int tok = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int chk = 2 * np + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vaddr + chunk_off(tok, chk), b0, b1, b2, b3);
          mma_16816(o[2 * np], ph[2 * ks], pl[2 * ks], ph[2 * ks + 1], pl[2 * ks + 1], b0, b1);
          mma_16816(o[2 * np + 1], ph[2 * ks], pl[2 * ks], ph[2 * ks + 1], pl[2 * ks + 1], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      bulk_wait_read_all();
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (j + 1 < nblk_w) issue_v(nxt);
    cur = nxt;
  }
  if (aborted) {
    // drain: copies already issued for this warp's stage must land before the CTA exits
    if (lane == 0) {
      bulk_wait_all();
      mbar_wait(&full_k[warp], 0, vp.status);
      mbar_wait(&full_k[warp], 1, vp.status);
      mbar_wait(&full_v[warp], 0, vp.status);
      mbar_wait(&full_v[warp], 1, vp.status);
    }
    return;
  }
  if (seg >= 0) {
    write_record(seg, false);
    last_written = seg;
  }
  neutral_upto(seg_last + 1);
  if (lane == 0) bulk_wait_all();
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
  auto rec = [&](int c, int w) { return vp.rec + (((int64_t)(c + q) * kWarps + w) * G + hh) * (2 + D); };
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c)
    if (!empty(c))
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, rec(c, w)[0]);
  for (int dim = threadIdx.x; dim < D; dim += blockDim.x) {
    float av = 0.f, lv = 0.f;
    if (M != -INFINITY) {
      for (int c = c0; c <= c1; ++c) {
        if (empty(c)) continue;
        for (int w = 0; w < kWarps; ++w) {
          const float* rc = rec(c, w);
          if (rc[0] == -INFINITY) continue;
          const float sc = exp2f(rc[0] - M);
          av = fmaf(rc[2 + dim], sc, av);
          lv = fmaf(rc[1], sc, lv);
        }
      }
    }
    vp.out[((int64_t)s * vp.h_q + h) * D + dim] = lv > 0.f ? av / lv : 0.f;
  }
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

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over rows of d bf16 values: boxes of 64 columns x 32 rows, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  memset(m, 0, sizeof(*m));
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (rows < 32) rows = 32;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int G>
cudaError_t launch_dg(const Ctx& c, int mode, const CUtensorMap* maps, const ViewParams& vp, const SessionArgs& a,
                      cudaStream_t st) {
  using Q = Geo<D>;
  const size_t smem = (size_t)kWarps * 2 * Q::PAGE + (size_t)32 * 4 * Q::CPR * sizeof(float4) + 1024;
  cudaError_t e = cudaSuccess;
  if (vp.total > 0) {
    void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const ViewParams,
                 const SessionArgs) =
        mode == 0 ? view_kernel<D, G, 0> : (mode == 1 ? view_kernel<D, G, 1> : view_kernel<D, G, 2>);
    if ((e = ensure_smem(kern, c.device, smem)) != cudaSuccess) return e;
    kern<<<vp.P, kWarps * 32, smem, st>>>(maps[0], maps[1], maps[2], maps[3], vp, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  combine_kernel<D, G><<<vp.n_sessions * vp.h_q, D, 0, st>>>(vp, a, mode != 0);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Ctx& c, int mode, const CUtensorMap* maps, const ViewParams& vp, const SessionArgs& a,
                     cudaStream_t st) {
  switch (c.group) {
    case 1: return launch_dg<D, 1>(c, mode, maps, vp, a, st);
    case 2: return launch_dg<D, 2>(c, mode, maps, vp, a, st);
    case 3: return launch_dg<D, 3>(c, mode, maps, vp, a, st);
    case 4: return launch_dg<D, 4>(c, mode, maps, vp, a, st);
    case 5: return launch_dg<D, 5>(c, mode, maps, vp, a, st);
    case 6: return launch_dg<D, 6>(c, mode, maps, vp, a, st);
    case 7: return launch_dg<D, 7>(c, mode, maps, vp, a, st);
    case 8: return launch_dg<D, 8>(c, mode, maps, vp, a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_view(const Ctx& c, int mode, const uint16_t* k_src, const uint16_t* v_src, int64_t n_pages,
                        const int32_t* bt, int n_sessions, const SessionArgs& a, const int32_t* kept,
                        const uint16_t* q, uint16_t* k_view, uint16_t* v_view, int32_t* view_len, float* out,
                        cudaStream_t st) {
  ViewParams vp;
  vp.bt = bt;
  vp.max_blocks = c.p.max_blocks;
  vp.n_pages = n_pages;
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
  // tensor maps: sources (pool pages, or the view for mode 1) and destinations (the view)
  const uint64_t view_rows = (uint64_t)n_sessions * c.p.h_kv * 32 * c.budget;
  const uint64_t pool_rows = (uint64_t)n_pages * c.p.h_kv * 32;
  if (pool_rows > 0x7FFFFFFFull || view_rows > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  CUtensorMap maps[4];
  cudaError_t e;
  if (mode == 1) {
    if ((e = make_map(&maps[0], k_src, view_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[1], v_src, view_rows, c.p.d)) != cudaSuccess) return e;
    maps[2] = maps[0];
    maps[3] = maps[1];
  } else {
    if ((e = make_map(&maps[0], k_src, pool_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[1], v_src, pool_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[2], k_view, view_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[3], v_view, view_rows, c.p.d)) != cudaSuccess) return e;
  }
  return c.p.d == 128 ? launch_d<128>(c, mode, maps, vp, a, st) : launch_d<64>(c, mode, maps, vp, a, st);
}

cudaError_t launch_rope_tables(const Ctx& c, cudaStream_t st) {
  rope_table_kernel<<<256, 256, 0, st>>>(reinterpret_cast<float2*>(c.rope_base), c.budget + 1,
                                         reinterpret_cast<float2*>(c.rope_off), c.rope_base_hl, c.rope_off_hl, c.p.d,
                                         (double)c.p.rope_theta);
  return cudaGetLastError();
}

}  // namespace kvm
