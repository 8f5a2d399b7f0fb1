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
// number of pages.  Each CTA is warp-specialised:
//   - a producer warp resolves 32 blocks at a time (kept id -> page, one lane
//     each, the next 32 resolved while the current 32 are issued) and keeps a
//     ring of NS shared-memory stages full: per block one stage receives the K
//     and V pages by TMA tiled loads (64-column boxes, 128-byte swizzle) and,
//     when writing a view, the block's rows of the RoPE base tables by 1-D bulk
//     copies, all completing on the stage's `full` mbarrier;
//   - four rotation warps (eight for FP8 pages, below) take every fourth block of the share: each rotates
//     K in place at view positions 32*i + r (cos/sin composed in fp32 from the
//     staged per-slot row and the per-offset values, which a lane keeps in
//     registers because it always rotates the same (row, pair) slots; both
//     tables filled in fp64; pairs whose rotation cancels are redone in
//     float-float from the hi/lo halves), rounds to bf16, writes the rotated K and the
//     untouched V to the view with TMA tiled stores, marks the stage `rotated`
//     and frees its share of the stage once the stores have read it;
//   - two attention warps take every other block: each waits for the rotated
//     page, computes the scores with mma.sync (m16n8k16, bf16 -> fp32; A rows
//     0..7 hold the rotated, scaled query heads rounded to bf16, rows 8..15
//     their bf16 residuals, so one MMA gives an fp32-accurate score), keeps an
//     online softmax per head in the log2 domain (the running maximum is raised
//     only when it grows by more than 8) and accumulates P.V with mma.sync, P
//     split the same way, then frees its share of the stage.
// FP8 pages (fused mode): eight rotation warps, and the producer fills a ring
// of code slots instead of the stages (the K and V code pages and the block's
// base table row, by 1-D bulk copies); the rotation warp that owns the block
// decodes it into its stage (K rotated, V scaled and rounded to bf16), frees
// the code slot at once, and the stage goes on as for bf16 pages.  The
// per-offset cos/sin then come from a shared-memory copy of the table.
// NS is a multiple of both warp counts, so every rotation and every attention
// warp owns whole stages and meets their rounds strictly in order: a wait on a
// stage barrier is never more than one phase ahead, which the parity waits
// need.  The 7 warps of the bf16 modes fit two per SM sub-partition, so every
// warp may hold up to 255 registers; the rotation (about four times the
// attention's work per block) gets four warps.  FP8 pages: 11 warps, at most
// three per sub-partition, 168 registers each.
// No warp reads global memory on the per-block path.  Each attention warp
// writes one partial record (max, sum, output) per segment (session, KV head)
// of its CTA's share — a neutral record for a segment it had no block of — in
// the record group (cta + segment), which is unique to the pair.  At the end
// the CTA folds its attention warps' records of each segment into one CTA record
// (log-sum-exp), then counts itself in on each of its segments with one
// atomic add; the CTA that arrives last on a segment (no CTA ever waits)
// merges that segment's CTA records with batched independent loads and writes
// the G output rows, then resets the segment's counter for the next call.
// Every mbarrier wait is bounded; a timeout sets KVM_DEV_TIMEOUT, the warp
// stops, the producer waits (bounded) for its copies in flight, and the CTA
// does not count itself in, so the outputs of its segments are left unwritten
// (the status word says why).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr int kAttn = kViewWarps;  // attention warps per CTA (attention-record slots)
// Rotation warps per CTA (warps 0 .. rot_warps - 1): four for bf16 pages; eight for FP8 pages, whose decoding
// doubles the rotation warps' work per block.  The producer is the warp after the attention warps.
template <bool F8>
constexpr int rot_warps() {
  return F8 ? 8 : 4;
}
template <bool F8>
constexpr int view_threads() {
  return (rot_warps<F8>() + kAttn + 1) * 32;
}

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
  uint32_t* seg_count;         // [n_sessions * h_kv] arrival counters (zero between calls)
  const float2* rope_base;     // [budget + 1][d/2] (cos, sin) rounded to fp32
  const float2* rope_base_lo;  // [budget + 1][d/2] what the rounding dropped (cos, sin)
  const float2* rope_off;      // [32][d/2]
  const float2* rope_off_lo;   // [32][d/2]
  float* out;
  const float* k_scale;  // FP8 pages: [n_pages][h_kv] scale of each K page
  const float* v_scale;
  const uint8_t* k8;     // FP8 pages: [n_pages][h_kv][32][d] codes
  const uint8_t* v8;
  uint32_t* status;
  int64_t total;  // kept blocks over all (session, KV head)
  int any_empty;  // some session keeps no block
  int budget;
  int h_kv;
  int h_q;
  int n_sessions;
  int P;  // CTAs
  float q_scale;  // log2(e) / sqrt(d)
  uint64_t wait_ns;  // wall-clock limit of the pipeline waits (the drain of copies in flight keeps the full limit)
  int stall;         // failure-path test: the rotation of flat block 0 first waits on a barrier nothing completes
};

// Attention record of one (CTA, segment, warp, query head): max, sum, 2 pad, output[D] (16-byte aligned).
template <int D>
constexpr int kRecFloats = 4 + D;

template <int D, bool F8 = false>
struct Geo {
  static constexpr int BOXES = D / 64;          // 64-column (128-byte) boxes per page row
  static constexpr uint32_t BOX = 32 * 128;     // bytes of one box (32 rows)
  static constexpr uint32_t PAGE = 32 * D * 2;  // bytes of one K (or V) page in bf16
  static constexpr uint32_t CPAGE = 32 * D;     // bytes of one page of FP8 codes
  // a stage: the bf16 K and V pages (as loaded, or decoded from FP8 pages)
  static constexpr uint32_t STAGE = 2 * PAGE;
  static constexpr int CPR = D / 16;            // rotation items (chunk pairs) per row
  static constexpr int RPP = 32 / CPR;          // rows per rotation pass
  static constexpr int PASSES = CPR;            // rotation passes per page
  static constexpr int KS = D / 16;             // MMA k-steps over the head dimension
  static constexpr int NO = D / 8;              // output n-tiles
  static constexpr int NS = F8 ? (D == 128 ? 8 : 16) : (D == 128 ? 12 : 24);  // a multiple of both warp counts
  static constexpr uint32_t TAB = D / 2 * 8;     // bytes of one table row ((cos, sin) per pair)
  // FP8 pages: the loads fill a ring of their own, NC code slots (the K and V code pages, then the block's base
  // table row), which a rotation warp frees as soon as it has decoded the block into a stage; the stage then
  // only waits for the view stores and the attention.  bf16 pages: the loads fill the stages (NC = NS).  NC is
  // a multiple of the rotation warps, so each code slot, like each stage, belongs to one rotation warp.
  static constexpr int NC = NS;
  static constexpr uint32_t CSLOT = 2 * CPAGE + TAB;  // bytes of one code slot
  static constexpr uint32_t OFS = 32 * TAB;           // FP8: the per-offset (cos, sin) table, [32 rows][d/2]
  // shared memory, from the 1024-byte-aligned base
  static constexpr uint32_t OFF_CODE = NS * STAGE;                        // FP8: [NC] code slots
  static constexpr uint32_t OFF_OFS = OFF_CODE + (F8 ? NC * CSLOT : 0);   // FP8: offset table (swizzled)
  static constexpr uint32_t OFF_TAB = OFF_OFS + (F8 ? OFS : 0);           // bf16: [NS][hi | lo] table rows
  static constexpr uint32_t OFF_META = OFF_TAB + (F8 ? 0 : NS * 2 * TAB); // [NS] int: tokens of the block
  static constexpr uint32_t OFF_CMETA = OFF_META + NS * 4;                // FP8: [NC] int, per code slot
  static constexpr uint32_t OFF_SCALE = OFF_CMETA + (F8 ? NC * 4 : 0);    // FP8: [NC] float2 page scales
  static constexpr uint32_t BYTES = OFF_SCALE + (F8 ? NC * 8 : 0) + 1024; // + alignment slack
  static_assert(CSLOT % 16 == 0 && OFF_OFS % 16 == 0 && OFF_SCALE % 8 == 0, "bulk-copy and vector alignment");
  static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};

// Moves [src, src + bytes) into L2 (no completion to wait for); src and bytes multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ int64_t cta_begin(int c, int64_t total, int P) { return (int64_t)c * total / P; }
// CTA whose share contains flat block f (shares are [floor(cT/P), floor((c+1)T/P))).
__device__ __forceinline__ int cta_of(int64_t f, int64_t total, int P) {
  return (int)(((f + 1) * (int64_t)P - 1) / total);
}

struct Cursor {
  int s, g, i;
};
// (session, KV head, slot) of flat block f; a session's share is h_kv * n_keep < 2^31 blocks.
__device__ __forceinline__ Cursor locate(int64_t f, const SessionArgs& a, int n_sessions) {
  int s = 0;
  while (s + 1 < n_sessions && a.seg_base[s + 1] <= f) ++s;
  const int local = (int)(f - a.seg_base[s]);
  const int nk = a.n_keep[s];
  const int g = local / nk;
  return Cursor{s, g, local - g * nk};
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

template <int D, int G, int MODE, bool F8 = false>
__global__ void __launch_bounds__(view_threads<F8>(), 1)
    view_kernel(const __grid_constant__ CUtensorMap tm_ksrc, const __grid_constant__ CUtensorMap tm_vsrc,
                const __grid_constant__ CUtensorMap tm_kdst, const __grid_constant__ CUtensorMap tm_vdst,
                const ViewParams vp, const SessionArgs a) {
  using Q = Geo<D, F8>;
  static_assert(!F8 || MODE == 2, "FP8 pages are a source of the fused mode");
  constexpr bool kWrite = MODE != 1;
  constexpr bool kAttend = MODE != 0;
  constexpr int NS = Q::NS;
  constexpr int NC = Q::NC;  // slots the loads fill: code slots (FP8 pages), else the stages themselves
  constexpr int kRot = rot_warps<F8>();
  constexpr int kProducer = kRot + kAttn;
  constexpr int kThreads = view_threads<F8>();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_addr(smem);
  int* meta = reinterpret_cast<int*>(smem + Q::OFF_META);
  int* cmeta = F8 ? reinterpret_cast<int*>(smem + Q::OFF_CMETA) : meta;  // tokens per loaded slot
  float2* meta_scale = reinterpret_cast<float2*>(smem + Q::OFF_SCALE);
  // full: per loaded slot; rotated, empty: per stage; cempty (FP8): per code slot, freed by its rotation warp
  __shared__ __align__(8) uint64_t full[NC], rotated[NS], empty[NS], cempty[F8 ? NC : 1];
  __shared__ __align__(8) uint64_t never;  // failure-path test only: initialised, never arrived on

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  if (tid == 0) {
    for (int cs = 0; cs < NC; ++cs) {
      mbar_init(&full[cs], 1);
      if (F8) mbar_init(&cempty[cs], 1);
    }
    for (int st = 0; st < NS; ++st) {
      mbar_init(&rotated[st], 1);
      mbar_init(&empty[st], (kWrite ? 1 : 0) + (kAttend ? 1 : 0));  // the stage's rotation and attention warps
    }
    mbar_init(&never, 1);
    mbar_fence_init();
  }
  // A rotation lane always rotates the same pairs of every block: rows r = lane / CPR + RPP * pass, pairs
  // k = 8 cc + v (v < 8) with cc = lane % CPR.  Their offset cos/sin (r * theta_k, block-independent, from the
  // context's table) stay in registers for the whole kernel: of[pass][u] holds pairs 2u and 2u + 1.  They are
  // loaded before the wait on the preceding kernel, which wrote none of them.
  // Each is held as two packed pairs (cos of pairs 2u and 2u + 1; sin of the same), the operands of the paired
  // fp32 instructions below.
  // FP8 pages: the table sits in shared memory instead (the eight rotation warps have no room for it in
  // registers); a lane reads its pass's four float4 (cos, sin of pairs 2u and 2u + 1) from a layout whose float4
  // index u is XOR-swizzled with the lane's chunk pair (and, for d = 64, its row parity), so the eight lanes of a
  // quarter warp hit eight different bank groups.
  uint64_t ofc[Q::PASSES][4], ofs[Q::PASSES][4];
  auto ofs_swz = [](int r, int cc) { return ((cc >> 1) & 3) ^ (D == 64 ? (r & 1) << 1 : 0); };
  if constexpr (F8) {
    float4* o4 = reinterpret_cast<float4*>(smem + Q::OFF_OFS);
    const float4* src = reinterpret_cast<const float4*>(vp.rope_off);
    for (int i = tid; i < 32 * (D / 4); i += kThreads) {
      const int r = i / (D / 4), j = i % (D / 4), cc = j >> 2, u = j & 3;
      o4[r * (D / 4) + 4 * cc + (u ^ ofs_swz(r, cc))] = __ldg(src + i);
    }
  } else if (kWrite && warp < kRot) {
    const int cc = lane % Q::CPR;
#pragma unroll
    for (int pass = 0; pass < Q::PASSES; ++pass)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2* t = vp.rope_off + (lane / Q::CPR + Q::RPP * pass) * (D / 2) + 8 * cc + 2 * u;
        const float2 o0 = __ldg(t), o1 = __ldg(t + 1);
        ofc[pass][u] = pk2(o0.x, o1.x);
        ofs[pass][u] = pk2(o0.y, o1.y);
      }
  }
  // While the preceding kernel finishes, warm L2 with the block-table rows of this CTA's sessions (the producer's
  // first page lookups then hit L2): the CTAs sharing a session each take one slice of its row, so the row is
  // requested once.  A prefetch only moves lines into L2, the point of coherence, so it cannot make a lookup see
  // an older table; only whole 16-byte pieces inside each row are prefetched.
  if (MODE != 1 && warp == kProducer && lane == 0 && vp.total > 0) {
    const int64_t f0 = cta_begin(c, vp.total, vp.P), f1 = cta_begin(c + 1, vp.total, vp.P);
    if (f0 < f1) {
      const int s0 = locate(f0, a, vp.n_sessions).s, s1 = locate(f1 - 1, a, vp.n_sessions).s;
      for (int s = s0; s <= s1; ++s) {
        if (a.seg_base[s + 1] <= a.seg_base[s]) continue;
        const int cA = cta_of(a.seg_base[s], vp.total, vp.P), cB = cta_of(a.seg_base[s + 1] - 1, vp.total, vp.P);
        const char* row = reinterpret_cast<const char*>(vp.bt + (int64_t)s * vp.max_blocks);
        const int64_t row_bytes = ((int64_t)a.n_blk[s] * 4) & ~(int64_t)15;
        const int64_t n = cB - cA + 1, chunk = ((row_bytes + n - 1) / n + 15) & ~(int64_t)15;
        const int64_t off = (int64_t)(c - cA) * chunk;
        if ((reinterpret_cast<uintptr_t>(row) & 15) == 0 && off < row_bytes)
          prefetch_l2(row + off, (uint32_t)(chunk < row_bytes - off ? chunk : row_bytes - off));
      }
    }
  }
  griddep_wait();  // kept ids, queries, views and outputs belong to the stream order from here on
  if (vp.any_empty) {
    // sessions with no kept block (empty history): zero output rows and view lengths
    const int64_t per_s = (int64_t)vp.h_q * D, n_out = vp.n_sessions * per_s;
    for (int64_t idx = (int64_t)c * blockDim.x + tid; idx < n_out; idx += (int64_t)vp.P * blockDim.x) {
      const int s = (int)(idx / per_s), hd = (int)(idx % per_s);
      if (a.n_keep[s] != 0) continue;
      if (kAttend) vp.out[idx] = 0.f;
      if (hd % (G * D) == 0) vp.view_len[s * vp.h_kv + hd / (G * D)] = 0;
    }
  }
  const int64_t fa = cta_begin(c, vp.total, vp.P), fb = cta_begin(c + 1, vp.total, vp.P);
  if (fa >= fb) return;
  const int64_t nb = fb - fa;  // blocks of this CTA
  const int Lcap = 32 * vp.budget;

  __syncthreads();

  const Cursor firstc = locate(fa, a, vp.n_sessions), lastc = locate(fb - 1, a, vp.n_sessions);
  const int seg_first = firstc.s * vp.h_kv + firstc.g;
  const int seg_last = lastc.s * vp.h_kv + lastc.g;
  KVM_DEBUG_CHECK(seg_first <= seg_last && c + seg_last < vp.P + vp.n_sessions * vp.h_kv, vp.status);
  bool aborted = false;
  int64_t issued = 0;  // producer: blocks whose copies were issued

  static_assert(NS % kRot == 0 && NS % kAttn == 0 && NC % kRot == 0,
                "each rotation and each attention warp owns whole stages, each rotation warp whole code slots");
  if (warp == kProducer) {
    // ============================================================ producer
    // lane l resolves block jb + l: tokens present (0 = skip), source tile row, view slot
    auto resolve = [&](int64_t jb, int& valid, int& ysrc, int& slot, float& sk, float& sv) {
      valid = 0;
      ysrc = 0;
      slot = 0;
      sk = sv = 0.f;
      const int64_t j = jb + lane;
      if (j >= nb) return;
      const Cursor cu = locate(fa + j, a, vp.n_sessions);
      const int q = cu.s * vp.h_kv + cu.g;
      slot = cu.i;
      if (MODE == 1) {
        int L = vp.view_len[q];
        L = L < 0 ? 0 : (L > Lcap ? Lcap : L);  // caller-supplied: the attention warp reports a bad value
        valid = max(0, min(32, L - 32 * cu.i));
        ysrc = q * Lcap + 32 * cu.i;
      } else {
        const int id = vp.kept[(int64_t)q * vp.budget + cu.i];
        const int prev = cu.i > 0 ? vp.kept[(int64_t)q * vp.budget + cu.i - 1] : -1;
        if (id >= 0 && id < a.n_blk[cu.s] && id > prev) {  // kept ids ascend within a list
          const int32_t page = vp.bt[(int64_t)cu.s * vp.max_blocks + id];
          if (page >= 0 && page < vp.n_pages) {
            valid = block_tokens(id, a, cu.s);
            ysrc = (int)(((int64_t)page * vp.h_kv + cu.g) * 32);
            if (F8) {
              sk = vp.k_scale[(int64_t)page * vp.h_kv + cu.g];
              sv = vp.v_scale[(int64_t)page * vp.h_kv + cu.g];
            }
          } else {
            atomicOr(vp.status, KVM_DEV_BAD_PAGE);
          }
        } else {
          atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
        }
      }
    };
    int v_cur, y_cur, i_cur;
    float sk_cur, sv_cur;
    resolve(0, v_cur, y_cur, i_cur, sk_cur, sv_cur);
    for (int64_t jb = 0; jb < nb && !aborted; jb += 32) {
      int v_nxt = 0, y_nxt = 0, i_nxt = 0;
      float sk_nxt = 0.f, sv_nxt = 0.f;
      if (jb + 32 < nb) resolve(jb + 32, v_nxt, y_nxt, i_nxt, sk_nxt, sv_nxt);  // in flight while this batch is issued
      const int cnt = (int)(nb - jb < 32 ? nb - jb : 32);
      for (int l = 0; l < cnt; ++l) {
        const int valid = __shfl_sync(0xffffffffu, v_cur, l);
        const int ysrc = __shfl_sync(0xffffffffu, y_cur, l);
        const int slot = __shfl_sync(0xffffffffu, i_cur, l);
        const float sk = F8 ? __shfl_sync(0xffffffffu, sk_cur, l) : 0.f;
        const float sv = F8 ? __shfl_sync(0xffffffffu, sv_cur, l) : 0.f;
        const int64_t jj = jb + l;
        const int st = (int)(jj % NC);  // the slot this block's loads fill
        const uint32_t round = (uint32_t)(jj / NC);
        int ok = 1;
        if (lane == 0) {
          if (round > 0) ok = mbar_wait(F8 ? &cempty[st] : &empty[st], (round - 1) & 1, vp.status, vp.wait_ns);
          if (ok) {
            cmeta[st] = valid;
            unsigned char* kdst = F8 ? smem + Q::OFF_CODE + st * Q::CSLOT : smem + st * Q::STAGE;
            if (valid > 0) {
              if constexpr (F8) {
                // the two code pages (contiguous 32 x d bytes each) and the base table's hi row by 1-D bulk
                // copies into the code slot
                meta_scale[st] = make_float2(sk, sv);
                mbar_arrive_expect_tx(&full[st], 2 * Q::CPAGE + Q::TAB);
                bulk_g2s(kdst, vp.k8 + (int64_t)ysrc * D, Q::CPAGE, &full[st]);
                bulk_g2s(kdst + Q::CPAGE, vp.v8 + (int64_t)ysrc * D, Q::CPAGE, &full[st]);
                bulk_g2s(kdst + 2 * Q::CPAGE, vp.rope_base + (int64_t)slot * (D / 2), Q::TAB, &full[st]);
              } else {
                mbar_arrive_expect_tx(&full[st], 2 * Q::PAGE + (kWrite ? 2 * Q::TAB : 0));
#pragma unroll
                for (int b = 0; b < Q::BOXES; ++b) {
                  tma_load_2d(kdst + b * Q::BOX, &tm_ksrc, 64 * b, ysrc, &full[st]);
                  tma_load_2d(kdst + Q::PAGE + b * Q::BOX, &tm_vsrc, 64 * b, ysrc, &full[st]);
                }
              }
              if (kWrite && !F8) {
                unsigned char* tdst = smem + Q::OFF_TAB + st * 2 * Q::TAB;
                bulk_g2s(tdst, vp.rope_base + (int64_t)slot * (D / 2), Q::TAB, &full[st]);
                bulk_g2s(tdst + Q::TAB, vp.rope_base_lo + (int64_t)slot * (D / 2), Q::TAB, &full[st]);
              }
            } else {
              mbar_arrive(&full[st]);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          aborted = true;
          break;
        }
        issued = jj + 1;
      }
      v_cur = v_nxt;
      y_cur = y_nxt;
      i_cur = i_nxt;
      sk_cur = sk_nxt;
      sv_cur = sv_nxt;
    }
  } else if (warp < kRot) {
    // ============================================================ rotation warps
    if (kWrite) {
      const int cc = lane % Q::CPR;
      int prev_st = -1;  // stage of this warp's previous block, freed one block later
      for (int64_t jj = warp; jj < nb; jj += kRot) {
        const int st = (int)(jj % NS);
        const uint32_t phase = (uint32_t)((jj / NS) & 1);
        const int cslot = (int)(jj % NC);  // the slot the block was loaded into (the stage itself for bf16 pages)
        const uint32_t cphase = (uint32_t)((jj / NC) & 1);
        const Cursor cu = locate(fa + jj, a, vp.n_sessions);
        const int q = cu.s * vp.h_kv + cu.g;
        const int64_t ydst = (int64_t)q * Lcap + 32 * cu.i;
        KVM_DEBUG_CHECK(cu.i < vp.budget && ydst + 32 <= (int64_t)vp.n_sessions * vp.h_kv * Lcap, vp.status);
        const uint32_t vaddr = sbase + st * Q::STAGE + Q::PAGE;
        bool bad = !mbar_wait(&full[cslot], cphase, vp.status, vp.wait_ns);
        if (F8 && jj >= NS) {
          // FP8 pages: the stage is written here, so block jj - NS must be done with it: this warp's own view
          // stores of that block have read it (its share, given now), and its attention warp has arrived
          if (lane == 0) {
            bulk_wait_read<NS / kRot - 1>();  // this warp's later blocks' stores may still be reading
            mbar_arrive(&empty[st]);
          }
          __syncwarp();
          bad = bad || !mbar_wait(&empty[st], phase ^ 1u, vp.status, vp.wait_ns);
        }
        bad = bad || (vp.stall && fa + jj == 0 && !mbar_wait(&never, 0, vp.status, vp.wait_ns));
        if (__any_sync(0xffffffffu, bad)) {
          aborted = true;
          break;
        }
        const int valid = cmeta[cslot];
        if (cu.i == 0 && lane == 0) {  // the segment's view length, written by the rotation warp of its block 0
          const int nk = a.n_keep[cu.s];
          const int last = vp.kept[(int64_t)q * vp.budget + nk - 1];
          vp.view_len[q] = 32 * (nk - 1) + ((last >= 0 && last < a.n_blk[cu.s]) ? block_tokens(last, a, cu.s) : 32);
        }
        if (valid > 0) {
            unsigned char* kst = smem + st * Q::STAGE;
            uint4* kq = reinterpret_cast<uint4*>(kst);  // the stage's K page as 16-byte chunks
            // the block's base table row: in its code slot (FP8 pages) or beside its stage
            const unsigned char* tab_hi =
                F8 ? smem + Q::OFF_CODE + cslot * Q::CSLOT + 2 * Q::CPAGE : smem + Q::OFF_TAB + st * 2 * Q::TAB;
            const float4* __restrict__ tabh = reinterpret_cast<const float4*>(tab_hi);
            // the block's base cos/sin for this lane's 8 pairs, as packed pairs (2u, 2u + 1)
            uint64_t bc[4], bs[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float4 t = tabh[4 * cc + u];  // (cos, sin) of pair 2u, then of pair 2u + 1
              bc[u] = pk2(t.x, t.z);
              bs[u] = pk2(t.y, t.w);
            }
            // one pass = row r = lane / CPR + RPP * pass, chunks cc and cc + d/16 (8 pairs).  Each pair of pairs is
            // rotated with
            // the paired fp32 instructions, every element rounded exactly as by the scalar operations:
            //   cs = fma(bc, oc, -bs * os), sn = fma(bs, oc, bc * os), f1 = fma(x1, cs, -x2 * sn),
            //   f2 = fma(x2, cs, x1 * sn).
            // Accuracy: with the fp32 tables (each within 2^-24 relative of the fp64 value) the composed cos/sin
            // are within 4 * 2^-24 of exact and the rotated f within 2^-24 (5 (|x1| + |x2|) + |f|), less than one
            // bf16 ulp of f (> 2^-8 |f|) whenever |f| >= 2^-13 (|x1| + |x2|).  A pass holding a pair below that
            // (the rotation cancels) keeps the original bits of its row in the stage and is redone in
            // float-float after the passes, so every stored key is within one ulp of the exact rotation.
            if constexpr (F8) {
            // FP8 pages: K is decoded (code * scale, fp32) as it is rotated, with the same paired-fp32 rotation
            // as bf16 pages; each rotated value is stored, and a pair that cancels is redone in float-float after
            // the passes from its codes.  V is decoded and rounded to bf16 into the stage's V page, which the
            // view store and the attention then read.
            const unsigned char* codes = smem + Q::OFF_CODE + cslot * Q::CSLOT;
            const float2 scl = meta_scale[cslot];
            const float4* o4 = reinterpret_cast<const float4*>(smem + Q::OFF_OFS);
            uint32_t redo_all = 0;  // bit pass: the pass holds a pair whose rotation cancels
            // (two passes per iteration: the whole kernel's code then stays within the instruction cache, which
            // the fully unrolled FP8 decode and rotation of eight warps did not)
#pragma unroll 2
            for (int pass = 0; pass < Q::PASSES; ++pass) {
              const int r = lane / Q::CPR + Q::RPP * pass;
              const uint2 ca = *reinterpret_cast<const uint2*>(codes + r * D + 8 * cc);
              const uint2 cb = *reinterpret_cast<const uint2*>(codes + r * D + D / 2 + 8 * cc);
              const uint32_t cw[4] = {ca.x, ca.y, cb.x, cb.y};
              float xa_f[8], xb_f[8];  // elements 8cc + v and their rotation partners d/2 further
#pragma unroll
              for (int k2 = 0; k2 < 4; ++k2) {
                const float2 lo = dequant_e4m3x2(cw[k2], scl.x), hi = dequant_e4m3x2(cw[k2] >> 16, scl.x);
                float* dst = k2 < 2 ? xa_f + 4 * k2 : xb_f + 4 * (k2 - 2);
                dst[0] = lo.x;
                dst[1] = lo.y;
                dst[2] = hi.x;
                dst[3] = hi.y;
              }
              uint32_t oa[4], ob[4];
              bool cancel = false;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float4 t = o4[r * (D / 4) + 4 * cc + (u ^ ofs_swz(r, cc))];
                const uint64_t oc2 = pk2(t.x, t.z), os2 = pk2(t.y, t.w);
                const uint64_t cs = fma2(bc[u], oc2, mul2(bs[u] ^ 0x8000000080000000ull, os2));
                const uint64_t sn = fma2(bs[u], oc2, mul2(bc[u], os2));
                const float x1l = xa_f[2 * u], x1h = xa_f[2 * u + 1], x2l = xb_f[2 * u], x2h = xb_f[2 * u + 1];
                const uint64_t x1 = pk2(x1l, x1h), x2 = pk2(x2l, x2h), nx2 = pk2(-x2l, -x2h);
                float f1l, f1h, f2l, f2h;
                up2(fma2(x1, cs, mul2(nx2, sn)), f1l, f1h);
                up2(fma2(x2, cs, mul2(x1, sn)), f2l, f2h);
                cancel |= fminf(fabsf(f1l), fabsf(f2l)) * 0x1p13f < fabsf(x1l) + fabsf(x2l);
                cancel |= fminf(fabsf(f1h), fabsf(f2h)) * 0x1p13f < fabsf(x1h) + fabsf(x2h);
                oa[u] = pack_bf16x2(f1l, f1h);
                ob[u] = pack_bf16x2(f2l, f2h);
              }
              kq[chunk_off(r, cc) >> 4] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
              kq[chunk_off(r, cc + D / 16) >> 4] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
              redo_all |= cancel ? 1u << pass : 0u;
            }
#pragma unroll 2
            for (int pass = 0; pass < Q::PASSES; ++pass) {
              const int r = lane / Q::CPR + Q::RPP * pass;
              const uint2 va = *reinterpret_cast<const uint2*>(codes + Q::CPAGE + r * D + 8 * cc);
              const uint2 vb = *reinterpret_cast<const uint2*>(codes + Q::CPAGE + r * D + D / 2 + 8 * cc);
              const uint32_t vw[4] = {va.x, va.y, vb.x, vb.y};
              uint32_t vo[8];
#pragma unroll
              for (int k2 = 0; k2 < 4; ++k2) {
                const float2 wl = dequant_e4m3x2(vw[k2], scl.y), wh = dequant_e4m3x2(vw[k2] >> 16, scl.y);
                vo[2 * k2] = pack_bf16x2(wl.x, wl.y);
                vo[2 * k2 + 1] = pack_bf16x2(wh.x, wh.y);
              }
              sts128(vaddr + chunk_off(r, cc), make_uint4(vo[0], vo[1], vo[2], vo[3]));
              sts128(vaddr + chunk_off(r, cc + D / 16), make_uint4(vo[4], vo[5], vo[6], vo[7]));
            }
            if (redo_all) {  // rare: each pair of a flagged pass rotated again from its codes, in float-float if it cancels
              const float2* tabl = vp.rope_base_lo + (int64_t)cu.i * (D / 2);  // not staged: rare path
              const float2* tabh2 = reinterpret_cast<const float2*>(tabh);
#pragma unroll 1
              for (uint32_t m = redo_all; m; m &= m - 1) {
                const int pass = __ffs(m) - 1;
                const int r = lane / Q::CPR + Q::RPP * pass;
#pragma unroll 1
                for (int v = 0; v < 8; ++v) {
                  const int k = 8 * cc + v;
                  const float x1 = dequant_e4m3x2(codes[r * D + k], scl.x).x;
                  const float x2 = dequant_e4m3x2(codes[r * D + D / 2 + k], scl.x).x;
                  const float2 bh = tabh2[k], oh = __ldg(vp.rope_off + r * (D / 2) + k);
                  float cs, sn;
                  rope_cs(bh, oh.x, oh.y, cs, sn);
                  if (!(fminf(fabsf(fmaf(x1, cs, -x2 * sn)), fabsf(fmaf(x2, cs, x1 * sn))) * 0x1p13f <
                        fabsf(x1) + fabsf(x2)))
                    continue;  // this pair was stored correctly by the pass
                  const float2 bl = __ldg(tabl + k), ol = __ldg(vp.rope_off_lo + r * (D / 2) + k);
                  float y1, y2;
                  rotate_exact(x1, x2, make_float4(bh.x, bl.x, bh.y, bl.y), make_float4(oh.x, ol.x, oh.y, ol.y), y1,
                               y2);
                  const uint32_t y = pack_bf16x2(y1, y2);
                  *(reinterpret_cast<uint16_t*>(kst + chunk_off(r, cc)) + v) = (uint16_t)(y & 0xFFFFu);
                  *(reinterpret_cast<uint16_t*>(kst + chunk_off(r, cc + D / 16)) + v) = (uint16_t)(y >> 16);
                }
              }
            }
            } else {
            uint4 wa = kq[chunk_off(lane / Q::CPR, cc) >> 4], wb = kq[chunk_off(lane / Q::CPR, cc + D / 16) >> 4];
            uint32_t redo_all = 0;  // bit pass
#pragma unroll
            for (int pass = 0; pass < Q::PASSES; ++pass) {
              const int r = lane / Q::CPR + Q::RPP * pass;
              if (pass > 0) {
                wa = kq[chunk_off(r, cc) >> 4];
                wb = kq[chunk_off(r, cc + D / 16) >> 4];
              }
              const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w}, xb[4] = {wb.x, wb.y, wb.z, wb.w};
              uint32_t oa[4], ob[4];
              bool cancel = false;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint64_t cs = fma2(bc[u], ofc[pass][u], mul2(bs[u] ^ 0x8000000080000000ull, ofs[pass][u]));
                const uint64_t sn = fma2(bs[u], ofc[pass][u], mul2(bc[u], ofs[pass][u]));
                const float x1l = bf16lo(xa[u]), x1h = bf16hi(xa[u]), x2l = bf16lo(xb[u]), x2h = bf16hi(xb[u]);
                const uint64_t x1 = pk2(x1l, x1h), x2 = pk2(x2l, x2h), nx2 = pk2(-x2l, -x2h);
                float f1l, f1h, f2l, f2h;
                up2(fma2(x1, cs, mul2(nx2, sn)), f1l, f1h);
                up2(fma2(x2, cs, mul2(x1, sn)), f2l, f2h);
                cancel |= fminf(fabsf(f1l), fabsf(f2l)) * 0x1p13f < fabsf(x1l) + fabsf(x2l);
                cancel |= fminf(fabsf(f1h), fabsf(f2h)) * 0x1p13f < fabsf(x1h) + fabsf(x2h);
                oa[u] = pack_bf16x2(f1l, f1h);
                ob[u] = pack_bf16x2(f2l, f2h);
              }
              if (cancel) {  // the row's chunks keep their original bits until the fix-up below
                redo_all |= 1u << pass;
              } else {
                kq[chunk_off(r, cc) >> 4] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
                kq[chunk_off(r, cc + D / 16) >> 4] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
              }
            }
            if (redo_all) {  // rare: float-float rotation of the flagged passes' pairs, read back from the stage
              const float2* tabl = reinterpret_cast<const float2*>(smem + Q::OFF_TAB + st * 2 * Q::TAB + Q::TAB);
              const float2* tabh2 = reinterpret_cast<const float2*>(tabh);
#pragma unroll 1
              for (uint32_t m = redo_all; m; m &= m - 1) {
                const int pass = __ffs(m) - 1;
                const int r = lane / Q::CPR + Q::RPP * pass;
#pragma unroll 1
                for (int v = 0; v < 8; ++v) {
                  const int k = 8 * cc + v;
                  uint16_t* e1 = reinterpret_cast<uint16_t*>(kst + chunk_off(r, cc)) + v;
                  uint16_t* e2 = reinterpret_cast<uint16_t*>(kst + chunk_off(r, cc + D / 16)) + v;
                  const float x1 = __uint_as_float((uint32_t)*e1 << 16), x2 = __uint_as_float((uint32_t)*e2 << 16);
                  const float2 bh = tabh2[k], bl = tabl[k];
                  const float2 oh = __ldg(vp.rope_off + r * (D / 2) + k), ol = __ldg(vp.rope_off_lo + r * (D / 2) + k);
                  float y1, y2;
                  rotate_exact(x1, x2, make_float4(bh.x, bl.x, bh.y, bl.y), make_float4(oh.x, ol.x, oh.y, ol.y), y1,
                               y2);
                  const uint32_t y = pack_bf16x2(y1, y2);
                  *e1 = (uint16_t)(y & 0xFFFFu);
                  *e2 = (uint16_t)(y >> 16);
                }
              }
            }
            }
            if (valid < 32) {  // partial block: plain stores of the rows present, from the stage
              __syncwarp();
#pragma unroll 1
              for (int pass = 0; pass < Q::PASSES; ++pass) {
                const int r = lane / Q::CPR + Q::RPP * pass;
                if (r < valid) {
                  uint16_t* kd = vp.k_view + (ydst + r) * D;
                  uint16_t* vd = vp.v_view + (ydst + r) * D;
                  *reinterpret_cast<uint4*>(kd + 8 * cc) = kq[chunk_off(r, cc) >> 4];
                  *reinterpret_cast<uint4*>(kd + D / 2 + 8 * cc) = kq[chunk_off(r, cc + D / 16) >> 4];
                  *reinterpret_cast<uint4*>(vd + 8 * cc) = lds128(vaddr + chunk_off(r, cc));
                  *reinterpret_cast<uint4*>(vd + D / 2 + 8 * cc) = lds128(vaddr + chunk_off(r, cc + D / 16));
                }
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (valid == 32 && lane == 0) {
#pragma unroll
              for (int b = 0; b < Q::BOXES; ++b) {
                tma_store_2d(&tm_kdst, 64 * b, (int)ydst, smem + st * Q::STAGE + b * Q::BOX);
                tma_store_2d(&tm_vdst, 64 * b, (int)ydst, smem + st * Q::STAGE + Q::PAGE + b * Q::BOX);
              }
            }
        }
        if constexpr (F8) {
          // the block's codes and table row are consumed: its code slot may be refilled.  The stage's token count
          // goes with the rotated arrival below.
          __syncwarp();
          if (lane == 0) {
            meta[st] = valid;
            mbar_arrive(&cempty[cslot]);
          }
        }
        // The attention warp may read the rotated page now.  This block's view stores form one bulk group (empty
        // when there are none); the stage is free once the group has read its source.  Fused: the stage's
        // attention warp holds it for a while anyway, so this warp frees the stage of its previous block after
        // issuing this block's stores and never waits for stores it has just issued (FP8 pages: one stage per
        // warp, freed just before the warp's next block is decoded into it).  Materialising only, the stage is
        // freed at once (its load refill is then the one thing waiting on it).
        if (lane == 0) {
          bulk_commit();
          if constexpr (kAttend) {
            mbar_arrive(&rotated[st]);
            if (!F8 && prev_st >= 0) {
              bulk_wait_read<1>();
              mbar_arrive(&empty[prev_st]);
            }
          } else {
            bulk_wait_read<0>();
            mbar_arrive(&empty[st]);
          }
        }
        prev_st = (kAttend && !F8) ? st : -1;
        __syncwarp();
      }
      if (kAttend && !aborted && prev_st >= 0 && lane == 0) {
        bulk_wait_read<0>();
        mbar_arrive(&empty[prev_st]);
      }
    }
  } else if (warp < kProducer) {
    // ============================================================ attention warps
    const int aw = warp - kRot;               // attention-record slot
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group (query head) and column pair
    uint32_t qa[Q::KS][4];                     // query A fragments: rows 0..7 bf16 hi, rows 8..15 bf16 residual
    float o[Q::NO][4];                         // output accumulators: [0..1] hi part, [2..3] residual part
    float m_run = -INFINITY, l_run = 0.f;      // head gq, log2 domain; l is this thread's partial sum
    int seg = -1, last_written = seg_first - 1;

    // At the end of each of the CTA's segments (every one in [seg_first, seg_last], in order, neutral where a
    // warp had no block of it) the two attention warps meet: warp 1 leaves its state in shared memory, warp 0
    // combines it with its own (log-sum-exp, warp 0 first) and writes the CTA record of the segment.  Both warps
    // make the same sequence of calls on every path, aborted ones included, so the named barriers pair up.
    static_assert(kAttn == 2, "the segment records combine exactly two attention warps");
    __shared__ float2 xs_ml[32];
    __shared__ float2 xs_o[Q::NO][32];
    auto write_record = [&](int sq, bool neutral) {
      float l = neutral ? 0.f : l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const float m = neutral ? -INFINITY : m_run;
      if (aw == 1) {
        xs_ml[lane] = make_float2(m, l);
#pragma unroll
        for (int n = 0; n < Q::NO; ++n)
          xs_o[n][lane] = neutral ? make_float2(0.f, 0.f) : make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
      }
      named_sync(1, 2 * 32);  // warp 1's state is in shared memory
      if (aw == 0 && gq < G) {
        const float2 ml1 = xs_ml[lane];
        const float M = fmaxf(m, ml1.x);
        float lv = 0.f, sc0 = 0.f, sc1 = 0.f;
        if (M != -INFINITY) {
          sc0 = m == -INFINITY ? 0.f : exp2f(m - M);
          sc1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - M);
          lv = fmaf(l, sc0, lv);
          lv = fmaf(ml1.y, sc1, lv);
        }
        float* rec = vp.rec + (((int64_t)(c + sq) * (kAttn + 1) + kAttn) * G + gq) * kRecFloats<D>;
        if (tq == 0) *reinterpret_cast<float2*>(rec) = make_float2(M, lv);
#pragma unroll
        for (int n = 0; n < Q::NO; ++n) {
          const float2 b = xs_o[n][lane];
          float2 r = make_float2(0.f, 0.f);
          if (M != -INFINITY) {
            const float ax = neutral ? 0.f : o[n][0] + o[n][2], ay = neutral ? 0.f : o[n][1] + o[n][3];
            r.x = fmaf(ax, sc0, r.x);
            r.x = fmaf(b.x, sc1, r.x);
            r.y = fmaf(ay, sc0, r.y);
            r.y = fmaf(b.y, sc1, r.y);
          }
          *reinterpret_cast<float2*>(rec + 4 + 8 * n + 2 * tq) = r;
        }
      }
      named_sync(1, 2 * 32);  // warp 0 has read the buffer
    };
    auto neutral_upto = [&](int sq_end) {  // neutral records for segments (last_written, sq_end)
      for (int sq = last_written + 1; sq < sq_end; ++sq) write_record(sq, true);
      if (sq_end - 1 > last_written) last_written = sq_end - 1;
    };

    auto begin_segment = [&](const Cursor& cu, int q) {
      const int nk = a.n_keep[cu.s];
      int L;
      if (MODE == 1) {
        L = vp.view_len[q];
        if (L < 0 || L > Lcap) {  // caller-supplied: clamp so the table reads stay in range
          if (lane == 0) atomicOr(vp.status, KVM_DEV_BAD_BLOCK);
          L = L < 0 ? 0 : Lcap;
        }
      } else {
        const int last = vp.kept[(int64_t)q * vp.budget + nk - 1];
        L = 32 * (nk - 1) + ((last >= 0 && last < a.n_blk[cu.s]) ? block_tokens(last, a, cu.s) : 32);
      }
      // RoPE(q, L) for this thread's fragment elements: head gq, dims 16kk + 2tq + {0,1,8,9} (kk < KS/2),
      // each paired with the same dim + d/2, which sits in k-step kk + KS/2 at the same place
      const float2* bb = vp.rope_base + (int64_t)(L >> 5) * (D / 2);
      const float2* oo = vp.rope_off + (L & 31) * (D / 2);
      const uint16_t* qh = vp.q + ((int64_t)cu.s * vp.h_q + cu.g * G + (gq < G ? gq : 0)) * D;
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

    if (kAttend) {
      for (int64_t jj = aw; jj < nb; jj += kAttn) {
        const int st = (int)(jj % NS);
        const uint32_t phase = (uint32_t)((jj / NS) & 1);
        const Cursor cu = locate(fa + jj, a, vp.n_sessions);
        const int q = cu.s * vp.h_kv + cu.g;
        if (q != seg) {
          if (seg >= 0) {
            write_record(seg, false);
            last_written = seg;
          }
          neutral_upto(q);
          seg = q;
          begin_segment(cu, q);
        }
        const uint32_t kaddr = sbase + st * Q::STAGE, vaddr = kaddr + Q::PAGE;
        // the rotated page (fused) or the view page as loaded (attention over a given view)
        if (__any_sync(0xffffffffu, !mbar_wait(kWrite ? &rotated[st] : &full[st], phase, vp.status, vp.wait_ns))) {
          aborted = true;
          break;
        }
        const int valid = meta[st];
        if (valid > 0) {
            // ---- scores S = q . K^T for the block's 32 tokens (4 n-tiles of 8)
            float sc[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
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
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // every path closes the remaining segments, so that both warps meet at the same barriers (after an
      // abort the records are not used: the CTA leaves before counting itself in)
      if (seg >= 0) {
        write_record(seg, false);
        last_written = seg;
      }
      neutral_upto(seg_last + 1);
    }
  }

  griddep_launch_dependents();  // the next kernel may be scheduled while this one merges and drains
  // The view stores' shared-memory sources are read (the writes themselves complete with the grid; nothing in
  // this kernel reads the view).  The attention warps' records are read below by this CTA only, after the
  // barrier; the CTA record the other CTAs read is fenced before the CTA counts itself in.
  if (lane == 0) bulk_wait_read_all();
  if (__syncthreads_or(aborted)) {
    if (warp == kProducer && lane == 0) {
      // copies still in flight into a stage must land before the CTA exits: wait (bounded) for the
      // last round issued on each stage
      for (int st = 0; st < NC; ++st)
        if (issued > st) mbar_wait(&full[st], (uint32_t)(((issued - 1 - st) / NC) & 1), vp.status);
    }
    return;
  }
  if (!kAttend) return;

  // ------------------------------------------------------------ merge
  // Records: per (CTA c, segment sq) a group of kAttn + 1 slots at ((c + sq) * (kAttn + 1)) * G; slot kAttn
  // holds the CTA's state of the segment, written by attention warp 0 at the segment's end (thread i of a merge
  // owns head i / (D/4), dims 4 * (i % (D/4)) .. + 3).
  constexpr int kSlots = kAttn + 1;
  constexpr int Q4 = D / 4;
  const bool all_live = vp.total >= vp.P;  // then no CTA share is empty
  auto live_cta = [&](int cc) { return all_live || cta_begin(cc, vp.total, vp.P) < cta_begin(cc + 1, vp.total, vp.P); };
  auto rec_at = [&](int cc, int sq, int slot, int h) {
    return vp.rec + ((((int64_t)(cc + sq) * kSlots + slot) * G) + h) * kRecFloats<D>;
  };
  // count this CTA in on each of its segments (one atomic per segment, in parallel; acquire-release, so the
  // records written before the barrier above are published with it, and the CTA that completes a segment
  // sees every other CTA's record); that CTA merges the segment
  __shared__ int s_last[64];
  for (int sq0 = seg_first; sq0 <= seg_last; sq0 += 64) {
    const int n_here = min(64, seg_last - sq0 + 1);
    if (tid < n_here) {
      const int sq = sq0 + tid;
      const int s = sq / vp.h_kv, g = sq % vp.h_kv;
      const int nk = a.n_keep[s];
      const int64_t start = a.seg_base[s] + (int64_t)g * nk;
      const int c0 = cta_of(start, vp.total, vp.P), c1 = cta_of(start + nk - 1, vp.total, vp.P);
      uint32_t n_cov = 0;
      if (all_live)
        n_cov = c1 - c0 + 1;
      else
        for (int cc = c0; cc <= c1; ++cc) n_cov += live_cta(cc);
      const uint32_t prev = atom_add_acq_rel_gpu(&vp.seg_count[sq], 1u);
      s_last[tid] = prev + 1 == n_cov;
      if (prev + 1 == n_cov) vp.seg_count[sq] = 0;  // every CTA of the segment has counted: ready for the next call
    }
    __syncthreads();
    // 3. merge of the CTA records of each completed segment, up to 24 CTAs per round of independent loads
    for (int k = 0; k < n_here; ++k) {
      if (!s_last[k]) continue;
      const int sq = sq0 + k;
      const int s = sq / vp.h_kv, g = sq % vp.h_kv;
      const int nk = a.n_keep[s];
      const int64_t start = a.seg_base[s] + (int64_t)g * nk;
      const int c0 = cta_of(start, vp.total, vp.P), c1 = cta_of(start + nk - 1, vp.total, vp.P);
      for (int i = tid; i < G * Q4; i += kThreads) {
        const int h = i / Q4, d4 = i % Q4;
        float m_acc = -INFINITY, l_acc = 0.f;
        float4 o_acc = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kBatch = 24;  // records loaded together (one round of independent loads)
        for (int cb = c0; cb <= c1; cb += kBatch) {
          float2 ml[kBatch];
          float4 ov[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int cc = cb + u;
            ml[u] = make_float2(-INFINITY, 0.f);
            ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (cc <= c1 && live_cta(cc)) {
              const float* r = rec_at(cc, sq, kAttn, h);
              ml[u] = __ldcg(reinterpret_cast<const float2*>(r));
              ov[u] = __ldcg(reinterpret_cast<const float4*>(r + 4) + d4);
            }
          }
          float mb = m_acc;
#pragma unroll
          for (int u = 0; u < kBatch; ++u) mb = fmaxf(mb, ml[u].x);
          if (mb == -INFINITY) continue;  // only neutral records so far
          const float a0 = exp2f(m_acc - mb);  // 0 while m_acc is -inf
          l_acc *= a0;
          o_acc.x *= a0;
          o_acc.y *= a0;
          o_acc.z *= a0;
          o_acc.w *= a0;
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float a1 = exp2f(ml[u].x - mb);  // 0 for neutral records (m = -inf)
            l_acc = fmaf(ml[u].y, a1, l_acc);
            o_acc.x = fmaf(ov[u].x, a1, o_acc.x);
            o_acc.y = fmaf(ov[u].y, a1, o_acc.y);
            o_acc.z = fmaf(ov[u].z, a1, o_acc.z);
            o_acc.w = fmaf(ov[u].w, a1, o_acc.w);
          }
          m_acc = mb;
        }
        const float inv = l_acc > 0.f ? 1.f / l_acc : 0.f;
        reinterpret_cast<float4*>(vp.out + ((int64_t)s * vp.h_q + g * G + h) * D)[d4] =
            make_float4(o_acc.x * inv, o_acc.y * inv, o_acc.z * inv, o_acc.w * inv);
      }
    }
    __syncthreads();  // s_last is re-written for the next 64 segments
  }
}

// RoPE tables computed in fp64: base[slot][i] = (cos, sin)(32*slot*theta_i), off[r][i] = (cos, sin)(r*theta_i),
// theta_i = rope_theta^(-2i/d); each stored as the fp32 rounding (hi) and the fp32 rounding of what that
// dropped (lo), so hi + lo holds the value to ~2^-48.
__global__ void rope_table_kernel(float2* base, float2* base_lo, int n_slots, float2* off, float2* off_lo, int d,
                                  double rope_theta) {
  const int half = d / 2;
  const int64_t n = (int64_t)(n_slots + 32) * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = idx / half;
    const int i = (int)(idx % half);
    const double inv_freq = pow(rope_theta, -2.0 * i / d);
    const bool is_base = row < n_slots;
    double sn, cs;
    sincos((is_base ? 32.0 * (double)row : (double)(row - n_slots)) * inv_freq, &sn, &cs);
    const float ch = (float)cs, sh = (float)sn;
    const float2 hi = make_float2(ch, sh), lo = make_float2((float)(cs - (double)ch), (float)(sn - (double)sh));
    if (is_base) {
      base[row * half + i] = hi;
      base_lo[row * half + i] = lo;
    } else {
      off[(row - n_slots) * half + i] = hi;
      off_lo[(row - n_slots) * half + i] = lo;
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
  static_assert(Geo<D>::BYTES <= 227 * 1024 && Geo<D, true>::BYTES <= 227 * 1024, "view kernel shared memory");
  if (vp.total == 0 && !vp.any_empty) return cudaSuccess;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const ViewParams,
               const SessionArgs) =
      mode == 0 ? view_kernel<D, G, 0>
                : (mode == 1 ? view_kernel<D, G, 1> : (mode == 2 ? view_kernel<D, G, 2> : view_kernel<D, G, 2, true>));
  const uint32_t bytes = mode == 3 ? Geo<D, true>::BYTES : Geo<D>::BYTES;
  cudaError_t e = ensure_smem(kern, c.device, bytes);
  if (e != cudaSuccess) return e;
  const int threads = mode == 3 ? view_threads<true>() : view_threads<false>();
  return launch_pdl(kern, dim3(vp.P), dim3(threads), bytes, st, 1, maps[0], maps[1], maps[2], maps[3], vp, a);
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
                        cudaStream_t st, const float* k_scale, const float* v_scale) {
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
  vp.seg_count = c.seg_count;
  vp.rope_base = reinterpret_cast<const float2*>(c.rope_base);
  vp.rope_off = reinterpret_cast<const float2*>(c.rope_off);
  vp.rope_base_lo = reinterpret_cast<const float2*>(c.rope_base_lo);
  vp.rope_off_lo = reinterpret_cast<const float2*>(c.rope_off_lo);
  vp.out = out;
  vp.k_scale = k_scale;
  vp.v_scale = v_scale;
  vp.k8 = reinterpret_cast<const uint8_t*>(k_src);
  vp.v8 = reinterpret_cast<const uint8_t*>(v_src);
  vp.status = c.status;
  vp.total = a.seg_base[n_sessions];
  vp.any_empty = 0;
  for (int s = 0; s < n_sessions; ++s) vp.any_empty |= a.n_keep[s] == 0;
  vp.budget = c.budget;
  vp.h_kv = c.p.h_kv;
  vp.h_q = c.p.h_q;
  vp.n_sessions = n_sessions;
  // one CTA per SM, but never more CTAs than kept blocks: every CTA then has a non-empty share (a small view
  // would otherwise leave most CTAs idle and make the merge walk over empty shares)
  vp.P = (int)(vp.total > 0 && vp.total < c.view_ctas ? vp.total : c.view_ctas);
  vp.q_scale = (float)(1.4426950408889634 / sqrt((double)c.p.d));
  vp.wait_ns = c.wait_ns;
  vp.stall = c.stall_first_wait;
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
  } else if (mode == 3) {  // FP8 code pages come in by 1-D bulk copies: only the view maps are used
    if ((e = make_map(&maps[2], k_view, view_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[3], v_view, view_rows, c.p.d)) != cudaSuccess) return e;
    maps[0] = maps[2];
    maps[1] = maps[3];
  } else {
    if ((e = make_map(&maps[0], k_src, pool_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[1], v_src, pool_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[2], k_view, view_rows, c.p.d)) != cudaSuccess) return e;
    if ((e = make_map(&maps[3], v_view, view_rows, c.p.d)) != cudaSuccess) return e;
  }
  return c.p.d == 128 ? launch_d<128>(c, mode, maps, vp, a, st) : launch_d<64>(c, mode, maps, vp, a, st);
}

cudaError_t launch_rope_tables(const Ctx& c, cudaStream_t st) {
  rope_table_kernel<<<256, 256, 0, st>>>(reinterpret_cast<float2*>(c.rope_base),
                                         reinterpret_cast<float2*>(c.rope_base_lo), c.budget + 1,
                                         reinterpret_cast<float2*>(c.rope_off), reinterpret_cast<float2*>(c.rope_off_lo),
                                         c.p.d, (double)c.p.rope_theta);
  return cudaGetLastError();
}

// 4-D map over `rows` rows of d bf16 values whose boxes land in shared memory in the tensor cores' no-swizzle
// core-matrix order: dims (8 columns, 8 rows, d/8 column groups, rows/8 row groups), strides (2 B, 2d B, 16 B,
// 16d B), one box = 64 rows = 8 row groups.  Element (r, c) of a box is then at
// ((r / 8) * (d / 8) + c / 8) * 64 + (r % 8) * 8 + c % 8: 8 x 16-byte core matrices, adjacent along the columns
// 128 bytes apart and along the rows d * 16 bytes apart.  Rows past `rows` read as zeros.
cudaError_t make_core_matrix_map(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  memset(m, 0, sizeof(*m));
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (rows % 8 != 0 || d % 8 != 0) return cudaErrorInvalidValue;
  const cuuint64_t dims[4] = {8, 8, (cuuint64_t)d / 8, (cuuint64_t)rows / 8};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, 16, (cuuint64_t)d * 16};
  const cuuint32_t box[4] = {8, 8, (cuuint32_t)d / 8, 8};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kvm
