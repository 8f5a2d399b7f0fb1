// Attention of a step's query tokens over the execution view, on the
// 5th-generation tensor cores (tcgen05 + TMEM).
//
// Evolve review of KVMem, "Strengths": recall is scheduled once per agent
// step; KVMEM reproduction README, "Local reproduction": the view replaces
// full attention.  The step's T tokens are the history's last T tokens, so
// token t sits at view position p_t = L - T + t (the view's recent blocks hold
// it); its query, rotated at p_t, attends the view slots j <= p_t.  Per KV
// head g the R = T*G query rows (row r = t*G + hh) form a dense
// R x L x d contraction twice (scores, then P.V):
//   pack    queries rotated at p_t and scaled by log2(e)/sqrt(d), split into a
//           bf16 part and its bf16 residual, in the no-swizzle K-major
//           core-matrix layout (8 rows x 16 bytes per core matrix);
//   K, V    64-token tiles come straight from the view through 4-D tensor-map
//           boxes that land in the same core-matrix layout: a K tile is the
//           K-major B operand of the scores, a V tile the MN-major B operand
//           of P.V (no transposed copy); in the last tile the rows past the
//           view length are zeroed in shared memory before P.V reads them;
//   attend  per 128 query rows, over 64-token tiles of the view:
//             S  = Q_hi K^T + Q_lo K^T          (one fp32 TMEM accumulator)
//             P  = exp2(S - m) per row          (online softmax in registers)
//             O += P_hi V + P_lo V              (fp32 TMEM accumulator)
//           with the split operands giving fp32-accurate products on bf16 MMAs.
// Warp roles: warp 0 issues the copies, warp 1 owns TMEM and issues the
// MMAs (S of the next tile is issued before P.V of this one, into a second S
// buffer), warps 2..9 run the softmax in two streams (even and odd tiles), each
// thread owning one query row of its stream (a warp can only read its quarter
// of the 128 TMEM lanes).  A stream reads S, keeps its running maximum (raised
// only when it grows by more than 8, then its accumulator is rescaled in TMEM)
// and writes P to shared memory; at the end the two streams' states are merged
// and O / l is written to the output.
// Every mbarrier wait is bounded.
#include "kvm_device.cuh"
#include "kvm_internal.h"

namespace kvm {
namespace {

constexpr int kSoftWarps = 8;                   // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kSoftWarps;  // producer, MMA issuer, softmax warps
constexpr int kRows = 128;                      // query rows per CTA (MMA M)
constexpr int kTile = 64;                       // view tokens per tile (S: N = 64; P.V: K = 64)
static_assert(kTile == 64, "the softmax reductions are written for 64-token tiles");
constexpr uint32_t kTmemCols = 512;             // S/P[4] x 64 columns + O_0, O_1 (d columns each)

// Element (r, c) of a [rows][cols] bf16 matrix in the K-major core-matrix layout (cols = K).
__device__ __forceinline__ int64_t cm_index(int64_t r, int c, int cols) {
  return ((r >> 3) * (cols >> 3) + (c >> 3)) * 64 + (r & 7) * 8 + (c & 7);
}

// The view length the kernels work with: a length outside [n_q, Lcap] is reported by the query packing and
// clamped into that range, so every access stays inside the view buffers.
__device__ __forceinline__ int clamp_view_len(int L, int n_q, int Lcap) { return L < n_q ? n_q : (L > Lcap ? Lcap : L); }

// Query rows of KV head (s, g): rotated at p_t, scaled, split -> hi / lo packed [rows_pad][D].
template <int D>
__global__ void step_pack_q_kernel(const uint16_t* __restrict__ q, const int32_t* __restrict__ view_len, int n_q,
                                   int h_q, int h_kv, int group, int rows_pad, int Lcap,
                                   const float2* __restrict__ rope_base, const float2* __restrict__ rope_off,
                                   float q_scale, uint16_t* __restrict__ q_hi, uint16_t* __restrict__ q_lo,
                                   uint32_t* __restrict__ status) {
  griddep_wait();
  const int sg = blockIdx.y, s = sg / h_kv, g = sg % h_kv;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // (row, pair i < D/2)
  if (idx >= rows_pad * (D / 2)) return;
  const int row = idx / (D / 2), i = idx % (D / 2);
  float y1 = 0.f, y2 = 0.f;
  if (row < n_q * group) {
    const int L0 = view_len[sg];
    if ((L0 < n_q || L0 > Lcap) && i == 0) atomicOr(status, KVM_DEV_BAD_VIEW);
    const int L = clamp_view_len(L0, n_q, Lcap);
    const int t = row / group, hh = row % group;
    const int pos = L - n_q + t;
    const uint16_t* qh = q + (((int64_t)s * n_q + t) * h_q + g * group + hh) * D;
    const float x1 = __uint_as_float((uint32_t)qh[i] << 16), x2 = __uint_as_float((uint32_t)qh[i + D / 2] << 16);
    const float2 b = rope_base[(int64_t)(pos >> 5) * (D / 2) + i], o = rope_off[(pos & 31) * (D / 2) + i];
    const float cs = fmaf(b.x, o.x, -b.y * o.y), sn = fmaf(b.y, o.x, b.x * o.y);
    y1 = (x1 * cs - x2 * sn) * q_scale;
    y2 = (x2 * cs + x1 * sn) * q_scale;
  }
  const uint32_t h = pack_bf16x2(y1, y2);
  const uint32_t l = pack_bf16x2(y1 - bf16lo(h), y2 - bf16hi(h));
  uint16_t* dh = q_hi + (int64_t)sg * rows_pad * D;
  uint16_t* dl = q_lo + (int64_t)sg * rows_pad * D;
  dh[cm_index(row, i, D)] = (uint16_t)(h & 0xFFFFu);
  dh[cm_index(row, i + D / 2, D)] = (uint16_t)(h >> 16);
  dl[cm_index(row, i, D)] = (uint16_t)(l & 0xFFFFu);
  dl[cm_index(row, i + D / 2, D)] = (uint16_t)(l >> 16);
}

constexpr int kStages = 4;  // K tile stages and V tile stages in shared memory
constexpr int kSP = 4;      // S/P buffers in TMEM: two per stream

struct AttnBars {
  uint64_t q_full, k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[kSP], p_full[kSP], pv_done[kSP], drain, v_tail;
  uint64_t xch[4];  // per lane quarter: both softmax warps have published their row state
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A * B^T for one K = 16 slice with A in tensor memory (row i in lane i, two bf16 of
// consecutive K per 32-bit column: 8 columns per slice) and B described in shared memory.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int D>
constexpr size_t attn_smem_bytes() {
  return 2 * (size_t)kRows * D * 2 + 2 * (size_t)kStages * kTile * D * 2;
}
// dynamic + static (barriers and the row exchange buffer, under 3 KiB) within the 227 KiB a CTA may use
static_assert(attn_smem_bytes<128>() + 3 * 1024 <= 227 * 1024, "step attention: shared memory per CTA");

// grid (rows_pad / 128, chunks, S * h_kv): CTA (x, y, z) attends row tile x of KV head z over the view tiles
// of chunk y; with more than one chunk each CTA leaves an unnormalised partial state (O, max, sum) and the CTA
// completing a row tile merges the partials.
//
// Pipeline of tile j: stream j & 1 owns the softmax warps and accumulator O of tile j; S(j) and then P(j) live
// in TMEM buffer j % 4 (two per stream); K/V tiles rotate over kStages stages:
//   MMA issuer:  [P.V(j-2) done] S(j+2) = Q K(j+2)^T into buffer (j+2) % 4
//                [P(j) written]  O_(j&1) += P(j) V(j), P read from TMEM
//   softmax of stream j & 1:  [S(j) done] read S(j); [P.V(j-2) done] rescale O if the maximum rose;
//                write P(j) over S(j) in TMEM (bf16 part in the first 32 columns, residual in the last 32)
// so each stream's softmax overlaps the other stream's MMAs, and no probability passes through shared memory.
// Every barrier is waited on at most one phase behind its newest completed phase (each buffer's next phase
// needs a step the waiter has not taken).
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) step_attn_kernel(
    const uint16_t* __restrict__ q_hi, const uint16_t* __restrict__ q_lo, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ view_len, int n_q, int rows_pad, int Lcap,
    int h_kv, int h_q, int kv_chunk, float* __restrict__ part, uint32_t* __restrict__ cnt, float* __restrict__ out,
    uint32_t* __restrict__ status) {
  constexpr uint32_t Q_BYTES = kRows * D * 2, KV_BYTES = kTile * D * 2;
  // core matrices: K-major operands (Q, K) step 128 bytes along K and D * 16 bytes across 8-row groups; the
  // MN-major V tile steps 128 bytes along MN (dims) and D * 16 bytes along K (8-token groups)
  constexpr uint32_t SBO_Q = D / 8 * 128, LBO = 128, LBO_V = D * 16, SBO_V = 128;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(kRows, kTile);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(kRows, D) | (1u << 16);  // B (V) is MN-major
  extern __shared__ __align__(128) unsigned char smem[];  // no-swizzle operands need 16-byte alignment
  unsigned char* qh_s = smem;
  unsigned char* ql_s = qh_s + Q_BYTES;
  unsigned char* v_s = ql_s + Q_BYTES;            // [kStages] V tiles
  unsigned char* k_s = v_s + kStages * KV_BYTES;  // [kStages] K tiles
  __shared__ AttnBars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float xval[2][2][kRows];  // [max, sum][stream][row]: each stream's softmax state at the end

  griddep_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = blockIdx.z, s = sg / h_kv, g = sg % h_kv;
  const int row0 = blockIdx.x * kRows;
  const int L = clamp_view_len(view_len[sg], n_q, Lcap);
  // tiles up to the last view position any row of this CTA attends (the step's token rows are ordered by t)
  const int last_row = min(n_q * G, row0 + kRows) - 1;
  const int nt_full = (L - n_q + last_row / G + kTile) / kTile;
  // this CTA's chunk of the row tile's view tiles: [kv0, kv0 + nt)
  const int splits = gridDim.y, kv0 = blockIdx.y * kv_chunk;
  const int nt = min(nt_full - kv0, kv_chunk);
  if (nt <= 0) return;  // past the view: the chunk count of this row tile does not include it
  KVM_DEBUG_CHECK(row0 < rows_pad && (int64_t)(kv0 + nt) * kTile <= (int64_t)Lcap + kTile, status);
  __shared__ int s_last;

  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < kSP; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], kSoftWarps / 2);
      mbar_init(&bars.pv_done[i], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars.xch[i], 2);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.v_tail, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tm_o = tmem + kSP * kTile;  // O_0 (even tiles), then O_1 (odd tiles)

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // K tiles run two tiles ahead of V tiles (scores are computed two tiles ahead of P.V)
    mbar_arrive_expect_tx(&bars.q_full, 2 * Q_BYTES);
    bulk_g2s(qh_s, q_hi + ((int64_t)sg * rows_pad + row0) * D, Q_BYTES, &bars.q_full);
    bulk_g2s(ql_s, q_lo + ((int64_t)sg * rows_pad + row0) * D, Q_BYTES, &bars.q_full);
    int nk = 0, nv = 0;  // tiles whose K / V copy was issued
    for (int i = 0; i < nt + 2 && !abort_flag; ++i) {
      if (i < nt) {
        const int sk = i % kStages;
        if (i >= kStages && !mbar_wait(&bars.k_empty[sk], (i / kStages - 1) & 1, status)) {
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&bars.k_full[sk], KV_BYTES);
        tma_load_4d(k_s + sk * KV_BYTES, &tm_k, 0, 0, 0, (sg * Lcap + (kv0 + i) * kTile) / 8, &bars.k_full[sk]);
        nk = i + 1;
      }
      const int jv = i - 2;
      if (jv >= 0) {
        const int sv = jv % kStages;
        if (jv >= kStages && !mbar_wait(&bars.v_empty[sv], (jv / kStages - 1) & 1, status)) {
          abort_flag = 1;
          break;
        }
        const int tok0 = (kv0 + jv) * kTile, y = (sg * Lcap + tok0) / 8;
        unsigned char* vt = v_s + sv * KV_BYTES;
        if (tok0 + kTile <= L) {
          mbar_arrive_expect_tx(&bars.v_full[sv], KV_BYTES);
          tma_load_4d(vt, &tm_v, 0, 0, 0, y, &bars.v_full[sv]);
        } else {
          // the view's last tile: its rows past the view length (unwritten view slots, possibly not finite) are
          // zeroed before P.V, whose probabilities there are zero, reads them
          mbar_arrive_expect_tx(&bars.v_tail, KV_BYTES);
          tma_load_4d(vt, &tm_v, 0, 0, 0, y, &bars.v_tail);
          if (!mbar_wait(&bars.v_tail, 0, status)) {
            abort_flag = 1;
            break;
          }
          for (int r = L - tok0; r < kTile; ++r)
#pragma unroll 4
            for (int c8 = 0; c8 < D / 8; ++c8)
              *reinterpret_cast<uint4*>(vt + ((r >> 3) * (D / 8) + c8) * 128 + (r & 7) * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();  // visible to the tensor cores
          mbar_arrive(&bars.v_full[sv]);
        }
        nv = jv + 1;
      }
    }
    // copies in flight must land before the CTA can exit
    mbar_wait(&bars.q_full, 0, status);
    for (int i = max(0, nk - kStages); i < nk; ++i) mbar_wait(&bars.k_full[i % kStages], (i / kStages) & 1, status);
    for (int i = max(0, nv - kStages); i < nv; ++i) mbar_wait(&bars.v_full[i % kStages], (i / kStages) & 1, status);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t qh_a = smem_addr(qh_s), ql_a = smem_addr(ql_s);
    // S(j) into TMEM buffer j % 4 once P.V(j - 4), the last reader of that buffer, is done
    auto issue_s = [&](int j) -> bool {
      const int sk = j % kStages, sb = j % kSP;
      if (!mbar_wait(&bars.k_full[sk], (j / kStages) & 1, status)) return false;
      if (j >= kSP && !mbar_wait(&bars.pv_done[sb], (j / kSP - 1) & 1, status)) return false;
      tc_fence_after();
      const uint32_t k_a = smem_addr(k_s + sk * KV_BYTES);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16(tmem + sb * kTile, smem_desc(qh_a + kk * 256, LBO, SBO_Q), smem_desc(k_a + kk * 256, LBO, SBO_Q),
                 IDESC_S, kk > 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16(tmem + sb * kTile, smem_desc(ql_a + kk * 256, LBO, SBO_Q), smem_desc(k_a + kk * 256, LBO, SBO_Q),
                 IDESC_S, 1);
      mma_commit(&bars.s_full[sb]);
      mma_commit(&bars.k_empty[sk]);
      return true;
    };
    bool ok = mbar_wait(&bars.q_full, 0, status);
    for (int j = 0; ok && j < 2 && j < nt; ++j) ok = issue_s(j);
    for (int j = 0; ok && j < nt && !abort_flag; ++j) {
      const int sv = j % kStages, pb = j % kSP;
      if (j + 2 < nt && !issue_s(j + 2)) {
        ok = false;
        break;
      }
      if (!mbar_wait(&bars.p_full[pb], (j / kSP) & 1, status) || !mbar_wait(&bars.v_full[sv], (j / kStages) & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t v_a = smem_addr(v_s + sv * KV_BYTES);
      const uint32_t p_t = tmem + pb * kTile;  // P(j): bf16 part in columns 0..31, residual in 32..63
      const uint32_t o = tm_o + (j & 1) * D;   // this tile's stream accumulator
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        // 16 tokens per MMA: two 8-token core-matrix groups along K
        mma_bf16_tmem_a(o, p_t + kk * 8, smem_desc(v_a + kk * 2 * LBO_V, LBO_V, SBO_V), IDESC_O, (j >= 2 || kk > 0));
        mma_bf16_tmem_a(o, p_t + kTile / 2 + kk * 8, smem_desc(v_a + kk * 2 * LBO_V, LBO_V, SBO_V), IDESC_O, 1);
      }
      mma_commit(&bars.pv_done[pb]);
      mma_commit(&bars.v_empty[sv]);
    }
    if (!ok) abort_flag = 1;
    // every issued MMA has completed before TMEM is released
    mma_commit(&bars.drain);
    mbar_wait(&bars.drain, 0, status);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / epilogue, one query row per thread
    // Two streams: warps 2..5 take the even tiles, warps 6..9 the odd ones, each with its own running maximum
    // m, sum l and accumulator (O_0 or O_1), so one stream's softmax overlaps the other's MMAs.  The streams
    // are merged once, at the end.
    const int quarter = warp & 3, stream = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
    const int row = row0 + r;
    const bool valid_row = row < n_q * G;
    const int t = row / G, hh = row % G;
    const int pos = valid_row ? L - n_q + t : -1;  // this row's view position; it attends slots <= pos
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t my_o = tm_o + lane_base + stream * D;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = stream; j < nt; j += 2) {
      const int sb = j % kSP;
      const uint32_t my_s = tmem + lane_base + sb * kTile;
      if (__any_sync(0xffffffffu, abort_flag) || !mbar_wait_warp(&bars.s_full[sb], (j / kSP) & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(my_s, sv[0]);
      tmem_ld32(my_s + 32, sv[1]);
      tmem_wait_ld();
      const int tok0 = (kv0 + j) * kTile;
      float x[kTile];
      if (__all_sync(0xffffffffu, tok0 + kTile - 1 <= pos)) {  // no masked column in this tile
#pragma unroll
        for (int c = 0; c < kTile; ++c) x[c] = __uint_as_float(sv[c >> 5][c & 31]);
      } else {
#pragma unroll
        for (int c = 0; c < kTile; ++c) x[c] = tok0 + c <= pos ? __uint_as_float(sv[c >> 5][c & 31]) : -INFINITY;
      }
      // tree maximum (short dependency chains)
      float mx[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) mx[i] = fmaxf(fmaxf(x[i], x[i + 16]), fmaxf(x[i + 32], x[i + 48]));
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) mx[i] = fmaxf(mx[i], mx[i + w]);
      const float mt = mx[0];
      // raise the reference only when it grows by more than 8 (a factor 256): O is then rescaled in TMEM
      const float m_new = (mt > m + 8.f) ? mt : m;
      const float corr = m_new == m ? 1.f : fast_exp2(m - m_new);  // 0 while m was -inf
      if (j >= 2 && __any_sync(0xffffffffu, m_new != m)) {
        // the stream's accumulator must be quiescent: P.V(j - 2), its last, is done
        if (!mbar_wait_warp(&bars.pv_done[(j - 2) % kSP], ((j - 2) / kSP) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(my_o + cc * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
          tmem_st32(my_o + cc * 32, ov);
        }
      }
      l *= corr;
      m = m_new;
      // P = exp2(S - m), split into bf16 + residual, written over S(j): two bf16 of consecutive tokens per column
      const bool live = m != -INFINITY;  // padding rows: zeros
      float ls[4] = {0.f, 0.f, 0.f, 0.f};  // partial sums (short dependency chains)
      uint32_t ph[kTile / 2], pl[kTile / 2];
#pragma unroll
      for (int c = 0; c < kTile / 2; ++c) {
        const float p0 = live ? fast_exp2(x[2 * c] - m) : 0.f;
        const float p1 = live ? fast_exp2(x[2 * c + 1] - m) : 0.f;
        ls[c & 3] += p0 + p1;
        ph[c] = pack_bf16x2(p0, p1);
        pl[c] = pack_bf16x2(p0 - bf16lo(ph[c]), p1 - bf16hi(ph[c]));
      }
      tmem_st32(my_s, ph);
      tmem_st32(my_s + kTile / 2, pl);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[sb]);
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
    }
    if (!ok) abort_flag = 1;
    if (ok && nt > 0) {
      // merge the streams: O = (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) / (l_0 2^(m_0 - M) + l_1 2^(m_1 - M));
      // a stream without tiles (nt == 1) has m = -inf and an accumulator that was never written
      xval[0][stream][r] = m;
      xval[1][stream][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.xch[quarter]);
      const int last = (nt - 1) - ((nt - 1 - stream) & 1);  // this stream's last tile
      const int other_last = (nt - 1) - ((nt - 1 - (stream ^ 1)) & 1);
      // both streams' accumulators are read: wait for each stream's last P.V
      ok = mbar_wait_warp(&bars.xch[quarter], 0, status) &&
           (last < 0 || mbar_wait_warp(&bars.pv_done[last % kSP], (last / kSP) & 1, status)) &&
           (other_last < 0 || mbar_wait_warp(&bars.pv_done[other_last % kSP], (other_last / kSP) & 1, status));
      if (ok) {
        tc_fence_after();
        const float m0 = xval[0][0][r], m1 = xval[0][1][r];
        const float M = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M), f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
        const float lt = xval[1][0][r] * f0 + xval[1][1][r] * f1;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const bool split = splits > 1;  // a chunk of the row: unnormalised partial state, merged below
        const float w0 = split ? f0 : f0 * inv, w1 = split ? f1 : f1 * inv;
        const bool use1 = nt > 1;  // O_1 holds data only when the odd stream had a tile
        float* pu = part + ((int64_t)(sg * gridDim.x + blockIdx.x) * splits + blockIdx.y) * (kRows * (D + 2));
        if (split && stream == 0) *reinterpret_cast<float2*>(pu + kRows * D + 2 * r) = make_float2(M, lt);
        float* dst = split ? pu + (int64_t)r * D : out + (((int64_t)s * n_q + t) * h_q + g * G + hh) * D;
        // the two warps of a quarter split the d columns
#pragma unroll 1
        for (int cc = stream * (D / 64); cc < (stream + 1) * (D / 64); ++cc) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tm_o + lane_base + cc * 32, o0);
          tmem_ld32(tm_o + lane_base + D + cc * 32, o1);
          tmem_wait_ld();
          if (valid_row || split) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 v;
              v.x = __uint_as_float(o0[i]) * w0 + (use1 ? __uint_as_float(o1[i]) * w1 : 0.f);
              v.y = __uint_as_float(o0[i + 1]) * w0 + (use1 ? __uint_as_float(o1[i + 1]) * w1 : 0.f);
              v.z = __uint_as_float(o0[i + 2]) * w0 + (use1 ? __uint_as_float(o1[i + 2]) * w1 : 0.f);
              v.w = __uint_as_float(o0[i + 3]) * w0 + (use1 ? __uint_as_float(o1[i + 3]) * w1 : 0.f);
              *reinterpret_cast<float4*>(dst + cc * 32 + i) = v;
            }
          }
        }
      }
    }
  }
  if (splits > 1) __threadfence();  // this thread's partial rows, before the chunk is counted
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (splits > 1) {
    // the CTA that completes a row tile's chunks merges them (no CTA waits on another)
    const int rt_id = sg * gridDim.x + blockIdx.x;
    const int expected = (nt_full + kv_chunk - 1) / kv_chunk;
    if (tid == 0) s_last = atomicAdd(&cnt[rt_id], 1u) + 1 == (uint32_t)expected;
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float* pr = part + (int64_t)rt_id * splits * (kRows * (D + 2));
      for (int item = tid; item < kRows * (D / 4); item += kThreads) {
        const int r = item / (D / 4), c4 = item % (D / 4), row = row0 + r;
        if (row >= n_q * G) continue;
        float Mx = -INFINITY;
        for (int k = 0; k < expected; ++k) Mx = fmaxf(Mx, __ldcg(pr + (int64_t)k * (kRows * (D + 2)) + kRows * D + 2 * r));
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < expected; ++k) {
          const float* pk = pr + (int64_t)k * (kRows * (D + 2));
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(pk + kRows * D + 2 * r));
          if (ml.x == -INFINITY) continue;
          const float w = fast_exp2(ml.x - Mx);
          Ls += w * ml.y;
          const float4 o = __ldcg(reinterpret_cast<const float4*>(pk + (int64_t)r * D) + c4);
          acc.x += w * o.x;
          acc.y += w * o.y;
          acc.z += w * o.z;
          acc.w += w * o.w;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const int t = row / G, hh = row % G;
        reinterpret_cast<float4*>(out + (((int64_t)s * n_q + t) * h_q + g * G + hh) * D)[c4] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
      if (tid == 0) cnt[rt_id] = 0;  // ready for the next call
    }
  }
}

template <int D, int G>
cudaError_t launch_dg(const Ctx& c, const uint16_t* q, int n_q, const uint16_t* k_view, const uint16_t* v_view,
                      const int32_t* view_len, int n_sessions, float* out, cudaStream_t st) {
  const int SG = n_sessions * c.p.h_kv;
  const int rows_pad = (n_q * G + kRows - 1) / kRows * kRows;  // query rows per KV head, padded to the CTA tile
  const int Lcap = 32 * c.budget;
  cudaError_t e;
  const int nqp = rows_pad * (D / 2);
  if ((e = launch_pdl(step_pack_q_kernel<D>, dim3((nqp + 255) / 256, SG), dim3(256), 0, st, 1, q, view_len, n_q,
                      c.p.h_q, c.p.h_kv, G, rows_pad, Lcap, reinterpret_cast<const float2*>(c.rope_base),
                      reinterpret_cast<const float2*>(c.rope_off), (float)(1.4426950408889634 / sqrt((double)D)),
                      c.attn_q, c.attn_q + (int64_t)SG * rows_pad * D, c.status)) != cudaSuccess)
    return e;
  // K and V tiles of every KV head's view, read in place (rows past the last head read as zeros)
  CUtensorMap tm_k, tm_v;
  if ((e = make_core_matrix_map(&tm_k, k_view, (uint64_t)SG * Lcap, D)) != cudaSuccess ||
      (e = make_core_matrix_map(&tm_v, v_view, (uint64_t)SG * Lcap, D)) != cudaSuccess)
    return e;
  const size_t smem = attn_smem_bytes<D>();
  auto ka = step_attn_kernel<D, G>;
  if ((e = ensure_smem(ka, c.device, smem)) != cudaSuccess) return e;
  // Split each row tile's view tiles into chunks when the row tiles alone leave SMs idle: the chunk count
  // minimises (CTA waves) x (chunk length + a fixed cost per chunk), within the partial-state scratch.
  const int rt = rows_pad / kRows * SG;
  const int tiles_max = (Lcap + kTile - 1) / kTile;
  int splits = 1;
  if (2 * rt <= c.attn_units_cap && rt < c.num_sms) {
    double best = 1e30;
    for (int sp = 1; sp <= 16 && sp * rt <= c.attn_units_cap && sp <= tiles_max; ++sp) {
      const double waves = (double)((rt * sp + c.num_sms - 1) / c.num_sms);
      const double cost = waves * (1.0 / sp + 0.03);
      if (cost < best - 1e-9) {
        best = cost;
        splits = sp;
      }
    }
  }
  const int kv_chunk = (tiles_max + splits - 1) / splits;
  return launch_pdl(ka, dim3(rows_pad / kRows, splits, SG), dim3(kThreads), smem, st, 1, (const uint16_t*)c.attn_q,
                    (const uint16_t*)(c.attn_q + (int64_t)SG * rows_pad * D), tm_k, tm_v, view_len, n_q, rows_pad,
                    Lcap, c.p.h_kv, c.p.h_q, kv_chunk, c.attn_part, c.attn_cnt, out, c.status);
}

template <int D>
cudaError_t launch_d(const Ctx& c, const uint16_t* q, int n_q, const uint16_t* k_view, const uint16_t* v_view,
                     const int32_t* view_len, int n_sessions, float* out, cudaStream_t st) {
  switch (c.group) {
    case 1: return launch_dg<D, 1>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 2: return launch_dg<D, 2>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 3: return launch_dg<D, 3>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 4: return launch_dg<D, 4>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 5: return launch_dg<D, 5>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 6: return launch_dg<D, 6>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 7: return launch_dg<D, 7>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
    case 8: return launch_dg<D, 8>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_step_attn(const Ctx& c, const uint16_t* q, int n_q, const uint16_t* k_view, const uint16_t* v_view,
                             const int32_t* view_len, int n_sessions, float* out, cudaStream_t st) {
  return c.p.d == 128 ? launch_d<128>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st)
                      : launch_d<64>(c, q, n_q, k_view, v_view, view_len, n_sessions, out, st);
}

}  // namespace kvm
