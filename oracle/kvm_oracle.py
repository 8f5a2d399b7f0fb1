"""Oracle for the KVMem decode hot path: a plain, slow, fp64 CPU restatement.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs import this module.  The CUDA
library never calls it, and it shares no code with the CUDA library: the two
meet only at the seeded inputs of the ``synth`` package.

Sources (web pages on KVMem, arXiv 2609.04852):
  [README] "KVMEM: Virtualizing a million-token agent workspace with paged KV"
           (auto-research reproduction README)
  [REVIEW] "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU"
           (Evolve review)

Every function states the passage it follows.  Where the pages leave a step
open, the reading taken is marked READING.  The CPU tests in
tests/test_oracle_pins.py pin each function against brute force, closed
forms, invariants or library routines.

Layouts (bf16 is carried as its uint16 bit pattern):
  pool      uint16 [n_pages][h_kv][32][d]   pre-RoPE keys / values; a page holds one block of every KV head
  page_of   int32  [n_blk]                  logical block -> physical page (the block table row)
  index     f64    [h_kv][n_blk][d]         Mean-K vectors
  q         uint16 [h_q][d]                 post-q-norm, pre-RoPE query (one decode token)
"""
from __future__ import annotations

import numpy as np

BLOCK = 32  # tokens per block: [REVIEW] "Summary" (relevant 32-token blocks)


# --------------------------------------------------------------------------- bf16
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (bf16 = the top 16 bits of an IEEE fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round fp64 values to bf16 (8 significant bits), nearest-even, in one step.

    READING: every bf16 conversion rounds to nearest even.  Rounding straight
    from fp64 (not via fp32) avoids double rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # |x| = m * 2**e with m in [0.5, 1)
    q = np.maximum(e - 8, -133)             # spacing of 8-bit significands; bf16 subnormal floor
    r = np.rint(np.ldexp(x, -q))            # ties to even
    y = np.ldexp(r, q).astype(np.float32)   # exact: r has at most 8 bits
    return (y.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------- paging
def paged_tokens(pool, page_of, head: int, n_tok: int) -> np.ndarray:
    """Tokens [n_tok][d] of one head, read through the block table.

    [README] "Background and main changes": history is kept as paged KV; block
    b of the history lives in physical page page_of[b].
    """
    n_blk = -(-n_tok // BLOCK)
    pages = np.asarray(pool)[np.asarray(page_of)[:n_blk], head]      # [n_blk][32][d]
    return pages.reshape(n_blk * BLOCK, pages.shape[-1])[:n_tok]


# --------------------------------------------------------------------------- step 1: index
def mean_k_index(keys_bits) -> np.ndarray:
    """Mean-K vectors k_bar_b = mean of the keys in block b: [n_blk][d].

    [README] "Core equation" (index vector k_bar_b) and [REVIEW] "Summary"
    (position-independent Mean-K index over 32-token blocks).  The keys are
    pre-RoPE, so the mean does not depend on where the block sits.
    READING: a partial last block is the mean over the tokens present.
    """
    k = bf16_to_f64(keys_bits)
    n_tok, d = k.shape
    n_full = n_tok // BLOCK
    out = np.empty((-(-n_tok // BLOCK), d))
    out[:n_full] = k[:n_full * BLOCK].reshape(n_full, BLOCK, d).mean(axis=1)
    if n_tok % BLOCK:
        out[n_full] = k[n_full * BLOCK:].mean(axis=0)
    return out


def mean_k_index_bf16(keys_bits) -> np.ndarray:
    """Mean-K vectors as the bf16 operand of step-level (tensor-core) scoring: uint16 [n_blk][d].

    READING: the step-level scoring contraction takes bf16 operands, so the
    index vector is rounded to bf16 (nearest even) first.  The oracle rounds
    the exact mean (``mean_k_index``); a kernel that rounds its fp32 mean can
    land one bf16 step away where the exact mean lies within the fp32 error
    of a rounding midpoint, and the parity tests bound that effect.
    """
    return f64_to_bf16(mean_k_index(keys_bits))


def index_append(index, keys_bits, tok_begin: int, n_tok: int) -> np.ndarray:
    """Index after tokens [tok_begin, tok_begin + n_tok) were appended.

    Every block the range touches is recomputed from the keys present (no
    running-sum state); other rows are left as they were.  ``keys_bits`` holds
    all tokens of the history up to tok_begin + n_tok.
    """
    total = tok_begin + n_tok
    new = np.array(index, dtype=np.float64, copy=True)
    n_blk = -(-total // BLOCK)
    if new.shape[0] < n_blk:
        new = np.concatenate([new, np.zeros((n_blk - new.shape[0], new.shape[1]))])
    if n_tok == 0:
        return new
    for b in range(tok_begin // BLOCK, n_blk):
        rows = np.asarray(keys_bits)[b * BLOCK:min(total, b * BLOCK + BLOCK)]
        new[b] = bf16_to_f64(rows).mean(axis=0)
    return new


# --------------------------------------------------------------------------- quantised KV pages (FP8 E4M3)
# [README] "Background and main changes" (the deployment runs the model in NVFP4) -- the pages give no
# precision for the paged KV itself.  READING for the quantised-page variant: FP8 E4M3 codes (the OCP 8-bit
# floating-point format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, exponent 15
# with mantissa 7 is NaN, largest finite 448) with one fp32 scale per (page, KV head), for K and for V
# separately; a value is code * scale.  Both quantisation decisions (the scale and each code) are taken in
# fp32, the precision of the kernels.
E4M3_MAX = 448.0


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of E4M3 codes: (-1)^s 2^(e-7) (1 + m/8) for e > 0, (-1)^s 2^-6 (m/8) for e = 0."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e, m = (c >> 3) & 0xF, c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


_E4M3_POS = e4m3_to_f64(np.arange(127, dtype=np.uint8))   # the finite non-negative values, ascending


def f32_to_e4m3(x) -> np.ndarray:
    """Round (fp32) values to E4M3 codes: nearest, ties to even, magnitudes beyond 448 saturate to 448.

    The spacing of E4M3 values is 2^(E-3) in the binade [2^E, 2^(E+1)) for E >= -6, and 2^-9 below 2^-6
    (subnormals); rounding |x| on that grid with ties to even gives the nearest value, then the code is looked
    up.  The sign is kept (negative zero included); NaN gives the NaN code 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                            # a = f 2^e, f in [0.5, 1): binade exponent E = e - 1
    q = np.maximum(e - 4, -9)                     # log2 of the spacing
    v = np.minimum(np.ldexp(np.rint(np.ldexp(a, -q)), q), E4M3_MAX)
    v = np.where(np.isnan(a), 0.0, v)
    code = np.searchsorted(_E4M3_POS, v).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def quantize_page(x_bits):
    """One page of one KV head, bf16 [32][d] -> (E4M3 codes uint8 [32][d], fp32 scale).

    READING: scale = amax / 448 in fp32 (amax = the largest |x| of the page as stored, all 32 rows); each
    code = E4M3(x / scale) with the division in fp32; a page of zeros gets scale 1.  The largest element
    then maps to +-448 exactly.
    """
    x = bf16_to_f64(x_bits).astype(np.float32)
    amax = np.float32(np.max(np.abs(x)))
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    return f32_to_e4m3(np.float32(x) / scale), scale


def quantize_pool(pool_bits):
    """Every page of a pool: (codes uint8 [n_pages][h_kv][32][d], scales fp32 [n_pages][h_kv])."""
    pool_bits = np.asarray(pool_bits)
    n_pages, h_kv = pool_bits.shape[:2]
    codes = np.empty(pool_bits.shape, dtype=np.uint8)
    scales = np.empty((n_pages, h_kv), dtype=np.float32)
    for p in range(n_pages):
        for g in range(h_kv):
            codes[p, g], scales[p, g] = quantize_page(pool_bits[p, g])
    return codes, scales


def dequantize(codes, scale) -> np.ndarray:
    """Values of quantised elements: the fp32 product code * scale (one rounding), as fp64."""
    return (e4m3_to_f64(codes).astype(np.float32) * np.float32(scale)).astype(np.float64)


def paged_dequant_tokens(codes_pool, scales, page_of, head: int, n_tok: int) -> np.ndarray:
    """Dequantised tokens [n_tok][d] of one head, read through the block table."""
    n_blk = -(-n_tok // BLOCK)
    pages = np.asarray(page_of)[:n_blk]
    vals = np.stack([dequantize(np.asarray(codes_pool)[p, head], np.asarray(scales)[p, head]) for p in pages])
    return vals.reshape(n_blk * BLOCK, vals.shape[-1])[:n_tok]


def mean_k_index_of(keys) -> np.ndarray:
    """Mean-K vectors of keys given as values (fp64 [n_tok][d]): the definition of mean_k_index."""
    k = np.asarray(keys, dtype=np.float64)
    n_tok, d = k.shape
    n_full = n_tok // BLOCK
    out = np.empty((-(-n_tok // BLOCK), d))
    out[:n_full] = k[:n_full * BLOCK].reshape(n_full, BLOCK, d).mean(axis=1)
    if n_tok % BLOCK:
        out[n_full] = k[n_full * BLOCK:].mean(axis=0)
    return out


def materialize_values(keys, values, ids, n_tok: int, theta: float):
    """Execution view of one KV head from keys / values given as values (dequantised pages):
    (K_view bits, V_view bits), each [L][d].  As ``materialize``, with the value view rounded to bf16
    (nearest even) since the dequantised values are not bf16.
    """
    rows = view_rows(ids, n_tok)
    k_view = f64_to_bf16(rope(np.asarray(keys, dtype=np.float64)[rows], np.arange(rows.size), theta))
    v_view = f64_to_bf16(np.asarray(values, dtype=np.float64)[rows])
    return k_view, v_view


# --------------------------------------------------------------------------- step 2: scores
def block_scores(q_bits, index) -> np.ndarray:
    """s[h, b] = <q_h, k_bar_b of h's KV head> / sqrt(d): [h_q][n_blk].

    [README] "Core equation": s_b = <q, k_bar_b>/sqrt(d).  [README] "2026-09-08
    validation correction": the query is the normalised one (the inputs are
    post-q-norm).  Query head h reads KV head h // (h_q / h_kv).
    """
    q = bf16_to_f64(q_bits)
    h_q, d = q.shape
    h_kv = index.shape[0]
    group = h_q // h_kv
    s = np.empty((h_q, index.shape[1]))
    for h in range(h_q):
        s[h] = index[h // group] @ q[h] / np.sqrt(d)
    return s


def gqa_softmax_sum(s, h_kv: int) -> np.ndarray:
    """Gs[g, b] = sum over the heads h of group g of softmax_b(s[h, :])[b].

    [README] "2026-09-08 validation correction": the withdrawn run averaged the
    GQA query heads before the softmax; the corrected method takes the softmax
    per head first.  READING: the softmax runs over all blocks of the history
    (sink and recent included); the probabilities are then summed, not
    averaged, over the group.
    """
    s = np.asarray(s, dtype=np.float64)
    h_q, n_blk = s.shape
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p.reshape(h_kv, h_q // h_kv, n_blk).sum(axis=1)


def step_group_scores_bf16(q_steps_bits, index_bf16_bits) -> np.ndarray:
    """Step-level group scores with the bf16 index operand (fp64 arithmetic on the bf16 values)."""
    return step_group_scores(q_steps_bits, bf16_to_f64(index_bf16_bits))


def step_group_scores(q_steps_bits, index) -> np.ndarray:
    """Step-level scoring of several query tokens at once: Gs summed over queries.

    [REVIEW] "Strengths" (step-level recall scheduling: one selection per agent
    step).  READING: each (query token, head) row gets its own softmax over
    blocks; Gs[g, b] sums the probabilities over the step's query tokens and
    over the heads of group g.
    """
    q_steps_bits = np.asarray(q_steps_bits)
    h_kv = index.shape[0]
    total = np.zeros((h_kv, index.shape[1]))
    for t in range(q_steps_bits.shape[0]):
        total += gqa_softmax_sum(block_scores(q_steps_bits[t], index), h_kv)
    return total


def withdrawn_group_scores(q_bits, index) -> np.ndarray:
    """The withdrawn scoring, kept only as a contrast: the group's query heads
    are averaged (without re-normalising) before one softmax per KV head.

    [README] "2026-09-08 validation correction" (the variant the authors withdrew).
    """
    q = bf16_to_f64(q_bits)
    h_q, d = q.shape
    h_kv = index.shape[0]
    qbar = q.reshape(h_kv, h_q // h_kv, d).mean(axis=1)
    out = np.empty((h_kv, index.shape[1]))
    for g in range(h_kv):
        s = index[g] @ qbar[g] / np.sqrt(d)
        p = np.exp(s - s.max())
        out[g] = p / p.sum()
    return out


# --------------------------------------------------------------------------- step 3: selection
def select_blocks(gs_row, n_blk: int, n_sink: int, n_recent: int, top_k: int) -> np.ndarray:
    """Kept block ids of one KV head, ascending.

    [README] "Core equation": the selected KV is concatenated within the block
    budget.  READINGS: blocks [0, n_sink) (sink) and the last n_recent blocks
    are always kept; the top_k best of the remaining candidates by group score
    are added, the lower id winning a tie; if the history has no more blocks
    than the budget, every block is kept.  Output is in original order.
    """
    if n_blk <= n_sink + n_recent + top_k:
        return np.arange(n_blk, dtype=np.int64)
    gs_row = np.asarray(gs_row, dtype=np.float64)
    cand = np.arange(n_sink, n_blk - n_recent, dtype=np.int64)
    order = np.lexsort((cand, -gs_row[cand]))       # score descending, then id ascending
    chosen = cand[order[:top_k]]
    forced = np.concatenate([np.arange(n_sink), np.arange(n_blk - n_recent, n_blk)]).astype(np.int64)
    return np.sort(np.concatenate([forced, chosen]))


def kth_candidate_score(gs_row, n_blk: int, n_sink: int, n_recent: int, top_k: int) -> float:
    """Group score of the last candidate selected (the boundary of the top-k)."""
    if n_blk <= n_sink + n_recent + top_k:
        return float("nan")
    cand = np.asarray(gs_row, dtype=np.float64)[n_sink:n_blk - n_recent]
    return float(np.sort(cand)[::-1][top_k - 1])


# --------------------------------------------------------------------------- step 4: view
def rope(x, pos, theta: float) -> np.ndarray:
    """Rotary position embedding at position(s) ``pos``, fp64.

    [REVIEW] "Summary" / "Scope & Claims" (position-consistent re-RoPE).
    READING: the rotate-half pairing of Qwen models, dimension i paired with
    i + d/2, angle pos * theta**(-2i/d), the full head dimension rotated.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def view_rows(ids, n_tok: int) -> np.ndarray:
    """History token of each view slot: the kept blocks' tokens, in block order."""
    rows = [np.arange(b * BLOCK, min(n_tok, b * BLOCK + BLOCK)) for b in np.asarray(ids, dtype=np.int64)]
    return np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)


def materialize(keys_bits, values_bits, ids, n_tok: int, theta: float):
    """Execution view of one KV head: (K_view bits, V_view bits), each [L][d].

    [README] "Core equation" (selected KV concatenated, address space and
    execution window kept apart) and [REVIEW] "Summary" (blocks restored with
    re-RoPE into a bounded view).  View slot j holds the j-th kept token; its
    key is rotated at view position j and rounded to bf16; its value is copied.
    """
    rows = view_rows(ids, n_tok)
    k = bf16_to_f64(np.asarray(keys_bits)[rows])
    k_view = f64_to_bf16(rope(k, np.arange(rows.size), theta))
    v_view = np.array(np.asarray(values_bits)[rows], dtype=np.uint16)
    return k_view, v_view


def decode_attention(q_bits, k_view_bits, v_view_bits, theta: float) -> np.ndarray:
    """Single-token attention of a group's query heads over the view: [G][d].

    [README] "Local reproduction" (the view replaces full attention) and
    "2026-09-08 validation correction" (RoPE applied to the query).
    READING: the query sits at view position L, the slot after the view; its
    softmax scale is 1/sqrt(d).  An empty view gives zeros.
    """
    q = bf16_to_f64(q_bits)
    g, d = q.shape
    L = np.asarray(k_view_bits).shape[0]
    if L == 0:
        return np.zeros((g, d))
    qr = rope(q, L, theta)
    k = bf16_to_f64(k_view_bits)
    v = bf16_to_f64(v_view_bits)
    s = qr @ k.T / np.sqrt(d)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def step_view_attention(q_steps_bits, k_view_bits, v_view_bits, theta: float) -> np.ndarray:
    """Attention of a step's T query tokens (the group's heads) over the view: [T][G][d].

    [REVIEW] "Strengths" (recall scheduled once per agent step) and [README]
    "Local reproduction" (the view replaces full attention).  READING: the
    step's tokens are the history's last T tokens, so token t sits at view
    position p_t = L - T + t (the recent blocks of the view hold them); its
    query is rotated at p_t and attends the view slots j <= p_t (causal within
    the step); softmax scale 1/sqrt(d).
    """
    q = bf16_to_f64(q_steps_bits)                 # [T][G][d]
    T, g, d = q.shape
    k = bf16_to_f64(k_view_bits)
    v = bf16_to_f64(v_view_bits)
    L = k.shape[0]
    if L < T:
        raise ValueError("the view must hold the step's tokens")
    out = np.zeros((T, g, d))
    for t in range(T):
        pos = L - T + t
        qr = rope(q[t], pos, theta)
        s = qr @ k[:pos + 1].T / np.sqrt(d)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out[t] = p @ v[:pos + 1]
    return out


# --------------------------------------------------------------------------- attention-mass diagnostic
def block_attention_mass(q_bits, keys_bits, theta: float) -> np.ndarray:
    """Full-attention mass of each history block, summed over a group's query heads: [n_blk].

    [README] "Background and main changes" (a few blocks hold most of the attention: the top 8 of about 103
    blocks held 66.5% of it).  READING: exact attention over the whole history, the query at position
    N = n_tok (the slot after the history, as in decode attention with every block kept) and each key at its
    history position t, scale 1/sqrt(d); mass[b] = sum over the group's heads h and the block's tokens t of
    softmax_t(<RoPE(q_h, N), RoPE(k_t, t)>/sqrt(d)).  Each head's weights sum to 1, so sum_b mass[b] = G.
    """
    q = bf16_to_f64(q_bits)                          # [G][d]
    k = bf16_to_f64(keys_bits)                       # [n_tok][d]
    n_tok, d = k.shape
    qr = rope(q, n_tok, theta)
    kr = rope(k, np.arange(n_tok), theta)
    s = qr @ kr.T / np.sqrt(d)                       # [G][n_tok]
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    n_blk = -(-n_tok // BLOCK)
    pad = np.zeros((p.shape[0], n_blk * BLOCK - n_tok))
    return np.concatenate([p, pad], axis=1).reshape(p.shape[0], n_blk, BLOCK).sum(axis=(0, 2))


def top_mass_share(mass, group: int, k: int = 8) -> float:
    """Share of the group's attention mass held by its k largest blocks (mass sums to `group`)."""
    m = np.sort(np.asarray(mass, dtype=np.float64))[::-1]
    return float(m[:k].sum() / group)


# --------------------------------------------------------------------------- one layer
def kvmem_layer(k_pool, v_pool, page_of, q_bits, n_tok: int, n_sink: int, n_recent: int, top_k: int,
                theta: float, attend: bool = True, heads=None):
    """The whole per-layer path for one session, in the pages' order.

    q_bits is [h_q][d] (one decode token) or [T][h_q][d] (a step of T tokens;
    then no attention).  ``heads`` limits the view/attention work to some KV
    heads (the scores always cover all heads).  Returns a dict with
    index [h_kv][n_blk][d], gs [h_kv][n_blk], ids {g: [n_keep]},
    k_view/v_view {g: [L][d] bits} and out [h_q][d] (rows of the heads done).
    """
    h_kv = np.asarray(k_pool).shape[1]
    q_bits = np.asarray(q_bits)
    multi = q_bits.ndim == 3
    h_q = q_bits.shape[-2]
    group = h_q // h_kv
    n_blk = -(-n_tok // BLOCK)
    keys = [paged_tokens(k_pool, page_of, g, n_tok) for g in range(h_kv)]
    index = np.stack([mean_k_index(keys[g]) for g in range(h_kv)]) if n_blk else np.zeros((h_kv, 0, q_bits.shape[-1]))
    if n_blk == 0:
        gs = np.zeros((h_kv, 0))
    elif multi:
        gs = step_group_scores(q_bits, index)
    else:
        gs = gqa_softmax_sum(block_scores(q_bits, index), h_kv)
    res = {"index": index, "gs": gs, "ids": {}, "k_view": {}, "v_view": {}}
    out = np.zeros((h_q, q_bits.shape[-1]))
    for g in (range(h_kv) if heads is None else heads):
        ids = select_blocks(gs[g], n_blk, n_sink, n_recent, top_k)
        vals = paged_tokens(v_pool, page_of, g, n_tok)
        kv, vv = materialize(keys[g], vals, ids, n_tok, theta)
        res["ids"][g], res["k_view"][g], res["v_view"][g] = ids, kv, vv
        if attend and not multi:
            out[g * group:(g + 1) * group] = decode_attention(q_bits[g * group:(g + 1) * group], kv, vv, theta)
    res["out"] = out
    return res
