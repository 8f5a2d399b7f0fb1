"""Shared helpers for the parity tests: device buffers from synth inputs, the
oracle's results for the same inputs, and the comparison rules.

Tolerances (each derived from the arithmetic; the pages fix none of them):
  index       |kbar_gpu - kbar| <= 2^-18 * mean_t |k_t,i|   (fp32 sum of <= 32 terms: <= 31 * 2^-24, doubled)
  head score  |s_gpu - s| <= 1e-5 * max(|s|, sum_i |q_i kbar_i| / sqrt(d))
  group score |Gs_gpu - Gs| <= 1e-4 * Gs + 1e-9
              (softmax of scores each off by <= 1e-5 of a magnitude bound of ~4: the exponent moves by
               <= 4e-5 per head and the normaliser by as much again, so ~1e-4 relative)
  kept ids    identical, except blocks whose oracle group score is within 1e-4 * tau of the oracle's
              k-th candidate score tau; same count, forced blocks present, ascending
  step scores (bf16 index operand) the oracle rounds the exact mean to bf16, the kernel its fp32 mean;
              the two can differ by one bf16 step where the exact mean lies within the fp32 error
              (the index bound above) of a rounding midpoint.  That moves a score by at most
              beta = sum_i |q_i| delta_i / sqrt(d) (delta_i the possible step), each probability by at
              most a factor exp(beta + zeta) (zeta the normaliser's share), and adds
              sum_rows p (exp(beta + zeta) - 1) to the group-score tolerance and to the id window
  V view      bit-exact
  K view      within 1 bf16 ulp (fp32 vs fp64 rotation can straddle a rounding boundary)
  out         |out_gpu - out| <= 1e-3
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import kvm_oracle as O
import sparse_attention_decode_04_b300 as K

BF16 = torch.bfloat16


def dev_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(BF16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class LayerOnDevice:
    """Device copies of one layer's inputs plus the step's output buffers."""

    def __init__(self, w: synth.Workload, li: synth.LayerInputs, ctx: K.Context, device="cuda"):
        self.w, self.li, self.ctx = w, li, ctx
        S, hk, d = w.n_sessions, w.h_kv, w.d
        self.k_pool = dev_u16(li.k_pool, device)
        self.v_pool = dev_u16(li.v_pool, device)
        bt = np.full((S, ctx.max_blocks), -1, dtype=np.int32)
        bt[:, :li.block_table.shape[1]] = li.block_table
        self.bt = torch.from_numpy(bt).to(device)
        self.q = dev_u16(li.q if w.n_q > 1 else li.q[:, 0], device)
        self.index = torch.zeros((S, hk, ctx.max_blocks, d), dtype=torch.float32, device=device)
        self.kept = torch.full((S, hk, ctx.budget), -7, dtype=torch.int32, device=device)
        self.gs = torch.zeros((S, hk, ctx.max_blocks), dtype=torch.float32, device=device)
        self.hs = torch.zeros((S, w.h_q, ctx.max_blocks), dtype=torch.float32, device=device)
        self.k_view = torch.zeros((S, hk, 32 * ctx.budget, d), dtype=BF16, device=device)
        self.v_view = torch.zeros((S, hk, 32 * ctx.budget, d), dtype=BF16, device=device)
        self.view_len = torch.full((S, hk), -7, dtype=torch.int32, device=device)
        self.out = torch.full((S, w.h_q, d), float("nan"), dtype=torch.float32, device=device)
        self.n_tok = [w.n_tok] * S
        self.n_pages = w.n_pages

    def index_build(self):
        K.kvm_index_append(self.ctx, self.k_pool, self.n_pages, self.bt, [0] * len(self.n_tok), self.n_tok,
                           self.index)

    def score_select(self, scores=True):
        K.kvm_score_select(self.ctx, self.q, self.w.n_q, self.index, self.n_tok, self.kept,
                           self.gs if scores else None, self.hs if (scores and self.w.n_q == 1) else None)

    def materialize(self, kept=None):
        K.kvm_materialize(self.ctx, self.k_pool, self.v_pool, self.n_pages, self.bt, self.n_tok,
                          self.kept if kept is None else kept, self.k_view, self.v_view, self.view_len)

    def attend(self):
        K.kvm_decode_attn(self.ctx, self.q, self.k_view, self.v_view, self.view_len, len(self.n_tok), self.out)

    def fused(self, kept=None):
        K.kvm_materialize_attn(self.ctx, self.k_pool, self.v_pool, self.n_pages, self.bt, self.n_tok,
                               self.kept if kept is None else kept, self.q, self.k_view, self.v_view,
                               self.view_len, self.out)


def oracle_layer(w: synth.Workload, li: synth.LayerInputs, session: int = 0, heads=None, attend=True):
    q = li.q[session] if w.n_q > 1 else li.q[session, 0]
    return O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[session], q, w.n_tok, w.n_sink, w.n_recent,
                         w.top_k, w.rope_theta, attend=attend and w.n_q == 1, heads=heads)


def oracle_keys(w, li, session, head):
    return O.paged_tokens(li.k_pool, li.block_table[session], head, w.n_tok)


# ------------------------------------------------------------------ comparisons
def check_index(gpu_idx: np.ndarray, keys_bits: np.ndarray, ora_idx: np.ndarray):
    k = np.abs(O.bf16_to_f64(keys_bits))
    n_tok, d = k.shape
    n_blk = ora_idx.shape[0]
    pad = np.zeros((n_blk * 32 - n_tok, d))
    cnt = np.minimum(32, n_tok - 32 * np.arange(n_blk))[:, None]
    mean_abs = np.concatenate([k, pad]).reshape(n_blk, 32, d).sum(axis=1) / cnt
    err = np.abs(gpu_idx.astype(np.float64) - ora_idx)
    bad = err > 2.0 ** -18 * mean_abs
    assert not bad.any(), f"index: {bad.sum()} elements off, worst {err.max():.3e}"


def check_head_scores(gpu_s: np.ndarray, q_bits: np.ndarray, index: np.ndarray, ora_s: np.ndarray):
    q = O.bf16_to_f64(q_bits)
    h_q, d = q.shape
    group = h_q // index.shape[0]
    bound = np.stack([np.abs(index[h // group]) @ np.abs(q[h]) for h in range(h_q)]) / np.sqrt(d)
    tol = 1e-5 * np.maximum(np.abs(ora_s), bound)
    err = np.abs(gpu_s.astype(np.float64) - ora_s)
    assert (err <= tol).all(), f"head scores: {(err > tol).sum()} off, worst ratio {(err / tol).max():.3f}"


def check_group_scores(gpu_gs: np.ndarray, ora_gs: np.ndarray, extra=None):
    """extra: per-block tolerance added for a known operand difference (step scoring), else None."""
    err = np.abs(gpu_gs.astype(np.float64) - ora_gs)
    tol = 1e-4 * ora_gs + 1e-9 + (0.0 if extra is None else extra)
    assert (err <= tol).all(), f"group scores: {(err > tol).sum()} off, worst ratio {(err / tol).max():.3f}"


def index_operand_slack(keys_bits: np.ndarray, to_exact: bool = False) -> np.ndarray:
    """Per element of the bf16 index operand, how far the kernel's value can be from the oracle's: [n_blk][d].

    The kernel rounds an fp32 mean that lies within the index bound e = 2^-18 mean_t |k_t,i| of the exact mean
    m, and round-to-nearest is monotone, so its bf16 value lies in [bf16(m - e), bf16(m + e)].  Against the
    oracle's bf16(m) that is at most bf16(m + e) - bf16(m - e) (zero unless a midpoint lies within e of m);
    against the unrounded m (to_exact) the largest distance of either end from m.
    """
    k = np.abs(O.bf16_to_f64(keys_bits))
    n_tok, d = k.shape
    m = O.mean_k_index(keys_bits)
    n_blk = m.shape[0]
    pad = np.zeros((n_blk * 32 - n_tok, d))
    cnt = np.minimum(32, n_tok - 32 * np.arange(n_blk))[:, None]
    e = 2.0 ** -18 * np.concatenate([k, pad]).reshape(n_blk, 32, d).sum(axis=1) / cnt
    lo = O.bf16_to_f64(O.f64_to_bf16(m - e))
    hi = O.bf16_to_f64(O.f64_to_bf16(m + e))
    if to_exact:
        return np.maximum(np.abs(hi - m), np.abs(lo - m))
    return hi - lo


def step_operand_tolerance(q_group_bits: np.ndarray, index_vals: np.ndarray, slack: np.ndarray) -> np.ndarray:
    """Group-score tolerance from index-operand differences of at most `slack`: [n_blk].

    q_group_bits [T][G][d] (the group's query heads for every step token), index_vals [n_blk][d] the oracle's
    operand values.  For each (token, head) row: beta_b = sum_i |q_i| slack_bi / sqrt(d) bounds the score
    change of block b, zeta = log sum_b p_b exp(beta_b) the normaliser's, so p_b moves by at most
    p_b (exp(beta_b + zeta) - 1); the bound is that summed over the rows.
    """
    q = O.bf16_to_f64(q_group_bits)
    T, G, d = q.shape
    tol = np.zeros(index_vals.shape[0])
    for t in range(T):
        s = index_vals @ q[t].T / np.sqrt(d)                  # [n_blk][G]
        beta = slack @ np.abs(q[t]).T / np.sqrt(d)
        p = np.exp(s - s.max(axis=0))
        p /= p.sum(axis=0)
        zeta = np.log((p * np.exp(beta)).sum(axis=0))
        tol += (p * np.expm1(beta + zeta)).sum(axis=1)
    return tol


def check_ids(gpu_ids: np.ndarray, ora_ids: np.ndarray, gs: np.ndarray, w: synth.Workload, extra=None) -> bool:
    """Returns True when the lists are identical; asserts the allowed-difference rule otherwise.

    extra: per-block group-score tolerance from a known operand difference (step scoring).  A block b then
    differs legitimately if |Gs_b - tau| <= 1e-4 tau + extra_b + max over the differing blocks of extra:
    swapping b with a block c across the boundary needs Gs_b - Gs_c within both their tolerances."""
    n_keep = len(ora_ids)
    assert gpu_ids.shape[0] >= n_keep
    assert (gpu_ids[n_keep:] == -1).all(), "padding after n_keep must be -1"
    g = gpu_ids[:n_keep]
    assert (np.diff(g) > 0).all(), "ids must ascend"
    if np.array_equal(g, ora_ids):
        return True
    n_blk = w.n_blk
    forced = set(range(min(w.n_sink, n_blk))) | set(range(max(0, n_blk - w.n_recent), n_blk))
    assert forced <= set(g.tolist())
    tau = O.kth_candidate_score(gs, n_blk, w.n_sink, w.n_recent, w.top_k)
    diff = set(g.tolist()) ^ set(ora_ids.tolist())
    ex = np.zeros(len(gs)) if extra is None else np.asarray(extra, dtype=np.float64)
    ex_max = max(ex[b] for b in diff) if diff else 0.0
    near = [b for b in diff if abs(gs[b] - tau) <= 1e-4 * tau + ex[b] + ex_max]
    assert len(near) == len(diff), f"ids differ away from the boundary: {sorted(diff)} (tau={tau})"
    return False


def check_view(gpu_k: np.ndarray, gpu_v: np.ndarray, ora_k: np.ndarray, ora_v: np.ndarray):
    L = ora_k.shape[0]
    assert np.array_equal(gpu_v[:L], ora_v), "V view must be bit-exact"
    a, b = O.bf16_to_f64(gpu_k[:L]), O.bf16_to_f64(ora_k)
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(a), np.abs(b)))[1] - 8)
    bad = np.abs(a - b) > ulp
    assert not bad.any(), f"K view: {bad.sum()} elements beyond 1 ulp"
    return int((a != b).sum())


def check_out(gpu_out: np.ndarray, ora_out: np.ndarray):
    err = np.abs(gpu_out.astype(np.float64) - ora_out)
    assert np.isfinite(gpu_out).all() and err.max() <= 1e-3, f"out: worst abs error {err.max():.3e}"
    return float(err.max())


def kept_tensor(ids_per_head: dict, S_h_budget, device="cuda") -> torch.Tensor:
    """int32 [S][h_kv][budget] from {(s, g): ids}, -1 padded (test-chosen kept lists)."""
    S, hk, budget = S_h_budget
    t = np.full((S, hk, budget), -1, dtype=np.int32)
    for (s, g), ids in ids_per_head.items():
        t[s, g, :len(ids)] = ids
    return torch.from_numpy(t).to(device)
