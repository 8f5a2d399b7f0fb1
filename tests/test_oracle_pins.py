"""Pins for the CPU oracle: each check comes from outside the oracle's own code.

Brute force on tiny inputs (per-token loops, exact rationals), closed forms
worked by hand, invariants of the mathematics, and special cases that reduce
to library routines.  A plausible mistake in the oracle (a dropped 1/sqrt(d),
a softmax over the wrong axis, heads averaged instead of summed, a wrong RoPE
pairing or sign, an off-by-one view position, a wrong tie-break) fails at
least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import synth
from oracle import kvm_oracle as O

RNG = np.random.default_rng(12345)


def rand_bf16(shape, scale=1.0):
    return O.f64_to_bf16(RNG.normal(0.0, scale, size=shape))


# ----------------------------------------------------------------------------- bf16
def test_bf16_exact_values_and_ties():
    assert O.f64_to_bf16([1.0, -2.0, 0.0, 0.5, 3.0]).tolist() == [0x3F80, 0xC000, 0x0000, 0x3F00, 0x4040]
    # 1 + 2^-8 sits halfway between 1 and 1 + 2^-7: ties go to the even pattern 0x3F80.
    assert int(O.f64_to_bf16(1 + 2.0 ** -8)) == 0x3F80
    # 1 + 3*2^-8 is halfway between 0x3F81 and 0x3F82: even is 0x3F82.
    assert int(O.f64_to_bf16(1 + 3 * 2.0 ** -8)) == 0x3F82
    # Just above the tie: must round up.  Going through fp32 first would lose the 2^-40 and tie down.
    assert int(O.f64_to_bf16(1 + 2.0 ** -8 + 2.0 ** -40)) == 0x3F81
    assert int(O.f64_to_bf16(-(1 + 2.0 ** -8 + 2.0 ** -40))) == 0xBF81


def test_bf16_matches_torch_from_fp32():
    x = RNG.normal(0, 3, size=20000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), ref)


def test_bf16_roundtrip_all_finite_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = O.bf16_to_f64(bits)
    fin = np.isfinite(vals)
    back = O.f64_to_bf16(vals[fin])
    # -0.0 and +0.0 both survive with their sign
    assert np.array_equal(back, bits[fin])


# ----------------------------------------------------------------------------- Mean-K
def test_mean_k_equals_exact_rational_mean():
    keys = rand_bf16((3 * 32 + 7, 8))          # two full blocks ... and a partial tail block
    idx = O.mean_k_index(keys)
    vals = O.bf16_to_f64(keys)
    assert idx.shape == (4, 8)
    for b in range(4):
        rows = range(b * 32, min(len(vals), b * 32 + 32))
        for i in range(8):
            exact = sum(Fraction(float(vals[t, i])) for t in rows) / len(rows)
            assert abs(Fraction(float(idx[b, i])) - exact) <= abs(exact) * Fraction(1, 2 ** 52)


def _bf16_nearest_even_of_rational(x: Fraction) -> int:
    """bf16 bit pattern nearest to an exact rational, ties to the even pattern, by enumerating the
    representable neighbours (normal range only, which the test data stays in)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): neighbours 1 + m/128 and 1 + (m+1)/128
    m = int((a - 1) * 128)
    lo, hi = Fraction(128 + m, 128), Fraction(128 + m + 1, 128)
    dl, dh = a - lo, hi - a
    pick = m if dl < dh else (m + 1 if dh < dl else (m if m % 2 == 0 else m + 1))
    if pick == 128:                      # rounded up to the next binade
        pick, e = 0, e + 1
    return sign | ((e + 127) << 7) | pick


def test_bf16_index_operand_is_the_rounded_exact_mean():
    """The bf16 operand of step scoring is the exact rational mean of each block's keys rounded to the
    nearest bf16 (ties to even), found here by enumerating neighbours in exact arithmetic."""
    keys = rand_bf16((5 * 32 + 11, 24), scale=2.0)
    got = O.mean_k_index_bf16(keys)
    vals = O.bf16_to_f64(keys)
    assert got.shape == (6, 24)
    for b in range(6):
        rows = range(b * 32, min(len(vals), b * 32 + 32))
        for i in range(24):
            exact = sum(Fraction(float(vals[t, i])) for t in rows) / len(rows)
            assert int(got[b, i]) == _bf16_nearest_even_of_rational(exact), (b, i)
    # a block whose exact mean sits on a midpoint: 31 keys of 1 and one of 1 + 2^-3 give a mean of
    # 1 + 2^-8 (halfway between 1 and 1 + 2^-7) and round to the even pattern 0x3F80; 1 + 3 * 2^-3 for the
    # odd key gives 1 + 3 * 2^-8, halfway between 0x3F81 and 0x3F82, which rounds to 0x3F82
    tie = O.f64_to_bf16(np.array([[1.0]] * 31 + [[1.125]]))
    assert int(O.mean_k_index_bf16(tie)[0, 0]) == 0x3F80
    tie2 = O.f64_to_bf16(np.array([[1.0]] * 31 + [[1.375]]))
    assert int(O.mean_k_index_bf16(tie2)[0, 0]) == 0x3F82


def test_index_append_matches_full_build_and_is_position_free():
    keys = rand_bf16((300, 16))
    full = O.mean_k_index(keys)
    idx = O.mean_k_index(keys[:45])
    for a, b in [(45, 70), (70, 64), (134, 1), (135, 165)]:
        idx = O.index_append(idx, keys[:a + b], a, b)
    assert np.array_equal(idx, full)
    # Zero-length append changes nothing.
    assert np.array_equal(O.index_append(full, keys, 300, 0), full)


# ----------------------------------------------------------------------------- scores
def test_block_score_is_mean_of_per_token_scores():
    """s_b = <q, mean_t k_t>/sqrt(d) must equal mean_t <q, k_t>/sqrt(d) (linearity), by per-token loops."""
    h_q, h_kv, d, n_tok = 6, 2, 16, 96
    keys = [rand_bf16((n_tok, d)) for _ in range(h_kv)]
    q = rand_bf16((h_q, d))
    idx = np.stack([O.mean_k_index(k) for k in keys])
    s = O.block_scores(q, idx)
    qf = O.bf16_to_f64(q)
    for h in range(h_q):
        kv = O.bf16_to_f64(keys[h // 3])
        for b in range(n_tok // 32):
            per_tok = [sum(qf[h, i] * kv[t, i] for i in range(d)) / math.sqrt(d) for t in range(b * 32, b * 32 + 32)]
            assert s[h, b] == pytest.approx(sum(per_tok) / 32, rel=1e-12, abs=1e-14)


def test_softmax_single_head_group_is_library_softmax():
    s = RNG.normal(0, 4, size=(3, 50))
    gs = O.gqa_softmax_sum(s, 3)
    assert np.allclose(gs, scipy.special.softmax(s, axis=1), rtol=1e-14, atol=0)


def test_group_sum_closed_forms():
    ln3 = math.log(3.0)
    # Two heads in one group: p1 = (1/4, 3/4), p2 = (3/4, 1/4): the sum is (1, 1).
    assert np.allclose(O.gqa_softmax_sum(np.array([[0.0, ln3], [ln3, 0.0]]), 1), [[1.0, 1.0]], atol=1e-15)
    # p1 = (1/4, 3/4), p2 = (1/2, 1/2): the sum is (3/4, 5/4); an average would give half of that.
    assert np.allclose(O.gqa_softmax_sum(np.array([[0.0, ln3], [7.0, 7.0]]), 1), [[0.75, 1.25]], atol=1e-15)
    # Two groups keep apart: rows 0-1 -> group 0, rows 2-3 -> group 1.
    s = np.array([[0.0, ln3], [ln3, 0.0], [0.0, 0.0], [0.0, ln3]])
    assert np.allclose(O.gqa_softmax_sum(s, 2), [[1.0, 1.0], [0.75, 1.25]], atol=1e-15)


def test_group_scores_sum_to_group_size():
    s = RNG.normal(0, 2, size=(40, 777))
    gs = O.gqa_softmax_sum(s, 8)
    assert np.allclose(gs.sum(axis=1), 5.0, rtol=1e-13)


def test_withdrawn_averaging_is_distinguishable():
    """Head A likes block 0, head B block 1, both like block 3 moderately.

    Per-head softmax then sum ranks blocks 0 and 1 first; averaging the query
    heads first ranks block 3 first.  Closed form worked by hand.
    """
    r2 = math.sqrt(2.0)
    q = O.f64_to_bf16([[1.0, 0.0], [0.0, 1.0]])                        # h_q = 2, h_kv = 1, d = 2
    idx = np.array([[[5 * r2, 0.0], [0.0, 5 * r2], [0.0, 0.0], [2.6 * r2, 2.6 * r2]]])
    s = O.block_scores(q, idx)
    assert np.allclose(s, [[5, 0, 0, 2.6], [0, 5, 0, 2.6]], atol=1e-12)
    za = math.exp(5) + 2 + math.exp(2.6)
    expect = np.array([(math.exp(5) + 1) / za, (1 + math.exp(5)) / za, 2 / za, 2 * math.exp(2.6) / za])
    gs = O.gqa_softmax_sum(s, 1)
    assert np.allclose(gs[0], expect, rtol=1e-13)
    wd = O.withdrawn_group_scores(q, idx)
    # averaged query (1/2, 1/2): scores (5/2, 5/2, 0, 2.6) over sqrt(2) * sqrt(2) = 2, softmax worked by hand
    zw = 2 * math.exp(2.5) + 1 + math.exp(2.6)
    assert np.allclose(wd[0], [math.exp(2.5) / zw, math.exp(2.5) / zw, 1 / zw, math.exp(2.6) / zw], rtol=1e-13)
    assert int(np.argmax(gs[0])) in (0, 1) and int(np.argmax(wd[0])) == 3


def test_withdrawn_scoring_averages_not_sums_and_keeps_groups_apart():
    """Hand-worked vectors for two KV groups of three query heads.  The averaged query halves and thirds the
    scores; a sum of the heads (three times the mean) or a mean over the wrong group gives another vector."""
    q = O.f64_to_bf16([[2.0, 0.0], [1.0, 0.0], [0.0, 0.0],             # group 0: mean (1, 0)
                       [0.0, 3.0], [0.0, 0.0], [0.0, 0.0]])            # group 1: mean (0, 1)
    r2 = math.sqrt(2.0)
    idx = np.array([[[r2, 0.0], [0.0, r2], [2 * r2, 0.0]],             # group 0: scores (1, 0, 2)
                    [[0.0, r2], [r2, 0.0], [0.0, -r2]]])               # group 1: scores (1, 0, -1)
    wd = O.withdrawn_group_scores(q, idx)
    z0 = math.e + 1 + math.e ** 2
    z1 = math.e + 1 + math.exp(-1)
    want = np.array([[math.e / z0, 1 / z0, math.e ** 2 / z0], [math.e / z1, 1 / z1, math.exp(-1) / z1]])
    assert np.allclose(wd, want, rtol=1e-14)
    # a sum of the heads would give scores (3, 0, 6) for group 0: a different vector
    zs = math.exp(3) + 1 + math.exp(6)
    assert not np.allclose(wd[0], [math.exp(3) / zs, 1 / zs, math.exp(6) / zs], rtol=1e-3)
    assert np.allclose(wd.sum(axis=1), 1.0, rtol=1e-14)                 # one softmax per KV head


def test_step_scores_single_token_and_mass():
    idx = RNG.normal(0, 0.3, size=(2, 40, 8))
    qs = rand_bf16((3, 4, 8))
    one = O.step_group_scores(qs[:1], idx)
    assert np.array_equal(one, O.gqa_softmax_sum(O.block_scores(qs[0], idx), 2))
    assert np.allclose(O.step_group_scores(qs, idx).sum(axis=1), 3 * 2, rtol=1e-13)


# ----------------------------------------------------------------------------- selection
def brute_select(gs, n_blk, n_sink, n_recent, top_k):
    if n_blk <= n_sink + n_recent + top_k:
        return list(range(n_blk))
    keep = set(range(n_sink)) | set(range(n_blk - n_recent, n_blk))
    cands = sorted(range(n_sink, n_blk - n_recent), key=lambda b: (-gs[b], b))
    return sorted(keep | set(cands[:top_k]))


@pytest.mark.parametrize("n_blk,n_sink,n_recent,top_k", [
    (50, 1, 2, 7), (50, 4, 8, 20), (50, 0, 0, 5), (12, 4, 4, 4), (11, 4, 4, 4), (3, 4, 8, 2), (0, 1, 2, 3),
    (40, 0, 5, 10), (40, 6, 0, 10)])
def test_select_matches_brute_force_with_ties(n_blk, n_sink, n_recent, top_k):
    gs = np.round(RNG.uniform(0, 1, size=n_blk), 1)          # many exact ties
    ids = O.select_blocks(gs, n_blk, n_sink, n_recent, top_k)
    assert ids.tolist() == brute_select(gs, n_blk, n_sink, n_recent, top_k)
    assert len(ids) == min(n_blk, n_sink + n_recent + top_k)
    assert np.all(np.diff(ids) > 0)


def test_select_tie_goes_to_lower_id():
    gs = np.zeros(20)
    gs[[7, 9, 11, 13]] = 1.0
    assert O.select_blocks(gs, 20, 1, 1, 2).tolist() == [0, 7, 9, 19]


def brute_kth(gs, n_blk, n_sink, n_recent, top_k):
    """The k-th largest candidate score by counting: the value v with #{c: gs_c > v} < k <= #{c: gs_c >= v}."""
    if n_blk <= n_sink + n_recent + top_k:
        return float("nan")
    cands = [float(gs[b]) for b in range(n_sink, n_blk - n_recent)]
    for v in cands:
        above = sum(1 for x in cands if x > v)
        at_or_above = sum(1 for x in cands if x >= v)
        if above < top_k <= at_or_above:
            return v
    raise AssertionError("no k-th value")


@pytest.mark.parametrize("n_blk,n_sink,n_recent,top_k", [
    (60, 2, 3, 1), (60, 2, 3, 7), (60, 2, 3, 54), (60, 0, 0, 1), (60, 0, 0, 59), (40, 4, 4, 31), (40, 4, 4, 32)])
def test_kth_candidate_score_by_counting(n_blk, n_sink, n_recent, top_k):
    """The boundary score against a counting loop, with exact ties (values on a 0.1 grid), top_k = 1, top_k one
    short of the candidate count, and top_k equal to it (every block kept: no boundary, NaN)."""
    gs = np.round(RNG.uniform(0, 1, size=n_blk), 1)
    # the forced blocks hold the largest scores: they must not be counted among the candidates
    gs[:n_sink] = 5.0
    gs[n_blk - n_recent:] = 7.0
    got = O.kth_candidate_score(gs, n_blk, n_sink, n_recent, top_k)
    want = brute_kth(gs, n_blk, n_sink, n_recent, top_k)
    if math.isnan(want):
        assert math.isnan(got)
        assert len(O.select_blocks(gs, n_blk, n_sink, n_recent, top_k)) == n_blk
        return
    assert got == want
    # the boundary is the smallest score among the chosen candidates
    ids = O.select_blocks(gs, n_blk, n_sink, n_recent, top_k)
    chosen = [b for b in ids if n_sink <= b < n_blk - n_recent]
    assert len(chosen) == top_k and min(gs[chosen]) == got


def test_kth_candidate_score_hand_cases():
    gs = np.array([9.0, 0.3, 0.8, 0.8, 0.1, 0.5, 9.0])      # sink 0 and recent 6 hold the largest scores
    assert O.kth_candidate_score(gs, 7, 1, 1, 1) == 0.8
    assert O.kth_candidate_score(gs, 7, 1, 1, 2) == 0.8      # tie: the second 0.8
    assert O.kth_candidate_score(gs, 7, 1, 1, 3) == 0.5
    assert O.kth_candidate_score(gs, 7, 1, 1, 4) == 0.3
    assert math.isnan(O.kth_candidate_score(gs, 7, 1, 1, 5))  # budget covers every block


# ----------------------------------------------------------------------------- RoPE
def test_rope_matches_complex_rotation():
    """RoFormer's complex form: z_i = x_i + i x_{i+d/2} is multiplied by exp(i p theta^(-2i/d))."""
    d, theta = 16, 1e4
    x = RNG.normal(size=(5, d))
    pos = np.array([0.0, 1.0, 7.0, 1000.0, 65535.0])
    got = O.rope(x, pos, theta)
    for r in range(5):
        for i in range(d // 2):
            z = complex(x[r, i], x[r, i + d // 2]) * np.exp(1j * pos[r] * theta ** (-2.0 * i / d))
            assert got[r, i] == pytest.approx(z.real, abs=1e-9)
            assert got[r, i + d // 2] == pytest.approx(z.imag, abs=1e-9)


def test_rope_invariants():
    d, theta = 128, 1e6
    x = RNG.normal(size=(7, d))
    assert np.array_equal(O.rope(x, 0, theta), x)                      # identity at p = 0
    for p0, p in [(0, 5), (31, 32), (4096, 65535), (1048000, 1048575)]:
        # RoPE(x, p) = R(p - p0) applied to RoPE(x, p0)
        assert np.allclose(O.rope(O.rope(x, p0, theta), p - p0, theta), O.rope(x, p, theta), atol=1e-9)
    assert np.allclose(np.linalg.norm(O.rope(x, 12345, theta), axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    q, k = RNG.normal(size=d), RNG.normal(size=d)
    a = O.rope(q, 100, theta) @ O.rope(k, 40, theta)
    b = O.rope(q, 1060, theta) @ O.rope(k, 1000, theta)
    assert a == pytest.approx(b, rel=1e-9)                              # depends on m - n only


# ----------------------------------------------------------------------------- view + attention
def test_materialize_positions_and_copies():
    d, n_tok, theta = 8, 5 * 32 + 9, 1e4
    keys, vals = rand_bf16((n_tok, d)), rand_bf16((n_tok, d))
    ids = np.array([0, 2, 5])                                          # block 5 is the 9-token tail
    kv, vv = O.materialize(keys, vals, ids, n_tok, theta)
    rows = list(range(0, 32)) + list(range(64, 96)) + list(range(160, 169))
    assert kv.shape == (73, d) and np.array_equal(vv, vals[rows])
    for j, t in enumerate(rows):
        expect = O.f64_to_bf16(O.rope(O.bf16_to_f64(keys[t]), j, theta))
        assert np.array_equal(kv[j], expect)


def brute_full_attention(q_bits, keys_bits, vals_bits, theta):
    """Standard decode over a conventional post-RoPE bf16 KV cache, token by token."""
    qf, kf, vf = O.bf16_to_f64(q_bits), O.bf16_to_f64(keys_bits), O.bf16_to_f64(vals_bits)
    n, d = kf.shape
    out = []
    for h in range(qf.shape[0]):
        qr = O.rope(qf[h], n, theta)
        logits = []
        for t in range(n):
            kt = O.bf16_to_f64(O.f64_to_bf16(O.rope(kf[t], t, theta)))
            logits.append(sum(qr[i] * kt[i] for i in range(d)) / math.sqrt(d))
        m = max(logits)
        w = [math.exp(v - m) for v in logits]
        z = sum(w)
        out.append([sum(w[t] * vf[t, i] for t in range(n)) / z for i in range(d)])
    return np.array(out)


def test_all_blocks_kept_equals_full_attention():
    d, n_tok, theta = 16, 3 * 32 + 5, 1e4
    keys, vals, q = rand_bf16((n_tok, d)), rand_bf16((n_tok, d)), rand_bf16((2, d))
    ids = O.select_blocks(np.zeros(4), 4, 1, 1, 8)                     # budget covers every block
    kv, vv = O.materialize(keys, vals, ids, n_tok, theta)
    got = O.decode_attention(q, kv, vv, theta)
    assert np.allclose(got, brute_full_attention(q, keys, vals, theta), rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    d, theta = 8, 1e4
    q, v = rand_bf16((3, d)), rand_bf16((1, d))
    k = rand_bf16((1, d))
    assert np.allclose(O.decode_attention(q, k, v, theta), O.bf16_to_f64(v).repeat(3, 0), atol=0)   # L = 1
    vals = rand_bf16((40, d))
    zeros = np.zeros((40, d), dtype=np.uint16)                          # all keys zero: uniform weights
    assert np.allclose(O.decode_attention(q, zeros, vals, theta), O.bf16_to_f64(vals).mean(0), rtol=1e-13)
    assert np.array_equal(O.decode_attention(q, zeros[:0], vals[:0], theta), np.zeros((3, d)))


# ----------------------------------------------------------------------------- planted recovery
def _recovered(w, layer=0):
    li = synth.layer_inputs(w, layer)
    res = O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[0], li.q[0, 0], w.n_tok, w.n_sink,
                        w.n_recent, w.top_k, w.rope_theta, heads=[])
    hits = []
    for g in range(w.h_kv):
        ids = O.select_blocks(res["gs"][g], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        hits.append(len(set(ids.tolist()) & set(li.planted[0, g].tolist())))
    return hits


def test_planted_blocks_recovered_on_tiny_seed0():
    assert _recovered(synth.WORKLOADS["tiny_8k_g4_d64"]) [0] >= 3


def test_clean_variant_recovers_every_planted_block():
    w = synth.WORKLOADS["tiny_8k_g4_d64"].with_(eps_scale=0.1, q_noise_var=0.0)
    assert _recovered(w) == [4]
    # GQA geometry, 4 planted topics per KV head: signal <mu_b, sum mu> ~ 32 against cross-talk std ~ 5.7.
    w2 = synth.WORKLOADS["gqa40x8_256k"].with_(n_tok=32768, top_k=64, n_planted=4, eps_scale=0.1, q_noise_var=0.0)
    assert _recovered(w2) == [4] * 8


# --------------------------------------------------------------------------- step attention over the view
def test_step_attention_is_causal_within_the_step():
    rng = np.random.default_rng(3)
    T, G, d, L = 5, 2, 16, 40
    q = rand_bf16((T, G, d))
    k = rand_bf16((L, d))
    v = rand_bf16((L, d))
    out = O.step_view_attention(q, k, v, 1e4)
    # slots after a token's own position never reach it; its own slot and earlier ones do
    for t in range(T):
        pos = L - T + t
        v2 = v.copy()
        v2[pos + 1:] = O.f64_to_bf16(rng.normal(size=(L - pos - 1, d)))
        out2 = O.step_view_attention(q, k, v2, 1e4)
        assert np.array_equal(out2[t], out[t])
        v3 = v.copy()
        v3[pos] = O.f64_to_bf16(rng.normal(size=d) + 3.0)
        assert not np.allclose(O.step_view_attention(q, k, v3, 1e4)[t], out[t])


def test_step_attention_positions_match_decode_attention_by_relative_distance():
    """Token t of the step (query at view position p, keys at 0..p) and decode attention over slots 0..p
    (query at p + 1) see the same relative distances once the keys are moved one position on (RoPE
    composition).  The moved keys are re-rounded to bf16, hence the loose tolerance; an off-by-one in the
    step's positions changes high-frequency logits by about a radian and fails it."""
    T, G, d, L = 3, 2, 16, 24
    q = rand_bf16((T, G, d))
    k = rand_bf16((L, d))
    v = rand_bf16((L, d))
    out = O.step_view_attention(q, k, v, 1e4)
    for t in range(T):
        pos = L - T + t
        moved = O.f64_to_bf16(O.rope(O.bf16_to_f64(k[:pos + 1]), np.ones(pos + 1), 1e4))
        ref = O.decode_attention(q[t], moved, v[:pos + 1], 1e4)
        assert np.allclose(out[t], ref, atol=2e-2)


def test_step_attention_uniform_keys_average_the_causal_window():
    T, G, d, L = 4, 3, 8, 12
    q = rand_bf16((T, G, d))
    k = np.zeros((L, d), dtype=np.uint16)                 # zero keys: every logit is 0
    v = rand_bf16((L, d))
    out = O.step_view_attention(q, k, v, 1e4)
    vf = O.bf16_to_f64(v)
    for t in range(T):
        pos = L - T + t
        assert np.allclose(out[t], np.broadcast_to(vf[:pos + 1].mean(axis=0), (G, d)), atol=1e-14)


def test_step_attention_matches_library_softmax_hand_case():
    # T = 2, L = 2, d = 2, theta irrelevant at position 0 for token 0 (RoPE at 0 is the identity)
    q = O.f64_to_bf16([[[1.0, 0.0]], [[0.0, 2.0]]])      # [T][G=1][d]
    k = O.f64_to_bf16([[2.0, 0.0], [0.0, 1.0]])
    v = O.f64_to_bf16([[1.0, -1.0], [3.0, 5.0]])
    out = O.step_view_attention(q, k, v, 1e4)
    assert np.allclose(out[0, 0], [1.0, -1.0], atol=1e-15)   # token 0 sees slot 0 only
    # token 1 at position 1: q rotated by angle 1 * theta^0 = 1 rad on the (0, 1) pair
    c, s_ = np.cos(1.0), np.sin(1.0)
    qr = np.array([0.0 * c - 2.0 * s_, 2.0 * c + 0.0 * s_])
    logits = np.array([qr @ [2.0, 0.0], qr @ [0.0, 1.0]]) / np.sqrt(2.0)
    w = np.exp(logits - logits.max())
    w /= w.sum()
    assert np.allclose(out[1, 0], w @ np.array([[1.0, -1.0], [3.0, 5.0]]), atol=1e-14)


# ----------------------------------------------------------------------------- FP8 E4M3 pages
def _torch_e4m3_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_library_and_hand_values():
    v = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    lib = _torch_e4m3_table()
    assert np.array_equal(np.isnan(v), np.isnan(lib)) and np.isnan(v).sum() == 2      # 0x7F and 0xFF
    fin = ~np.isnan(v)
    assert np.array_equal(v[fin], lib[fin])
    # by hand from the format: 1.0 = 2^(7-7), the largest normal 2^8 * 1.75, the smallest normal and subnormal
    assert (v[0x38], v[0xB8], v[0x7E], v[0x08], v[0x01], v[0x07]) == (1.0, -1.0, 448.0, 2.0 ** -6, 2.0 ** -9,
                                                                         7 * 2.0 ** -9)


def test_e4m3_encode_is_nearest_even_by_brute_force():
    vals = O.e4m3_to_f64(np.arange(127, dtype=np.uint8))            # finite non-negative, ascending
    x = np.concatenate([RNG.uniform(-448, 448, 3000), RNG.uniform(-0.05, 0.05, 3000),
                        (vals[:-1] + vals[1:]) / 2, -(vals[:-1] + vals[1:]) / 2]).astype(np.float32)
    got = O.f32_to_e4m3(x)
    for xi, gi in zip(x.astype(np.float64), got):
        d = np.abs(vals - abs(xi))
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]   # tie: even mantissa
        assert gi == (code | (0x80 if np.signbit(xi) else 0)), (xi, gi, code)
    # the library's conversion agrees inside the finite range
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)


def test_e4m3_saturates_beyond_448():
    assert O.f32_to_e4m3([448.0, 449.0, 463.9, 464.0, 1e6, -1e6]).tolist() == [0x7E] * 5 + [0xFE]


def test_quantize_page_scale_and_the_largest_element():
    x = rand_bf16((32, 64), 0.7)
    codes, scale = O.quantize_page(x)
    vals = O.bf16_to_f64(x)
    amax = np.float32(np.abs(vals).max())
    assert scale == np.float32(amax / np.float32(448.0))
    i = np.unravel_index(np.argmax(np.abs(vals)), vals.shape)
    assert abs(O.e4m3_to_f64(codes[i])) == 448.0
    # every dequantised element within half a code spacing (relative 2^-4) or half a subnormal step
    deq = O.dequantize(codes, scale)
    assert np.all(np.abs(deq - vals) <= np.maximum(np.abs(vals) * 2.0 ** -4, 2.0 ** -10 * scale) * 1.0001)
    zc, zs = O.quantize_page(np.zeros((32, 64), dtype=np.uint16))
    assert zs == np.float32(1.0) and not zc.any()


def test_representable_pages_survive_quantisation_exactly():
    """Values that are E4M3 values times a power of two, with the largest at 448 * 2^k, have scale 2^k: the
    dequantised pages equal the bf16 pages, so the index and the view are those of the bf16 path."""
    k = -6
    codes = RNG.integers(0, 127, size=(4, 32, 64)).astype(np.uint8) | (RNG.integers(0, 2, (4, 32, 64)) << 7).astype(np.uint8)
    codes[:, 0, 0] = 0x7E                                          # the page maximum: 448
    x = O.f64_to_bf16(O.e4m3_to_f64(codes) * 2.0 ** k)              # exact in bf16
    pool = x[:, None]                                               # [n_pages][h_kv=1][32][d]
    qc, qs = O.quantize_pool(pool)
    assert np.all(qs == np.float32(2.0 ** k)) and np.array_equal(qc[:, 0], codes)
    page_of = np.array([2, 0, 3, 1])
    n_tok = 4 * 32 - 5
    deq = O.paged_dequant_tokens(qc, qs, page_of, 0, n_tok)
    bits = O.paged_tokens(pool, page_of, 0, n_tok)
    assert np.array_equal(deq, O.bf16_to_f64(bits))
    assert np.array_equal(O.mean_k_index_of(deq), O.mean_k_index(bits))
    kv, vv = O.materialize_values(deq, deq, [0, 2, 3], n_tok, 1e4)
    kb, vb = O.materialize(bits, bits, [0, 2, 3], n_tok, 1e4)
    assert np.array_equal(kv, kb) and np.array_equal(vv, vb)


# ----------------------------------------------------------------------------- attention-mass diagnostic
def test_attention_mass_brute_force_tiny():
    """Per-token loops with the math library: rotate each pair by hand, exponentiate, sum per block."""
    d, G, n_tok, theta = 8, 2, 70, 100.0
    q = rand_bf16((G, d), 1.0)
    k = rand_bf16((n_tok, d), 1.0)
    qv, kv = O.bf16_to_f64(q), O.bf16_to_f64(k)

    def rot(x, pos):
        out = [0.0] * d
        for i in range(d // 2):
            a = pos * theta ** (-2.0 * i / d)
            out[i] = x[i] * math.cos(a) - x[i + d // 2] * math.sin(a)
            out[i + d // 2] = x[i + d // 2] * math.cos(a) + x[i] * math.sin(a)
        return out

    want = [0.0] * 3
    for h in range(G):
        qr = rot(list(qv[h]), n_tok)
        sc = [sum(a * b for a, b in zip(qr, rot(list(kv[t]), t))) / math.sqrt(d) for t in range(n_tok)]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        z = sum(w)
        for t in range(n_tok):
            want[t // 32] += w[t] / z
    got = O.block_attention_mass(q, k, theta)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def test_attention_mass_sums_to_group_and_uniform_keys_spread_evenly():
    q = rand_bf16((5, 64), 1.0)
    k = rand_bf16((32 * 9 + 11, 64), 1.0)
    m = O.block_attention_mass(q, k, 1e4)
    assert m.shape == (10,) and abs(m.sum() - 5.0) < 1e-12
    # identical zero keys: every token gets 1/n_tok, so a block's mass is G * (its tokens) / n_tok
    z = np.zeros((32 * 9 + 11, 64), dtype=np.uint16)
    mu = O.block_attention_mass(q, z, 1e4)
    want = 5.0 * np.array([32] * 9 + [11]) / (32 * 9 + 11)
    assert np.allclose(mu, want, rtol=1e-12)


def test_attention_mass_depends_on_relative_positions_only():
    """Rotary attention sees relative positions only: the same history with the query at N + 96 and every key
    at t + 96 (rotated by hand here) gives the same block masses."""
    d, G, theta = 16, 2, 1e4
    q = rand_bf16((G, d), 1.0)
    k = rand_bf16((100, d), 1.0)
    base = O.block_attention_mass(q, k, theta)
    qv, kv = O.bf16_to_f64(q), O.bf16_to_f64(k)
    qr = O.rope(qv, 100 + 96, theta)
    kr = O.rope(kv, np.arange(100) + 96, theta)
    s = qr @ kr.T / np.sqrt(d)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    shifted = np.concatenate([p, np.zeros((G, 28))], axis=1).reshape(G, 4, 32).sum(axis=(0, 2))
    assert np.allclose(base, shifted, rtol=1e-9)


def test_top_mass_share():
    m = np.array([0.5, 0.1, 1.0, 0.2, 0.2])
    assert O.top_mass_share(m, 2, k=2) == pytest.approx(0.75)
