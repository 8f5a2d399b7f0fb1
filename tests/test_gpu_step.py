"""Step-level (multi-query) scoring on the tensor cores against the oracle.

The contraction takes bf16 operands (the scoring precision the step-level
workload states), so the oracle scores, in fp64, the bf16 rounding of the
exact Mean-K vectors.  The kernel rounds its fp32 index instead, which can
differ by one bf16 step where the exact mean lies near a rounding midpoint;
harness.step_operand_tolerance bounds what that does to each group score and
widens the group-score tolerance and the id window by exactly that bound.
At full size the ids are also checked against the pure fp64 oracle (no bf16
rounding of the index at all), with the window the rounding itself allows.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O

from harness import check_group_scores, check_ids, dev_u16, index_operand_slack, step_operand_tolerance

pytestmark = pytest.mark.gpu


def run_step(w, li):
    ctx = K.Context.for_workload(w)
    S = w.n_sessions
    kp = dev_u16(li.k_pool)
    bt = torch.from_numpy(li.block_table).cuda()
    q = dev_u16(li.q)                                                  # [S][n_q][h_q][d]
    index = torch.zeros((S, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device="cuda")
    kept = torch.full((S, w.h_kv, ctx.budget), -7, dtype=torch.int32, device="cuda")
    gs = torch.zeros((S, w.h_kv, w.n_blk), dtype=torch.float32, device="cuda")
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [0] * S, [w.n_tok] * S, index)
    K.kvm_score_select(ctx, q, w.n_q, index, [w.n_tok] * S, kept, gs)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    # second call without group-score output must select the same blocks
    kept2 = torch.full_like(kept, -7)
    K.kvm_score_select(ctx, q, w.n_q, index, [w.n_tok] * S, kept2)
    torch.cuda.synchronize()
    assert torch.equal(kept, kept2)
    ctx.close()
    return gs.cpu().numpy(), kept.cpu().numpy()


def oracle_step(w, li, s, heads, exact=False):
    """Per KV head g: (oracle group scores, the operand tolerance of the GPU's bf16 index against them).

    exact=False: the oracle scores the bf16 rounding of the exact mean; exact=True: the unrounded mean."""
    G = w.group
    res = {}
    for g in heads:
        keys = O.paged_tokens(li.k_pool, li.block_table[s], g, w.n_tok)
        qg = li.q[s][:, G * g:G * (g + 1)]
        if exact:
            idx = O.mean_k_index(keys)
            gs = O.step_group_scores(qg, idx[None])[0]
        else:
            idx = O.bf16_to_f64(O.mean_k_index_bf16(keys))
            gs = O.step_group_scores_bf16(qg, O.mean_k_index_bf16(keys)[None])[0]
        res[g] = (gs, step_operand_tolerance(qg, idx, index_operand_slack(keys, to_exact=exact)))
    return res


@pytest.mark.parametrize("d,h_q,h_kv,n_q", [(128, 8, 2, 40), (64, 12, 3, 33), (128, 5, 1, 256)])
def test_step_scores_small_ragged(d, h_q, h_kv, n_q):
    w = synth.Workload("step_small", h_q=h_q, h_kv=h_kv, d=d, n_tok=300 * 32 + 7, n_sink=3, n_recent=5, top_k=40,
                       rope_theta=1e6, n_planted=4, seed=31, n_q=n_q, attend=False)
    li = synth.layer_inputs(w, 0)
    gs, kept = run_step(w, li)
    ora = oracle_step(w, li, 0, range(w.h_kv))
    assert np.allclose(ora[0][0].sum(), n_q * w.group, rtol=1e-9)
    for g in range(w.h_kv):
        gs_o, extra = ora[g]
        assert extra.max() < 1e-2 * gs_o.max()          # the slack is a few blocks' share, not a blanket
        check_group_scores(gs[0, g], gs_o, extra)
        ids = O.select_blocks(gs_o, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        check_ids(kept[0, g], ids, gs_o, w, extra)


@pytest.mark.slow
def test_step_scores_full_size_256_queries_1m_tokens():
    w = synth.WORKLOADS["step256q_1m"]
    li = synth.layer_inputs(w, 0)
    gs, kept = run_step(w, li)
    heads = [0, 5]                                     # sampled KV heads (the oracle scores them in full)
    ora = oracle_step(w, li, 0, heads)
    same = 0
    for g in heads:
        gs_o, extra = ora[g]
        check_group_scores(gs[0, g], gs_o, extra)
        ids = O.select_blocks(gs_o, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        same += check_ids(kept[0, g], ids, gs_o, w, extra)
        # planted blocks of this head are found by the step's queries
        assert len(set(kept[0, g].tolist()) & set(li.planted[0, g].tolist())) >= 12
    assert same >= 1
    # the pure fp64 oracle (index never rounded to bf16): group scores and ids within what the bf16 rounding of
    # the index operand allows
    ora64 = oracle_step(w, li, 0, heads, exact=True)
    for g in heads:
        gs64, extra64 = ora64[g]
        check_group_scores(gs[0, g], gs64, extra64)
        ids64 = O.select_blocks(gs64, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        check_ids(kept[0, g], ids64, gs64, w, extra64)


def test_bf16_copy_of_the_index_and_the_conversion_give_identical_scores():
    """The appends' bf16 copy of the index (kept for the multi-query scoring) holds exactly the rounding the
    conversion of the fp32 index gives: scores and ids are bit-identical whichever the call uses.  The copy is
    used only when it holds every scored block of the index it was appended to."""
    w = synth.Workload("step_copy", h_q=8, h_kv=2, d=128, n_tok=300 * 32 + 7, n_sink=3, n_recent=5, top_k=40,
                       rope_theta=1e6, n_planted=4, seed=37, n_q=40, attend=False)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    kp = dev_u16(li.k_pool)
    bt = torch.from_numpy(li.block_table).cuda()
    q = dev_u16(li.q)
    n = w.n_tok

    def score(index):
        kept = torch.full((1, w.h_kv, ctx.budget), -7, dtype=torch.int32, device="cuda")
        gs = torch.zeros((1, w.h_kv, w.n_blk), dtype=torch.float32, device="cuda")
        K.kvm_score_select(ctx, q, w.n_q, index, [n], kept, gs)
        torch.cuda.synchronize()
        assert K.kvm_device_status(ctx) == 0
        return gs, kept

    index = torch.zeros((1, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device="cuda")
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [0], [5000], index)          # two ragged appends
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [5000], [n - 5000], index)
    gs1, kept1 = score(index)                                                 # from the appends' copy
    other = torch.zeros_like(index)
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [0], [0], other)              # the copy now follows `other`
    gs2, kept2 = score(index)                                                 # converted by the call
    assert torch.equal(gs1, gs2) and torch.equal(kept1, kept2)
    # an index whose later rows were written by other means: the copy lacks them, so the call converts
    index3 = torch.zeros_like(index)
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [0], [4000], index3)          # blocks 0..124
    index3[:, :, 125:] = index[:, :, 125:]
    gs3, kept3 = score(index3)
    assert torch.equal(gs1, gs3) and torch.equal(kept1, kept3)
    # and the result matches the oracle
    ora = oracle_step(w, li, 0, range(w.h_kv))
    for g in range(w.h_kv):
        gs_o, tol = ora[g]
        check_group_scores(gs1[0, g].cpu().numpy(), gs_o, tol)
        ids = O.select_blocks(gs_o, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        check_ids(kept1[0, g].cpu().numpy(), ids, gs_o, w, tol)
    ctx.close()
