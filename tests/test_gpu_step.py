"""Step-level (multi-query) scoring on the tensor cores against the oracle.

The contraction takes bf16 operands; the oracle forms the bf16 index operand
the way the kernel does (fp32 mean, then nearest-even bf16) and scores in
fp64.  Tolerances: group scores 1e-4 relative (see harness.py), kept ids by
the near-boundary rule.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O

from harness import check_group_scores, check_ids, dev_u16

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


def oracle_step(w, li, s, heads):
    idx16 = np.stack([O.mean_k_index_bf16(O.paged_tokens(li.k_pool, li.block_table[s], g, w.n_tok))
                      for g in range(w.h_kv)])
    gs = O.step_group_scores_bf16(li.q[s], idx16)
    return {g: gs[g] for g in heads}


@pytest.mark.parametrize("d,h_q,h_kv,n_q", [(128, 8, 2, 40), (64, 12, 3, 33), (128, 5, 1, 256)])
def test_step_scores_small_ragged(d, h_q, h_kv, n_q):
    w = synth.Workload("step_small", h_q=h_q, h_kv=h_kv, d=d, n_tok=300 * 32 + 7, n_sink=3, n_recent=5, top_k=40,
                       rope_theta=1e6, n_planted=4, seed=31, n_q=n_q, attend=False)
    li = synth.layer_inputs(w, 0)
    gs, kept = run_step(w, li)
    ora = oracle_step(w, li, 0, range(w.h_kv))
    assert np.allclose(ora[0].sum(), n_q * w.group, rtol=1e-9)
    for g in range(w.h_kv):
        check_group_scores(gs[0, g], ora[g])
        ids = O.select_blocks(ora[g], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        check_ids(kept[0, g], ids, ora[g], w)


@pytest.mark.slow
def test_step_scores_full_size_256_queries_1m_tokens():
    w = synth.WORKLOADS["step256q_1m"]
    li = synth.layer_inputs(w, 0)
    gs, kept = run_step(w, li)
    heads = [0, 5]                                     # sampled KV heads (the oracle scores them in full)
    ora = oracle_step(w, li, 0, heads)
    same = 0
    for g in heads:
        check_group_scores(gs[0, g], ora[g])
        ids = O.select_blocks(ora[g], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        same += check_ids(kept[0, g], ids, ora[g], w)
        # planted blocks of this head are found by the step's queries
        assert len(set(kept[0, g].tolist()) & set(li.planted[0, g].tolist())) >= 12
    assert same >= 1
