"""The selection controls through the C ABI against the oracle, and their
contrast with the method at the same block budget.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O

from harness import LayerOnDevice, check_group_scores, check_ids, oracle_keys

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_tok", [("tiny_8k_g4_d64", None), ("gqa40x8_256k", 40000)])
def test_withdrawn_averaged_scoring_matches_oracle(name, n_tok):
    w = synth.WORKLOADS[name]
    if n_tok:
        w = w.with_(n_tok=n_tok)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build()
    kept = torch.full_like(dev.kept, -7)
    gs = torch.zeros_like(dev.gs)
    K.kvm_select_control(ctx, K.CONTROL_WITHDRAWN_AVERAGE, dev.q, dev.index, dev.n_tok, kept, gs)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    idx = np.stack([O.mean_k_index(oracle_keys(w, li, 0, g)) for g in range(w.h_kv)])
    ora = O.withdrawn_group_scores(li.q[0, 0], idx)
    assert np.allclose(ora.sum(axis=1), 1.0, rtol=1e-12)     # one softmax per KV head
    for g in range(w.h_kv):
        check_group_scores(gs[0, g, :w.n_blk].cpu().numpy(), ora[g])
        ids = O.select_blocks(ora[g], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        check_ids(kept[0, g].cpu().numpy(), ids, ora[g], w)
    ctx.close()


def test_recent_only_keeps_the_last_budget_blocks():
    base = synth.Workload("recent", h_q=8, h_kv=2, d=128, n_tok=5000, n_sink=1, n_recent=2, top_k=30,
                          rope_theta=1e6, n_planted=4, seed=3)
    lens = [700, 0, 5000, 33 * 32 + 5]
    ctx = K.Context(base.h_q, base.h_kv, base.d, base.n_sink, base.n_recent, base.top_k, base.rope_theta,
                    max_blocks=base.n_blk, max_sessions=len(lens))
    kept = torch.full((len(lens), base.h_kv, ctx.budget), -7, dtype=torch.int32, device="cuda")
    K.kvm_select_control(ctx, K.CONTROL_RECENT_ONLY, None, None, lens, kept)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    for s, n in enumerate(lens):
        n_blk = -(-n // 32)
        n_keep = min(n_blk, ctx.budget)
        want = np.full(ctx.budget, -1)
        want[:n_keep] = np.arange(n_blk - n_keep, n_blk)
        for g in range(base.h_kv):
            assert np.array_equal(kept[s, g].cpu().numpy(), want)
    ctx.close()


@pytest.mark.parametrize("name,n_tok", [("tiny_8k_g4_d64", None), ("gqa40x8_256k", 40000)])
def test_recent_only_keeps_less_relevance_than_kvmem(name, n_tok):
    """At the same budget, the blocks KVMem keeps hold the planted relevant blocks and the most group-score
    mass; the recent-only blocks hold the planted ones only by chance.  (The pages compare task loss on a real
    model; on these synthetic keys the relevance lives in the pre-RoPE space the index scores, so that is
    where the contrast is checked.)"""
    w = synth.WORKLOADS[name]
    if n_tok:
        w = w.with_(n_tok=n_tok)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build()
    dev.score_select()
    recent = torch.full_like(dev.kept, -7)
    K.kvm_select_control(ctx, K.CONTROL_RECENT_ONLY, None, None, dev.n_tok, recent)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    mass_k = mass_r = 0.0
    planted_k = planted_r = 0
    for g in range(w.h_kv):
        ids_k = dev.kept[0, g].cpu().numpy()
        ids_r = recent[0, g].cpu().numpy()
        ids_k, ids_r = ids_k[ids_k >= 0], ids_r[ids_r >= 0]
        assert len(ids_k) == len(ids_r) == w.n_keep                 # the same budget
        gs = dev.gs[0, g, :w.n_blk].cpu().numpy().astype(np.float64)
        mass_k += gs[ids_k].sum()
        mass_r += gs[ids_r].sum()
        planted = set(li.planted[0, g].tolist())
        planted_k += len(planted & set(ids_k.tolist()))
        planted_r += len(planted & set(ids_r.tolist()))
    assert mass_k > mass_r
    assert planted_k >= (3 * w.n_planted * w.h_kv) // 4 and planted_k > planted_r
    ctx.close()
