"""Page tiers beyond the bf16 HBM pool, through the C ABI against the oracle.

FP8 E4M3 pages: codes and scales bit-exact (both sides decide them in fp32),
the Mean-K index of the dequantised keys within the index tolerance, the view
from quantised pages (V bit-exact, K within one bf16 ulp) and attention over
it within 1e-3.  Host-resident pages: the view gathered over the host link is
checked the same way.  Kept lists are the oracle's own (or chosen by the
test), so no oracle input comes from the device path.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O
from synth import device as synth_dev

from harness import check_group_scores, check_ids, check_out, check_view, dev_u16, host_u16, kept_tensor

pytestmark = pytest.mark.gpu

BLOCK = 32


def check_index_values(gpu_idx, keys, ora_idx):
    """|k_bar_gpu - k_bar| <= 2^-18 * mean_t |k_t,i| per element (fp32 sum of <= 32 terms)."""
    k = np.abs(np.asarray(keys, dtype=np.float64))
    n_tok, d = k.shape
    n_blk = ora_idx.shape[0]
    pad = np.zeros((n_blk * BLOCK - n_tok, d))
    cnt = np.minimum(BLOCK, n_tok - BLOCK * np.arange(n_blk))[:, None]
    mean_abs = np.concatenate([k, pad]).reshape(n_blk, BLOCK, d).sum(axis=1) / cnt
    err = np.abs(np.asarray(gpu_idx, dtype=np.float64) - ora_idx)
    assert (err <= 2.0 ** -18 * mean_abs).all(), f"index: worst error {err.max():.3e}"


def _quantized_layer(w, li, ctx):
    """Device bf16 pools -> device FP8 pools through kvm_quantize_pages (every page, in a shuffled order)."""
    kp, vp = dev_u16(li.k_pool), dev_u16(li.v_pool)
    n_pages = li.k_pool.shape[0]
    order = torch.from_numpy(np.random.default_rng(5).permutation(n_pages).astype(np.int32)).cuda()
    k8 = torch.zeros(tuple(li.k_pool.shape), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    ks = torch.zeros((n_pages, w.h_kv), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    K.kvm_quantize_pages(ctx, kp, n_pages, order, k8, ks)
    K.kvm_quantize_pages(ctx, vp, n_pages, order, v8, vs)
    return k8, ks, v8, vs


@pytest.mark.parametrize("name,n_tok", [("tiny_8k_g4_d64", None), ("gqa40x8_256k", 20000 + 17)])
def test_quantize_pages_codes_and_scales_bit_exact(name, n_tok):
    w = synth.WORKLOADS[name]
    if n_tok:
        w = w.with_(n_tok=n_tok)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    k8, ks, v8, vs = _quantized_layer(w, li, ctx)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    ok_codes, ok_scales = O.quantize_pool(li.k_pool)
    ov_codes, ov_scales = O.quantize_pool(li.v_pool)
    assert np.array_equal(ks.cpu().numpy(), ok_scales) and np.array_equal(vs.cpu().numpy(), ov_scales)
    assert np.array_equal(k8.cpu().numpy(), ok_codes) and np.array_equal(v8.cpu().numpy(), ov_codes)
    ctx.close()


@pytest.mark.parametrize("name,n_tok", [("tiny_8k_g4_d64", 8192 - 9), ("gqa40x8_256k", 20000 + 17)])
def test_fp8_index_view_and_attention_match_oracle(name, n_tok):
    """Index over quantised keys (history, then a ragged append), the oracle's selection on it, the view from
    quantised pages and decode attention over that view."""
    w = synth.WORKLOADS[name].with_(n_tok=n_tok)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    k8, ks, v8, vs = _quantized_layer(w, li, ctx)
    bt = torch.from_numpy(li.block_table).cuda()
    S = 1
    index = torch.zeros((S, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device="cuda")
    n_hist = n_tok - 45
    K.kvm_index_append_fp8(ctx, k8, ks, w.n_pages, bt, [0], [n_hist], index)
    K.kvm_index_append_fp8(ctx, k8, ks, w.n_pages, bt, [n_hist], [45], index)
    k_codes, k_scales = O.quantize_pool(li.k_pool)
    v_codes, v_scales = O.quantize_pool(li.v_pool)
    G = w.group
    ids, keys, vals = {}, {}, {}
    for g in range(w.h_kv):
        keys[g] = O.paged_dequant_tokens(k_codes, k_scales, li.block_table[0], g, n_tok)
        vals[g] = O.paged_dequant_tokens(v_codes, v_scales, li.block_table[0], g, n_tok)
        idx = O.mean_k_index_of(keys[g])
        gs = O.gqa_softmax_sum(O.block_scores(li.q[0, 0, G * g:G * (g + 1)], idx[None]), 1)[0]
        ids[g] = O.select_blocks(gs, w.n_blk, w.n_sink, w.n_recent, w.top_k)
    kept = kept_tensor({(0, g): ids[g] for g in range(w.h_kv)}, (S, w.h_kv, ctx.budget))
    k_view = torch.zeros((S, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device="cuda")
    v_view = torch.zeros_like(k_view)
    view_len = torch.full((S, w.h_kv), -7, dtype=torch.int32, device="cuda")
    K.kvm_materialize_fp8(ctx, k8, ks, v8, vs, w.n_pages, bt, [n_tok], kept, k_view, v_view, view_len)
    q = dev_u16(li.q[:, 0])
    out = torch.full((S, w.h_q, w.d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_decode_attn(ctx, q, k_view, v_view, view_len, S, out)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    # the same view and attention in one pass (kvm_materialize_attn_fp8), into fresh buffers
    k_view2 = torch.zeros_like(k_view)
    v_view2 = torch.zeros_like(v_view)
    view_len2 = torch.full_like(view_len, -7)
    out2 = torch.full_like(out, float("nan"))
    K.kvm_materialize_attn_fp8(ctx, k8, ks, v8, vs, w.n_pages, bt, [n_tok], kept, q, k_view2, v_view2, view_len2, out2)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    for g in range(w.h_kv):
        check_index_values(index[0, g].cpu().numpy(), keys[g], O.mean_k_index_of(keys[g]))
        kv, vv = O.materialize_values(keys[g], vals[g], ids[g], n_tok, w.rope_theta)
        ref = O.decode_attention(li.q[0, 0, G * g:G * (g + 1)], kv, vv, w.rope_theta)
        for kvd, vvd, vld, od in ((k_view, v_view, view_len, out), (k_view2, v_view2, view_len2, out2)):
            assert int(vld[0, g]) == kv.shape[0]
            check_view(host_u16(kvd[0, g]), host_u16(vvd[0, g]), kv, vv)
            check_out(od[0, G * g:G * (g + 1)].cpu().numpy(), ref)
    # V from either path is the same bf16 rounding of the same fp32 values: bit-identical
    assert torch.equal(v_view.view(torch.int16), v_view2.view(torch.int16))
    ctx.close()


def _pinned(a: np.ndarray) -> torch.Tensor:
    t = torch.empty(a.shape, dtype=torch.int16, pin_memory=True)
    t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)))
    return t.view(torch.bfloat16)


@pytest.mark.parametrize("name,n_tok,sessions", [("tiny_8k_g4_d64", 8192 - 3, 1), ("gqa40x8_256k", 12000 + 5, 2)])
def test_host_resident_pages_give_the_oracle_view(name, n_tok, sessions):
    """Pools in pinned host memory; the gather reads the kept rows over the host link."""
    w = synth.WORKLOADS[name].with_(n_tok=n_tok, n_sessions=sessions,
                                    session_seeds=tuple(40 + s for s in range(sessions)))
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    kh, vh = _pinned(li.k_pool), _pinned(li.v_pool)
    bt = torch.from_numpy(li.block_table).cuda()
    rng = np.random.default_rng(17)
    ids = {}
    for s in range(sessions):
        for g in range(w.h_kv):
            # a kept list chosen by the test: forced blocks plus random others (the last block is partial)
            forced = set(range(w.n_sink)) | set(range(w.n_blk - w.n_recent, w.n_blk))
            rest = sorted(set(range(w.n_blk)) - forced)
            ids[(s, g)] = np.array(sorted(forced | set(rng.choice(rest, w.n_keep - len(forced), replace=False)
                                                       .tolist())), dtype=np.int32)
    kept = kept_tensor(ids, (sessions, w.h_kv, ctx.budget))
    k_view = torch.zeros((sessions, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device="cuda")
    v_view = torch.zeros_like(k_view)
    view_len = torch.full((sessions, w.h_kv), -7, dtype=torch.int32, device="cuda")
    K.kvm_materialize_host(ctx, kh, vh, w.n_pages, bt, [n_tok] * sessions, kept, k_view, v_view, view_len)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    for (s, g), kid in ids.items():
        keys = O.paged_tokens(li.k_pool, li.block_table[s], g, n_tok)
        vals = O.paged_tokens(li.v_pool, li.block_table[s], g, n_tok)
        kv, vv = O.materialize(keys, vals, kid, n_tok, w.rope_theta)
        assert int(view_len[s, g]) == kv.shape[0] == w.view_tokens
        check_view(host_u16(k_view[s, g]), host_u16(v_view[s, g]), kv, vv)
    # a device pointer is not a host pool
    with pytest.raises(K.KvmError):
        K.kvm_materialize_host(ctx, k_view, v_view, w.n_pages, bt, [n_tok] * sessions, kept, k_view, v_view,
                               view_len)
    ctx.close()


@pytest.mark.slow
def test_fp8_full_size_1m_token_layer_sampled_heads():
    """One layer of the 1M-token workspace with FP8 pages, in the launch configuration the bench times: index
    over the quantised history, score and select, the view from quantised pages, decode attention; two KV heads
    recomputed by the oracle."""
    w = synth.WORKLOADS["ws1m_16layer"]
    layer = 2
    ctx = K.Context.for_workload(w)
    bt_np = synth.block_table(w)
    bt = torch.from_numpy(bt_np).cuda()
    k8 = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((w.n_pages, w.h_kv), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    kp = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    synth_dev.fill_kv_pool(w, layer, bt, kp.view(torch.int16), vp.view(torch.int16))
    all_pages = torch.arange(w.n_pages, dtype=torch.int32, device="cuda")
    K.kvm_quantize_pages(ctx, kp, w.n_pages, all_pages, k8, ks)
    K.kvm_quantize_pages(ctx, vp, w.n_pages, all_pages, v8, vs)
    torch.cuda.synchronize()
    del kp, vp
    index = torch.zeros((1, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device="cuda")
    K.kvm_index_append_fp8(ctx, k8, ks, w.n_pages, bt, [0], [w.n_tok], index)
    q_np = synth.queries(w, layer)
    q = dev_u16(q_np[:, 0])
    kept = torch.full((1, w.h_kv, ctx.budget), -7, dtype=torch.int32, device="cuda")
    gs = torch.zeros((1, w.h_kv, w.n_blk), dtype=torch.float32, device="cuda")
    K.kvm_score_select(ctx, q, 1, index, [w.n_tok], kept, gs)
    k_view = torch.empty((1, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device="cuda")
    v_view = torch.empty_like(k_view)
    view_len = torch.full((1, w.h_kv), -7, dtype=torch.int32, device="cuda")
    K.kvm_materialize_fp8(ctx, k8, ks, v8, vs, w.n_pages, bt, [w.n_tok], kept, k_view, v_view, view_len)
    out = torch.full((1, w.h_q, w.d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_decode_attn(ctx, q, k_view, v_view, view_len, 1, out)
    # the fused FP8 call (the bench's launch configuration for FP8 pages), into its own buffers
    k_view2 = torch.empty_like(k_view)
    v_view2 = torch.empty_like(v_view)
    view_len2 = torch.full_like(view_len, -7)
    out2 = torch.full_like(out, float("nan"))
    K.kvm_materialize_attn_fp8(ctx, k8, ks, v8, vs, w.n_pages, bt, [w.n_tok], kept, q, k_view2, v_view2, view_len2,
                               out2)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    assert torch.equal(view_len, view_len2) and torch.equal(v_view.view(torch.int16), v_view2.view(torch.int16))
    G = w.group
    same = 0
    for g in (1, 6):
        kh, vh = synth.kv_pool(w, layer, bt_np, sessions=[0], heads=(g, g + 1))
        pages = bt_np[0][:w.n_blk]
        kc = np.zeros((w.n_pages, 1, BLOCK, w.d), dtype=np.uint8)
        vc = np.zeros_like(kc)
        ksc = np.zeros((w.n_pages, 1), dtype=np.float32)
        vsc = np.zeros_like(ksc)
        for p in pages:
            kc[p, 0], ksc[p, 0] = O.quantize_page(kh[p, g])
            vc[p, 0], vsc[p, 0] = O.quantize_page(vh[p, g])
        del kh, vh
        assert np.array_equal(ks.cpu().numpy()[pages, g], ksc[pages, 0])
        keys = O.paged_dequant_tokens(kc, ksc, bt_np[0], 0, w.n_tok)
        vals = O.paged_dequant_tokens(vc, vsc, bt_np[0], 0, w.n_tok)
        idx = O.mean_k_index_of(keys)
        check_index_values(index[0, g].cpu().numpy(), keys, idx)
        qg = q_np[0, 0, G * g:G * (g + 1)]
        gso = O.gqa_softmax_sum(O.block_scores(qg, idx[None]), 1)[0]
        check_group_scores(gs[0, g].cpu().numpy(), gso)
        ids = O.select_blocks(gso, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        if not check_ids(kept[0, g].cpu().numpy(), ids, gso, w):
            continue
        same += 1
        kv, vv = O.materialize_values(keys, vals, ids, w.n_tok, w.rope_theta)
        ref = O.decode_attention(qg, kv, vv, w.rope_theta)
        for kvd, vvd, od in ((k_view, v_view, out), (k_view2, v_view2, out2)):
            check_view(host_u16(kvd[0, g]), host_u16(vvd[0, g]), kv, vv)
            check_out(od[0, G * g:G * (g + 1)].cpu().numpy(), ref)
    assert same >= 1
    ctx.close()
