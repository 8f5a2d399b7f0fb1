"""Step attention over the view (tensor cores) against the oracle.

The step's tokens are the history's last n_q tokens: token t sits at view
position L - n_q + t and attends the slots up to its own.  Views are built
from the oracle's own kept lists (so no oracle input comes from the device
path) or written directly from seeded random values; the GPU's output is
compared element by element with the oracle's fp64 attention, within the
1e-3 absolute bound of harness.py (products are fp32-accurate on the device,
so the observed error is far below it).
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O
from synth import device as synth_dev

from harness import LayerOnDevice, check_out, check_view, dev_u16, host_u16, kept_tensor

pytestmark = pytest.mark.gpu

BLOCK = 32


def _step_ids(w, li, s):
    """The oracle's step-level selection for every KV head of session s."""
    idx16 = np.stack([O.mean_k_index_bf16(O.paged_tokens(li.k_pool, li.block_table[s], g, w.n_tok))
                      for g in range(w.h_kv)])
    gs = O.step_group_scores_bf16(li.q[s], idx16)
    return {g: O.select_blocks(gs[g], w.n_blk, w.n_sink, w.n_recent, w.top_k) for g in range(w.h_kv)}


@pytest.mark.parametrize("d,h_q,h_kv,n_q,n_tok", [(128, 8, 2, 40, 300 * 32 + 7), (64, 12, 3, 33, 200 * 32 + 19),
                                                  (128, 5, 1, 130, 90 * 32)])
def test_step_attention_small_ragged(d, h_q, h_kv, n_q, n_tok):
    """Index, step scores, the oracle's kept lists materialised on the device, then step attention: every
    output row against the oracle (ragged views over several 64-token tiles, ragged 128-row query tiles)."""
    w = synth.Workload("step_attn_small", h_q=h_q, h_kv=h_kv, d=d, n_tok=n_tok, n_sink=3, n_recent=5, top_k=40,
                       rope_theta=1e6, n_planted=4, seed=37, n_q=n_q, attend=False)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    ids = _step_ids(w, li, 0)
    dev.materialize(kept=kept_tensor({(0, g): ids[g] for g in range(h_kv)}, (1, h_kv, ctx.budget)))
    out = torch.full((1, n_q, h_q, d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_step_attn(ctx, dev.q, n_q, dev.k_view, dev.v_view, dev.view_len, 1, out)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    G = w.group
    for g in range(h_kv):
        keys = O.paged_tokens(li.k_pool, li.block_table[0], g, w.n_tok)
        vals = O.paged_tokens(li.v_pool, li.block_table[0], g, w.n_tok)
        kv, vv = O.materialize(keys, vals, ids[g], w.n_tok, w.rope_theta)
        assert int(dev.view_len[0, g]) == kv.shape[0] == w.view_tokens
        check_view(host_u16(dev.k_view[0, g]), host_u16(dev.v_view[0, g]), kv, vv)
        ref = O.step_view_attention(li.q[0][:, G * g:G * (g + 1)], kv, vv, w.rope_theta)
        err = check_out(out[0, :, G * g:G * (g + 1)].cpu().numpy(), ref)
        assert err < 1e-4                    # fp32-accurate products: far inside the 1e-3 bound
    ctx.close()


def _random_view(rng, S, h_kv, cap, d, lens):
    """Seeded bf16 view: keys ~ N(0, 1) (so scores spread over several units), values ~ N(0, 1); the slots past
    each view length hold NaN bit patterns, which the kernel must never read."""
    k = O.f64_to_bf16(rng.standard_normal((S, h_kv, cap, d)))
    v = O.f64_to_bf16(rng.standard_normal((S, h_kv, cap, d)))
    for s in range(S):
        for g in range(h_kv):
            k[s, g, lens[s][g]:] = 0x7FC1
            v[s, g, lens[s][g]:] = 0x7FC1
    return k, v


def test_step_attention_sessions_ragged_lengths_and_edges():
    """Several sessions in one launch; per head a different view length: the step covering the whole view
    (L == n_q), one token past a tile edge, exact tile multiples, and the full capacity."""
    rng = np.random.default_rng(2024)
    h_q, h_kv, d, n_q, theta = 16, 2, 128, 37, 1e4
    n_sink, n_recent, top_k = 1, 2, 17               # budget 20 blocks = 640 slots
    cap = BLOCK * (n_sink + n_recent + top_k)
    lens = [[640, 333], [n_q, 65], [64 * 3, 129]]
    S = len(lens)
    ctx = K.Context(h_q, h_kv, d, n_sink, n_recent, top_k, theta, max_blocks=64, max_sessions=S, max_queries=n_q)
    k, v = _random_view(rng, S, h_kv, cap, d, lens)
    q = O.f64_to_bf16(rng.standard_normal((S, n_q, h_q, d)) * 1.5)
    out = torch.full((S, n_q, h_q, d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_step_attn(ctx, dev_u16(q), n_q, dev_u16(k), dev_u16(v),
                    torch.tensor(lens, dtype=torch.int32, device="cuda"), S, out)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    G = h_q // h_kv
    for s in range(S):
        for g in range(h_kv):
            L = lens[s][g]
            ref = O.step_view_attention(q[s][:, G * g:G * (g + 1)], k[s, g, :L], v[s, g, :L], theta)
            err = check_out(out[s, :, G * g:G * (g + 1)].cpu().numpy(), ref)
            assert err < 1e-4, (s, g, err)
    ctx.close()


def test_single_token_step_attends_the_whole_view():
    """n_q = 1: the token is the view's last slot and attends every slot, itself included."""
    rng = np.random.default_rng(7)
    h_q, h_kv, d, theta = 8, 1, 64, 1e6
    lens = [[1000]]
    ctx = K.Context(h_q, h_kv, d, 0, 1, 39, theta, max_blocks=64, max_sessions=1, max_queries=2)
    k, v = _random_view(rng, 1, h_kv, BLOCK * 40, d, lens)
    q = O.f64_to_bf16(rng.standard_normal((1, 1, h_q, d)) * 2.0)
    out = torch.full((1, 1, h_q, d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_step_attn(ctx, dev_u16(q), 1, dev_u16(k), dev_u16(v), torch.tensor(lens, dtype=torch.int32,
                    device="cuda"), 1, out)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    ref = O.step_view_attention(q[0], k[0, 0, :1000], v[0, 0, :1000], theta)
    assert check_out(out[0].cpu().numpy(), ref) < 1e-4
    ctx.close()


def test_view_shorter_than_the_step_is_reported_not_read_past():
    """A view_len below n_q (or past the capacity) sets the status bit; every access stays in the buffers."""
    h_q, h_kv, d, n_q = 4, 1, 64, 20
    ctx = K.Context(h_q, h_kv, d, 0, 1, 3, 1e4, max_blocks=8, max_sessions=2, max_queries=n_q)
    cap = BLOCK * 4
    k = torch.zeros((2, h_kv, cap, d), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, n_q, h_q, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((2, n_q, h_q, d), dtype=torch.float32, device="cuda")
    K.kvm_step_attn(ctx, q, n_q, k, k, torch.tensor([[5], [cap + 9]], dtype=torch.int32, device="cuda"), 2, out)
    assert K.kvm_device_status(ctx) == K.DEV_BAD_VIEW
    with pytest.raises(K.KvmError):
        K.kvm_step_attn(ctx, q, cap + 1, k, k, torch.tensor([[cap], [cap]], dtype=torch.int32, device="cuda"), 2,
                        out)
    ctx.close()


def test_repeated_step_attention_calls_give_identical_outputs():
    rng = np.random.default_rng(11)
    h_q, h_kv, d, n_q = 10, 2, 128, 64
    lens = [[700, 451]]
    ctx = K.Context(h_q, h_kv, d, 2, 2, 20, 1e6, max_blocks=64, max_sessions=1, max_queries=n_q)
    k, v = _random_view(rng, 1, h_kv, BLOCK * 24, d, lens)
    q = dev_u16(O.f64_to_bf16(rng.standard_normal((1, n_q, h_q, d))))
    vl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kd, vd = dev_u16(k), dev_u16(v)
    outs = []
    for _ in range(3):
        o = torch.full((1, n_q, h_q, d), float("nan"), dtype=torch.float32, device="cuda")
        K.kvm_step_attn(ctx, q, n_q, kd, vd, vl, 1, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    ctx.close()


def _seeded_kept(w, rng):
    """A valid kept list for the full-size geometry chosen by the test: the forced sink and recent blocks plus
    top_k other blocks drawn at random, ascending."""
    n_blk = w.n_blk
    forced = set(range(w.n_sink)) | set(range(n_blk - w.n_recent, n_blk))
    rest = np.array(sorted(set(range(n_blk)) - forced))
    pick = rng.choice(rest, size=w.top_k, replace=False)
    return np.array(sorted(forced | set(pick.tolist())), dtype=np.int32)


@pytest.mark.slow
def test_step_attention_full_size_256_queries_65k_view_sampled_heads():
    """The 256-token step over a 65,536-token view per KV head (40 query heads, 8 KV heads, d 128) from a
    1,048,576-token history, in the launch configuration the bench times; two KV heads recomputed by the
    oracle in full (all 256 x 5 rows)."""
    w = synth.WORKLOADS["step256q_1m"]
    layer = 0
    rng = np.random.default_rng(99)
    ids = {g: _seeded_kept(w, rng) for g in range(w.h_kv)}
    ctx = K.Context.for_workload(w)
    bt_np = synth.block_table(w)
    bt = torch.from_numpy(bt_np).cuda()
    kp = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    synth_dev.fill_kv_pool(w, layer, bt, kp.view(torch.int16), vp.view(torch.int16))
    kept = kept_tensor({(0, g): ids[g] for g in range(w.h_kv)}, (1, w.h_kv, ctx.budget))
    k_view = torch.empty((1, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device="cuda")
    v_view = torch.empty_like(k_view)
    view_len = torch.full((1, w.h_kv), -7, dtype=torch.int32, device="cuda")
    K.kvm_materialize(ctx, kp, vp, w.n_pages, bt, [w.n_tok], kept, k_view, v_view, view_len)
    del kp, vp
    q_np = synth.queries(w, layer)                                  # [1][256][h_q][d]
    q = dev_u16(q_np)
    out = torch.full((1, w.n_q, w.h_q, w.d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvm_step_attn(ctx, q, w.n_q, k_view, v_view, view_len, 1, out)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    G = w.group
    for g in (0, 5):
        kh, vh = synth.kv_pool(w, layer, bt_np, sessions=[0], heads=(g, g + 1))
        keys = O.paged_tokens(kh, bt_np[0], g, w.n_tok)
        vals = O.paged_tokens(vh, bt_np[0], g, w.n_tok)
        del kh, vh
        kv, vv = O.materialize(keys, vals, ids[g], w.n_tok, w.rope_theta)
        assert int(view_len[0, g]) == kv.shape[0] == w.view_tokens
        ref = O.step_view_attention(q_np[0][:, G * g:G * (g + 1)], kv, vv, w.rope_theta)
        check_out(out[0, :, G * g:G * (g + 1)].cpu().numpy(), ref)
    ctx.close()
