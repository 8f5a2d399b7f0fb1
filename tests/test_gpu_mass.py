"""The attention-mass diagnostic through the C ABI against the oracle.

Tolerance: |mass_gpu - mass| <= 1e-4 * mass + 1e-7 per block (scores from fp32 rotations composed from
fp64-filled tables, about 2^-22 relative, then fp32 exponentials and sums; the same derivation as the group
scores' 1e-4).  Every row sums to the group size.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O
from synth import device as synth_dev

from harness import dev_u16

pytestmark = pytest.mark.gpu

BLOCK = 32


def check_mass(gpu, ora):
    err = np.abs(np.asarray(gpu, dtype=np.float64) - ora)
    tol = 1e-4 * ora + 1e-7
    assert (err <= tol).all(), f"mass: {(err > tol).sum()} blocks off, worst ratio {(err / tol).max():.3f}"


@pytest.mark.parametrize("name,n_tok,sessions", [("tiny_8k_g4_d64", 8192 - 5, 1), ("gqa40x8_256k", 20000 + 13, 2)])
def test_attention_mass_matches_oracle(name, n_tok, sessions):
    w = synth.WORKLOADS[name].with_(n_tok=n_tok, n_sessions=sessions,
                                    session_seeds=tuple(60 + s for s in range(sessions)))
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    mass = torch.full((sessions, w.h_kv, ctx.max_blocks), -1.0, dtype=torch.float32, device="cuda")
    K.kvm_attention_mass(ctx, dev_u16(li.q[:, 0]), dev_u16(li.k_pool), w.n_pages,
                         torch.from_numpy(li.block_table).cuda(), [n_tok] * sessions, mass)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    G = w.group
    for s in range(sessions):
        for g in range(w.h_kv):
            keys = O.paged_tokens(li.k_pool, li.block_table[s], g, n_tok)
            ora = O.block_attention_mass(li.q[s, 0, G * g:G * (g + 1)], keys, w.rope_theta)
            got = mass[s, g, :w.n_blk].cpu().numpy()
            check_mass(got, ora)
            assert abs(got.astype(np.float64).sum() - G) < 1e-4 * G
    ctx.close()


@pytest.mark.slow
def test_attention_mass_full_size_1m_tokens_sampled_heads():
    """One layer of the 1M-token workspace (32,768 blocks per KV head), two KV heads against the oracle; the
    top-8 share of the planted-topic synthetic history is reported."""
    w = synth.WORKLOADS["ws1m_16layer"]
    layer = 1
    ctx = K.Context.for_workload(w)
    bt_np = synth.block_table(w)
    bt = torch.from_numpy(bt_np).cuda()
    kp = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    synth_dev.fill_kv_pool(w, layer, bt, kp.view(torch.int16), vp.view(torch.int16))
    del vp
    q_np = synth.queries(w, layer)
    mass = torch.zeros((1, w.h_kv, w.n_blk), dtype=torch.float32, device="cuda")
    K.kvm_attention_mass(ctx, dev_u16(q_np[:, 0]), kp, w.n_pages, bt, [w.n_tok], mass)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    G = w.group
    for g in (2, 7):
        kh, _ = synth.kv_pool(w, layer, bt_np, sessions=[0], heads=(g, g + 1))
        keys = O.paged_tokens(kh, bt_np[0], g, w.n_tok)
        del kh
        ora = O.block_attention_mass(q_np[0, 0, G * g:G * (g + 1)], keys, w.rope_theta)
        got = mass[0, g].cpu().numpy()
        check_mass(got, ora)
        print(f"KV head {g}: top-8 share {O.top_mass_share(got, G):.4f} (oracle {O.top_mass_share(ora, G):.4f})")
    ctx.close()
