"""Guard bytes around every buffer the device path writes.

Each output buffer is a window into a larger allocation whose other bytes hold a known pattern; after the
calls, the pattern must be intact on both sides of every window, and inside the views past each head's view
length (slots a head does not use are never written).  This catches a tensor-map extent, a store index or a
row stride that runs past its buffer, which the value comparisons of the parity tests cannot see when the
stray bytes land in memory no test reads.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K

from harness import dev_u16

pytestmark = pytest.mark.gpu

GUARD = 4096                 # elements of pattern on each side of a window
PATTERN16 = 0x5A5A           # bf16 / int16 windows
PATTERN32 = 0x7FA5A5A5       # fp32 / int32 windows (a NaN payload no kernel writes)


class Guarded:
    """A window of `shape` and `dtype` inside an allocation filled with the pattern."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape))
        wide = torch.int16 if dtype in (torch.bfloat16, torch.int16) else torch.int32
        pat = PATTERN16 if wide == torch.int16 else PATTERN32
        if wide == torch.int16:
            pat = pat - 0x10000 if pat >= 0x8000 else pat
        self.raw = torch.full((n + 2 * GUARD,), pat, dtype=wide, device="cuda")
        self.pat = pat
        self.window = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.window.fill_(fill)

    def assert_guards(self, name):
        lo, hi = self.raw[:GUARD], self.raw[-GUARD:]
        assert bool((lo == self.pat).all()), f"{name}: bytes before the buffer were written"
        assert bool((hi == self.pat).all()), f"{name}: bytes after the buffer were written"


def _two_session_case():
    """Session 0: 5000 tokens (selection active); session 1: 700 tokens (every block kept, view shorter than
    the budget); one pool."""
    base = synth.Workload("canary", h_q=8, h_kv=2, d=128, n_tok=5000, n_sessions=1, n_sink=1, n_recent=2,
                          top_k=30, rope_theta=1e6, n_planted=4, seed=61)
    lens = [5000, 700]
    per = [synth.layer_inputs(base.with_(n_tok=max(n, 512), seed=61 + s), 0) for s, n in enumerate(lens)]
    bt = np.full((2, base.n_blk), -1, dtype=np.int32)
    off = 0
    for s, p in enumerate(per):
        bt[s, :p.block_table.shape[1]] = p.block_table[0] + off
        off += p.k_pool.shape[0]
    kp = np.concatenate([p.k_pool for p in per], axis=0)
    vp = np.concatenate([p.v_pool for p in per], axis=0)
    q = np.stack([p.q[0, 0] for p in per])
    return base, lens, kp, vp, bt, q


@pytest.mark.parametrize("mode", ["fused", "unfused", "fp8"])
def test_no_write_outside_the_output_buffers(mode):
    base, lens, kp, vp, bt, q = _two_session_case()
    S, hk, d, hq = 2, base.h_kv, base.d, base.h_q
    ctx = K.Context(hq, hk, d, base.n_sink, base.n_recent, base.top_k, base.rope_theta,
                    max_blocks=base.n_blk, max_sessions=S)
    budget = ctx.budget
    n_pages = kp.shape[0]
    kpd, vpd, btd, qd = dev_u16(kp), dev_u16(vp), torch.from_numpy(bt).cuda(), dev_u16(q)
    index = Guarded((S, hk, base.n_blk, d), torch.float32, 0.0)
    kept = Guarded((S, hk, budget), torch.int32)
    gs = Guarded((S, hk, base.n_blk), torch.float32, 0.0)
    hs = Guarded((S, hq, base.n_blk), torch.float32, 0.0)
    kv = Guarded((S, hk, 32 * budget, d), torch.bfloat16)
    vv = Guarded((S, hk, 32 * budget, d), torch.bfloat16)
    vlen = Guarded((S, hk), torch.int32)
    out = Guarded((S, hq, d), torch.float32)
    if mode == "fp8":
        # FP8 codes (one byte each) in int16-patterned allocations, viewed as bytes
        k8g = Guarded((n_pages * hk * 32 * d // 2,), torch.int16)
        v8g = Guarded((n_pages * hk * 32 * d // 2,), torch.int16)
        k8 = k8g.window.view(torch.uint8).view(n_pages, hk, 32, d)
        v8 = v8g.window.view(torch.uint8).view(n_pages, hk, 32, d)
        ks = Guarded((n_pages, hk), torch.float32)
        vs = Guarded((n_pages, hk), torch.float32)
        pages = torch.arange(n_pages, dtype=torch.int32, device="cuda")
        K.kvm_quantize_pages(ctx, kpd, n_pages, pages, k8, ks.window)
        K.kvm_quantize_pages(ctx, vpd, n_pages, pages, v8, vs.window)
        K.kvm_index_append_fp8(ctx, k8, ks.window, n_pages, btd, [0, 0], lens, index.window)
    else:
        K.kvm_index_append(ctx, kpd, n_pages, btd, [0, 0], lens, index.window)
    K.kvm_score_select(ctx, qd, 1, index.window, lens, kept.window, gs.window, hs.window)
    if mode == "fused":
        K.kvm_materialize_attn(ctx, kpd, vpd, n_pages, btd, lens, kept.window, qd, kv.window, vv.window,
                               vlen.window, out.window)
    elif mode == "unfused":
        K.kvm_materialize(ctx, kpd, vpd, n_pages, btd, lens, kept.window, kv.window, vv.window, vlen.window)
        K.kvm_decode_attn(ctx, qd, kv.window, vv.window, vlen.window, S, out.window)
    else:
        K.kvm_materialize_attn_fp8(ctx, k8, ks.window, v8, vs.window, n_pages, btd, lens, kept.window, qd,
                                   kv.window, vv.window, vlen.window, out.window)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    named = {"index": index, "kept": kept, "group scores": gs, "head scores": hs, "K view": kv, "V view": vv,
             "view lengths": vlen, "output": out}
    if mode == "fp8":
        named.update({"K codes": k8g, "V codes": v8g, "K scales": ks, "V scales": vs})
    for name, g in named.items():
        g.assert_guards(name)
    # inside the views: the slots past each head's view length keep the pattern
    L = vlen.window.cpu().numpy()
    assert L[1].max() < 32 * budget, "the short session must leave view slots unused"
    for s in range(S):
        for h in range(hk):
            for buf, name in ((kv, "K view"), (vv, "V view")):
                tail = buf.window[s, h, L[s, h]:].view(torch.int16)
                assert bool((tail == buf.pat).all()), f"{name} ({s}, {h}) written past its view length {L[s, h]}"
    # the kept lists end with -1 where fewer blocks exist than the budget; nothing is left unwritten
    assert not bool((kept.window == PATTERN32).any()), "a kept-list slot was never written"
    ctx.close()
