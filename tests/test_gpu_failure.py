"""Failure paths of the view calls, on the GPU, without faulting or hanging it.

- A pipeline wait that runs out (a barrier nothing completes, with a short
  wall-clock limit set through kvm_set_wait_limit) is reported as
  KVM_DEV_TIMEOUT in the status word; clearing the word also resets the
  per-call merge counters, and the next call on the same context matches the
  oracle again.
- Kept ids outside the history, or out of ascending order, are reported as
  KVM_DEV_BAD_BLOCK and their slots are skipped: every other view slot and the
  attention over the valid slots still match the oracle.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K
from oracle import kvm_oracle as O

from harness import LayerOnDevice, check_out, check_view, host_u16, kept_tensor, oracle_keys

pytestmark = pytest.mark.gpu


def test_view_wait_timeout_is_reported_and_the_context_recovers():
    from test_gpu_parity import compare_layer
    w = synth.WORKLOADS["gqa40x8_256k"].with_(n_tok=40000)      # every CTA of the view kernel has blocks
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build()
    dev.score_select()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    K.kvm_set_wait_limit(ctx, 100_000, True)       # 0.1 ms; the first rotation wait can never complete
    dev.out.fill_(float("nan"))
    dev.fused()
    st = K.kvm_device_status(ctx, clear=False)
    assert st & K.DEV_TIMEOUT, f"status 0x{st:x}"
    # the C call reports it as a timeout, and clearing resets the word (and the merge counters)
    assert K.kvm_device_status(ctx, clear=True) & K.DEV_TIMEOUT
    assert K.kvm_device_status(ctx) == 0
    K.kvm_set_wait_limit(ctx)                      # back to the normal limit, no stall
    dev.out.fill_(float("nan"))
    dev.fused()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    assert compare_layer(w, li, dev, heads=[0, 3, 7]) >= 2
    # and once more: the counters of the recovered call were left at zero for the next one
    first = dev.out.clone()
    dev.fused()
    torch.cuda.synchronize()
    assert torch.equal(dev.out, first)
    ctx.close()



def test_fp8_view_wait_timeout_is_reported_and_the_context_recovers():
    """The same on the FP8 view path, whose loads fill a ring of code slots and whose rotation warps wait for their
    stages: the timed-out call reports KVM_DEV_TIMEOUT, and the next calls give the first call's view and output
    bit for bit."""
    w = synth.WORKLOADS["gqa40x8_256k"].with_(n_tok=40000)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build()
    dev.score_select()
    n = dev.n_pages
    pages = torch.arange(n, dtype=torch.int32, device="cuda")
    k8 = torch.empty((n, w.h_kv, 32, w.d), dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((n, w.h_kv), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    K.kvm_quantize_pages(ctx, dev.k_pool, n, pages, k8, ks)
    K.kvm_quantize_pages(ctx, dev.v_pool, n, pages, v8, vs)

    def fused8():
        K.kvm_materialize_attn_fp8(ctx, k8, ks, v8, vs, n, dev.bt, dev.n_tok, dev.kept, dev.q, dev.k_view,
                                   dev.v_view, dev.view_len, dev.out)

    fused8()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    out0, kview0, vview0 = dev.out.clone(), dev.k_view.clone(), dev.v_view.clone()
    K.kvm_set_wait_limit(ctx, 100_000, True)       # 0.1 ms; the first rotation wait can never complete
    dev.out.fill_(float("nan"))
    fused8()
    assert K.kvm_device_status(ctx, clear=True) & K.DEV_TIMEOUT
    assert K.kvm_device_status(ctx) == 0
    K.kvm_set_wait_limit(ctx)
    for _ in range(2):
        dev.out.fill_(float("nan"))
        fused8()
        torch.cuda.synchronize()
        assert K.kvm_device_status(ctx) == 0
        assert torch.equal(dev.out, out0)
        assert torch.equal(dev.k_view, kview0) and torch.equal(dev.v_view, vview0)
    ctx.close()

def _expected_view_and_out(w, li, slots, q_group, L):
    """View rows and attention output for {slot: block id} (the valid slots), query at position L."""
    keys = oracle_keys(w, li, 0, 0)
    vals = O.paged_tokens(li.v_pool, li.block_table[0], 0, w.n_tok)
    rows_k, rows_v = {}, {}
    for i, b in slots.items():
        t = np.arange(b * 32, min(w.n_tok, b * 32 + 32))
        rows_k[i] = O.f64_to_bf16(O.rope(O.bf16_to_f64(keys[t]), 32 * i + np.arange(len(t)), w.rope_theta))
        rows_v[i] = vals[t]
    kf = O.bf16_to_f64(np.concatenate([rows_k[i] for i in sorted(slots)]))
    vf = O.bf16_to_f64(np.concatenate([rows_v[i] for i in sorted(slots)]))
    qr = O.rope(O.bf16_to_f64(q_group), L, w.rope_theta)
    s = qr @ kf.T / np.sqrt(w.d)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return rows_k, rows_v, p @ vf


@pytest.mark.parametrize("fault", ["out_of_range", "not_ascending"])
def test_bad_kept_ids_are_reported_and_skipped(fault):
    w = synth.WORKLOADS["tiny_8k_g4_d64"]
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    keys = oracle_keys(w, li, 0, 0)
    gs = O.gqa_softmax_sum(O.block_scores(li.q[0, 0], O.mean_k_index(keys)[None]), 1)[0]
    ids = O.select_blocks(gs, w.n_blk, w.n_sink, w.n_recent, w.top_k).copy()
    bad = 6
    if fault == "out_of_range":
        ids[bad] = w.n_blk + 3
    else:
        ids[bad - 1], ids[bad] = ids[bad], ids[bad - 1]  # slot bad-1 now holds the larger id: slot bad is out of order
    # the documented rule: a slot is skipped when its id is outside the history or not above the entry before it
    # (so an out-of-range entry also makes the next slot, which is not above it, a skipped one)
    skipped = {i for i in range(len(ids)) if not (0 <= ids[i] < w.n_blk) or (i > 0 and ids[i] <= ids[i - 1])}
    assert bad in skipped
    slots = {i: int(b) for i, b in enumerate(ids) if i not in skipped}
    dev.k_view.fill_(0)
    dev.v_view.fill_(0)
    dev.fused(kept_tensor({(0, 0): ids}, (1, 1, ctx.budget)))
    st = K.kvm_device_status(ctx, clear=True)
    assert st & K.DEV_BAD_BLOCK and not st & (K.DEV_BAD_PAGE | K.DEV_TIMEOUT), f"status 0x{st:x}"
    L = 32 * len(ids)                                   # the last kept block is full
    assert int(dev.view_len[0, 0]) == L
    rows_k, rows_v, out = _expected_view_and_out(w, li, slots, li.q[0, 0], L)
    kv, vv = host_u16(dev.k_view[0, 0]), host_u16(dev.v_view[0, 0])
    for i in slots:
        check_view(kv[32 * i:32 * i + 32], vv[32 * i:32 * i + 32], rows_k[i], rows_v[i])
    for i in skipped:  # skipped slots are not written
        assert not kv[32 * i:32 * i + 32].any() and not vv[32 * i:32 * i + 32].any()
    check_out(dev.out[0].cpu().numpy(), out)
    assert K.kvm_device_status(ctx) == 0
    ctx.close()
