"""The allocation-free score+select entry point agrees with kvm_score_select.

kvm_score_select_noalloc serves callers that cannot allocate device memory
(a runtime whose pool owns all device memory, or code that must not
synchronise the device), so it keeps its scratch in a fixed array inside the
library instead of a context.  This file is collected last on purpose: it
reuses that shared array across calls, and a failure here should not hide the
results of the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import sparse_attention_decode_04_b300 as K

from harness import LayerOnDevice, check_group_scores

pytestmark = pytest.mark.gpu


def _params(w):
    return K.Params(w.h_q, w.h_kv, w.d, w.n_sink, w.n_recent, w.top_k, w.rope_theta, w.n_blk, 1, 1)


@pytest.mark.parametrize("name", ["tiny_8k_g4_d64", "gqa40x8_256k"])
def test_noalloc_matches_context_entry_point_on_two_calls(name):
    w = synth.WORKLOADS[name]
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build()
    dev.score_select()                       # the existing entry point (context scratch)
    torch.cuda.synchronize()
    ref_ids = dev.kept.cpu().numpy()
    ref_gs = dev.gs.cpu().numpy()
    p = _params(w)
    K.kvm_noalloc_status(clear=True)           # start from a clear word, whatever ran before in this process
    for call in range(2):                    # two calls in a row share the library's scratch array
        kept = torch.full_like(dev.kept, -7)
        gs = torch.full_like(dev.gs, float("nan"))
        K.kvm_score_select_noalloc(p, dev.q, dev.index, [w.n_tok], kept, gs)
        torch.cuda.synchronize()
        # no device-side error was recorded by the call (the word is readable, and stays set until cleared)
        assert K.kvm_noalloc_status(clear=False) == 0
        assert np.array_equal(kept.cpu().numpy(), ref_ids), f"call {call}: kept ids differ"
        got = gs.cpu().numpy()
        for g in range(w.h_kv):
            check_group_scores(got[0, g, :w.n_blk], ref_gs[0, g, :w.n_blk].astype(np.float64))
    ctx.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synth.WORKLOADS["ws1m_16layer"]
    p = K.Params(w.h_q, w.h_kv, w.d, w.n_sink, w.n_recent, w.top_k, w.rope_theta, 8 * 40960, 1, 1)
    q = torch.zeros((2, w.h_q, w.d), dtype=torch.bfloat16, device="cuda")
    index = torch.zeros((2, w.h_kv, 16, w.d), dtype=torch.float32, device="cuda")   # never read
    kept = torch.zeros((2, w.h_kv, w.budget), dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvmError) as e:
        K.kvm_score_select_noalloc(p, q, index, [32, 32], kept)
    assert e.value.status == 2 and "at most" in str(e.value)
    assert torch.all(kept == 0)
