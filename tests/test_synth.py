"""The seeded input generator: Philox known answers and the workload recipe's statistics."""
import numpy as np

import synth
from oracle import kvm_oracle as O


def test_philox_known_answers():
    # Known-answer vectors published with Random123 for Philox4x32-10.
    assert synth.philox4x32_10([0, 0, 0, 0], [0, 0]) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)
    assert synth.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)
    assert synth.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]) == (
        0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)


def test_recipe_statistics_and_determinism():
    w = synth.WORKLOADS["tiny_8k_g4_d64"]
    a = synth.layer_inputs(w, 0)
    b = synth.layer_inputs(w, 0)
    assert np.array_equal(a.k_pool, b.k_pool) and np.array_equal(a.q, b.q)
    k = O.bf16_to_f64(a.k_pool)
    assert abs(np.mean(k ** 2) - 1.0) < 1e-2                   # keys are RMS-normalised
    v = O.bf16_to_f64(a.v_pool)
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1.0) < 0.02
    q = O.bf16_to_f64(a.q)
    assert np.allclose(np.mean(q ** 2, axis=-1), 1.0, atol=1e-2)
    # within a block, keys share the topic: same-block key pairs correlate, cross-block ones do not
    kk = k[:, 0].reshape(-1, 32, w.d)
    same = np.mean(np.sum(kk[:, 0] * kk[:, 1], axis=-1)) / w.d
    cross = np.mean(np.sum(kk[:-1, 0] * kk[1:, 0], axis=-1)) / w.d
    assert 0.15 < same < 0.25 and abs(cross) < 0.03          # 0.25 / 1.25 = 0.2 expected
    assert sorted(set(a.block_table[0].tolist())) == list(range(w.n_blk))
    assert a.planted.shape == (1, 1, 4) and np.all(np.diff(a.planted[0, 0]) > 0)
    assert np.all((a.planted >= w.n_sink) & (a.planted < w.n_blk - w.n_recent))


def test_layers_and_sessions_differ_and_append_pages_are_fresh():
    w = synth.WORKLOADS["ws1m_16layer"].with_(n_tok=4096, append_tok=512, n_layers=2)
    bt = synth.block_table(w)
    assert bt[0, -16:].tolist() == list(range(w.n_blk - 16, w.n_blk))
    assert sorted(bt[0].tolist()) == list(range(w.n_blk))
    k0, _ = synth.kv_pool(w, 0, bt)
    k1, _ = synth.kv_pool(w, 1, bt)
    assert not np.array_equal(k0, k1)
    w4 = synth.WORKLOADS["batch8x256k_8layer"].with_(n_tok=1024)
    bt4 = synth.block_table(w4)
    assert sorted(bt4.reshape(-1).tolist()) == list(range(w4.n_pages))
