"""The oracle still reproduces its stored results (tests/golden/, written by make_golden.py)."""
import json
import os

import numpy as np

import synth
from oracle import kvm_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_tiny_layer_matches_stored():
    g = _load("tiny_8k_g4_d64_layer0.json")
    w = synth.WORKLOADS[g["workload"]]
    li = synth.layer_inputs(w, 0)
    assert li.planted[0, 0].tolist() == g["planted"]
    r = O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[0], li.q[0, 0], w.n_tok, w.n_sink, w.n_recent,
                      w.top_k, w.rope_theta)
    assert r["ids"][0].tolist() == g["kept_ids"]
    gs = np.array([float.fromhex(x) for x in g["group_scores"]])
    assert np.allclose(r["gs"][0], gs, rtol=1e-12, atol=0)
    out = np.array([[float.fromhex(x) for x in row] for row in g["out"]])
    assert np.allclose(r["out"], out, rtol=1e-12, atol=1e-15)
    assert r["k_view"][0][0].tolist() == g["k_view_row0"]
    assert r["k_view"][0][-1].tolist() == g["k_view_last"]
    # every planted block is in the view
    assert set(g["planted"]) <= set(g["kept_ids"])


def test_gqa_256k_recovery_matches_stored():
    g = _load("gqa40x8_256k_recovery.json")
    w = synth.WORKLOADS[g["workload"]]
    li = synth.layer_inputs(w, 0)
    r = O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[0], li.q[0, 0], w.n_tok, w.n_sink, w.n_recent,
                      w.top_k, w.rope_theta, heads=[])
    hits = []
    for h in range(w.h_kv):
        ids = O.select_blocks(r["gs"][h], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        hits.append(len(set(ids.tolist()) & set(li.planted[0, h].tolist())))
    assert hits == g["planted_recovered_per_kv_head"]
    assert min(hits) >= 12          # at least 3/4 of the planted blocks per head
