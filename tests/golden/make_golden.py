"""Writes the stored oracle results under tests/golden/.

Inputs come from the seeded ``synth`` generator; every stored value is
computed by ``oracle.kvm_oracle`` alone.  The pages print no worked example of
any step, so these files freeze the oracle's own results on two workloads
(they guard against regressions; the pins in test_oracle_pins.py are what
tie the oracle to the pages and the mathematics).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import kvm_oracle as O  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def tiny():
    w = synth.WORKLOADS["tiny_8k_g4_d64"]
    li = synth.layer_inputs(w, 0)
    r = O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[0], li.q[0, 0], w.n_tok, w.n_sink, w.n_recent,
                      w.top_k, w.rope_theta)
    return {
        "workload": w.name,
        "source": "oracle.kvm_oracle.kvmem_layer on synth.layer_inputs(tiny_8k_g4_d64, layer 0)",
        "planted": li.planted[0, 0].tolist(),
        "kept_ids": r["ids"][0].tolist(),
        "group_scores": [float.hex(float(x)) for x in r["gs"][0]],
        "out": [[float.hex(float(x)) for x in row] for row in r["out"]],
        "k_view_row0": [int(x) for x in r["k_view"][0][0]],
        "k_view_last": [int(x) for x in r["k_view"][0][-1]],
    }


def gqa_recovery():
    w = synth.WORKLOADS["gqa40x8_256k"]
    li = synth.layer_inputs(w, 0)
    r = O.kvmem_layer(li.k_pool, li.v_pool, li.block_table[0], li.q[0, 0], w.n_tok, w.n_sink, w.n_recent,
                      w.top_k, w.rope_theta, heads=[])
    hits, kth = [], []
    for g in range(w.h_kv):
        ids = O.select_blocks(r["gs"][g], w.n_blk, w.n_sink, w.n_recent, w.top_k)
        hits.append(len(set(ids.tolist()) & set(li.planted[0, g].tolist())))
        kth.append(float.hex(O.kth_candidate_score(r["gs"][g], w.n_blk, w.n_sink, w.n_recent, w.top_k)))
    return {"workload": w.name,
            "source": "oracle.kvm_oracle scores + select_blocks on synth.layer_inputs(gqa40x8_256k, layer 0)",
            "planted_recovered_per_kv_head": hits, "n_planted": w.n_planted, "kth_group_score": kth}


if __name__ == "__main__":
    for name, fn in [("tiny_8k_g4_d64_layer0.json", tiny), ("gqa40x8_256k_recovery.json", gqa_recovery)]:
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=1)
        print("wrote", name)
