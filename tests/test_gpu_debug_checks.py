"""The debug build (libkvm_debug.so: kernels check the indices they compute and report a bad one through the
status word) on the parity cases: no check fires, and every output is bit-identical to the release build's.

The debug build runs in a child process (a process loads one build of the library)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
import synth
import sparse_attention_decode_04_b300 as K
from harness import LayerOnDevice, dev_u16

out = {"debug_checks": K.kvm_debug_checks()}
import hashlib
def digest(t):
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    a = np.ascontiguousarray(t.cpu().numpy())
    return [a.dtype.str, list(a.shape), hashlib.sha256(a.view(np.uint8).tobytes()).hexdigest()]

# decode path: tiny and a 3-session call (all kept, empty, normal), fused and unfused
for name in ("tiny_8k_g4_d64", "gqa40x8_256k"):
    w = synth.WORKLOADS[name]
    if name != "tiny_8k_g4_d64":
        w = w.with_(n_tok=40000)
    li = synth.layer_inputs(w, 0)
    ctx = K.Context.for_workload(w)
    dev = LayerOnDevice(w, li, ctx)
    dev.index_build(); dev.score_select(); dev.fused()
    torch.cuda.synchronize()
    st = K.kvm_device_status(ctx)
    out[name] = {"status": st, "index": digest(dev.index), "kept": digest(dev.kept), "gs": digest(dev.gs),
                 "k_view": digest(dev.k_view), "v_view": digest(dev.v_view), "out": digest(dev.out)}
    dev.materialize(); dev.attend()
    torch.cuda.synchronize()
    out[name]["status2"] = K.kvm_device_status(ctx)
    out[name]["out_unfused"] = digest(dev.out)
    ctx.close()
# step scoring + step attention
w = synth.Workload("dbg_step", h_q=8, h_kv=2, d=128, n_tok=300 * 32 + 7, n_sink=3, n_recent=5, top_k=40,
                   rope_theta=1e6, n_planted=4, seed=31, n_q=40, attend=False)
li = synth.layer_inputs(w, 0)
ctx = K.Context.for_workload(w)
dev = LayerOnDevice(w, li, ctx)
dev.index_build(); dev.score_select(); dev.materialize()
qs = dev_u16(li.q)
o = torch.empty((1, w.n_q, w.h_q, w.d), dtype=torch.float32, device="cuda")
K.kvm_step_attn(ctx, qs, w.n_q, dev.k_view, dev.v_view, dev.view_len, 1, o)
torch.cuda.synchronize()
out["step"] = {"status": K.kvm_device_status(ctx), "kept": digest(dev.kept), "gs": digest(dev.gs), "out": digest(o)}
ctx.close()
print("RESULT " + json.dumps(out))
'''


def run(variant):
    env = dict(os.environ)
    if variant == "debug":
        env["KVM_LIBRARY"] = "debug"
    else:
        env.pop("KVM_LIBRARY", None)
    code = "ROOT = " + repr(ROOT) + "\n" + CASES
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


def test_debug_build_checks_pass_and_results_are_identical():
    from sparse_attention_decode_04_b300 import build as B
    B.build(debug=True)
    rel, dbg = run("release"), run("debug")
    assert rel["debug_checks"] == 0 and dbg["debug_checks"] == 1
    for case in ("tiny_8k_g4_d64", "gqa40x8_256k", "step"):
        assert dbg[case]["status"] == 0, f"{case}: debug status 0x{dbg[case]['status']:x}"
        assert dbg[case] == rel[case], f"{case}: the debug build's results differ"
