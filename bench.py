"""Benchmark of the KVMem decode hot path on B300: one JSON line on stdout.

Default workload (ws1m_16layer): 40 query heads / 8 KV heads, d = 128, a
1,048,576-token history per layer with 16 layers resident in HBM (64 GiB of
bf16 K/V pages + 2 GiB fp32 Mean-K index), a 65,536-token view per layer
(4 sink + 32 recent + 2012 top-k blocks), one decode query per layer.  One
step = the step's 512 new tokens appended to every layer's index (kvm_index_append_layers: one
launch for all layers, as no layer's append depends on an earlier layer), then for each of the 16
layers, in order:
    kvm_score_select -> kvm_materialize_attn (gather + re-RoPE view, decode attention).
Metric: step latency per layer (us) and the HBM GB/s of the bytes each layer
must touch (index read + appended keys + kept K/V read + view write).

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl kvm|reference]
                    [--workload NAME] [--layers N] [--no-e2e] [--no-cpu-baseline]
                    [--profile-step]

--impl reference times the CPU oracle on a bounded sample of the same workload
(one KV head of one layer per step) on the host's cores.
Under torchrun (N > 1) every rank runs its own independent replica (separate
sessions: the path shards with no exchange); rank 0 prints the line with the
maximum time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "select+materialize+attend step µs and HBM GB/s at 1M-token history, per layer"
STEP_METRIC = ("step-level select+materialize+attend µs per layer: 256 query tokens scored together over a "
               "1M-token history, then their causal attention over the 65,536-token view")
BLOCK = 32


def must_touch_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes one layer of a step must move (all sessions)."""
    per_sess = 0
    idx_read = w.h_kv * w.n_blk * w.d * 4
    app_blocks = -(-w.append_tok // BLOCK) if w.append_tok else 0
    app = w.append_tok * w.h_kv * w.d * 2 + app_blocks * w.h_kv * w.d * 4
    view = w.h_kv * w.view_tokens * w.d * 2          # one of K or V
    per_sess = idx_read + app + 2 * view + 2 * view  # kept K/V read + K/V view written
    return per_sess * w.n_sessions


def view_call_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes of one kvm_materialize_attn call (kept K/V read + view written)."""
    return 4 * w.h_kv * w.view_tokens * w.d * 2 * w.n_sessions


def max_over_ranks(values, world: int, device):
    """Each timing's maximum over all ranks (every rank calls this; identity on one rank)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_gbps(bytes_per_rank_layer: int, us_layer_slowest: float, world: int) -> float:
    """Whole-job GB/s: every rank moved its own bytes in the slowest rank's time (weak scaling)."""
    return bytes_per_rank_layer * world / (us_layer_slowest * 1e-6) / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle timing
_UNIT = {}  # the sampled layer's inputs, shared with the forked workers (copy on write)


def _oracle_unit(unit):
    """One (session, KV head) unit of one layer's step, by the oracle; returns the kept block count."""
    from oracle import kvm_oracle as O
    s, g = unit
    w, k, v, bt, q = _UNIT["w"], _UNIT["k"], _UNIT["v"], _UNIT["bt"], _UNIT["q"]
    G = w.group
    keys = O.paged_tokens(k, bt[s], g, w.n_tok)
    vals = O.paged_tokens(v, bt[s], g, w.n_tok)
    if w.n_q > 1:  # a step of query tokens: step scores, select, materialise, step attention
        qs = q[s][:, G * g:G * (g + 1)]
        gs = O.step_group_scores(qs, _UNIT["hist_index"][unit][None])[0]
        ids = O.select_blocks(gs, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        kv, vv = O.materialize(keys, vals, ids, w.n_tok, w.rope_theta)
        O.step_view_attention(qs, kv, vv, w.rope_theta)
    else:  # the decode step: append, score, select, materialise, attend
        idx = _UNIT["hist_index"][unit]
        if w.append_tok:
            idx = O.index_append(idx, keys, w.n_tok - w.append_tok, w.append_tok)
        qg = q[s, 0, G * g:G * (g + 1)]
        gs = O.gqa_softmax_sum(O.block_scores(qg, idx[None]), 1)[0]
        ids = O.select_blocks(gs, w.n_blk, w.n_sink, w.n_recent, w.top_k)
        kv, vv = O.materialize(keys, vals, ids, w.n_tok, w.rope_theta)
        O.decode_attention(qg, kv, vv, w.rope_theta)
    return len(ids)


def _oracle_worker(conn, my_units):
    """Worker process: builds the index state of its units (untimed), then runs them on every request."""
    from oracle import kvm_oracle as O
    w, k, bt = _UNIT["w"], _UNIT["k"], _UNIT["bt"]
    n_hist = w.n_tok - w.append_tok
    n_idx = n_hist if w.append_tok else w.n_tok
    for s, g in my_units:  # the index before the step, built outside the timed region as on the GPU
        parts = []  # block by block in pieces (the blocks are independent), so the temporaries stay small
        for b0 in range(0, -(-n_idx // 32), 2048):
            t0 = b0 * 32
            t1 = min(n_idx, t0 + 2048 * 32)
            parts.append(O.mean_k_index(O.paged_tokens(k, bt[s][b0:], g, t1 - t0)))
        _UNIT["hist_index"][(s, g)] = np.concatenate(parts) if parts else np.zeros((0, w.d))
    conn.send("ready")
    n_keep = 0
    while conn.recv() == "go":
        for u in my_units:
            n_keep = _oracle_unit(u)
        conn.send(n_keep)


def _oracle_child(name: str, reps: int, warmup: int, q_tokens: int):
    """Child-process body (no GPU): times the oracle on every (session, KV head) unit of layer 0, the units
    spread over one forked worker process per host core (each worker always runs the same units), and prints
    JSON."""
    import multiprocessing as mp
    w = synth.WORKLOADS[name]
    if q_tokens and w.n_q > q_tokens:
        w = w.with_(n_q=q_tokens)
    bt = synth.block_table(w)
    k, v = synth.kv_pool(w, 0, bt)
    q = synth.queries(w, 0)
    units = [(s, g) for s in range(w.n_sessions) for g in range(w.h_kv)]
    _UNIT.update(w=w, k=k, v=v, bt=bt, q=q, hist_index={})
    n_workers = max(1, min(os.cpu_count() or 1, len(units)))
    # forked once the inputs exist (this process never touches a GPU), so the workers share them
    ctx = mp.get_context("fork")
    pipes, procs = [], []
    for i in range(n_workers):
        a, b = ctx.Pipe()
        p = ctx.Process(target=_oracle_worker, args=(b, units[i::n_workers]), daemon=True)
        p.start()
        pipes.append(a)
        procs.append(p)
    for a in pipes:
        assert a.recv() == "ready"
    walls, n_keep = [], 0
    for i in range(warmup + reps):
        t0 = time.perf_counter()
        for a in pipes:
            a.send("go")
        n_keep = [a.recv() for a in pipes][0]
        if i >= warmup:
            walls.append(time.perf_counter() - t0)
    for a in pipes:
        a.send("stop")
    for p in procs:
        p.join(timeout=10)
    print(json.dumps({"seconds": statistics.median(walls), "n_keep": n_keep, "reps": len(walls),
                      "workers": n_workers, "units": len(units), "n_q": w.n_q}), flush=True)


def oracle_sample(w: synth.Workload, reps: int, warmup: int):
    """Times the oracle on one whole layer of the workload (every (session, KV head) unit, in parallel on the
    host's cores), in a child process with every BLAS / OpenMP pool pinned to one thread per worker.  For a step
    of many query tokens only the first 16 tokens are sampled (the rest of the step scales the score and the
    attention work linearly).

    Returns (seconds per layer, worker processes used, description).
    """
    q_tokens = 16 if w.n_q > 16 else 0
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", w.name, str(reps), str(warmup),
                        str(q_tokens)], capture_output=True, text=True, env=env, check=True)
    res = json.loads(r.stdout.strip().splitlines()[-1])
    units = res["units"]
    if w.n_q > 1:
        desc = (f"oracle (numpy fp64) on layer 0 of {w.name}: the first {res['n_q']} of the step's {w.n_q} query "
                f"tokens (step scores over {w.n_blk} blocks, select, materialise {res['n_keep']} blocks, causal "
                f"attention over the view) for all {units} (session, KV head) units, {res['workers']} worker "
                f"processes of one thread each, wall time per layer (median of {res['reps']})")
    else:
        desc = (f"oracle (numpy fp64) on layer 0 of {w.name}: append {w.append_tok} tokens, score {w.n_blk} blocks "
                f"for {w.group} query heads, select, materialise {res['n_keep']} blocks, attend, for all {units} "
                f"(session, KV head) units, {res['workers']} worker processes of one thread each, wall time per "
                f"layer (median of {res['reps']})")
    return res["seconds"], res["workers"], desc


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    layer_s, workers, desc = oracle_sample(w, args.steps, args.warmup)
    scale = w.n_q / min(w.n_q, 16) if w.n_q > 1 else 1.0  # a step's sample covers its first 16 query tokens
    if scale != 1.0:
        desc += f"; scaled by {scale:g} to the step's {w.n_q} query tokens"
    us_layer = layer_s * scale * 1e6
    gbs = must_touch_bytes(w) / (us_layer * 1e-6) / 1e9
    line = {"impl": "reference", "metric": METRIC if w.n_q == 1 else STEP_METRIC, "value": round(us_layer, 1),
            "unit": "us/layer",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            # one timed step is one layer of the workload (all of its units), measured, not extrapolated
            "ms_per_step": round(us_layer / 1e3, 3), "layers_per_step": 1,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": "layer 0 of the workload per step, every (session, KV head) unit"},
            "hbm_gbps_equivalent": round(gbs, 3),
            "cpu_baseline": {"value": round(us_layer, 1), "unit": "us/layer", "cores": workers, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(us_layer, 1), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU bench
def run_kvm(args, w):
    import torch
    import torch.distributed as dist

    import sparse_attention_decode_04_b300 as K
    from synth import device as synth_dev

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    S, L = w.n_sessions, w.n_layers
    ctx = K.Context.for_workload(w)
    n_pages = w.n_pages
    n_hist = w.n_tok - w.append_tok
    bt = torch.from_numpy(synth.block_table(w)).to(dev)
    kp, vp, index, qs = [], [], [], []
    out_all = torch.empty((L, S, w.h_q, w.d), dtype=torch.float32, device=dev)  # every layer's output, contiguous
    outs = [out_all[layer] for layer in range(L)]
    for layer in range(L):
        k = torch.empty((n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        synth_dev.fill_kv_pool(w, layer, bt, k.view(torch.int16), v.view(torch.int16))
        kp.append(k)
        vp.append(v)
        q = synth.queries(w, layer)
        qs.append(torch.from_numpy(q[:, 0].view(np.int16)).to(dev).view(torch.bfloat16).contiguous())
        idx = torch.zeros((S, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device=dev)
        K.kvm_index_append(ctx, k, n_pages, bt, [0] * S, [n_hist] * S, idx)  # the history before this step
        index.append(idx)
    kept = [torch.empty((S, w.h_kv, ctx.budget), dtype=torch.int32, device=dev) for _ in range(L)]
    k_view = torch.empty((S, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device=dev)
    v_view = torch.empty_like(k_view)
    view_len = torch.empty((S, w.h_kv), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    # the full history index build of one layer (setup work, timed on its own): the same call again, which
    # rewrites layer 0's index with the same values
    build_ms = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        K.kvm_index_append(ctx, kp[0], n_pages, bt, [0] * S, [n_hist] * S, index[0], stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        build_ms.append(e0.elapsed_time(e1))
    assert K.kvm_device_status(ctx) == 0
    build_us = float(np.median(build_ms)) * 1e3
    build_bytes = S * n_hist * w.h_kv * w.d * 2 + S * w.h_kv * (-(-n_hist // BLOCK)) * w.d * 4
    n_tok = [w.n_tok] * S
    # [one append launch for every layer,] then per layer score + select (recent-only: one kernel) and the fused
    # view kernel
    launches_per_step = (1 if w.append_tok else 0) + L * ((1 if args.selection == "recent" else 2) + 1)

    def call_append(layer):
        if w.append_tok:
            K.kvm_index_append(ctx, kp[layer], n_pages, bt, [n_hist] * S, [w.append_tok] * S, index[layer])

    def call_select(layer):
        if args.selection == "kvmem":
            K.kvm_score_select(ctx, qs[layer], 1, index[layer], n_tok, kept[layer])
        else:  # the pages' controls at the same budget
            control = K.CONTROL_RECENT_ONLY if args.selection == "recent" else K.CONTROL_WITHDRAWN_AVERAGE
            K.kvm_select_control(ctx, control, qs[layer], index[layer], n_tok, kept[layer])

    def call_view(layer):
        K.kvm_materialize_attn(ctx, kp[layer], vp[layer], n_pages, bt, n_tok, kept[layer], qs[layer], k_view,
                               v_view, view_len, outs[layer])

    # The step's new tokens have their keys for every layer when the step starts, so no layer's index append
    # waits on an earlier layer's output: every layer's append runs in one launch at the start of the step
    # (kvm_index_append_layers), and from there on each kernel follows the previous one on one stream, so under
    # programmatic dependent launch each may start early and prefetch while the previous one finishes.
    def append_all():
        if w.append_tok:
            K.kvm_index_append_layers(ctx, kp, n_pages, bt, [n_hist] * S, [w.append_tok] * S, index)

    def step():
        append_all()
        for layer in range(L):
            call_select(layer)
            call_view(layer)

    # (the append stage is the one launch for every layer, divided over the layers like the others)
    stage_fns = {"index_append": lambda layer: append_all() if layer == 0 else None, "score_select": call_select,
                 "materialize_attn": call_view}
    if not w.append_tok:
        del stage_fns["index_append"]  # nothing is appended inside this workload's step

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0

    if args.profile_step:
        # one eager step between cudaProfilerStart/Stop, for `ncu --profile-from-start off`
        torch.cuda.profiler.start()
        step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        if rank == 0:
            print(json.dumps({"profile_step": w.name, "launches": launches_per_step}), flush=True)
        return

    # CUDA graphs: one whole step (all layers), and each stage alone over all layers (per-call durations)
    side = torch.cuda.Stream()
    side.wait_stream(stream)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()  # warm the side stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize()
        return g

    graph = capture(step) if not args.no_graph else None
    stage_graphs = {}
    if not args.no_graph:
        for name, fn in stage_fns.items():
            stage_graphs[name] = capture(lambda fn=fn: [fn(layer) for layer in range(L)])
    for _ in range(max(1, args.warmup)):
        if graph is not None:
            graph.replay()
        else:
            step()
    torch.cuda.synchronize()

    gpu_index = local
    if os.environ.get("CUDA_VISIBLE_DEVICES"):
        try:
            gpu_index = int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
        except ValueError:
            gpu_index = local
    sampler = ClockSampler(gpu_index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    with sampler:
        time.sleep(0.3)
        step_ms = timed(graph.replay if graph is not None else step, args.steps)
        stage_ms = {name: timed(g.replay, args.steps) for name, g in stage_graphs.items()}
    st = K.kvm_device_status(ctx)
    if st != 0:
        raise RuntimeError(f"device status 0x{st:x} after the timed region")
    stage_us = {name: round(ms * 1e3 / L, 2) for name, ms in stage_ms.items()}
    eager_ms = timed(step, max(1, min(args.steps, 3)))

    step_ms, eager_ms = max_over_ranks([step_ms, eager_ms], world, dev)

    us_layer = step_ms * 1e3 / L
    bytes_layer = must_touch_bytes(w)
    gbs = job_gbps(bytes_layer, us_layer, world)
    peak, peak_kind = load_peaks()
    vb = view_call_bytes(w)
    view_us = stage_us.get("materialize_attn") or us_layer
    achieved = vb / (view_us * 1e-6) / 1e9

    # end-to-end through the public API with host buffers: H2D of the step's queries and new K/V pages,
    # D2H of every layer's attention output
    e2e = None
    if not args.no_e2e:
        app_blocks = -(-w.append_tok // BLOCK) if w.append_tok else 0
        first_new_page = [int(x) for x in synth.block_table(w)[:, w.n_blk - app_blocks]] if app_blocks else []
        q_host = torch.empty((L, S, w.h_q, w.d), dtype=torch.bfloat16).pin_memory()
        for layer in range(L):
            q_host[layer].copy_(qs[layer].cpu())
        new_k = [kp[layer][first_new_page[0]:first_new_page[0] + app_blocks].cpu().pin_memory() for layer in range(L)] \
            if app_blocks and S == 1 else None
        new_v = [vp[layer][first_new_page[0]:first_new_page[0] + app_blocks].cpu().pin_memory() for layer in range(L)] \
            if app_blocks and S == 1 else None
        out_host = torch.empty((L, S, w.h_q, w.d), dtype=torch.float32).pin_memory()
        q_dev = torch.empty((L, S, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
        h2d = q_host.numel() * 2 + (sum(t.numel() * 2 for t in new_k) * 2 if new_k else 0)
        d2h = out_host.numel() * 4

        def copy_new_pages(layer):
            if new_k:
                p0 = first_new_page[0]
                kp[layer][p0:p0 + app_blocks].copy_(new_k[layer], non_blocking=True)
                vp[layer][p0:p0 + app_blocks].copy_(new_v[layer], non_blocking=True)

        # The new pages' copies run on a stream of their own, back to back on the copy engine, ahead of the
        # layers that need them.
        copy_stream = torch.cuda.Stream()
        copy_done = [torch.cuda.Event() for _ in range(L)]

        def e2e_step():
            main = torch.cuda.current_stream()
            q_dev.copy_(q_host, non_blocking=True)
            copy_stream.wait_stream(main)
            with torch.cuda.stream(copy_stream):
                for layer in range(L):
                    copy_new_pages(layer)
                    copy_done[layer].record(copy_stream)
            # Each layer's append runs on the main stream just before its scoring: its pages landed long before
            # (the copies run ahead of the layers), and an append left on a side stream would wait for SM room
            # behind the previous layer's persistent view kernel.
            for layer in range(L):
                main.wait_event(copy_done[layer])
                call_append(layer)
                if args.selection == "kvmem":
                    K.kvm_score_select(ctx, q_dev[layer], 1, index[layer], n_tok, kept[layer])
                else:
                    call_select(layer)
                K.kvm_materialize_attn(ctx, kp[layer], vp[layer], n_pages, bt, n_tok, kept[layer], q_dev[layer],
                                       k_view, v_view, view_len, outs[layer])
            out_host.copy_(out_all, non_blocking=True)  # one read-back of every layer's output
            torch.cuda.current_stream().wait_stream(copy_stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        # A serving loop replays the whole step as one CUDA graph: the host-to-device copies of the queries and
        # new pages, every C-ABI call, and the device-to-host copy of the outputs are nodes of the graph.
        e2e_graph = capture(e2e_step) if graph is not None else None
        run_e2e = e2e_graph.replay if e2e_graph is not None else e2e_step
        for _ in range(2):
            run_e2e()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        a0.record(stream)
        for _ in range(args.steps):
            run_e2e()
        a1.record(stream)
        torch.cuda.synchronize()
        wall = (time.perf_counter() - wall0) / args.steps
        e2e_ms = max(a0.elapsed_time(a1) / args.steps, wall * 1e3)
        e2e = {"value": round(e2e_ms * 1e3 / L, 2), "unit": "us/layer", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
               "cuda_graph": e2e_graph is not None}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        layer_s, workers, desc = oracle_sample(w, 1, 0)
        cpu = {"value": round(layer_s * 1e6, 1), "unit": "us/layer", "cores": workers, "kind": "oracle",
               "sample": desc}

    traffic = recorded_traffic(w.name, "view_kernel", VIEW_KERNEL_SOURCES)

    per_config = None
    if (rank == 0 and world == 1 and not args.no_per_config and w.name == "ws1m_16layer" and args.layers is None
            and args.selection == "kvmem"):
        # the other workloads run in child processes; this one's pools are released first
        kp.clear()
        vp.clear()
        index.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        per_config = per_config_entries(args)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(us_layer, 2), "unit": "us/layer", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d, "history_tokens": w.n_tok,
                       "layers": L, "sessions_per_gpu": S, "view_tokens": w.view_tokens, "append_tokens": w.append_tok,
                       "kv_dtype": "bf16", "cuda_graph": graph is not None, "selection": args.selection,
                       "l2": (f"each layer's step touches {bytes_layer / 2**20:.0f} MiB (the index, kept K/V pages "
                              f"and the views), more than the 126 MB L2: no flush" if bytes_layer > 126e6 else
                              f"each layer's step touches {bytes_layer / 2**20:.2f} MiB, which stays in L2: a "
                              f"launch-bound case, reported in microseconds only"),
                       "parallelism": f"replicas x{world}"},
            "hbm_gbps": round(gbs, 1), "must_touch_bytes_per_layer": bytes_layer,
            "hbm_frac_of_measured": round(bytes_layer / (us_layer * 1e-6) / 1e9 / peak, 4),
            "stages_us_per_layer": stage_us, "ms_per_step_eager_untimed": round(eager_ms, 4),
            "roofline": {"bound": "hbm", "kernel": "kvm_materialize_attn (view_kernel: gather + re-RoPE + view write + attention + merge)",
                         "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": vb},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps * (2 if stage_graphs else 1),
            "clocks": sampler.summary(),
            "per_config": per_config,
            "index_build": {"us_per_layer": round(build_us, 1), "tokens": S * n_hist, "bytes": build_bytes,
                            "gbps": round(build_bytes / (build_us * 1e-6) / 1e9, 1),
                            "frac_of_measured": round(build_bytes / (build_us * 1e-6) / 1e9 / peak, 4),
                            "note": "kvm_index_append over the whole history of one layer (keys read once, "
                                    "index written once), timed apart from the step"},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


PER_CONFIG = ("tiny_8k_g4_d64", "gqa40x8_256k", "batch8x256k_8layer", "step256q_1m")


def per_config_entries(args) -> dict:
    """The other workloads, each measured by this script in a child process of its own (so each one's device
    memory is freed before the next), summarised against the 60%-of-roofline bound on its must-touch bytes."""
    peak, peak_kind = load_peaks()
    out = {}
    for name in PER_CONFIG:
        w = synth.WORKLOADS[name]
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", name, "--steps", str(args.steps),
               "--warmup", str(args.warmup), "--no-e2e", "--no-cpu-baseline", "--no-per-config"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        if r.returncode != 0 or not lines:
            out[name] = {"error": (r.stderr.strip().splitlines() or ["no output"])[-1][:300]}
            continue
        d = json.loads(lines[-1])
        e = {"us_per_layer": d["value"], "stages_us": d.get("stages_us_per_layer", d.get("stages_us")),
             "roofline": d.get("roofline"), "clocks": d.get("clocks")}
        if w.n_q == 1:
            mt = must_touch_bytes(w)
            gbs = mt / (d["value"] * 1e-6) / 1e9
            e.update({"must_touch_bytes_per_layer": mt, "hbm_gbps": round(gbs, 1),
                      "frac_of_measured_hbm": round(gbs / peak, 4),
                      "bound_us_60pct_of_8TBs": round(mt / (0.6 * 8e12) * 1e6, 1),
                      "bound_us_60pct_of_measured": round(mt / (0.6 * peak * 1e9) * 1e6, 1)})
            e["meets_bound_60pct_of_8TBs"] = d["value"] <= e["bound_us_60pct_of_8TBs"]
            if name.startswith("tiny"):
                e["note"] = "launch-bound: 0.38 MB per layer; reported as microseconds only"
        else:
            e["step_scores"] = d.get("step_scores")
            e["note"] = "tensor-bound; roofline of the step attention against the measured bf16 peak"
        out[name] = e
    return out


def step_attn_flops(w: synth.Workload) -> int:
    """Algorithmic FLOPs of one kvm_step_attn call: per (query row, attended slot) a d-long dot product for the
    score and a d-long accumulation of the value, 2 FLOPs per multiply-add; token t attends L - n_q + t + 1 slots."""
    L, T = w.view_tokens, w.n_q
    attended = sum(L - T + t + 1 for t in range(T))
    return 4 * w.d * w.h_q * attended * w.n_sessions


def step_score_flops(w: synth.Workload) -> int:
    """Algorithmic FLOPs of the step scores: one (n_q * h_q) x n_blk x d contraction (2 FLOPs per multiply-add)."""
    return 2 * w.n_q * w.h_q * w.n_blk * w.d * w.n_sessions


def run_kvm_step(args, w):
    """One layer of a step of n_q query tokens: step scores + select, materialise, step attention."""
    import torch

    import sparse_attention_decode_04_b300 as K
    from synth import device as synth_dev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    S = w.n_sessions
    ctx = K.Context.for_workload(w)
    bt = torch.from_numpy(synth.block_table(w)).to(dev)
    kp = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    synth_dev.fill_kv_pool(w, 0, bt, kp.view(torch.int16), vp.view(torch.int16))
    q_np = synth.queries(w, 0)                                          # [S][n_q][h_q][d]
    q = torch.from_numpy(q_np.view(np.int16)).to(dev).view(torch.bfloat16).contiguous()
    index = torch.zeros((S, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device=dev)
    n_tok = [w.n_tok] * S
    K.kvm_index_append(ctx, kp, w.n_pages, bt, [0] * S, n_tok, index)
    kept = torch.empty((S, w.h_kv, ctx.budget), dtype=torch.int32, device=dev)
    k_view = torch.empty((S, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device=dev)
    v_view = torch.empty_like(k_view)
    view_len = torch.empty((S, w.h_kv), dtype=torch.int32, device=dev)
    out = torch.empty((S, w.n_q, w.h_q, w.d), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0

    def call_select(q_in=q):
        K.kvm_score_select(ctx, q_in, w.n_q, index, n_tok, kept)

    def call_materialize():
        K.kvm_materialize(ctx, kp, vp, w.n_pages, bt, n_tok, kept, k_view, v_view, view_len)

    def call_attn(q_in=q):
        K.kvm_step_attn(ctx, q_in, w.n_q, k_view, v_view, view_len, S, out)

    def step():
        call_select()
        call_materialize()
        call_attn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    if args.profile_step:
        torch.cuda.profiler.start()
        step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        if rank == 0:
            print(json.dumps({"profile_step": w.name}), flush=True)
        return

    side = torch.cuda.Stream()
    side.wait_stream(stream)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize()
        return g

    graph = capture(step)
    stage_graphs = {"score_select": capture(call_select), "materialize": capture(call_materialize),
                    "step_attn": capture(call_attn)}
    for _ in range(max(1, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    gpu_index = local
    if os.environ.get("CUDA_VISIBLE_DEVICES"):
        try:
            gpu_index = int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
        except ValueError:
            gpu_index = local
    sampler = ClockSampler(gpu_index)
    with sampler:
        time.sleep(0.3)
        step_ms = timed(graph.replay, args.steps)
        stage_ms = {name: timed(g.replay, args.steps) for name, g in stage_graphs.items()}
    st = K.kvm_device_status(ctx)
    if st != 0:
        raise RuntimeError(f"device status 0x{st:x} after the timed region")
    step_ms = max_over_ranks([step_ms], world, dev)[0]

    # end to end with host buffers: H2D of the step's queries, D2H of the attention output
    q_host = torch.from_numpy(q_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    q_dev = torch.empty_like(q)
    out_host = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()

    def e2e_step():
        q_dev.copy_(q_host, non_blocking=True)
        call_select(q_dev)
        call_materialize()
        call_attn(q_dev)
        out_host.copy_(out, non_blocking=True)

    e2e_graph = capture(e2e_step)
    for _ in range(2):
        e2e_graph.replay()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    e2e_ms = timed(e2e_graph.replay, args.steps)
    e2e_ms = max(e2e_ms, (time.perf_counter() - wall0) * 1e3 / args.steps)

    peak_tf = None
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peak_tf, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    if peak_tf is None:
        peak_tf, peak_kind = 1800.0, "fallback"
    attn_flops = step_attn_flops(w)
    attn_us = stage_ms["step_attn"] * 1e3
    achieved = attn_flops / (attn_us * 1e-6) / 1e12
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        layer_s, workers, desc = oracle_sample(w, 1, 0)
        # the sample covers the first query tokens of the step; the oracle's work is linear in them
        scale = w.n_q / min(w.n_q, 16)
        cpu = {"value": round(layer_s * scale * 1e6, 1), "unit": "us/layer", "cores": workers, "kind": "oracle",
               "sample": desc + f"; scaled by {scale:g} to the step's {w.n_q} query tokens"}
    if rank == 0:
        line = {
            "metric": STEP_METRIC, "value": round(step_ms * 1e3, 2), "unit": "us/layer", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 MMA (split operands), f32 accumulate",
            "data": "synthetic",
            "config": {"workload": w.name, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d, "history_tokens": w.n_tok,
                       "query_tokens": w.n_q, "sessions_per_gpu": S, "view_tokens": w.view_tokens,
                       "kv_dtype": "bf16", "cuda_graph": True,
                       "l2": "inputs larger than L2 (K/V pool 4 GiB, index 128 MiB, view 256 MiB), no flush",
                       "parallelism": f"replicas x{world}"},
            "stages_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
            "roofline": {"bound": "tensor", "kernel": "kvm_step_attn (query packing + tcgen05 attention reading "
                                                      "K and V from the view, timed together)",
                         "achieved": round(achieved, 1), "peak": peak_tf, "peak_kind": peak_kind, "unit": "TFLOP/s",
                         "frac": round(achieved / peak_tf, 4),
                         "traffic": recorded_traffic(w.name, "step_attn_kernel", STEP_ATTN_SOURCES),
                         "algorithmic_flops_per_launch": attn_flops,
                         "issued_mma_flops_per_launch": 2 * attn_flops},
            "step_scores": {"algorithmic_flops": step_score_flops(w),
                            "tflops_per_s": round(step_score_flops(w) / (stage_ms["score_select"] * 1e-3) / 1e12, 1)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": "us/layer", "h2d_bytes_per_step": q_host.numel() * 2,
                    "d2h_bytes_per_step": out_host.numel() * 4, "cuda_graph": True},
            # per step: step scores 5 + select 1, view kernel 1, step attention 3; timed as the whole-step graph
            # and again as the three stage graphs
            "gpu_launches": 20 * args.steps,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def run_kvm_tier(args, w):
    """The decode step with the pages in another tier: FP8 E4M3 pages in HBM (``--kv fp8``: index over the
    dequantised keys, view gathered with dequantisation) or bf16 pages in pinned host memory (``--kv host``: the
    view gathered over the host link; the index stays in HBM).  Per layer: [append,] score + select, gather,
    decode attention over the view."""
    import torch

    import sparse_attention_decode_04_b300 as K
    from synth import device as synth_dev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    host = args.kv == "host"
    if host:
        w = w.with_(append_tok=0)  # new tokens' pages would be written to HBM first; the tier holds the history
    S, L = w.n_sessions, w.n_layers
    ctx = K.Context.for_workload(w)
    n_pages = w.n_pages
    n_hist = w.n_tok - w.append_tok
    bt = torch.from_numpy(synth.block_table(w)).to(dev)
    all_pages = torch.arange(n_pages, dtype=torch.int32, device=dev)
    pools, index, qs, outs = [], [], [], []
    for layer in range(L):
        k = torch.empty((n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        synth_dev.fill_kv_pool(w, layer, bt, k.view(torch.int16), v.view(torch.int16))
        idx = torch.zeros((S, w.h_kv, w.n_blk, w.d), dtype=torch.float32, device=dev)
        if host:
            K.kvm_index_append(ctx, k, n_pages, bt, [0] * S, [n_hist] * S, idx)
            kh = torch.empty((n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, pin_memory=True)
            vh = torch.empty_like(kh, pin_memory=True)
            kh.copy_(k)
            vh.copy_(v)
            pools.append((kh, vh))
        else:
            k8 = torch.empty((n_pages, w.h_kv, BLOCK, w.d), dtype=torch.uint8, device=dev)
            v8 = torch.empty_like(k8)
            ks = torch.empty((n_pages, w.h_kv), dtype=torch.float32, device=dev)
            vs = torch.empty_like(ks)
            K.kvm_quantize_pages(ctx, k, n_pages, all_pages, k8, ks)
            K.kvm_quantize_pages(ctx, v, n_pages, all_pages, v8, vs)
            K.kvm_index_append_fp8(ctx, k8, ks, n_pages, bt, [0] * S, [n_hist] * S, idx)
            pools.append((k8, ks, v8, vs))
        torch.cuda.synchronize()
        del k, v
        index.append(idx)
        q = synth.queries(w, layer)
        qs.append(torch.from_numpy(q[:, 0].view(np.int16)).to(dev).view(torch.bfloat16).contiguous())
        outs.append(torch.empty((S, w.h_q, w.d), dtype=torch.float32, device=dev))
    torch.cuda.empty_cache()  # the bf16 pools were temporaries
    kept = torch.empty((S, w.h_kv, ctx.budget), dtype=torch.int32, device=dev)
    k_view = torch.empty((S, w.h_kv, BLOCK * ctx.budget, w.d), dtype=torch.bfloat16, device=dev)
    v_view = torch.empty_like(k_view)
    view_len = torch.empty((S, w.h_kv), dtype=torch.int32, device=dev)
    n_tok = [w.n_tok] * S
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0

    def call_append(layer):
        if w.append_tok and not host:
            k8, ks = pools[layer][0], pools[layer][1]
            K.kvm_index_append_fp8(ctx, k8, ks, n_pages, bt, [n_hist] * S, [w.append_tok] * S, index[layer])

    def call_select(layer):
        K.kvm_score_select(ctx, qs[layer], 1, index[layer], n_tok, kept)

    def call_gather(layer):
        if host:
            K.kvm_materialize_host(ctx, pools[layer][0], pools[layer][1], n_pages, bt, n_tok, kept, k_view, v_view,
                                   view_len)
        else:
            k8, ks, v8, vs = pools[layer]
            K.kvm_materialize_fp8(ctx, k8, ks, v8, vs, n_pages, bt, n_tok, kept, k_view, v_view, view_len)

    def call_attend(layer):
        K.kvm_decode_attn(ctx, qs[layer], k_view, v_view, view_len, S, outs[layer])

    def call_fused(layer):  # FP8 pages: the view and the attention in one pass
        k8, ks, v8, vs = pools[layer]
        K.kvm_materialize_attn_fp8(ctx, k8, ks, v8, vs, n_pages, bt, n_tok, kept, qs[layer], k_view, v_view,
                                   view_len, outs[layer])

    # As in the bf16 leg: every layer's append on a side stream at the start of the step; layer 0's scoring
    # waits for its own, layer 1's for all of them, and later kernels follow each other with no cross-stream edge.
    appends = bool(w.append_tok) and not host
    app_stream = torch.cuda.Stream()
    app_first = torch.cuda.Event()

    def step():
        main = torch.cuda.current_stream()
        if appends:
            app_stream.wait_stream(main)
            with torch.cuda.stream(app_stream):
                for layer in range(L):
                    call_append(layer)
                    if layer == 0:
                        app_first.record(app_stream)
        for layer in range(L):
            if appends and layer == 0:
                main.wait_event(app_first)
            if appends and layer == 1:
                main.wait_stream(app_stream)
            call_select(layer)
            if host:
                call_gather(layer)
                call_attend(layer)
            else:
                call_fused(layer)
        if appends and L == 1:
            main.wait_stream(app_stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    if args.profile_step:
        torch.cuda.profiler.start()
        step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        if rank == 0:
            print(json.dumps({"profile_step": w.name, "kv": args.kv}), flush=True)
        return
    side = torch.cuda.Stream()
    side.wait_stream(stream)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize()
        return g

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    graph = capture(step)
    stages = ({"score_select": call_select, "gather": call_gather, "decode_attn": call_attend} if host else
              {"score_select": call_select, "materialize_attn_fp8": call_fused})
    if w.append_tok and not host:
        stages["index_append"] = call_append
    stage_graphs = {n: capture(lambda fn=fn: [fn(layer) for layer in range(L)]) for n, fn in stages.items()}
    graph.replay()
    torch.cuda.synchronize()
    # the host link's own copy bandwidth in this run: pinned host -> device, 1 GiB, best of 3
    link_gbs = None
    if host:
        src = torch.empty(1 << 29, dtype=torch.int16, pin_memory=True)
        dst = torch.empty(1 << 29, dtype=torch.int16, device=dev)
        link_gbs = max(src.numel() * 2 / (timed(lambda: dst.copy_(src, non_blocking=True), 1) * 1e-3) / 1e9
                       for _ in range(3))
        del src, dst
    gpu_index = local
    if os.environ.get("CUDA_VISIBLE_DEVICES"):
        try:
            gpu_index = int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
        except ValueError:
            gpu_index = local
    sampler = ClockSampler(gpu_index)
    with sampler:
        time.sleep(0.3)
        step_ms = timed(graph.replay, args.steps)
        stage_ms = {n: timed(g.replay, args.steps) for n, g in stage_graphs.items()}
    st = K.kvm_device_status(ctx)
    if st != 0:
        raise RuntimeError(f"device status 0x{st:x} after the timed region")
    step_ms = max_over_ranks([step_ms], world, dev)[0]
    us_layer = step_ms * 1e3 / L
    gather_us = stage_ms["gather" if host else "materialize_attn_fp8"] * 1e3 / L
    view_bytes = 2 * w.h_kv * w.view_tokens * w.d * 2 * S            # K and V view written (bf16)
    if host:
        src_bytes = 2 * w.h_kv * w.view_tokens * w.d * 2 * S         # kept bf16 rows read over the link
        achieved = src_bytes / (gather_us * 1e-6) / 1e9
        roof = {"bound": "host link", "kernel": "kvm_materialize_host (gather_view_kernel, bf16 source)",
                "achieved": round(achieved, 1), "peak": round(link_gbs, 1),
                "peak_kind": "measured in this run (pinned host -> device copy of 1 GiB)", "unit": "GB/s",
                "frac": round(achieved / link_gbs, 4), "traffic": None, "algorithmic_bytes_per_launch": src_bytes,
                "note": "bytes counted are the kept rows crossing the host link; the view writes go to HBM"}
    else:
        peak, peak_kind = load_peaks()
        q_bytes = 2 * w.h_kv * w.view_tokens * w.d * S + 2 * w.h_kv * w.n_keep * 4 * S   # codes + scales
        gb = q_bytes + view_bytes
        achieved = gb / (gather_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": "kvm_materialize_attn_fp8 (view_kernel, E4M3 source: gather + dequantise "
                                          "+ re-RoPE + view write + attention + merge)",
                "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(w.name + "/fp8", "view_kernel", VIEW_KERNEL_SOURCES),
                "algorithmic_bytes_per_launch": gb}
    if rank == 0:
        tier = "FP8 E4M3 pages in HBM" if not host else "bf16 pages in pinned host memory"
        line = {
            "metric": f"select+materialize+attend step µs per layer at 1M-token history, {tier}",
            "value": round(us_layer, 2), "unit": "us/layer", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "kv": args.kv, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d,
                       "history_tokens": w.n_tok, "layers": L, "sessions_per_gpu": S,
                       "view_tokens": w.view_tokens, "append_tokens": w.append_tok, "cuda_graph": True,
                       "l2": "inputs larger than L2, no flush", "parallelism": f"replicas x{world}"},
            "stages_us_per_layer": {n: round(v * 1e3 / L, 2) for n, v in stage_ms.items()},
            "roofline": roof,
            "cpu_baseline": None, "e2e": None,
            # per layer: [append 1,] score 1 + select 1, then gather 1 + attention 1 (host) or the fused view 1
            # (FP8); the step graph and the stage graphs
            "gpu_launches": ((1 if (w.append_tok and not host) else 0) + (4 if host else 3)) * L * args.steps * 2,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


VIEW_KERNEL_SOURCES = ("sparse_attention_decode_04_b300/csrc/kvm_view.cu", "sparse_attention_decode_04_b300/csrc/kvm_device.cuh",
                       "sparse_attention_decode_04_b300/csrc/kvm_internal.h", "include/kvm.h")
GATHER_KERNEL_SOURCES = ("sparse_attention_decode_04_b300/csrc/kvm_gather.cu",) + VIEW_KERNEL_SOURCES[1:]
STEP_ATTN_SOURCES = ("sparse_attention_decode_04_b300/csrc/kvm_step_attn.cu",) + VIEW_KERNEL_SOURCES[1:]


def run_mass(args, w):
    """The attention-mass diagnostic over every layer of the workload: per layer, the full attention of the
    decode query over the whole history, reduced to per-block mass (one kvm_attention_mass call)."""
    import torch

    import sparse_attention_decode_04_b300 as K
    from synth import device as synth_dev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    S, L = w.n_sessions, w.n_layers
    ctx = K.Context.for_workload(w)
    bt = torch.from_numpy(synth.block_table(w)).to(dev)
    kp, qs = [], []
    for layer in range(L):
        k = torch.empty((w.n_pages, w.h_kv, BLOCK, w.d), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        synth_dev.fill_kv_pool(w, layer, bt, k.view(torch.int16), v.view(torch.int16))
        del v
        kp.append(k)
        q = synth.queries(w, layer)
        qs.append(torch.from_numpy(q[:, 0].view(np.int16)).to(dev).view(torch.bfloat16).contiguous())
    torch.cuda.empty_cache()
    mass = torch.zeros((L, S, w.h_kv, w.n_blk), dtype=torch.float32, device=dev)
    n_tok = [w.n_tok] * S

    def step():
        for layer in range(L):
            K.kvm_attention_mass(ctx, qs[layer], kp[layer], w.n_pages, bt, n_tok, mass[layer])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert K.kvm_device_status(ctx) == 0
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=side):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.3)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    us_layer = ms * 1e3 / L
    key_bytes = w.n_tok * w.h_kv * w.d * 2 * S  # every key of the layer read once
    peak, peak_kind = load_peaks()
    achieved = key_bytes / (us_layer * 1e-6) / 1e9
    # share of each group's mass held by its 8 largest blocks (a row sums to the group size)
    top8 = np.sort(mass.cpu().numpy().astype(np.float64), axis=-1)[..., ::-1][..., :8].sum(axis=-1) / w.group
    shares = top8.reshape(-1)
    if rank == 0:
        print(json.dumps({
            "metric": "attention-mass diagnostic µs per layer (full attention of the decode query over the history)",
            "value": round(us_layer, 2), "unit": "us/layer", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "layers": L, "sessions_per_gpu": S, "history_tokens": w.n_tok,
                       "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d, "cuda_graph": True},
            "roofline": {"bound": "hbm", "kernel": "kvm_attention_mass (mass_tile_kernel + mass_finalize_kernel)",
                         "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "algorithmic_bytes_per_launch": key_bytes},
            "top8_share": {"mean": round(float(np.mean(shares)), 4), "min": round(float(np.min(shares)), 4),
                           "max": round(float(np.max(shares)), 4),
                           "note": "synthetic topic-mixture keys; the pages' 66.5% is on a real model"},
            "gpu_launches": 2 * L * args.steps, "clocks": sampler.summary()}), flush=True)


def K_source_hash(files=VIEW_KERNEL_SOURCES) -> str:
    """Hash of the code (comments and whitespace dropped) a kernel is compiled from: a recorded ncu traffic
    figure is valid only while it is unchanged."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f)) as fh:
            code = re.sub(r"/\*.*?\*/", " ", fh.read(), flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str, files) -> int | None:
    """DRAM bytes per launch of `kernel` at `workload` from a `traffic` line under profiles/, if its code hash
    still matches."""
    prof_dir = os.path.join(ROOT, "profiles")
    want = K_source_hash(files)
    for fn in sorted(os.listdir(prof_dir)) if os.path.isdir(prof_dir) else []:
        if not fn.endswith(".md"):
            continue
        with open(os.path.join(prof_dir, fn)) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) >= 5 and parts[0] == "traffic" and parts[1] == workload and parts[2] == kernel:
                    kv = dict(p.split("=", 1) for p in parts[3:] if "=" in p)
                    if kv.get("source_hash") == want:
                        return int(kv["bytes_per_launch"])
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvm", choices=["kvm", "reference"])
    ap.add_argument("--workload", default="ws1m_16layer", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--selection", default="kvmem", choices=["kvmem", "recent", "withdrawn"],
                    help="kvmem (the method) or one of the pages' controls at the same budget: recent-only, or the "
                         "withdrawn head-averaged scoring")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only this many layers of the workload (profiling captures; each layer's launches are "
                         "the full-size ones)")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8", "host"],
                    help="page tier: bf16 pages in HBM (the method), FP8 E4M3 pages in HBM, or bf16 pages in "
                         "pinned host memory")
    ap.add_argument("--mass", action="store_true",
                    help="time the attention-mass diagnostic (full attention over the history, per-block mass)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' entries (per_config) of the default run")
    ap.add_argument("--profile-step", action="store_true",
                    help="after warm-up, run one step between cudaProfilerStart/Stop and exit (for ncu)")
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-child":
        _oracle_child(sys.argv[2], int(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5]))
        return
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = synth.WORKLOADS[args.workload]
    if args.layers is not None:
        w = w.with_(n_layers=max(1, min(args.layers, w.n_layers)))
    if args.impl == "reference":
        run_reference(args, w)
    elif args.mass:
        run_mass(args, w)
    elif w.n_q > 1:
        run_kvm_step(args, w)
    elif args.kv != "bf16":
        run_kvm_tier(args, w)
    else:
        run_kvm(args, w)


if __name__ == "__main__":
    main()
