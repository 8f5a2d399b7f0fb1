"""Seeded synthetic workloads for the KVMem decode hot path.

This package only makes inputs: the five workload shapes, paged bf16 K/V
pools, block tables, planted block sets and queries.  It holds none of the
method's arithmetic, so both the CUDA library and the CPU oracle are fed
from it.  The numbers come from ``kvm_synth.c`` (Philox4x32-10 counters and
Box-Muller normals, fp64), compiled on first use with the host gcc.

Recipe (topic-mixture keys, planted queries), per (session, layer, KV head):
  mu_b ~ N(0, 0.25 I) per 32-token block;  k_t = rms(mu_b + eps_t), eps ~ N(0, I)
  v_t ~ N(0, I);  q_h = rms(rms(sum_{b in P_g} mu_b) + eta_h), eta ~ N(0, 0.5 I)
All bf16 conversions round to nearest even.  P_g is drawn uniformly without
replacement from the selection candidates [n_sink, n_blk - n_recent).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

BLOCK = 32
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvm_synth.c")
_LIB_PATH = os.path.join(_HERE, "_kvm_synth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile kvm_synth.c into _kvm_synth.so (host gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, u32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_double
            lib.synth_philox4x32_10.argtypes = [P, P, P]
            lib.synth_philox4x32_10.restype = None
            lib.synth_bf16_rne.argtypes = [f64]
            lib.synth_bf16_rne.restype = ctypes.c_uint16
            lib.synth_topics.argtypes = [u32, i32, i32, i32, i32, P, i64, P]
            lib.synth_topics.restype = None
            lib.synth_kv_pages.argtypes = [u32, i32, i32, i32, i32, i64, i64, f64, P, i64, P, P, i32, i32, i32]
            lib.synth_kv_pages.restype = i32
            lib.synth_planted.argtypes = [u32, i32, i32, i32, i64, i64, i32, P]
            lib.synth_planted.restype = i32
            lib.synth_queries.argtypes = [u32, i32, i32, i32, i32, i32, i32, P, i32, f64, P]
            lib.synth_queries.restype = i32
            lib.synth_permutation.argtypes = [u32, u32, i64, P]
            lib.synth_permutation.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def philox4x32_10(ctr, key) -> tuple:
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    o = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return tuple(int(v) for v in o)


def bf16_rne_scalar(x: float) -> int:
    """The generator's own fp64 -> bf16 rounding (used for inputs only)."""
    return int(_load().synth_bf16_rne(float(x)))


def threads() -> int:
    return max(1, min(os.cpu_count() or 1, 64))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload: head geometry, history, budgets, seeds."""
    name: str
    h_q: int
    h_kv: int
    d: int
    n_tok: int                 # history tokens per session, including this step's appended tokens
    n_sessions: int = 1
    n_layers: int = 1
    n_sink: int = 4
    n_recent: int = 32
    top_k: int = 988
    rope_theta: float = 1e6
    n_planted: int = 16
    seed: int = 1
    session_seeds: tuple | None = None
    n_q: int = 1               # query tokens scored together (step-level scoring when > 1)
    append_tok: int = 0        # tokens appended and indexed inside each step
    attend: bool = True        # the step ends with decode attention over the view
    eps_scale: float = 1.0     # per-token key noise scale
    q_noise_var: float = 0.5   # per-head query noise variance

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def n_blk(self) -> int:
        return -(-self.n_tok // BLOCK)

    @property
    def budget(self) -> int:
        return self.n_sink + self.n_recent + self.top_k

    @property
    def n_keep(self) -> int:
        return min(self.n_blk, self.budget)

    @property
    def view_tokens(self) -> int:
        """Tokens in the view when the newest block is kept (always so when n_recent >= 1)."""
        if self.n_recent < 1 and self.n_tok % BLOCK and self.n_keep < self.n_blk:
            raise ValueError("view length depends on the selection")
        if self.n_tok % BLOCK == 0:
            return BLOCK * self.n_keep
        return BLOCK * (self.n_keep - 1) + self.n_tok % BLOCK

    @property
    def n_pages(self) -> int:
        """Physical pages per (layer, KV head): every session's blocks."""
        return self.n_sessions * self.n_blk

    def session_seed(self, s: int) -> int:
        return self.session_seeds[s] if self.session_seeds else self.seed

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, by what they are.  Budgets include the forced sink and
# recent blocks (so top_k = view blocks - n_sink - n_recent); the tiny case
# states "top-16 plus 1 sink and 2 recent".
WORKLOADS = {
    "tiny_8k_g4_d64": Workload("tiny_8k_g4_d64", h_q=4, h_kv=1, d=64, n_tok=8192, n_sink=1, n_recent=2,
                               top_k=16, rope_theta=1e4, n_planted=4, seed=0),
    "gqa40x8_256k": Workload("gqa40x8_256k", h_q=40, h_kv=8, d=128, n_tok=262144, n_sink=4, n_recent=32,
                             top_k=988, rope_theta=1e6, n_planted=16, seed=1),
    "ws1m_16layer": Workload("ws1m_16layer", h_q=40, h_kv=8, d=128, n_tok=1048576, n_layers=16, n_sink=4,
                             n_recent=32, top_k=2012, rope_theta=1e6, n_planted=16, seed=2, append_tok=512),
    "batch8x256k_8layer": Workload("batch8x256k_8layer", h_q=40, h_kv=8, d=128, n_tok=262144, n_sessions=8,
                                   n_layers=8, n_sink=4, n_recent=32, top_k=476, rope_theta=1e6, n_planted=16,
                                   seed=3, session_seeds=tuple(100 + s for s in range(8))),
    "step256q_1m": Workload("step256q_1m", h_q=40, h_kv=8, d=128, n_tok=1048576, n_sink=4, n_recent=32,
                            top_k=2012, rope_theta=1e6, n_planted=16, seed=4, n_q=256, attend=False),
}


def block_table(w: Workload) -> np.ndarray:
    """int32 [n_sessions][n_blk]: logical block -> physical page, shared by all layers and heads.

    Session s owns pages [s*n_blk, (s+1)*n_blk).  Its history blocks sit on a
    seeded random permutation of those pages; the blocks appended inside the
    step (append_tok) sit on consecutive fresh pages at the end of the range.
    """
    lib = _load()
    n_app = -(-w.append_tok // BLOCK) if w.append_tok else 0
    n_hist = w.n_blk - n_app
    bt = np.empty((w.n_sessions, w.n_blk), dtype=np.int32)
    for s in range(w.n_sessions):
        perm = np.empty(n_hist, dtype=np.int32)
        if lib.synth_permutation(w.session_seed(s), s, n_hist, _ptr(perm)) != 0:
            raise ValueError("bad permutation size")
        bt[s, :n_hist] = s * w.n_blk + perm
        bt[s, n_hist:] = s * w.n_blk + np.arange(n_hist, w.n_blk, dtype=np.int32)
    return bt


def planted(w: Workload, layer: int) -> np.ndarray:
    """int64 [n_sessions][h_kv][n_planted]: planted blocks, ascending per head."""
    lib = _load()
    out = np.empty((w.n_sessions, w.h_kv, w.n_planted), dtype=np.int64)
    lo, hi = w.n_sink, w.n_blk - w.n_recent
    for s in range(w.n_sessions):
        for g in range(w.h_kv):
            row = np.empty(w.n_planted, dtype=np.int64)
            if lib.synth_planted(w.session_seed(s), s, layer, g, lo, hi, w.n_planted, _ptr(row)) != 0:
                raise ValueError("not enough candidate blocks to plant")
            out[s, g] = row
    return out


def kv_pool(w: Workload, layer: int, bt: np.ndarray | None = None, sessions=None,
            out_k: np.ndarray | None = None, out_v: np.ndarray | None = None, t_range=None, heads=None):
    """bf16 bits (uint16) K and V pools [n_pages][h_kv][32][d] for one layer.

    t_range=(t0, t1) fills only those tokens of each session and heads=(lo, hi)
    only those KV heads (the rest of the arrays are left as given).
    """
    lib = _load()
    if bt is None:
        bt = block_table(w)
    shape = (w.n_pages, w.h_kv, BLOCK, w.d)
    k = out_k if out_k is not None else np.zeros(shape, dtype=np.uint16)
    v = out_v if out_v is not None else np.zeros(shape, dtype=np.uint16)
    assert k.shape == shape and v.shape == shape
    t0, t1 = t_range if t_range is not None else (0, w.n_tok)
    for s in (range(w.n_sessions) if sessions is None else sessions):
        row = np.ascontiguousarray(bt[s])
        h_lo, h_hi = heads if heads is not None else (0, w.h_kv)
        rc = lib.synth_kv_pages(w.session_seed(s), s, layer, w.h_kv, w.d, t0, t1, w.eps_scale,
                                _ptr(row), w.n_pages, _ptr(k), _ptr(v), threads(), h_lo, h_hi)
        if rc != 0:
            raise ValueError(f"synth_kv_pages failed ({rc})")
    return k, v


def queries(w: Workload, layer: int, plant: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits (uint16) [n_sessions][n_q][h_q][d]: post-q-norm, pre-RoPE queries."""
    lib = _load()
    if plant is None:
        plant = planted(w, layer)
    out = np.empty((w.n_sessions, w.n_q, w.h_q, w.d), dtype=np.uint16)
    for s in range(w.n_sessions):
        p = np.ascontiguousarray(plant[s])
        o = np.empty((w.n_q, w.h_q, w.d), dtype=np.uint16)
        if lib.synth_queries(w.session_seed(s), s, layer, w.h_q, w.h_kv, w.d, w.n_q, _ptr(p), w.n_planted,
                             w.q_noise_var, _ptr(o)) != 0:
            raise ValueError("synth_queries failed")
        out[s] = o
    return out


def topics(w: Workload, session: int, layer: int, head: int, blocks) -> np.ndarray:
    """fp64 [n][d]: the topic vectors mu_b the keys of these blocks were drawn around."""
    lib = _load()
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64))
    out = np.empty((b.size, w.d), dtype=np.float64)
    lib.synth_topics(w.session_seed(session), session, layer, head, w.d, _ptr(b), b.size, _ptr(out))
    return out


@dataclasses.dataclass
class LayerInputs:
    k_pool: np.ndarray       # uint16 [n_pages][h_kv][32][d]
    v_pool: np.ndarray       # uint16 [n_pages][h_kv][32][d]
    block_table: np.ndarray  # int32 [n_sessions][n_blk]
    q: np.ndarray            # uint16 [n_sessions][n_q][h_q][d]
    planted: np.ndarray      # int64 [n_sessions][h_kv][n_planted]


def layer_inputs(w: Workload, layer: int = 0, bt: np.ndarray | None = None) -> LayerInputs:
    if bt is None:
        bt = block_table(w)
    k, v = kv_pool(w, layer, bt)
    pl = planted(w, layer)
    return LayerInputs(k, v, bt, queries(w, layer, pl), pl)
