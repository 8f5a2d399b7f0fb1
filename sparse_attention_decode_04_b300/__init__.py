"""Python binding of libkvm.so, the KVMem decode hot path for B300 (sm_103a).

Argument marshalling only: every computation runs in the CUDA kernels behind
the C ABI declared in include/kvm.h.  Tensors are PyTorch CUDA tensors (torch
is used for device memory and streams); bf16 tensors may be passed as
torch.bfloat16 or as 16-bit integer bit patterns.  Host-side per-session
arrays (history lengths, append ranges) are Python sequences.

There is no fallback: if libkvm.so is missing the import of any entry point
raises, and a failing call raises KvmError with the library's message.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# KVM_LIBRARY=debug selects the debug build (device-side index checks reported through the status word)
LIB_PATH = os.path.join(PKG, "libkvm_debug.so" if os.environ.get("KVM_LIBRARY") == "debug" else "libkvm.so")
BLOCK = 32

KVM_OK = 0
STATUS_NAMES = {0: "KVM_OK", 1: "KVM_ERR_INVALID_ARG", 2: "KVM_ERR_SHAPE", 3: "KVM_ERR_BUDGET", 4: "KVM_ERR_CUDA",
                5: "KVM_ERR_TIMEOUT", 6: "KVM_ERR_DEVICE"}
DEV_BAD_PAGE, DEV_BAD_BLOCK, DEV_TIMEOUT, DEV_BAD_VIEW, DEV_DEBUG_CHECK = 0x1, 0x2, 0x4, 0x8, 0x10
CONTROL_RECENT_ONLY, CONTROL_WITHDRAWN_AVERAGE = 1, 2


class KvmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Params(ctypes.Structure):
    _fields_ = [("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("n_sink", ctypes.c_int32), ("n_recent", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("max_blocks", ctypes.c_int64), ("max_sessions", ctypes.c_int32),
                ("max_queries", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libkvm.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with: python -m sparse_attention_decode_04_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.kvm_status_string.argtypes = [ctypes.c_int]
        L.kvm_status_string.restype = ctypes.c_char_p
        L.kvm_last_error.argtypes = []
        L.kvm_last_error.restype = ctypes.c_char_p
        L.kvm_create.argtypes = [ctypes.POINTER(Params), ctypes.POINTER(P)]
        L.kvm_destroy.argtypes = [P]
        L.kvm_scratch_bytes.argtypes = [P]
        L.kvm_scratch_bytes.restype = ctypes.c_size_t
        L.kvm_index_append.argtypes = [P, P, i64, P, i32, P, P, P, P]
        L.kvm_score_select.argtypes = [P, P, i32, P, P, i32, P, P, P, P]
        L.kvm_materialize.argtypes = [P, P, P, i64, P, P, i32, P, P, P, P, P]
        L.kvm_decode_attn.argtypes = [P, P, P, P, P, i32, P, P]
        L.kvm_materialize_attn.argtypes = [P, P, P, i64, P, P, i32, P, P, P, P, P, P, P]
        L.kvm_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), i32, P]
        L.kvm_select_control.argtypes = [P, i32, P, P, P, i32, P, P, P]
        L.kvm_step_attn.argtypes = [P, P, i32, P, P, P, i32, P, P]
        L.kvm_quantize_pages.argtypes = [P, P, i64, P, i64, P, P, P]
        L.kvm_index_append_fp8.argtypes = [P, P, P, i64, P, i32, P, P, P, P]
        L.kvm_materialize_fp8.argtypes = [P, P, P, P, P, i64, P, P, i32, P, P, P, P, P]
        L.kvm_materialize_host.argtypes = [P, P, P, i64, P, P, i32, P, P, P, P, P]
        L.kvm_attention_mass.argtypes = [P, P, P, i64, P, P, i32, P, P]
        L.kvm_index_append_layers.argtypes = [P, i32, P, i64, P, i32, P, P, P, P]
        for name in ("kvm_create", "kvm_destroy", "kvm_index_append", "kvm_score_select", "kvm_materialize",
                     "kvm_decode_attn", "kvm_materialize_attn", "kvm_device_status", "kvm_select_control",
                     "kvm_step_attn", "kvm_quantize_pages", "kvm_index_append_fp8", "kvm_materialize_fp8",
                     "kvm_materialize_host", "kvm_attention_mass", "kvm_index_append_layers"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int):
    if status != KVM_OK:
        raise KvmError(status, lib().kvm_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkvm must be contiguous")
    return t.data_ptr()


def _i64(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Context:
    """A libkvm context: head geometry, budget, capacities and the device scratch."""

    def __init__(self, h_q: int, h_kv: int, d: int, n_sink: int, n_recent: int, top_k: int, rope_theta: float,
                 max_blocks: int, max_sessions: int = 1, max_queries: int = 1):
        self.params = Params(h_q, h_kv, d, n_sink, n_recent, top_k, rope_theta, max_blocks, max_sessions,
                             max_queries)
        h = ctypes.c_void_p()
        _check(lib().kvm_create(ctypes.byref(self.params), ctypes.byref(h)))
        self.handle = h
        self.h_q, self.h_kv, self.d = h_q, h_kv, d
        self.n_sink, self.n_recent, self.top_k = n_sink, n_recent, top_k
        self.budget = n_sink + n_recent + top_k
        self.max_blocks, self.max_sessions, self.max_queries = max_blocks, max_sessions, max_queries

    @classmethod
    def for_workload(cls, w, max_blocks=None, max_sessions=None):
        return cls(w.h_q, w.h_kv, w.d, w.n_sink, w.n_recent, w.top_k, w.rope_theta,
                   max_blocks or w.n_blk, max_sessions or w.n_sessions, w.n_q)

    @property
    def scratch_bytes(self) -> int:
        return int(lib().kvm_scratch_bytes(self.handle))

    def close(self):
        if getattr(self, "handle", None):
            _check(lib().kvm_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kvm_index_append(ctx: Context, k_pool, n_pages: int, block_table, tok_begin, n_tok, index, stream=None):
    n = len(n_tok)
    _check(lib().kvm_index_append(ctx.handle, _ptr(k_pool), int(n_pages), _ptr(block_table), n, _i64(tok_begin),
                                  _i64(n_tok), _ptr(index), _stream(stream)))


def kvm_index_append_layers(ctx: Context, k_pools, n_pages: int, block_table, tok_begin, n_tok, indexes,
                            stream=None):
    """kvm_index_append for several layers (lists of key pools and indexes, one per layer) in one launch."""
    if len(k_pools) != len(indexes):
        raise ValueError("one index per key pool")
    n, nl = len(n_tok), len(k_pools)
    pools = (ctypes.c_void_p * max(1, nl))(*[_ptr(t) for t in k_pools])
    idx = (ctypes.c_void_p * max(1, nl))(*[_ptr(t) for t in indexes])
    _check(lib().kvm_index_append_layers(ctx.handle, nl, pools, int(n_pages), _ptr(block_table), n, _i64(tok_begin),
                                         _i64(n_tok), idx, _stream(stream)))


def kvm_score_select(ctx: Context, q, n_q: int, index, n_tok, kept_ids, group_scores=None, head_scores=None,
                     stream=None):
    n = len(n_tok)
    _check(lib().kvm_score_select(ctx.handle, _ptr(q), int(n_q), _ptr(index), _i64(n_tok), n, _ptr(kept_ids),
                                  _ptr(group_scores), _ptr(head_scores), _stream(stream)))


def kvm_select_control(ctx: Context, control: int, q, index, n_tok, kept_ids, group_scores=None, stream=None):
    """The selection controls: CONTROL_RECENT_ONLY (q, index unused) or CONTROL_WITHDRAWN_AVERAGE."""
    n = len(n_tok)
    _check(lib().kvm_select_control(ctx.handle, int(control), _ptr(q), _ptr(index), _i64(n_tok), n, _ptr(kept_ids),
                                    _ptr(group_scores), _stream(stream)))


def kvm_materialize(ctx: Context, k_pool, v_pool, n_pages: int, block_table, n_tok, kept_ids, k_view, v_view,
                    view_len, stream=None):
    n = len(n_tok)
    _check(lib().kvm_materialize(ctx.handle, _ptr(k_pool), _ptr(v_pool), int(n_pages), _ptr(block_table),
                                 _i64(n_tok), n, _ptr(kept_ids), _ptr(k_view), _ptr(v_view), _ptr(view_len),
                                 _stream(stream)))


def kvm_decode_attn(ctx: Context, q, k_view, v_view, view_len, n_sessions: int, out, stream=None):
    _check(lib().kvm_decode_attn(ctx.handle, _ptr(q), _ptr(k_view), _ptr(v_view), _ptr(view_len), int(n_sessions),
                                 _ptr(out), _stream(stream)))


def kvm_materialize_attn(ctx: Context, k_pool, v_pool, n_pages: int, block_table, n_tok, kept_ids, q, k_view,
                         v_view, view_len, out, stream=None):
    n = len(n_tok)
    _check(lib().kvm_materialize_attn(ctx.handle, _ptr(k_pool), _ptr(v_pool), int(n_pages), _ptr(block_table),
                                      _i64(n_tok), n, _ptr(kept_ids), _ptr(q), _ptr(k_view), _ptr(v_view),
                                      _ptr(view_len), _ptr(out), _stream(stream)))


def kvm_step_attn(ctx: Context, q, n_q: int, k_view, v_view, view_len, n_sessions: int, out, stream=None):
    """Attention of a step's n_q query tokens (the history's last n_q tokens) over the view."""
    _check(lib().kvm_step_attn(ctx.handle, _ptr(q), int(n_q), _ptr(k_view), _ptr(v_view), _ptr(view_len),
                               int(n_sessions), _ptr(out), _stream(stream)))


def kvm_quantize_pages(ctx: Context, pool, n_pages: int, pages, pool8, scales, stream=None):
    """FP8 E4M3 codes and per-(page, KV head) fp32 scales of the listed pages (a device int32 tensor)."""
    _check(lib().kvm_quantize_pages(ctx.handle, _ptr(pool), int(n_pages), _ptr(pages), int(pages.numel()),
                                    _ptr(pool8), _ptr(scales), _stream(stream)))


def kvm_index_append_fp8(ctx: Context, k_pool8, k_scales, n_pages: int, block_table, tok_begin, n_tok, index,
                         stream=None):
    n = len(n_tok)
    _check(lib().kvm_index_append_fp8(ctx.handle, _ptr(k_pool8), _ptr(k_scales), int(n_pages), _ptr(block_table), n,
                                      _i64(tok_begin), _i64(n_tok), _ptr(index), _stream(stream)))


def kvm_materialize_fp8(ctx: Context, k_pool8, k_scales, v_pool8, v_scales, n_pages: int, block_table, n_tok,
                        kept_ids, k_view, v_view, view_len, stream=None):
    n = len(n_tok)
    _check(lib().kvm_materialize_fp8(ctx.handle, _ptr(k_pool8), _ptr(k_scales), _ptr(v_pool8), _ptr(v_scales),
                                     int(n_pages), _ptr(block_table), _i64(n_tok), n, _ptr(kept_ids), _ptr(k_view),
                                     _ptr(v_view), _ptr(view_len), _stream(stream)))


def kvm_materialize_attn_fp8(ctx: Context, k_pool8, k_scales, v_pool8, v_scales, n_pages: int, block_table, n_tok,
                             kept_ids, q, k_view, v_view, view_len, out, stream=None):
    """View from FP8 pages and decode attention over it in one pass (kvm_materialize_fp8 + kvm_decode_attn)."""
    L = lib()
    f = L.kvm_materialize_attn_fp8
    if f.argtypes is None:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        f.argtypes = [P, P, P, P, P, i64, P, P, i32, P, P, P, P, P, P, P]
        f.restype = ctypes.c_int
    n = len(n_tok)
    _check(f(ctx.handle, _ptr(k_pool8), _ptr(k_scales), _ptr(v_pool8), _ptr(v_scales), int(n_pages), _ptr(block_table),
             _i64(n_tok), n, _ptr(kept_ids), _ptr(q), _ptr(k_view), _ptr(v_view), _ptr(view_len), _ptr(out),
             _stream(stream)))


def kvm_materialize_host(ctx: Context, k_pool_host, v_pool_host, n_pages: int, block_table, n_tok, kept_ids,
                         k_view, v_view, view_len, stream=None):
    """The view from K/V pools in pinned, mapped host memory (e.g. torch.empty(..., pin_memory=True))."""
    n = len(n_tok)
    _check(lib().kvm_materialize_host(ctx.handle, _ptr(k_pool_host), _ptr(v_pool_host), int(n_pages),
                                      _ptr(block_table), _i64(n_tok), n, _ptr(kept_ids), _ptr(k_view), _ptr(v_view),
                                      _ptr(view_len), _stream(stream)))


def kvm_attention_mass(ctx: Context, q, k_pool, n_pages: int, block_table, n_tok, mass, stream=None):
    """Full-attention mass of every history block, summed over each KV head's query heads (a diagnostic)."""
    n = len(n_tok)
    _check(lib().kvm_attention_mass(ctx.handle, _ptr(q), _ptr(k_pool), int(n_pages), _ptr(block_table),
                                    _i64(n_tok), n, _ptr(mass), _stream(stream)))


def kvm_device_status(ctx: Context, clear: bool = True, stream=None) -> int:
    """Device status word (KVM_DEV_* bits) after synchronising the stream; never raises on a non-zero word."""
    out = ctypes.c_uint32(0)
    st = lib().kvm_device_status(ctx.handle, ctypes.byref(out), int(bool(clear)), _stream(stream))
    if st not in (0, 5, 6):
        _check(st)
    return int(out.value)


def kvm_score_select_noalloc(params: Params, q, index, n_tok, kept_ids, group_scores=None, stream=None):
    """Score and select for one decode query without any device allocation.

    For callers that cannot allocate device memory (and so cannot build a
    Context): the head geometry and budget come from `params`; the scratch is a
    fixed array inside libkvm.so (KVM_NOALLOC_SCRATCH_BYTES per GPU) that every
    call reuses, so calls that overlap on the GPU must be serialised.  The
    first call on a device should come before any stream capture.
    """
    L = lib()
    f = L.kvm_score_select_noalloc
    if f.argtypes is None:
        P = ctypes.c_void_p
        f.argtypes = [ctypes.POINTER(Params), P, P, P, ctypes.c_int32, P, P, P]
        f.restype = ctypes.c_int
    n = len(n_tok)
    _check(f(ctypes.byref(params), _ptr(q), _ptr(index), _i64(n_tok), n, _ptr(kept_ids), _ptr(group_scores),
             _stream(stream)))


def kvm_noalloc_status(clear: bool = True, stream=None) -> int:
    """Status word (KVM_DEV_* bits) of the allocation-free calls on the current device, after synchronising
    the stream; optionally cleared.  Never raises on a non-zero word."""
    L = lib()
    f = L.kvm_noalloc_status
    if f.argtypes is None:
        f.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32, ctypes.c_void_p]
        f.restype = ctypes.c_int
    out = ctypes.c_uint32(0)
    st = f(ctypes.byref(out), int(bool(clear)), _stream(stream))
    if st not in (0, 5, 6):
        _check(st)
    return int(out.value)


def kvm_debug_checks() -> bool:
    """True for the debug build of the library (device-side index checks)."""
    L = lib()
    f = L.kvm_debug_checks
    f.argtypes = []
    f.restype = ctypes.c_int32
    return bool(f())


def kvm_set_wait_limit(ctx: Context, wait_ns: int = 2_000_000_000, stall_first_wait: bool = False):
    """Failure-path testing: the view calls' pipeline-wait limit, and a first wait nothing completes."""
    L = lib()
    f = L.kvm_set_wait_limit
    if f.argtypes is None:
        f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32]
        f.restype = ctypes.c_int
    _check(f(ctx.handle, int(wait_ns), int(bool(stall_first_wait))))
