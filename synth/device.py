"""Device-side filling of paged K/V pools with the synth recipe (for large workloads).

Compiles kvm_synth_dev.cu (nvcc, sm_103a, -fmad=false) into _kvm_synth_dev.so
on first use.  The values equal those of synth.kv_pool (see the .cu header).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

from . import BLOCK, Workload

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvm_synth_dev.cu")
_LIB = os.path.join(_HERE, "_kvm_synth_dev.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.synth_dev_kv_pages.argtypes = [ctypes.c_uint32, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_double, P, ctypes.c_int64, P, P,
                                           P, P]
        lib.synth_dev_kv_pages.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_kv_pool(w: Workload, layer: int, block_table_dev, k_pool, v_pool, sessions=None, t_range=None):
    """Fills torch CUDA tensors k_pool/v_pool [n_pages][h_kv][32][d] for one layer (all given sessions)."""
    import torch
    lib = _load()
    bad = torch.zeros(1, dtype=torch.int32, device=k_pool.device)
    st = torch.cuda.current_stream().cuda_stream
    t0, t1 = t_range if t_range is not None else (0, w.n_tok)
    for s in (range(w.n_sessions) if sessions is None else sessions):
        row = block_table_dev[s]
        rc = lib.synth_dev_kv_pages(w.session_seed(s), s, layer, w.h_kv, w.d, t0, t1, w.eps_scale, row.data_ptr(),
                                    w.n_pages, k_pool.data_ptr(), v_pool.data_ptr(), bad.data_ptr(), st)
        if rc != 0:
            raise RuntimeError(f"synth_dev_kv_pages failed: cudaError {rc}")
    if int(bad.item()) != 0:
        raise ValueError("block table holds a page outside the pool")
    assert BLOCK == 32
