"""GPU side of the seeded input generator (``synth.cu``): fills large pools fast.

Produces exactly the values of ``ft_synth.expert_entry`` / ``ft_synth.normal_bf16`` and the
bytes of ``ft_synth.expert_entry_fp4``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import TAG_POOL, TAG_POOL_FP4, TAG_X, ENTRY_SIGMA, stream_key

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_DIR, "libft_synth.so")
SRC = os.path.join(_DIR, "synth.cu")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB):
        cmd = ["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
               "-fmad=false", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", SRC,
               "-o", LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} missing; run ft_synth.gpu.build()")
        _lib = ctypes.CDLL(LIB)
        _lib.fts_fill_host.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                       ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
        _lib.fts_fill_host.restype = ctypes.c_int
        _lib.fts_generate_device.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                             ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                             ctypes.c_void_p, ctypes.c_void_p]
        _lib.fts_generate_device.restype = ctypes.c_int
        _lib.fts_fill_host_fp4.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int]
        _lib.fts_fill_host_fp4.restype = ctypes.c_int
    return _lib


def fill_pool(dst_host_ptr: int, seed: int, L: int, E: int, d: int, d_ff: int,
              stage_entries: int = 64):
    """Write the [L][E][entry] pool of expert_entry(seed, l, e, d, d_ff) into host memory."""
    keys = np.array([stream_key(seed, TAG_POOL, l, e) for l in range(L) for e in range(E)],
                    dtype=np.uint64)
    rc = _load().fts_fill_host(keys.ctypes.data, len(keys), 3 * d * d_ff,
                               float(np.float32(ENTRY_SIGMA)), dst_host_ptr, stage_entries)
    if rc != 0:
        raise RuntimeError(f"fts_fill_host failed with CUDA error {rc}")


def fill_pool_fp4(dst_host_ptr: int, seed: int, L: int, E: int, d: int, d_ff: int,
                  stage_entries: int = 256):
    """Write the [L][E][entry] pool of expert_entry_fp4(seed, l, e, d, d_ff) into host memory."""
    keys = np.array([stream_key(seed, TAG_POOL_FP4, l, e) for l in range(L) for e in range(E)],
                    dtype=np.uint64)
    rc = _load().fts_fill_host_fp4(keys.ctypes.data, len(keys), 3 * d * d_ff // 2,
                                   3 * d * d_ff // 32, dst_host_ptr, stage_entries)
    if rc != 0:
        raise RuntimeError(f"fts_fill_host_fp4 failed with CUDA error {rc}")


def activations_device(dst_dev_ptr: int, seed: int, streams, T: int, d: int, stream=0):
    """Rows of activations(seed, s, T, d) for each s in ``streams``, back to back on the device."""
    keys = np.array([stream_key(seed, TAG_X, s) for s in streams], dtype=np.uint64)
    rc = _load().fts_generate_device(keys.ctypes.data, len(keys), T * d, 0, T * d, 1.0,
                                     dst_dev_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"fts_generate_device failed with CUDA error {rc}")
