"""Seeded synthetic inputs for the ternary linear layer and AdamW.

Shared by the CUDA path's tests and bench and by the CPU oracle's tests.  It
holds random-number generation and input formatting only; the generator and its
counter-based definition are described in ``synth.c``.  Tensor ids below give
every tensor of a workload its own stream; one workload uses one seed.

The workload recipes mirror the synthetic shapes of the layer's training step:
X ~ N(0,1) bf16 activations, dY ~ N(0, 0.01) bf16 upstream gradients, q uniform
integers in [-7, 7] (optionally with a share forced to zero), and per-column
scales uniform in a small positive range.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libtern_synth.so")

# tensor ids (one stream per tensor of a workload)
TID_X = 1
TID_DY = 2
TID_Q = 3
TID_SCALE = 4
TID_W = 5
TID_G = 6
TID_Q2 = 7
TID_SCALE2 = 8
TID_DY2 = 9


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, dbl, vp, ci = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                 ctypes.c_void_p, ctypes.c_int)
        lib.synth_normal_bf16.argtypes = [u64, u64, dbl, dbl, i64, i64, vp, ci]
        lib.synth_normal_f32.argtypes = [u64, u64, dbl, dbl, i64, i64, vp, ci]
        lib.synth_uniform_f32.argtypes = [u64, u64, dbl, dbl, i64, i64, vp, ci]
        lib.synth_int8.argtypes = [u64, u64, i64, i64, dbl, i64, i64, vp, ci]
        for f in (lib.synth_normal_bf16, lib.synth_normal_f32, lib.synth_uniform_f32, lib.synth_int8):
            f.restype = None
        lib.synth_key.argtypes = [u64, u64]
        lib.synth_key.restype = u64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal_bf16(seed, tid, n, mean=0.0, std=1.0, start=0, nthreads=0) -> np.ndarray:
    """n bf16 values (as uint16 bit patterns) ~ N(mean, std^2), elements [start, start+n)."""
    out = np.empty(int(n), dtype=np.uint16)
    _L().synth_normal_bf16(seed, tid, mean, std, start, n, _ptr(out), nthreads)
    return out


def normal_f32(seed, tid, n, mean=0.0, std=1.0, start=0, nthreads=0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float32)
    _L().synth_normal_f32(seed, tid, mean, std, start, n, _ptr(out), nthreads)
    return out


def uniform_f32(seed, tid, n, lo, hi, start=0, nthreads=0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float32)
    _L().synth_uniform_f32(seed, tid, lo, hi, start, n, _ptr(out), nthreads)
    return out


def int8_uniform(seed, tid, n, lo=-7, hi=7, zero_prob=0.0, start=0, nthreads=0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int8)
    _L().synth_int8(seed, tid, lo, hi, zero_prob, start, n, _ptr(out), nthreads)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

class LinearInputs:
    """One ternary linear layer's inputs: X [M,K] bf16, q [K,N] int8, scale [N] f32, dY [M,N] bf16."""

    def __init__(self, M, K, N, X, q, scale, dY):
        self.M, self.K, self.N = M, K, N
        self.X, self.q, self.scale, self.dY = X, q, scale, dY


def linear_inputs(M, K, N, seed=0, scale_lo=0.01, scale_hi=0.1, zero_prob=0.0,
                  dy_std=0.01, tids=(TID_X, TID_Q, TID_SCALE, TID_DY)) -> LinearInputs:
    tx, tq, ts, td = tids
    X = normal_bf16(seed, tx, M * K, 0.0, 1.0).reshape(M, K)
    q = int8_uniform(seed, tq, K * N, -7, 7, zero_prob).reshape(K, N)
    scale = uniform_f32(seed, ts, N, scale_lo, scale_hi)
    dY = normal_bf16(seed, td, M * N, 0.0, dy_std).reshape(M, N)
    return LinearInputs(M, K, N, X, q, scale, dY)


def rows_bf16(seed, tid, ncols, rows, mean=0.0, std=1.0) -> np.ndarray:
    """Selected rows of a row-major [*, ncols] bf16 normal tensor (random access)."""
    out = np.empty((len(rows), ncols), dtype=np.uint16)
    for i, r in enumerate(rows):
        out[i] = normal_bf16(seed, tid, ncols, mean, std, start=int(r) * ncols, nthreads=1)
    return out


def rows_int8(seed, tid, ncols, rows, lo=-7, hi=7, zero_prob=0.0) -> np.ndarray:
    out = np.empty((len(rows), ncols), dtype=np.int8)
    for i, r in enumerate(rows):
        out[i] = int8_uniform(seed, tid, ncols, lo, hi, zero_prob, start=int(r) * ncols, nthreads=1)
    return out


# Named configurations of the layer (M tokens, K input features, N output features).
TINY = dict(M=64, K=128, N=128, scale_lo=0.01, scale_hi=0.1, zero_prob=0.0)
RWKV_SHAPES = [(512, 512)] * 4 + [(512, 2048), (2048, 512)]   # (K, N) per projection, M = 8192
RWKV = dict(M=8192, scale_lo=0.01, scale_hi=0.1, zero_prob=0.0)
WIDE = dict(M=16384, K=2048, N=6144, scale_lo=0.005, scale_hi=0.05, zero_prob=0.4)
LARGE = dict(M=32768, K=4096, N=12288, scale_lo=0.005, scale_hi=0.05, zero_prob=0.0)
