"""CPU oracle (fp64, plain C) for the ternary linear layer and AdamW.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  It shares no code with the
CUDA library in ``bit_linear_gb300`` and never imports it; the two meet only in
the seeded inputs of ``tern_synth``.

The arithmetic lives in ``tern_oracle.c`` (each function cites the passage of
the pages it follows); this module compiles it with gcc and marshals numpy
arrays.  Every function returns fp64 results together with the sum of |term| of
each output's dot product, the denominator of the comparison tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tern_oracle.c")
_LIB = os.path.join(_HERE, "libtern_oracle.so")

SR4_THETA = 2      # train_gpu.cu: SR4_THETA
SR4_Q_CLAMP = 7    # train_gpu.cu: SR4_Q_CLAMP


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def use_library(path=None):
    """Point the oracle at another build of tern_oracle.c (the mutation tests plant
    mistakes in copies of the source); None restores the default build."""
    global _lib
    _lib = None if path is None else _bind(ctypes.CDLL(path))


def _bind(lib):
    vp, i64, ci, dbl, flt = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                             ctypes.c_float)
    sig = {
        "or_ternary": ([ci, ci], ci),
        "or_clamp": ([ci, ci], ci),
        "or_bf16_value": ([ctypes.c_uint16], dbl),
        "or_bf16_round": ([dbl], ctypes.c_uint16),
        "or_materialize": ([vp, vp, i64, i64, ci, ci, vp, vp, vp, vp, vp], None),
        "or_f16_value": ([ctypes.c_uint16], dbl),
        "or_f16_round": ([dbl], ctypes.c_uint16),
        "or_e4m3_value": ([ctypes.c_uint8], dbl),
        "or_e4m3_round": ([dbl], ctypes.c_uint8),
        "or_split8_planes": ([vp, vp, i64, i64, ci, ci, vp, vp], None),
        "or_fwd": ([vp, vp, vp, i64, i64, i64, ci, vp, vp, ci], None),
        "or_dx": ([vp, vp, vp, i64, i64, i64, ci, vp, vp, ci], None),
        "or_dw": ([vp, vp, vp, vp, i64, i64, i64, ci, vp, vp, vp, vp, ci], None),
        "or_fwd_at": ([vp, vp, flt, i64, ci, vp, vp], None),
        "or_dx_at": ([vp, vp, vp, i64, ci, vp, vp], None),
        "or_gq_at": ([vp, vp, flt, i64, vp, vp], None),
        "or_sgrad_at": ([vp, vp, vp, i64, i64, ci, vp, vp, ci], None),
        "or_adamw": ([vp, vp, vp, vp, i64, ci, dbl, dbl, dbl, dbl, dbl, dbl, ci, vp, vp, vp], None),
        "or_sumsq": ([vp, i64], dbl),
        "or_clip_factor": ([dbl, dbl], dbl),
        "or_mix64": ([ctypes.c_uint64], ctypes.c_uint64),
        "or_sr4_panel": ([vp, vp, vp, i64, i64, ci, ci, vp, vp], None),
        "or_sr4_uniform": ([ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64], flt),
        "or_sr4_scale": ([vp, i64, flt, flt], flt),
        "or_sr4_update": ([vp, vp, i64, flt, flt, ctypes.c_uint64, i64, ctypes.c_uint64, ci, ci, vp, vp],
                          None),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle needs C-contiguous numpy"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def ternary(q: int, theta: int = SR4_THETA) -> int:
    return _L().or_ternary(int(q), int(theta))


def clamp(q: int, c: int = SR4_Q_CLAMP) -> int:
    return _L().or_clamp(int(q), int(c))


def bf16_value(bits: int) -> float:
    return _L().or_bf16_value(int(bits))


def bf16_round(x: float) -> int:
    return int(_L().or_bf16_round(float(x)))


def f16_value(bits: int) -> float:
    return _L().or_f16_value(int(bits))


def f16_round(x: float) -> int:
    return int(_L().or_f16_round(float(x)))


def e4m3_value(bits: int) -> float:
    return _L().or_e4m3_value(int(bits))


def e4m3_round(x: float) -> int:
    return int(_L().or_e4m3_round(float(x)))


def split8_planes(q, scale, theta=SR4_THETA, q_clamp=SR4_Q_CLAMP):
    """The fp16 + e4m3 dX operands: returns (wh16 [K,N] uint16 binary16 bits,
    wl8 [K,N] uint8 e4m3 bits)."""
    q = _c(q, np.int8)
    K, N = q.shape
    scale = _c(scale, np.float32)
    wh16 = np.empty((K, N), np.uint16)
    wl8 = np.empty((K, N), np.uint8)
    _L().or_split8_planes(_p(q), _p(scale), K, N, int(theta), int(q_clamp), _p(wh16), _p(wl8))
    return wh16, wl8


def materialize(q, scale, theta=SR4_THETA, q_clamp=SR4_Q_CLAMP):
    """Returns dict(qc, packed [K,N/16] u32, t, whi, wlo [K,N] bf16 bits)."""
    q = _c(q, np.int8)
    K, N = q.shape
    scale = _c(scale, np.float32)
    out = dict(qc=np.empty((K, N), np.int8),
               packed=np.empty((K, N // 16), np.uint32) if N % 16 == 0 else None,
               t=np.empty((K, N), np.uint16), whi=np.empty((K, N), np.uint16),
               wlo=np.empty((K, N), np.uint16))
    _L().or_materialize(_p(q), _p(scale), K, N, theta, q_clamp, _p(out["qc"]), _p(out["packed"]),
                        _p(out["t"]), _p(out["whi"]), _p(out["wlo"]))
    return out


def fwd(X, q, scale, theta=SR4_THETA, nthreads=0):
    """Y [M,N] fp64 and its abs sums."""
    X, q, scale = _c(X, np.uint16), _c(q, np.int8), _c(scale, np.float32)
    M, K = X.shape
    N = q.shape[1]
    Y, Ya = np.empty((M, N)), np.empty((M, N))
    _L().or_fwd(_p(X), _p(q), _p(scale), M, K, N, theta, _p(Y), _p(Ya), nthreads)
    return Y, Ya


def dx(dY, q, scale, theta=SR4_THETA, nthreads=0):
    dY, q, scale = _c(dY, np.uint16), _c(q, np.int8), _c(scale, np.float32)
    M, N = dY.shape
    K = q.shape[0]
    out, oa = np.empty((M, K)), np.empty((M, K))
    _L().or_dx(_p(dY), _p(q), _p(scale), M, K, N, theta, _p(out), _p(oa), nthreads)
    return out, oa


def dw(X, dY, q, scale, theta=SR4_THETA, nthreads=0):
    """(gq, gq_abs) [K,N] and (sgrad, sgrad_abs) [N], fp64."""
    X, dY, q, scale = _c(X, np.uint16), _c(dY, np.uint16), _c(q, np.int8), _c(scale, np.float32)
    M, K = X.shape
    N = dY.shape[1]
    gq, gqa = np.empty((K, N)), np.empty((K, N))
    sg, sga = np.empty(N), np.empty(N)
    _L().or_dw(_p(X), _p(dY), _p(q), _p(scale), M, K, N, theta, _p(gq), _p(gqa), _p(sg), _p(sga),
               nthreads)
    return gq, gqa, sg, sga


def fwd_at(xrow, qcol, s, theta=SR4_THETA):
    xrow, qcol = _c(xrow, np.uint16), _c(qcol, np.int8)
    o, oa = ctypes.c_double(), ctypes.c_double()
    _L().or_fwd_at(_p(xrow), _p(qcol), float(s), len(xrow), theta, ctypes.byref(o), ctypes.byref(oa))
    return o.value, oa.value


def dx_at(dyrow, qrow, scale, theta=SR4_THETA):
    dyrow, qrow, scale = _c(dyrow, np.uint16), _c(qrow, np.int8), _c(scale, np.float32)
    o, oa = ctypes.c_double(), ctypes.c_double()
    _L().or_dx_at(_p(dyrow), _p(qrow), _p(scale), len(dyrow), theta, ctypes.byref(o), ctypes.byref(oa))
    return o.value, oa.value


def gq_at(xcol, dycol, s):
    xcol, dycol = _c(xcol, np.uint16), _c(dycol, np.uint16)
    o, oa = ctypes.c_double(), ctypes.c_double()
    _L().or_gq_at(_p(xcol), _p(dycol), float(s), len(xcol), ctypes.byref(o), ctypes.byref(oa))
    return o.value, oa.value


def sgrad_at(X, dycol, qcol, theta=SR4_THETA, nthreads=0):
    X, dycol, qcol = _c(X, np.uint16), _c(dycol, np.uint16), _c(qcol, np.int8)
    M, K = X.shape
    o, oa = ctypes.c_double(), ctypes.c_double()
    _L().or_sgrad_at(_p(X), _p(dycol), _p(qcol), M, K, theta, ctypes.byref(o), ctypes.byref(oa),
                     nthreads)
    return o.value, oa.value


def adamw(w, g, m, v, t, lr, b1, b2, eps, wd, gmul=1.0, decoupled=True):
    """One fp64 AdamW step; hyper-parameters are taken as fp32 then widened."""
    w, g, m, v = (_c(a, np.float32) for a in (w, g, m, v))
    n = w.size
    wo, mo, vo = np.empty(n), np.empty(n), np.empty(n)
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    _L().or_adamw(_p(w), _p(g), _p(m), _p(v), n, int(t), f32(lr), f32(b1), f32(b2), f32(eps), f32(wd),
                  f32(gmul), 1 if decoupled else 0, _p(wo), _p(mo), _p(vo))
    return wo, mo, vo


def sumsq(g) -> float:
    g = _c(g, np.float32)
    return float(_L().or_sumsq(_p(g), g.size))


def clip_factor(sumsq_total, max_norm) -> float:
    """-1 to skip the step (non-finite norm), else the gradient multiplier."""
    return float(_L().or_clip_factor(float(sumsq_total), float(max_norm)))


def adamw_clipped(tensors, t, lr, b1, b2, eps, wd, gmul=1.0, max_norm=0.0, decoupled=True):
    """AdamW over several (w, g, m, v) tensors with the global-norm clip and the
    non-finite skip: returns (list of (w, m, v) fp64, skipped)."""
    total = sum(sumsq(g) for _, g, _, _ in tensors)
    f = clip_factor(total, float(np.float32(max_norm)))
    if f < 0:
        return [tuple(np.asarray(a, np.float64) for a in (w, m, v)) for w, _, m, v in tensors], True
    gm = float(np.float32(np.float32(gmul) * np.float32(f)))
    return [adamw(w, g, m, v, t, lr, b1, b2, eps, wd, gm, decoupled) for w, g, m, v in tensors], False


# ----------------------------------------------------------------- SR4 (parity unpinned)

def mix64(z: int) -> int:
    return int(_L().or_mix64(int(z) & 0xFFFFFFFFFFFFFFFF))


def sr4_uniform(seed, counter, j) -> float:
    return float(_L().or_sr4_uniform(seed, counter, j))


def sr4_scale(gq, inv_bs=1.0, target_step=0.003) -> float:
    gq = _c(gq, np.float32)
    return float(_L().or_sr4_scale(_p(gq), gq.size, float(inv_bs), float(target_step)))


def sr4_update(q, gq, s, inv_bs=1.0, seed=42, idx_base=0, counter=0, q_clamp=SR4_Q_CLAMP, dither=True):
    """New q (int8) and the fp32 value y = x + u whose floor is the step taken."""
    q, gq = _c(q, np.int8), _c(gq, np.float32)
    out = np.empty_like(q)
    y = np.empty(q.shape, np.float32)
    _L().or_sr4_update(_p(q), _p(gq), q.size, float(inv_bs), float(s), int(seed), int(idx_base), int(counter),
                       int(q_clamp), 1 if dither else 0, _p(out), _p(y))
    return out, y


def sr4_panel(q, scale, q_prev=None, theta=SR4_THETA, q_clamp=SR4_Q_CLAMP):
    """(counts [neg, zero, pos, rail, dead, churn] uint64, scale [min, mean, max] fp64)."""
    q = _c(q, np.int8)
    K, N = q.shape
    qp = None if q_prev is None else _c(q_prev, np.int8)
    counts = np.zeros(6, np.uint64)
    st = np.zeros(3, np.float64)
    _L().or_sr4_panel(_p(q), _p(qp), _p(_c(scale, np.float32)), K, N, int(theta), int(q_clamp), _p(counts), _p(st))
    return counts, st
