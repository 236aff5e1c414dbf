"""Python binding of libtern, the sm_103a ternary-weight linear layer library.

Argument marshalling only: every step runs in the library's CUDA kernels (see
``include/tern.h`` for the C ABI).  PyTorch supplies device memory and the
current stream.  The functions carry the C names:

    tern_materialize(q, scale, tiles, theta=2, q_clamp=7, q_clamped=None)
    tern_linear_fwd(X, tiles, scale, Y)
    tern_linear_bwd(X, dY, tiles, scale, dX, gq, sgrad, workspace)
    adamw_step(w, g, m, v, t, lr, b1, b2, eps, wd, gmul=1.0, decoupled=True)

Materialize, MaterializeGrouped, GroupedForward, GroupedBackward and MultiAdamW are the same calls with
their arguments checked and marshalled once, for loops that repeat them on the
same buffers.

Importing this package loads ``lib/libtern.so``; if it is missing the import
fails (run ``bit_linear_gb300.build.build()`` or ``__graft_entry__.build()``).
There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libtern.so")

TERN_OK = 0
TERN_ERR_ARG = -1
TERN_ERR_ALIGN = -2
TERN_ERR_CUDA = -3
TERN_ERR_TIMEOUT = -4
TERN_ERR_WORKSPACE = -5
TERN_ERR_DEVICE = -6
TERN_ERR_SCRATCH_LIMIT = -7
TERN_NOALLOC_SCRATCH_BYTES = 8 << 20

TERN_TILE_PACKED, TERN_TILE_T, TERN_TILE_WHI, TERN_TILE_WLO, TERN_TILE_WHI16, TERN_TILE_WLO8 = 0, 1, 2, 3, 4, 5
TERN_ADAM_MAX_TENSORS = 64
TERN_BWD_ACCUMULATE = 1
TERN_BWD_DX_SPLIT8 = 2

# the C ABI's exported symbols (tests check the library exports every one)
ABI_SYMBOLS = ("tern_tiles_bytes", "tern_materialize", "tern_materialize_grouped", "tern_linear_fwd", "tern_linear_bwd_workspace_min",
               "tern_linear_bwd_workspace", "tern_linear_bwd_workspace_ex",
               "tern_linear_bwd", "tern_linear_bwd_ex", "tern_linear_bwd_noalloc", "tern_linear_fwd_grouped",
               "tern_linear_bwd_grouped_workspace", "tern_linear_bwd_grouped", "adamw_step", "tern_grad_sumsq_workspace",
               "tern_grad_sumsq", "adamw_step_multi", "tern_sr4_workspace", "tern_sr4_step", "tern_sr4_panel", "tern_strerror",
               "tern_device_status", "tern_device_diagnostics", "tern_selftest_wait_timeout")


class TernError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


class _Tiles(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("t_bf16", ctypes.c_void_p),
                ("whi_bf16", ctypes.c_void_p), ("wlo_bf16", ctypes.c_void_p),
                ("whi_f16", ctypes.c_void_p), ("wlo_e4m3", ctypes.c_void_p)]


class _MatLayer(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_clamped", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("out", ctypes.POINTER(_Tiles)), ("K", ctypes.c_int64), ("N", ctypes.c_int64)]


class _Layer(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("dY", ctypes.c_void_p), ("W", ctypes.POINTER(_Tiles)),
                ("scale", ctypes.c_void_p), ("Y", ctypes.c_void_p), ("dX", ctypes.c_void_p),
                ("gq", ctypes.c_void_p), ("sgrad", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("K", ctypes.c_int64), ("N", ctypes.c_int64), ("Y_bf16", ctypes.c_void_p),
                ("dX_bf16", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtern.so is not built ({LIB_PATH}); build it with bit_linear_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, ci, cf, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    tp = ctypes.POINTER(_Tiles)
    sigs = {
        "tern_tiles_bytes": ([i64, i64, ci], sz),
        "tern_materialize": ([vp, vp, vp, i64, i64, ci, ci, tp, vp], ci),
        "tern_materialize_grouped": ([ctypes.POINTER(_MatLayer), ci, ci, ci, vp], ci),
        "tern_linear_fwd": ([vp, tp, vp, vp, i64, i64, i64, vp], ci),
        "tern_linear_bwd_workspace_min": ([i64, i64, i64], sz),
        "tern_linear_bwd_workspace": ([i64, i64, i64], sz),
        "tern_linear_bwd_workspace_ex": ([i64, i64, i64, ctypes.c_uint], sz),
        "tern_linear_bwd": ([vp, vp, tp, vp, vp, vp, vp, vp, sz, i64, i64, i64, vp], ci),
        "tern_linear_bwd_ex": ([vp, vp, tp, vp, vp, vp, vp, vp, sz, i64, i64, i64, ctypes.c_uint, vp], ci),
        "tern_linear_bwd_noalloc": ([vp, vp, tp, vp, vp, vp, vp, i64, i64, i64, vp], ci),
        "tern_linear_fwd_grouped": ([ctypes.POINTER(_Layer), ci, vp], ci),
        "tern_linear_bwd_grouped_workspace": ([ctypes.POINTER(_Layer), ci], sz),
        "tern_linear_bwd_grouped": ([ctypes.POINTER(_Layer), ci, vp, sz, ctypes.c_uint, vp], ci),
        "adamw_step": ([vp, vp, vp, vp, i64, ci, cf, cf, cf, cf, cf, cf, ci, vp], ci),
        "tern_grad_sumsq_workspace": ([ctypes.POINTER(i64), ci], sz),
        "tern_grad_sumsq": ([ctypes.POINTER(vp), ctypes.POINTER(i64), ci, vp, vp, sz, vp], ci),
        "adamw_step_multi": ([ctypes.POINTER(vp)] * 4 + [ctypes.POINTER(i64), ci, vp, cf, cf, cf, cf, ci, vp, cf,
                                                          vp, vp], ci),
        "tern_sr4_workspace": ([i64], sz),
        "tern_sr4_step": ([vp, vp, i64, cf, cf, ctypes.c_uint64, i64, ctypes.c_uint64, ci, ci, vp, vp, sz, vp], ci),
        "tern_sr4_panel": ([vp, vp, vp, i64, i64, ci, ci, vp, vp, vp], ci),
        "tern_strerror": ([ci], ctypes.c_char_p),
        "tern_device_status": ([vp, ci], ci),
        "tern_device_diagnostics": ([ctypes.POINTER(i64), ci], ci),
        "tern_selftest_wait_timeout": ([ctypes.c_uint, vp], ci),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


lib = _load()


def strerror(status: int) -> str:
    return lib.tern_strerror(int(status)).decode()


def _check(status: int, where: str):
    if status != TERN_OK:
        raise TernError(status, where)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype, shape=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor of the given dtype (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


class Tiles:
    """Caller-owned weight encodings of one K x N ternary matrix (see tern.h, tern_tiles).

    packed int32 [K, N/16] (2-bit codes), t/whi/wlo bfloat16 [K, N]; the fp16 + e4m3 dX split
    whi_f16 float16 [K, N] and wlo_e4m3 uint8 [K, N] (e4m3 bit patterns).  Any member may be None.
    """

    def __init__(self, K, N, packed=None, t_bf16=None, whi_bf16=None, wlo_bf16=None, whi_f16=None, wlo_e4m3=None):
        self.K, self.N = int(K), int(N)
        self.packed, self.t_bf16, self.whi_bf16, self.wlo_bf16 = packed, t_bf16, whi_bf16, wlo_bf16
        self.whi_f16, self.wlo_e4m3 = whi_f16, wlo_e4m3

    @classmethod
    def empty(cls, K, N, device="cuda", packed=True, t=True, hi_lo=True, split8=False):
        K, N = int(K), int(N)
        mk = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        return cls(K, N,
                   mk((K, N // 16), torch.int32) if packed else None,
                   mk((K, N), torch.bfloat16) if t else None,
                   mk((K, N), torch.bfloat16) if hi_lo else None,
                   mk((K, N), torch.bfloat16) if hi_lo else None,
                   mk((K, N), torch.float16) if split8 else None,
                   mk((K, N), torch.uint8) if split8 else None)

    def _c(self) -> _Tiles:
        K, N = self.K, self.N
        return _Tiles(
            _ptr(self.packed, torch.int32, (K, N // 16), "tiles.packed"),
            _ptr(self.t_bf16, torch.bfloat16, (K, N), "tiles.t_bf16"),
            _ptr(self.whi_bf16, torch.bfloat16, (K, N), "tiles.whi_bf16"),
            _ptr(self.wlo_bf16, torch.bfloat16, (K, N), "tiles.wlo_bf16"),
            _ptr(self.whi_f16, torch.float16, (K, N), "tiles.whi_f16"),
            _ptr(self.wlo_e4m3, torch.uint8, (K, N), "tiles.wlo_e4m3"))


def tern_tiles_bytes(K, N, which) -> int:
    return int(lib.tern_tiles_bytes(int(K), int(N), int(which)))


class Materialize:
    """tern_materialize with its arguments marshalled once; see GroupedForward."""

    def __init__(self, q, scale, tiles: Tiles, theta=2, q_clamp=7, q_clamped=None):
        K, N = q.shape
        if (tiles.K, tiles.N) != (K, N):
            raise ValueError("tiles shape does not match q")
        self._ct = tiles._c()
        self._args = (_ptr(q, torch.int8, (K, N), "q"), _ptr(q_clamped, torch.int8, (K, N), "q_clamped"),
                      _ptr(scale, torch.float32, (N,), "scale"), K, N, int(theta), int(q_clamp),
                      ctypes.byref(self._ct))
        self._refs = (q, scale, tiles, q_clamped)

    def __call__(self, stream=None):
        _check(lib.tern_materialize(*self._args, _stream(stream)), "tern_materialize")


def tern_materialize(q, scale, tiles: Tiles, theta=2, q_clamp=7, q_clamped=None, stream=None):
    Materialize(q, scale, tiles, theta, q_clamp, q_clamped)(stream)


class MaterializeGrouped:
    """tern_materialize_grouped over weights given as dicts with q, scale, tiles and
    optionally q_clamped, arguments marshalled once; see GroupedForward."""

    def __init__(self, weights, theta=2, q_clamp=7):
        self._arr = (_MatLayer * len(weights))()
        self._keep = []
        for i, w in enumerate(weights):
            q, tiles = w["q"], w["tiles"]
            K, N = q.shape
            if (tiles.K, tiles.N) != (K, N):
                raise ValueError("tiles shape does not match q")
            ct = tiles._c()
            self._keep.append(ct)
            c = self._arr[i]
            c.q = _ptr(q, torch.int8, (K, N), "q")
            c.q_clamped = _ptr(w.get("q_clamped"), torch.int8, (K, N), "q_clamped")
            c.scale = _ptr(w.get("scale"), torch.float32, (N,), "scale")
            c.out = ctypes.pointer(ct)
            c.K, c.N = K, N
        self._n = len(weights)
        self._theta, self._clamp = int(theta), int(q_clamp)
        self._refs = list(weights)

    def __call__(self, stream=None):
        _check(lib.tern_materialize_grouped(self._arr, self._n, self._theta, self._clamp, _stream(stream)),
               "tern_materialize_grouped")


def tern_materialize_grouped(weights, theta=2, q_clamp=7, stream=None):
    MaterializeGrouped(weights, theta, q_clamp)(stream)


def tern_linear_fwd(X, tiles: Tiles, scale, Y, stream=None):
    M, K = X.shape
    N = tiles.N
    ct = tiles._c()
    _check(lib.tern_linear_fwd(_ptr(X, torch.bfloat16, (M, K), "X"), ctypes.byref(ct),
                               _ptr(scale, torch.float32, (N,), "scale"),
                               _ptr(Y, torch.float32, (M, N), "Y"), M, K, N, _stream(stream)),
           "tern_linear_fwd")


def tern_linear_bwd_workspace(M, K, N) -> int:
    return int(lib.tern_linear_bwd_workspace(int(M), int(K), int(N)))


def tern_linear_bwd_workspace_min(M, K, N) -> int:
    return int(lib.tern_linear_bwd_workspace_min(int(M), int(K), int(N)))


def tern_linear_bwd_workspace_ex(M, K, N, flags=0) -> int:
    return int(lib.tern_linear_bwd_workspace_ex(int(M), int(K), int(N), int(flags)))


def tern_linear_bwd(X, dY, tiles: Tiles, scale, dX, gq, sgrad, workspace, stream=None, accumulate=False,
                    split8=False):
    """accumulate=True adds TERN_BWD_ACCUMULATE (gq, sgrad +=), split8=True TERN_BWD_DX_SPLIT8 (dX from
    the fp16 + e4m3 split); either calls tern_linear_bwd_ex."""
    M, K = X.shape
    N = tiles.N
    ct = tiles._c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    ws_ptr = None if workspace is None else _ptr(workspace, workspace.dtype, None, "workspace")
    args = (_ptr(X, torch.bfloat16, (M, K), "X"), _ptr(dY, torch.bfloat16, (M, N), "dY"), ctypes.byref(ct),
            _ptr(scale, torch.float32, (N,), "scale"), _ptr(dX, torch.float32, (M, K), "dX"),
            _ptr(gq, torch.float32, (K, N), "gq"), _ptr(sgrad, torch.float32, (N,), "sgrad"), ws_ptr, ws_bytes,
            M, K, N)
    flags = (TERN_BWD_ACCUMULATE if accumulate else 0) | (TERN_BWD_DX_SPLIT8 if split8 else 0)
    if flags:
        _check(lib.tern_linear_bwd_ex(*args, flags, _stream(stream)), "tern_linear_bwd_ex")
    else:
        _check(lib.tern_linear_bwd(*args, _stream(stream)), "tern_linear_bwd")


def tern_linear_bwd_noalloc(X, dY, tiles: Tiles, scale, dX, gq, sgrad, stream=None):
    """tern_linear_bwd without a caller workspace, for callers that cannot allocate
    device memory: the sgrad partials live in a fixed 8 MiB array inside the
    library (see tern.h for the size limit and the rule that overlapping calls race)."""
    M, K = X.shape
    N = tiles.N
    ct = tiles._c()
    _check(lib.tern_linear_bwd_noalloc(_ptr(X, torch.bfloat16, (M, K), "X"), _ptr(dY, torch.bfloat16, (M, N), "dY"),
                                       ctypes.byref(ct), _ptr(scale, torch.float32, (N,), "scale"),
                                       _ptr(dX, torch.float32, (M, K), "dX"), _ptr(gq, torch.float32, (K, N), "gq"),
                                       _ptr(sgrad, torch.float32, (N,), "sgrad"), M, K, N, _stream(stream)),
           "tern_linear_bwd_noalloc")


def _layers(layers, backward):
    """ctypes array of tern_layer from dicts with keys X, tiles, scale and Y and/or Y_bf16
    (forward) or X, dY, tiles, scale and any of dX, dX_bf16, gq, sgrad (backward); a
    missing or None output is skipped.  The second value keeps the tern_tiles structs
    alive while the array is in use."""
    arr = (_Layer * len(layers))()
    keep = []
    for i, L in enumerate(layers):
        X, tiles = L["X"], L["tiles"]
        M, K = X.shape
        N = tiles.N
        ct = tiles._c()
        keep.append(ct)
        c = arr[i]
        c.X = _ptr(X, torch.bfloat16, (M, K), "X")
        c.W = ctypes.pointer(ct)
        c.scale = _ptr(L["scale"], torch.float32, (N,), "scale")
        c.M, c.K, c.N = M, K, N
        if backward:
            c.dY = _ptr(L["dY"], torch.bfloat16, (M, N), "dY")
            c.dX = _ptr(L.get("dX"), torch.float32, (M, K), "dX")
            c.dX_bf16 = _ptr(L.get("dX_bf16"), torch.bfloat16, (M, K), "dX_bf16")
            c.gq = _ptr(L.get("gq"), torch.float32, (K, N), "gq")
            c.sgrad = _ptr(L.get("sgrad"), torch.float32, (N,), "sgrad")
        else:
            c.Y = _ptr(L.get("Y"), torch.float32, (M, N), "Y")
            c.Y_bf16 = _ptr(L.get("Y_bf16"), torch.bfloat16, (M, N), "Y_bf16")
    return arr, keep


class GroupedForward:
    """tern_linear_fwd_grouped with its arguments checked and marshalled once: calling
    the object enqueues the grouped forward of the same buffers again (a training loop
    calls it every step).  It keeps references to the tensors it was given."""

    def __init__(self, layers):
        self._arr, self._keep = _layers(layers, False)
        self._n = len(layers)
        self._refs = list(layers)

    def __call__(self, stream=None):
        _check(lib.tern_linear_fwd_grouped(self._arr, self._n, _stream(stream)), "tern_linear_fwd_grouped")


class GroupedBackward:
    """tern_linear_bwd_grouped with its arguments (and workspace) marshalled once; see
    GroupedForward."""

    def __init__(self, layers, workspace, accumulate=False):
        self._arr, self._keep = _layers(layers, True)
        self._n = len(layers)
        self._ws = _ptr(workspace, workspace.dtype, None, "workspace")
        self._ws_bytes = workspace.numel() * workspace.element_size()
        self._flags = TERN_BWD_ACCUMULATE if accumulate else 0
        self._refs = (list(layers), workspace)

    def __call__(self, stream=None):
        _check(lib.tern_linear_bwd_grouped(self._arr, self._n, self._ws, self._ws_bytes, self._flags,
                                           _stream(stream)), "tern_linear_bwd_grouped")


def tern_linear_fwd_grouped(layers, stream=None):
    """Y = X * W_eff for every layer (dicts with X, tiles, scale, Y and/or Y_bf16), in grouped launches."""
    GroupedForward(layers)(stream)


def tern_linear_bwd_grouped_workspace(shapes) -> int:
    """Workspace bytes of tern_linear_bwd_grouped for layers of these (M, K, N) shapes."""
    arr = (_Layer * len(shapes))()
    for i, (M, K, N) in enumerate(shapes):
        arr[i].M, arr[i].K, arr[i].N = int(M), int(K), int(N)
    return int(lib.tern_linear_bwd_grouped_workspace(arr, len(shapes)))


def tern_linear_bwd_grouped(layers, workspace, stream=None, accumulate=False):
    """dX (fp32 and/or bf16), gq and sgrad for every layer (dicts with X, dY, tiles, scale, dX, dX_bf16,
    gq, sgrad)."""
    GroupedBackward(layers, workspace, accumulate)(stream)


def adamw_step(w, g, m, v, t, lr, b1, b2, eps, wd, gmul=1.0, decoupled=True, stream=None):
    n = w.numel()
    for name, x in (("g", g), ("m", m), ("v", v)):
        if x.numel() != n:
            raise ValueError(f"{name} has {x.numel()} elements, w has {n}")
    _check(lib.adamw_step(_ptr(w, torch.float32, None, "w"), _ptr(g, torch.float32, None, "g"),
                          _ptr(m, torch.float32, None, "m"), _ptr(v, torch.float32, None, "v"), n, int(t),
                          float(lr), float(b1), float(b2), float(eps), float(wd), float(gmul),
                          1 if decoupled else 0, _stream(stream)),
           "adamw_step")


def _ptr_array(ts, dtype, name):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t, dtype, None, f"{name}[{i}]")
    return arr


def _n_array(ts):
    return (ctypes.c_int64 * len(ts))(*[t.numel() for t in ts])


def tern_grad_sumsq_workspace(grads) -> int:
    n = _n_array(grads)
    return int(lib.tern_grad_sumsq_workspace(n, len(grads)))


def tern_grad_sumsq(grads, sumsq, workspace, stream=None):
    """sumsq (device float64 [1]) = sum of squares of every gradient tensor, fixed order."""
    n = _n_array(grads)
    _check(lib.tern_grad_sumsq(_ptr_array(grads, torch.float32, "g"), n, len(grads),
                               _ptr(sumsq, torch.float64, None, "sumsq"),
                               _ptr(workspace, workspace.dtype, None, "workspace"),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
           "tern_grad_sumsq")


class MultiAdamW:
    """adamw_step_multi with its arguments marshalled once (the per-step scalars stay in
    device memory, so the same call serves every step); see GroupedForward."""

    def __init__(self, ws, gs, ms, vs, scalars, b1, b2, eps, wd, decoupled=True, sumsq=None, max_norm=0.0,
                 skipped=None):
        k = len(ws)
        if not (len(gs) == len(ms) == len(vs) == k):
            raise ValueError("w, g, m, v lists differ in length")
        for i in range(k):
            if not (ws[i].numel() == gs[i].numel() == ms[i].numel() == vs[i].numel()):
                raise ValueError(f"tensor {i}: w, g, m, v sizes differ")
        self._args = (_ptr_array(ws, torch.float32, "w"), _ptr_array(gs, torch.float32, "g"),
                      _ptr_array(ms, torch.float32, "m"), _ptr_array(vs, torch.float32, "v"), _n_array(ws), k,
                      _ptr(scalars, torch.float32, (4,), "scalars"), float(b1), float(b2), float(eps), float(wd),
                      1 if decoupled else 0, _ptr(sumsq, torch.float64, None, "sumsq"), float(max_norm),
                      _ptr(skipped, torch.int32, None, "skipped"))
        self._refs = (list(ws), list(gs), list(ms), list(vs), scalars, sumsq, skipped)

    def __call__(self, stream=None):
        _check(lib.adamw_step_multi(*self._args, _stream(stream)), "adamw_step_multi")


def adamw_step_multi(ws, gs, ms, vs, scalars, b1, b2, eps, wd, decoupled=True, sumsq=None, max_norm=0.0,
                     skipped=None, stream=None):
    """AdamW over several tensors in one launch; `scalars` is a device float32 [4]
    tensor {lr, bc1, bc2, gmul}; `sumsq` (device float64 [1]) enables the global-norm
    clip (max_norm > 0) and the non-finite skip; `skipped` is a device int32 [1]."""
    MultiAdamW(ws, gs, ms, vs, scalars, b1, b2, eps, wd, decoupled, sumsq, max_norm, skipped)(stream)


def tern_sr4_workspace(numel) -> int:
    return int(lib.tern_sr4_workspace(int(numel)))


def tern_sr4_step(q, gq, workspace, inv_bs=1.0, target_step=0.003, seed=42, idx_base=0, counter=0, q_clamp=7,
                  use_dither=True, s_out=None, stream=None):
    """SR4 step: q (int8, in place) moves by stochastic rounding of -gq*inv_bs*s (see tern.h)."""
    n = q.numel()
    if gq.numel() != n:
        raise ValueError("q and gq differ in size")
    _check(lib.tern_sr4_step(_ptr(q, torch.int8, None, "q"), _ptr(gq, torch.float32, None, "gq"), n,
                             float(inv_bs), float(target_step), int(seed), int(idx_base), int(counter),
                             int(q_clamp), 1 if use_dither else 0, _ptr(s_out, torch.float32, None, "s_out"),
                             _ptr(workspace, workspace.dtype, None, "workspace"),
                             workspace.numel() * workspace.element_size(), _stream(stream)),
           "tern_sr4_step")


def tern_sr4_panel(q, scale, counts, scale_stats, packed_prev=None, theta=2, q_clamp=7, stream=None):
    """counts: device int64 [6] (neg, zero, pos, rail, dead, churn); scale_stats: device float64 [3]."""
    K, N = q.shape
    _check(lib.tern_sr4_panel(_ptr(q, torch.int8, (K, N), "q"),
                              _ptr(packed_prev, torch.int32, (K, N // 16), "packed_prev"),
                              _ptr(scale, torch.float32, (N,), "scale"), K, N, int(theta), int(q_clamp),
                              _ptr(counts, torch.int64, (6,), "counts"),
                              _ptr(scale_stats, torch.float64, (3,), "scale_stats"), _stream(stream)),
           "tern_sr4_panel")


def tern_device_status(stream=None, clear=True) -> int:
    """Synchronise the stream; TERN_ERR_TIMEOUT if a kernel gave up on a bounded wait."""
    return int(lib.tern_device_status(_stream(stream), 1 if clear else 0))


def tern_device_diagnostics(wait_ms=2000) -> dict:
    """The device-side failure records (see tern.h), read on the library's own
    non-blocking stream; usable while the caller's streams are stuck."""
    out = (ctypes.c_int64 * 8)()
    _check(lib.tern_device_diagnostics(out, int(wait_ms)), "tern_device_diagnostics")
    return {"status": out[0], "ctas_entered": out[1], "ctas_set_up": out[2], "ctas_exited": out[3],
            "first_give_up": {"site": out[4], "cta": out[5], "barrier": out[6], "parity": out[7]}}


def workspace_for(M, K, N, device="cuda") -> torch.Tensor:
    nbytes = tern_linear_bwd_workspace(M, K, N)
    return torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=device)
