"""The C-ABI library without a GPU: it builds, loads, exports every function the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._builder().build()
    import bit_linear_gb300 as bl
    return bl


def _declared():
    src = open(os.path.join(ROOT, "include", "tern.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("tern_materialize", "tern_linear_fwd", "tern_linear_bwd", "adamw_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(so, name), f"libtern.so does not export {name}"
    assert set(_declared()) == set(lib.ABI_SYMBOLS)


def test_strerror_covers_every_status(lib):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert lib.strerror(st) and lib.strerror(st) != "unknown status"
    assert lib.strerror(-99) == "unknown status"


def test_sizes(lib):
    assert lib.tern_tiles_bytes(4096, 12288, lib.TERN_TILE_PACKED) == 4096 * 768 * 4
    assert lib.tern_tiles_bytes(4096, 12288, lib.TERN_TILE_T) == 4096 * 12288 * 2
    assert lib.tern_tiles_bytes(7, 24, lib.TERN_TILE_T) == 0           # N not a multiple of 16
    assert lib.tern_tiles_bytes(7, 32, 9) == 0
    assert lib.tern_linear_bwd_workspace_min(32768, 4096, 12288) == 32 * 4 * 12288 * 4
    assert lib.tern_linear_bwd_workspace_min(64, 129, 16) == 2 * 4 * 16 * 4
    assert lib.tern_linear_bwd_workspace_min(0, 16, 16) == 0
    # plus at most 128 split tiles of 256 x 256 fp32 (pairs) for the G tail
    assert lib.tern_linear_bwd_workspace(32768, 4096, 12288) == 32 * 4 * 12288 * 4 + 128 * 256 * 256 * 4
    # K <= 128: single-CTA tiles (128 x 256), 1 tile x 1 k-block -> one split tile at most
    assert lib.tern_linear_bwd_workspace(64, 128, 16) == 256 * (-(-(1 * 4 * 16 * 4) // 256)) + 128 * 256 * 4
    assert lib.tern_linear_bwd_workspace(0, 16, 16) == 0
    # the fp16 + e4m3 dX planes and the split of dY (binary16, e4m3, the row exponents, the
    # column factors and their range, each rounded up to 256 bytes), which the G GEMM's
    # workspace shares
    assert lib.tern_tiles_bytes(4096, 12288, lib.TERN_TILE_WHI16) == 4096 * 12288 * 2
    assert lib.tern_tiles_bytes(4096, 12288, lib.TERN_TILE_WLO8) == 4096 * 12288
    assert lib.tern_linear_bwd_workspace_ex(32768, 4096, 12288, 0) == lib.tern_linear_bwd_workspace(32768, 4096, 12288)
    split = 32768 * 12288 * 3 + 32768 * 4 + 12288 * 4 + 256   # ... the column factors and their range
    assert lib.tern_linear_bwd_workspace_ex(32768, 4096, 12288, lib.TERN_BWD_DX_SPLIT8) == split
    assert lib.tern_linear_bwd_workspace_ex(64, 4096, 16, lib.TERN_BWD_DX_SPLIT8) == \
        lib.tern_linear_bwd_workspace(64, 4096, 16)       # the G workspace is the larger here
    assert lib.tern_linear_bwd_workspace_ex(64, 128, 128, 8) == 0      # unknown flag


P = ctypes.c_void_p


def _tiles(lib, base=0x10000):
    return lib._Tiles(P(base), P(base + 0x1000), P(base + 0x2000), P(base + 0x3000))


def test_forward_argument_checks(lib):
    f = lib.lib.tern_linear_fwd
    t = _tiles(lib)
    ok = (P(0x20000), ctypes.byref(t), P(0x30000), P(0x40000))
    assert f(None, ctypes.byref(t), P(0x30000), P(0x40000), 64, 128, 128, None) == lib.TERN_ERR_ARG
    assert f(*ok, 0, 128, 128, None) == lib.TERN_ERR_ARG           # M = 0
    assert f(*ok, 64, 8, 128, None) == lib.TERN_ERR_ARG            # K < 16
    assert f(*ok, 64, 24 + 16, 128, None) == lib.TERN_ERR_ALIGN    # K = 40
    assert f(*ok, 64, 128, 136, None) == lib.TERN_ERR_ALIGN        # N = 136
    assert f(P(0x20002), ctypes.byref(t), P(0x30000), P(0x40000), 64, 128, 128, None) == lib.TERN_ERR_ALIGN
    nul = lib._Tiles(None, None, P(0x12000), P(0x13000))          # neither the bf16 T nor the 2-bit codes
    assert f(P(0x20000), ctypes.byref(nul), P(0x30000), P(0x40000), 64, 128, 128, None) == lib.TERN_ERR_ARG
    mis = lib._Tiles(P(0x10004), None, None, None)                 # the 2-bit codes alone, misaligned
    assert f(P(0x20000), ctypes.byref(mis), P(0x30000), P(0x40000), 64, 128, 128, None) == lib.TERN_ERR_ALIGN


def test_backward_argument_checks(lib):
    f = lib.lib.tern_linear_bwd
    t = _tiles(lib)
    args = lambda dX, ws, n: (P(0x20000), P(0x21000), ctypes.byref(t), P(0x30000), dX, P(0x50000),  # noqa
                              P(0x60000), ws, n, 64, 128, 128, None)
    need = lib.tern_linear_bwd_workspace_min(64, 128, 128)
    assert f(*args(P(0x40000), P(0x70000), need - 4)) == lib.TERN_ERR_WORKSPACE
    assert f(*args(P(0x40000), None, need)) == lib.TERN_ERR_WORKSPACE
    nohl = lib._Tiles(None, P(0x11000), None, None)                 # dX asked without W_hi/W_lo or codes
    assert f(P(0x20000), P(0x21000), ctypes.byref(nohl), P(0x30000), P(0x40000), P(0x50000), None,
             P(0x70000), need, 64, 128, 128, None) == lib.TERN_ERR_ARG
    onehl = lib._Tiles(P(0x10000), None, P(0x12000), None)         # one of the two planes only
    assert f(P(0x20000), P(0x21000), ctypes.byref(onehl), P(0x30000), P(0x40000), None, None,
             P(0x70000), need, 64, 128, 128, None) == lib.TERN_ERR_ARG
    # the codes alone: dX expands W_hi / W_lo in the GEMM; N a multiple of 64 and a workspace
    codes = lib._Tiles(P(0x10000), None, None, None)
    assert f(P(0x20000), P(0x21000), ctypes.byref(codes), P(0x30000), P(0x40000), None, None,
             P(0x70000), need, 64, 128, 48, None) == lib.TERN_ERR_ALIGN
    assert f(P(0x20000), P(0x21000), ctypes.byref(codes), P(0x30000), P(0x40000), None, None,
             None, 0, 64, 128, 128, None) == lib.TERN_ERR_WORKSPACE
    assert f(P(0x20000), P(0x21000), ctypes.byref(t), P(0x30000), P(0x40004), P(0x50000), P(0x60000),
             P(0x70000), need, 64, 128, 128, None) == lib.TERN_ERR_ALIGN
    assert f(P(0x20000), P(0x21000), ctypes.byref(t), P(0x30000), None, None, None,
             None, 0, 64, 128, 128, None) == lib.TERN_ERR_ARG     # nothing requested
    nopk = lib._Tiles(None, P(0x11000), P(0x12000), P(0x13000))     # sgrad needs the 2-bit tiles
    assert f(P(0x20000), P(0x21000), ctypes.byref(nopk), P(0x30000), None, None, P(0x60000),
             P(0x70000), need, 64, 128, 128, None) == lib.TERN_ERR_ARG


def test_split8_backward_argument_checks(lib):
    f = lib.lib.tern_linear_bwd_ex
    M, K, N = 64, 128, 128
    split8 = lib._Tiles(P(0x10000), None, None, None, P(0x14000), P(0x15000))
    need = lib.tern_linear_bwd_workspace_ex(M, K, N, lib.TERN_BWD_DX_SPLIT8)
    call = lambda t, dX, ws, n, flags: f(P(0x20000), P(0x21000), ctypes.byref(t), P(0x30000), dX, None,  # noqa
                                         None, ws, n, M, K, N, flags, None)
    bf = _tiles(lib)                                                   # bf16 planes, no split planes
    assert call(bf, P(0x40000), P(0x70000), need, lib.TERN_BWD_DX_SPLIT8) == lib.TERN_ERR_ARG
    split_bytes = M * N * 2 + M * N + 256 + 512 + 256   # copies of dY, row exponents, column factors, range
    assert split_bytes <= need
    assert call(split8, P(0x40000), P(0x70000), split_bytes - 16, lib.TERN_BWD_DX_SPLIT8) == lib.TERN_ERR_WORKSPACE
    assert call(split8, P(0x40000), None, 0, lib.TERN_BWD_DX_SPLIT8) == lib.TERN_ERR_WORKSPACE
    assert call(split8, P(0x40000), P(0x70008), need, lib.TERN_BWD_DX_SPLIT8) == lib.TERN_ERR_ALIGN
    bad = lib._Tiles(P(0x10000), None, None, None, P(0x14000), P(0x15001))
    assert call(bad, P(0x40000), P(0x70000), need, lib.TERN_BWD_DX_SPLIT8) == lib.TERN_ERR_ALIGN
    assert call(split8, P(0x40000), P(0x70000), need, 4) == lib.TERN_ERR_ARG          # unknown flag
    only8 = lib._Tiles(None, None, None, None, P(0x14000), P(0x15000))
    assert call(only8, P(0x40000), P(0x70000), need, 0) == lib.TERN_ERR_ARG   # without the flag: planes or codes


def test_materialize_argument_checks(lib):
    f = lib.lib.tern_materialize
    t = _tiles(lib)
    q, s = P(0x20000), P(0x30000)
    assert f(q, None, s, 16, 32, 0, 7, ctypes.byref(t), None) == lib.TERN_ERR_ARG      # theta < 1
    assert f(q, None, s, 16, 32, 3, 2, ctypes.byref(t), None) == lib.TERN_ERR_ARG      # clamp < theta
    assert f(q, None, s, 16, 32, 2, 128, ctypes.byref(t), None) == lib.TERN_ERR_ARG    # clamp > 127
    assert f(q, None, None, 16, 32, 2, 7, ctypes.byref(t), None) == lib.TERN_ERR_ARG   # hi/lo need scale
    assert f(q, None, s, 16, 40, 2, 7, ctypes.byref(t), None) == lib.TERN_ERR_ALIGN
    assert f(P(0x20001), None, s, 16, 32, 2, 7, ctypes.byref(t), None) == lib.TERN_ERR_ALIGN
    assert f(q, None, s, 0, 32, 2, 7, ctypes.byref(t), None) == lib.TERN_ERR_ARG
    s8 = lib._Tiles(None, None, None, None, P(0x14000), None)         # split planes need scale
    assert f(q, None, None, 16, 32, 2, 7, ctypes.byref(s8), None) == lib.TERN_ERR_ARG
    s8 = lib._Tiles(None, None, None, None, None, P(0x15008))
    assert f(q, None, s, 16, 32, 2, 7, ctypes.byref(s8), None) == lib.TERN_ERR_ALIGN


def test_adamw_argument_checks(lib):
    f = lib.lib.adamw_step
    a = (P(0x10000), P(0x20000), P(0x30000), P(0x40000))
    hp = (1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1, None)
    assert f(*a, 0, 1, *hp) == lib.TERN_OK           # nothing to do: nothing enqueued
    assert f(*a, -1, 1, *hp) == lib.TERN_ERR_ARG
    assert f(*a, 10, 0, *hp) == lib.TERN_ERR_ARG     # t >= 1
    assert f(P(0x10008), *a[1:], 10, 1, *hp) == lib.TERN_ERR_ALIGN
    assert f(None, *a[1:], 10, 1, *hp) == lib.TERN_ERR_ARG


def test_noalloc_rejects_sizes_beyond_its_scratch_before_touching_the_device(lib):
    f = lib.lib.tern_linear_bwd_noalloc
    t = _tiles(lib)
    # ceil(4096/128) * 4 * 16400 partials > 2^21 floats of built-in scratch
    assert f(P(0x20000), P(0x21000), ctypes.byref(t), P(0x30000), None, None, P(0x60000),
             1, 4096, 16400, None) == lib.TERN_ERR_SCRATCH_LIMIT
    assert lib.strerror(lib.TERN_ERR_SCRATCH_LIMIT) != "unknown status"


def test_grouped_workspace_and_argument_checks(lib):
    shapes = [(1024, 512, 512)] * 4
    # sgrad partials of each layer (4 x 128-row blocks x 4 quarters x 512 columns), then
    # 256 split tiles of 256 x 256 fp32 (the group has 4 x 4 tiles x 16 k-blocks to split)
    assert lib.tern_linear_bwd_grouped_workspace(shapes) == 4 * (4 * 4 * 512 * 4) + 256 * 256 * 256 * 4
    assert lib.tern_linear_bwd_grouped_workspace([(0, 512, 512)]) == 0
    t = _tiles(lib)
    arr = (lib._Layer * 2)()
    for i in range(2):
        arr[i] = lib._Layer(P(0x20000), P(0x21000), ctypes.pointer(t), P(0x30000), P(0x40000), P(0x41000),
                            P(0x50000), P(0x60000), 64, 128, 128)
    f, b = lib.lib.tern_linear_fwd_grouped, lib.lib.tern_linear_bwd_grouped
    assert f(arr, 0, None) == lib.TERN_ERR_ARG
    assert f(None, 1, None) == lib.TERN_ERR_ARG
    arr[1].X = P(0x20002)
    assert f(arr, 2, None) == lib.TERN_ERR_ALIGN
    assert b(arr, 2, P(0x70000), 1 << 20, 0, None) == lib.TERN_ERR_ALIGN
    arr[1].X = P(0x20000)
    arr[1].K = 8
    assert f(arr, 2, None) == lib.TERN_ERR_ARG
    arr[1].K = 128
    assert b(arr, 2, None, 0, 0, None) == lib.TERN_ERR_WORKSPACE
    assert b(arr, 2, P(0x70000), 100, 0, None) == lib.TERN_ERR_WORKSPACE
    assert b(arr, 2, P(0x70000), 1 << 20, 4, None) == lib.TERN_ERR_ARG     # unknown flag


def test_multi_tensor_calls_take_at_most_the_table_size(lib):
    """adamw_step_multi and tern_grad_sumsq reject more than TERN_ADAM_MAX_TENSORS
    tensors (the per-tensor table travels in the launch's parameter block)."""
    k = lib.TERN_ADAM_MAX_TENSORS + 1
    ptrs = (ctypes.c_void_p * k)(*([0x10000] * k))
    ns = (ctypes.c_int64 * k)(*([16] * k))
    f = lib.lib.adamw_step_multi
    assert f(ptrs, ptrs, ptrs, ptrs, ns, k, P(0x20000), 0.9, 0.95, 1e-8, 0.1, 1, None, 0.0, None, None) == \
        lib.TERN_ERR_ARG
    assert lib.lib.tern_grad_sumsq(ptrs, ns, k, P(0x20000), P(0x30000), 1 << 20, None) == lib.TERN_ERR_ARG
    assert lib.lib.tern_grad_sumsq_workspace(ns, k) == 0
    assert lib.TERN_ADAM_MAX_TENSORS == 64


def test_grouped_materialize_argument_checks(lib):
    f = lib.lib.tern_materialize_grouped
    t = _tiles(lib)
    arr = (lib._MatLayer * 2)()
    for i in range(2):
        arr[i] = lib._MatLayer(P(0x20000), None, P(0x30000), ctypes.pointer(t), 64, 128)
    assert f(None, 2, 2, 7, None) == lib.TERN_ERR_ARG
    assert f(arr, 0, 2, 7, None) == lib.TERN_ERR_ARG
    assert f(arr, 2, 3, 2, None) == lib.TERN_ERR_ARG          # clamp < theta
    arr[1].N = 136                                             # not a multiple of 16
    assert f(arr, 2, 2, 7, None) == lib.TERN_ERR_ALIGN
    arr[1].N = 128
    arr[0].q = P(0x20004)                                      # misaligned
    assert f(arr, 2, 2, 7, None) == lib.TERN_ERR_ALIGN
