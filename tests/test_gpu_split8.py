"""dX from the fp16 + e4m3 split (TERN_BWD_DX_SPLIT8) against the fp64 oracle.

The weight planes h_c*T (binary16) and l_c*T (e4m3) are bit-exact against the
oracle's split8_planes; dX is within 1e-4 * sum|term| of the oracle's exact sum,
including the edge cases of the split: dY rows far below binary16's normal range
(the per-row exponent takes them out), scales at the ends of the synthetic range,
negative, zero and fp32-subnormal scales, and rows whose magnitudes span several
orders.  gq and sgrad, computed in the same call from a workspace the split shares,
are bit-equal to the call without the flag.
"""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import check_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def _scaled_rows(bits, factors):
    """bf16 bit rows times powers of two (exact while the values stay normal)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * factors[:, None].astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _run(bl, inp, theta=2, clamp=7, split8=True, dw=True):
    M, K, N = inp.M, inp.K, inp.N
    X, dY, q, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.q), dev(inp.scale)
    tiles = bl.Tiles.empty(K, N, t=False, hi_lo=not split8, split8=split8)
    bl.tern_materialize(q, scale, tiles, theta, clamp)
    nan = float("nan")
    dX = torch.full((M, K), nan, device="cuda")
    gq = torch.full((K, N), nan, device="cuda") if dw else None
    sgrad = torch.full((N,), nan, device="cuda") if dw else None
    flags = bl.TERN_BWD_DX_SPLIT8 if split8 else 0
    ws = torch.full((max(bl.tern_linear_bwd_workspace_ex(M, K, N, flags) // 4, 4),), nan, device="cuda")
    bl.tern_linear_bwd(X, dY, tiles, scale, dX, gq, sgrad, ws, split8=split8)
    torch.cuda.synchronize()
    assert bl.tern_device_status() == bl.TERN_OK
    return dX, gq, sgrad, tiles


def _check_dx(inp, dX, theta=2):
    ref, refa = oracle.dx(inp.dY, inp.q, inp.scale, theta)
    return check_close("dX(split8)", dX.cpu().numpy(), ref, refa)


# ----------------------------------------------------------------- the weight planes

@pytest.mark.parametrize("K,N", [(1, 16), (3, 48), (129, 4112), (256, 256), (40, 80)])
def test_split8_planes_bit_exact(cuda_lib, K, N):
    bl = cuda_lib
    q = syn.int8_uniform(7, 3, K * N, -128, 127).reshape(K, N)
    scale = syn.uniform_f32(7, 4, N, -0.1, 0.1)
    edge = np.array([0.0, -0.0, 1e-30, 2.0 ** -140, -3.0e4, 1.0, 0.005, 0.1, 65504.0, 1.9999999], np.float32)
    scale[:min(N, len(edge))] = edge[:min(N, len(edge))]
    wh, wl = oracle.split8_planes(q, scale, 2, 7)
    tiles = bl.Tiles(K, N, whi_f16=torch.full((K, N), 7.0, dtype=torch.float16, device="cuda"),
                     wlo_e4m3=torch.full((K, N), 0x55, dtype=torch.uint8, device="cuda"))
    bl.tern_materialize(dev(q), dev(scale), tiles, 2, 7)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tiles.whi_f16.view(torch.int16).cpu().numpy().view(np.uint16), wh)
    np.testing.assert_array_equal(tiles.wlo_e4m3.cpu().numpy(), wl)


def test_split8_planes_beside_the_other_encodings(cuda_lib):
    """All six planes in one call, with an in-place clamp: the split planes still follow q."""
    bl = cuda_lib
    K, N = 200, 528
    q = syn.int8_uniform(8, 3, K * N, -128, 127).reshape(K, N)
    scale = syn.uniform_f32(8, 4, N, -0.1, 0.1)
    ref = oracle.materialize(q, scale, 3, 7)
    wh, wl = oracle.split8_planes(q, scale, 3, 7)
    tiles = bl.Tiles.empty(K, N, split8=True)
    qd = dev(q)
    bl.tern_materialize(qd, dev(scale), tiles, 3, 7, q_clamped=qd)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qd.cpu().numpy(), ref["qc"])
    np.testing.assert_array_equal(tiles.packed.cpu().numpy().view(np.uint32), ref["packed"])
    np.testing.assert_array_equal(tiles.whi_bf16.view(torch.int16).cpu().numpy().view(np.uint16), ref["whi"])
    np.testing.assert_array_equal(tiles.whi_f16.view(torch.int16).cpu().numpy().view(np.uint16), wh)
    np.testing.assert_array_equal(tiles.wlo_e4m3.cpu().numpy(), wl)


def test_split8_planes_grouped(cuda_lib):
    bl = cuda_lib
    shapes = [(64, 128), (300, 64), (17, 4112)]
    ws, refs = [], []
    for i, (K, N) in enumerate(shapes):
        q = syn.int8_uniform(20 + i, 3, K * N, -7, 7).reshape(K, N)
        scale = syn.uniform_f32(20 + i, 4, N, -0.1, 0.1)
        tiles = bl.Tiles.empty(K, N, t=False, hi_lo=False, split8=True)
        ws.append(dict(q=dev(q), scale=dev(scale), tiles=tiles))
        refs.append(oracle.split8_planes(q, scale, 2, 7))
    bl.tern_materialize_grouped(ws, 2, 7)
    torch.cuda.synchronize()
    for w, (wh, wl) in zip(ws, refs):
        np.testing.assert_array_equal(w["tiles"].whi_f16.view(torch.int16).cpu().numpy().view(np.uint16), wh)
        np.testing.assert_array_equal(w["tiles"].wlo_e4m3.cpu().numpy(), wl)


# ----------------------------------------------------------------- dX, whole outputs

@pytest.mark.parametrize("M,K,N", [
    (64, 128, 128),      # tiny configuration
    (1, 16, 16),         # smallest legal layer
    (130, 144, 272),     # ragged in every dimension, several tiles
    (300, 528, 48),      # N below one k-block
    (257, 64, 784),
    (517, 400, 528),
    (100, 272, 1040),    # single-CTA tiles, ragged k-blocks
])
def test_split8_dx_matches_oracle(cuda_lib, M, K, N):
    inp = syn.linear_inputs(M, K, N, seed=M + 2 * K + N)
    dX, gq, sgrad, _ = _run(cuda_lib, inp)
    _check_dx(inp, dX)
    # gq and sgrad share the workspace with the split of dY: the same bits as without it
    _, gq0, sg0, _ = _run(cuda_lib, inp, split8=False)
    assert torch.equal(gq, gq0) and torch.equal(sgrad, sg0)


@pytest.mark.parametrize("K,N", [(512, 512), (512, 2048), (2048, 512)])
def test_split8_rwkv_block_projections(cuda_lib, K, N):
    inp = syn.linear_inputs(8192, K, N, seed=2, scale_lo=0.01, scale_hi=0.1)
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)


# ----------------------------------------------------------------- dX, the split's edge cases

def test_split8_tiny_and_huge_rows(cuda_lib):
    """Rows of dY scaled by 2^-120 .. 2^100: far outside binary16's range, brought back by
    the per-row exponent."""
    M, K, N = 96, 144, 272
    inp = syn.linear_inputs(M, K, N, seed=11)
    f = np.ldexp(1.0, np.resize(np.array([-120, -100, -60, -24, -17, 0, 20, 60, 100]), M))
    inp.dY = _scaled_rows(inp.dY, f)
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)
    zero = inp.dY.copy()
    zero[5] = 0
    inp.dY = zero
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)
    assert not dX[5].any().item()


@pytest.mark.parametrize("lo,hi", [(0.005, 0.0051), (0.099, 0.1), (-0.1, -0.005), (-0.1, 0.1)])
def test_split8_scale_ranges(cuda_lib, lo, hi):
    inp = syn.linear_inputs(200, 160, 336, seed=12, scale_lo=lo, scale_hi=hi)
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)


def test_split8_zero_subnormal_and_wide_scales(cuda_lib):
    inp = syn.linear_inputs(150, 96, 400, seed=13)
    s = inp.scale.copy()
    s[::9] = 0.0
    s[1::9] = 2.0 ** -140          # fp32 subnormal
    s[2::9] = -3.0e3
    s[3::9] = 1e-20
    inp.scale = s
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)


def test_split8_rows_spanning_orders_of_magnitude(cuda_lib):
    """Within a row, dY entries scaled by 2^-12 .. 2^12 at random (a 2^24 span)."""
    M, K, N = 128, 192, 1024
    inp = syn.linear_inputs(M, K, N, seed=14)
    rng = np.random.default_rng(14)
    e = rng.integers(-12, 13, (M, N))
    f = (inp.dY.astype(np.uint32) << 16).view(np.float32) * np.ldexp(1.0, e).astype(np.float32)
    inp.dY = (f.view(np.uint32) >> 16).astype(np.uint16)
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    _check_dx(inp, dX)


def test_split8_needs_its_planes_and_workspace(cuda_lib):
    bl = cuda_lib
    M, K, N = 64, 64, 64
    inp = syn.linear_inputs(M, K, N, seed=15)
    X, dY, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.scale)
    dX = torch.empty((M, K), device="cuda")
    no_planes = bl.Tiles.empty(K, N)   # bf16 planes only
    ws = torch.empty((bl.tern_linear_bwd_workspace_ex(M, K, N, bl.TERN_BWD_DX_SPLIT8) // 4,), device="cuda")
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd(X, dY, no_planes, scale, dX, None, None, ws, split8=True)
    assert e.value.status == bl.TERN_ERR_ARG
    tiles = bl.Tiles.empty(K, N, split8=True)
    small = torch.empty((16,), device="cuda")
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd(X, dY, tiles, scale, dX, None, None, small, split8=True)
    assert e.value.status == bl.TERN_ERR_WORKSPACE


# ----------------------------------------------------------------- full size, sampled

@pytest.mark.parametrize("name", ["large", "wide_up"])
def test_split8_full_size_sampled(cuda_lib, name):
    c = syn.LARGE if name == "large" else syn.WIDE
    M, K, N = c["M"], c["K"], c["N"]
    inp = syn.linear_inputs(M, K, N, seed=0, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"],
                            zero_prob=c["zero_prob"])
    dX, _, _, _ = _run(cuda_lib, inp, dw=False)
    dXd = dX.cpu().numpy()
    rng = np.random.default_rng(77)
    ms = np.concatenate([[0, M - 1, 0, M - 1], rng.integers(0, M, 4096)])
    rs = np.concatenate([[0, K - 1, K - 1, 0], rng.integers(0, K, 4096)])
    ref = np.array([oracle.dx_at(inp.dY[m], inp.q[r], inp.scale, 2) for m, r in zip(ms, rs)])
    check_close("dX(split8, sampled)", dXd[ms, rs], ref[:, 0], ref[:, 1])
