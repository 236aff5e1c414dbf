"""Grouped forward/backward (several independent layers per call) against the
oracle, layer by layer; Y and dX also bit-equal to the single-layer calls (the
same tiles, k-order and epilogue), gq and sgrad within the oracle tolerance
(their split G tiles may sum in another order)."""
import ctypes

import numpy as np
import pytest
import torch

import tern_synth as syn
from _parity import Layer, full_oracle_check

pytestmark = pytest.mark.gpu

# (M, K, N): single-CTA and CTA-pair tiles in both GEMM orientations, ragged edges
MIXED = [(300, 256, 384), (64, 144, 272), (1000, 512, 512), (257, 128, 1008), (8, 64, 48), (777, 128, 512),
         (129, 384, 256), (100, 256, 384), (513, 1024, 160), (2, 2048, 64)]


def _layers(shapes, seed0):
    out = []
    for i, (M, K, N) in enumerate(shapes):
        L = Layer(syn.linear_inputs(M, K, N, seed=seed0 + i))
        L.bl.tern_materialize(L.q, L.scale, L.tiles, 2, 7)
        out.append(L)
    return out


def _fwd_dicts(layers):
    return [dict(X=L.X, tiles=L.tiles, scale=L.scale, Y=L.Y) for L in layers]


def _bwd_dicts(layers):
    return [dict(X=L.X, dY=L.dY, tiles=L.tiles, scale=L.scale, dX=L.dX, gq=L.gq, sgrad=L.sgrad) for L in layers]


def _workspace(bl, layers, full=True):
    shapes = [(L.M, L.K, L.N) for L in layers]
    if full:
        nbytes = bl.tern_linear_bwd_grouped_workspace(shapes)
    else:   # the sgrad partials alone: no room to split G tiles
        nbytes = sum((bl.tern_linear_bwd_workspace_min(*s) + 255) // 256 * 256 for s in shapes)
    assert nbytes > 0
    return torch.full((nbytes // 4,), float("nan"), device="cuda")


@pytest.mark.parametrize("full_ws", [True, False])
def test_grouped_matches_oracle_and_single_calls(cuda_lib, full_ws):
    bl = cuda_lib
    layers = _layers(MIXED, 200)
    bl.tern_linear_fwd_grouped(_fwd_dicts(layers))
    bl.tern_linear_bwd_grouped(_bwd_dicts(layers), _workspace(bl, layers, full_ws))
    assert bl.tern_device_status() == bl.TERN_OK
    for L in layers:
        full_oracle_check(L)
    for L in layers:   # the single-layer calls give the same Y and dX bits
        Y1 = torch.empty_like(L.Y)
        dX1 = torch.empty_like(L.dX)
        bl.tern_linear_fwd(L.X, L.tiles, L.scale, Y1)
        bl.tern_linear_bwd(L.X, L.dY, L.tiles, L.scale, dX1, None, None, None)
        torch.cuda.synchronize()
        assert torch.equal(Y1, L.Y), (L.M, L.K, L.N)
        assert torch.equal(dX1, L.dX), (L.M, L.K, L.N)


def test_block_projections(cuda_lib):
    """Four square projections of one block's width and its two channel-mixing
    layers, as one grouped call each way, at 1024 tokens."""
    bl = cuda_lib
    layers = _layers([(1024, K, N) for K, N in syn.RWKV_SHAPES], 300)
    bl.tern_linear_fwd_grouped(_fwd_dicts(layers))
    bl.tern_linear_bwd_grouped(_bwd_dicts(layers), _workspace(bl, layers))
    assert bl.tern_device_status() == bl.TERN_OK
    for L in layers:
        full_oracle_check(L)


def test_grouped_accumulate_and_skipped_outputs(cuda_lib):
    """Two grouped calls with TERN_BWD_ACCUMULATE on the second double gq and
    sgrad; layers without dX, gq or sgrad leave those buffers untouched."""
    bl = cuda_lib
    layers = _layers([(300, 256, 384), (1000, 512, 512), (64, 144, 272)], 400)
    ref = _layers([(300, 256, 384), (1000, 512, 512), (64, 144, 272)], 400)
    ws = _workspace(bl, layers)
    d = _bwd_dicts(layers)
    bl.tern_linear_bwd_grouped(d, ws)
    bl.tern_linear_bwd_grouped(d, ws, accumulate=True)
    bl.tern_linear_bwd_grouped(_bwd_dicts(ref), _workspace(bl, ref))
    torch.cuda.synchronize()
    for L, R in zip(layers, ref):
        torch.testing.assert_close(L.gq, 2 * R.gq, rtol=1e-6, atol=1e-7)
        torch.testing.assert_close(L.sgrad, 2 * R.sgrad, rtol=1e-5, atol=1e-6)
    marker = float("nan")
    for L in layers:
        L.dX.fill_(marker)
        L.gq.fill_(marker)
        L.sgrad.fill_(marker)
    d = _bwd_dicts(layers)
    d[0]["dX"] = None
    d[1]["gq"] = None
    d[2]["sgrad"] = None
    bl.tern_linear_bwd_grouped(d, ws)
    torch.cuda.synchronize()
    assert torch.isnan(layers[0].dX).all() and torch.isnan(layers[1].gq).all() and torch.isnan(layers[2].sgrad).all()
    torch.testing.assert_close(layers[0].gq, ref[0].gq, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(layers[1].sgrad, ref[1].sgrad, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(layers[2].dX, ref[2].dX, rtol=0, atol=0)


def test_grouped_argument_errors_enqueue_nothing(cuda_lib):
    bl = cuda_lib
    layers = _layers([(64, 64, 64), (96, 128, 64)], 500)
    for L in layers:
        L.Y.fill_(7.0)
    arr, keep = bl._layers(_fwd_dicts(layers), False)
    arr[1].X = ctypes.c_void_p(layers[1].X.data_ptr() + 2)        # misaligned input in the second layer
    assert bl.lib.tern_linear_fwd_grouped(arr, 2, None) == bl.TERN_ERR_ALIGN
    arr[1].X = ctypes.c_void_p(layers[1].X.data_ptr())
    arr[1].N = 40                                                  # not a multiple of 16
    assert bl.lib.tern_linear_fwd_grouped(arr, 2, None) == bl.TERN_ERR_ALIGN
    assert bl.lib.tern_linear_fwd_grouped(arr, 0, None) == bl.TERN_ERR_ARG
    torch.cuda.synchronize()
    assert (layers[0].Y == 7.0).all() and (layers[1].Y == 7.0).all()
    barr, keep2 = bl._layers(_bwd_dicts(layers), True)
    assert bl.lib.tern_linear_bwd_grouped(barr, 2, None, 0, 0, None) == bl.TERN_ERR_WORKSPACE
    ws = _workspace(bl, layers, full=False)
    nb = ws.numel() * 4
    assert bl.lib.tern_linear_bwd_grouped(barr, 2, ctypes.c_void_p(ws.data_ptr()), nb - 256, 0, None) == \
        bl.TERN_ERR_WORKSPACE
    assert bl.lib.tern_linear_bwd_grouped(barr, 2, ctypes.c_void_p(ws.data_ptr()), nb, 2, None) == bl.TERN_ERR_ARG
    assert bl.lib.tern_linear_bwd_grouped(barr, 2, ctypes.c_void_p(ws.data_ptr()), nb, 0, None) == bl.TERN_OK
    assert bl.tern_device_status() == bl.TERN_OK


def _bf16_vs_oracle(name, got_bf16, ref, ref_abs):
    """A bf16 output is the fp32 result rounded to nearest even: within the GEMM
    tolerance of the oracle plus the rounding (at most 2^-8 of the value)."""
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    tol = 1e-4 * ref_abs
    bound = tol * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"{name}: max excess {np.max(err - bound):.3e}"


@pytest.mark.parametrize("shapes", [[(300, 256, 384), (1000, 512, 512)], [(64, 144, 272)], [(513, 1024, 160)]])
def test_bf16_outputs(cuda_lib, shapes):
    """Y_bf16 and dX_bf16 are the fp32 outputs rounded to nearest even (bit-exact
    against torch's CPU rounding of the fp32 results of the same call), within
    tolerance of the oracle, and the same bits when the fp32 output is skipped."""
    import oracle
    bl = cuda_lib
    layers = _layers(shapes, 600)
    yb = [torch.empty(L.M, L.N, dtype=torch.bfloat16, device="cuda") for L in layers]
    xb = [torch.empty(L.M, L.K, dtype=torch.bfloat16, device="cuda") for L in layers]
    f = _fwd_dicts(layers)
    b = _bwd_dicts(layers)
    for i in range(len(layers)):
        f[i]["Y_bf16"] = yb[i]
        b[i]["dX_bf16"] = xb[i]
    bl.tern_linear_fwd_grouped(f)
    bl.tern_linear_bwd_grouped(b, _workspace(bl, layers))
    assert bl.tern_device_status() == bl.TERN_OK
    for L, y16, x16 in zip(layers, yb, xb):
        assert torch.equal(y16.cpu().view(torch.int16), L.Y.cpu().to(torch.bfloat16).view(torch.int16))
        assert torch.equal(x16.cpu().view(torch.int16), L.dX.cpu().to(torch.bfloat16).view(torch.int16))
        inp = L.inp
        Yr, Ya = oracle.fwd(inp.X, inp.q, inp.scale)
        dXr, dXa = oracle.dx(inp.dY, inp.q, inp.scale)
        _bf16_vs_oracle("Y_bf16", y16, Yr, Ya)
        _bf16_vs_oracle("dX_bf16", x16, dXr, dXa)
    # bf16 only
    yb2 = [torch.empty_like(t) for t in yb]
    xb2 = [torch.empty_like(t) for t in xb]
    f2 = [dict(X=L.X, tiles=L.tiles, scale=L.scale, Y_bf16=t) for L, t in zip(layers, yb2)]
    b2 = [dict(X=L.X, dY=L.dY, tiles=L.tiles, scale=L.scale, dX_bf16=t) for L, t in zip(layers, xb2)]
    bl.tern_linear_fwd_grouped(f2)
    bl.tern_linear_bwd_grouped(b2, _workspace(bl, layers))
    torch.cuda.synchronize()
    for t, t2 in zip(yb + xb, yb2 + xb2):
        assert torch.equal(t.view(torch.int16), t2.view(torch.int16))


def test_two_layer_chain_through_bf16(cuda_lib):
    """Layer 1's Y_bf16 feeds layer 2 and layer 2's dX_bf16 is layer 1's dY: the
    chain's layer-2 output and layer-1 gradients equal the single calls made on
    the same bf16 intermediates (the intermediates themselves are checked above)."""
    bl = cuda_lib
    M, K1, N1 = 640, 256, 768
    a = syn.linear_inputs(M, K1, N1, seed=701)
    b = syn.linear_inputs(M, N1, K1, seed=702)
    L1, L2 = Layer(a), Layer(b)
    for L in (L1, L2):
        bl.tern_materialize(L.q, L.scale, L.tiles, 2, 7)
    X2 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    dY1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    bl.tern_linear_fwd_grouped([dict(X=L1.X, tiles=L1.tiles, scale=L1.scale, Y_bf16=X2)])
    bl.tern_linear_fwd_grouped([dict(X=X2, tiles=L2.tiles, scale=L2.scale, Y=L2.Y)])
    bl.tern_linear_bwd_grouped([dict(X=X2, dY=L2.dY, tiles=L2.tiles, scale=L2.scale, dX_bf16=dY1, gq=L2.gq,
                                     sgrad=L2.sgrad)], _workspace(bl, [L2]))
    bl.tern_linear_bwd_grouped([dict(X=L1.X, dY=dY1, tiles=L1.tiles, scale=L1.scale, dX=L1.dX, gq=L1.gq,
                                     sgrad=L1.sgrad)], _workspace(bl, [L1]))
    assert bl.tern_device_status() == bl.TERN_OK
    Y2 = torch.empty_like(L2.Y)
    dX1 = torch.empty_like(L1.dX)
    bl.tern_linear_fwd(X2, L2.tiles, L2.scale, Y2)
    bl.tern_linear_bwd(L1.X, dY1, L1.tiles, L1.scale, dX1, None, None, None)
    torch.cuda.synchronize()
    assert torch.equal(Y2, L2.Y) and torch.equal(dX1, L1.dX)
    assert torch.isfinite(L1.gq).all() and torch.isfinite(L2.sgrad).all()


def test_prepared_calls_repeat_the_plain_calls(cuda_lib):
    """Materialize, GroupedForward, GroupedBackward and MultiAdamW (arguments marshalled
    once) give the plain functions' results, call after call."""
    bl = cuda_lib
    layers = _layers(MIXED[:4], 700)
    ws = _workspace(bl, layers)
    fwd = bl.GroupedForward(_fwd_dicts(layers))
    bwd = bl.GroupedBackward(_bwd_dicts(layers), ws)
    mats = [bl.Materialize(L.q, L.scale, L.tiles, 2, 7) for L in layers]
    for _ in range(2):
        for m in mats:
            m()
        fwd()
        bwd()
        assert bl.tern_device_status() == bl.TERN_OK
        for L in layers:
            full_oracle_check(L)
    ref = [(L.Y.clone(), L.dX.clone()) for L in layers]
    bl.tern_linear_fwd_grouped(_fwd_dicts(layers))
    bl.tern_linear_bwd_grouped(_bwd_dicts(layers), ws)
    torch.cuda.synchronize()
    for L, (Y, dX) in zip(layers, ref):
        assert torch.equal(L.Y, Y) and torch.equal(L.dX, dX)
    n = [L.N for L in layers]
    w = [L.scale.clone() for L in layers]
    g = [L.sgrad.clone() for L in layers]
    m1, v1 = [torch.zeros(k, device="cuda") for k in n], [torch.zeros(k, device="cuda") for k in n]
    m2, v2 = [torch.zeros(k, device="cuda") for k in n], [torch.zeros(k, device="cuda") for k in n]
    w2 = [x.clone() for x in w]
    sc = torch.tensor([1e-3, 0.1, 0.05, 1.0], device="cuda")
    prep = bl.MultiAdamW(w, g, m1, v1, sc, 0.9, 0.95, 1e-8, 0.1)
    prep()
    prep()
    bl.adamw_step_multi(w2, g, m2, v2, sc, 0.9, 0.95, 1e-8, 0.1)
    bl.adamw_step_multi(w2, g, m2, v2, sc, 0.9, 0.95, 1e-8, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(w + m1 + v1, w2 + m2 + v2):
        assert torch.equal(a, b)


def test_single_layer_group_splits_the_last_wave_like_the_single_call(cuda_lib):
    """A grouped backward of one layer whose G tiles fill two waves and part of a third (the
    wide chain's up projection: 192 pair tiles on 76 pairs) runs the whole waves, then the
    last wave's tiles split along the token axis, as the single-layer call does: the same
    gq and sgrad bits, and the oracle's values on sampled entries."""
    from _parity import sampled_oracle_check
    bl = cuda_lib
    c = syn.WIDE
    inp = syn.linear_inputs(c["M"], c["K"], c["N"], seed=3, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"],
                            zero_prob=c["zero_prob"])
    L = Layer(inp)
    bl.tern_materialize(L.q, L.scale, L.tiles, 2, 7)
    bl.tern_linear_fwd(L.X, L.tiles, L.scale, L.Y)
    bl.tern_linear_bwd_grouped(_bwd_dicts([L]), _workspace(bl, [L]))
    assert bl.tern_device_status() == bl.TERN_OK
    gq1, sg1 = torch.empty_like(L.gq), torch.empty_like(L.sgrad)
    bl.tern_linear_bwd(L.X, L.dY, L.tiles, L.scale, None, gq1, sg1, L.ws)
    torch.cuda.synchronize()
    assert torch.equal(gq1, L.gq) and torch.equal(sg1, L.sgrad)
    sampled_oracle_check(L, n=1024, ncols=16)
