"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Bit-exact for the integer/byte work (clamp, ternary, 2-bit packing, bf16
operand planes); |gpu - oracle| <= 1e-4 * sum|term| element-wise for Y, dX,
gq and sgrad; AdamW within 1e-6 of (|w| + |dw|).  Outputs are NaN-filled
before each call so that an unwritten element fails.
"""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import Layer, check_close, dev, full_oracle_check, host_bits, sampled_oracle_check

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------- materialise

@pytest.mark.parametrize("K,N,theta,clamp", [
    (1, 16, 2, 7), (3, 48, 2, 7), (256, 256, 2, 7), (129, 4112, 1, 7), (64, 512, 3, 7),
    (17, 160, 7, 7), (32, 64, 8, 127), (40, 80, 2, 127)])
def test_materialize_bit_exact(cuda_lib, K, N, theta, clamp):
    bl = cuda_lib
    q = syn.int8_uniform(5, 3, K * N, -128, 127).reshape(K, N)      # full int8 range
    scale = syn.uniform_f32(5, 4, N, -0.1, 0.1)                      # both signs
    scale[::7] = 1.0                                                 # exact in bf16: s_lo = 0
    ref = oracle.materialize(q, scale, theta, clamp)
    tiles = bl.Tiles.empty(K, N)
    for t in (tiles.packed, tiles.t_bf16, tiles.whi_bf16, tiles.wlo_bf16):
        t.view(torch.int16).fill_(0x7FC1)
    qc = torch.full((K, N), 99, dtype=torch.int8, device="cuda")
    bl.tern_materialize(dev(q), dev(scale), tiles, theta, clamp, q_clamped=qc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qc.cpu().numpy(), ref["qc"])
    np.testing.assert_array_equal(tiles.packed.cpu().numpy().view(np.uint32), ref["packed"])
    np.testing.assert_array_equal(host_bits(tiles.t_bf16), ref["t"])
    np.testing.assert_array_equal(host_bits(tiles.whi_bf16), ref["whi"])
    np.testing.assert_array_equal(host_bits(tiles.wlo_bf16), ref["wlo"])


def test_materialize_every_int8_in_every_lane(cuda_lib):
    bl = cuda_lib
    q = np.arange(-128, 128, dtype=np.int16)
    q = np.stack([np.roll(q, j) for j in range(16)], axis=1).astype(np.int8)
    scale = np.linspace(0.01, 0.1, 16).astype(np.float32)
    for theta, clamp in [(1, 7), (2, 7), (3, 7), (7, 7), (2, 127)]:
        ref = oracle.materialize(q, scale, theta, clamp)
        tiles = bl.Tiles.empty(256, 16)
        bl.tern_materialize(dev(q), dev(scale), tiles, theta, clamp)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tiles.packed.cpu().numpy().view(np.uint32), ref["packed"])
        np.testing.assert_array_equal(host_bits(tiles.t_bf16), ref["t"])


def test_materialize_packed_only_and_inplace_clamp(cuda_lib):
    bl = cuda_lib
    K, N = 1000, 1008
    q = syn.int8_uniform(9, 3, K * N, -128, 127).reshape(K, N)
    ref = oracle.materialize(q, np.ones(N, np.float32), 2, 7)
    tiles = bl.Tiles(K, N, packed=torch.zeros((K, N // 16), dtype=torch.int32, device="cuda"))
    qd = dev(q)
    bl.tern_materialize(qd, None, tiles, 2, 7, q_clamped=qd)    # scale not needed without hi/lo planes
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tiles.packed.cpu().numpy().view(np.uint32), ref["packed"])
    np.testing.assert_array_equal(qd.cpu().numpy(), ref["qc"])


# ----------------------------------------------------------------- the layer, whole outputs

@pytest.mark.parametrize("M,K,N", [
    (64, 128, 128),      # tiny configuration
    (1, 16, 16),         # smallest legal layer
    (130, 144, 272),     # ragged in every dimension, several tiles
    (300, 528, 48),      # N below one tile
    (257, 64, 784),      # K below one k-block
    (517, 400, 528),
])
def test_layer_matches_oracle(cuda_lib, M, K, N):
    inp = syn.linear_inputs(M, K, N, seed=M + K + N)
    layer = Layer(inp).run()
    full_oracle_check(layer)


def test_tiny_configuration_with_adamw_on_scale(cuda_lib):
    bl = cuda_lib
    cfg = syn.TINY
    inp = syn.linear_inputs(cfg["M"], cfg["K"], cfg["N"], seed=0, scale_lo=0.01, scale_hi=0.1)
    layer = Layer(inp).run()
    full_oracle_check(layer)
    # AdamW on the scales with the scale gradient just computed (t = 1)
    _, _, sg, _ = oracle.dw(inp.X, inp.dY, inp.q, inp.scale)
    sgrad_gpu = layer.sgrad.cpu().numpy()
    m = torch.zeros(cfg["N"], device="cuda")
    v = torch.zeros(cfg["N"], device="cuda")
    w = layer.scale.clone()
    bl.adamw_step(w, layer.sgrad, m, v, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    z = np.zeros(cfg["N"], np.float32)
    wo, mo, vo = oracle.adamw(inp.scale, sgrad_gpu, z, z, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    _adam_close(w.cpu().numpy(), wo, inp.scale)
    _moments_close(m.cpu().numpy(), v.cpu().numpy(), mo, vo, z, z, sgrad_gpu, 1.0, inp.scale, True)


@pytest.mark.parametrize("K,N", [(512, 512), (512, 2048), (2048, 512)])
def test_rwkv_block_projections(cuda_lib, K, N):
    inp = syn.linear_inputs(8192, K, N, seed=1, scale_lo=0.01, scale_hi=0.1)
    layer = Layer(inp).run()
    full_oracle_check(layer)


def test_theta_8_zeroes_y_dx_sgrad(cuda_lib):
    inp = syn.linear_inputs(96, 64, 64, seed=3)
    layer = Layer(inp, theta=8, q_clamp=127).run()
    assert not layer.Y.any().item() and not layer.dX.any().item() and not layer.sgrad.any().item()
    full_oracle_check(layer)


def test_sgrad_is_deterministic(cuda_lib):
    inp = syn.linear_inputs(1000, 640, 528, seed=4)
    a = Layer(inp).run()
    s1, g1 = a.sgrad.clone(), a.gq.clone()
    a.run()
    assert torch.equal(s1, a.sgrad) and torch.equal(g1, a.gq)


def test_backward_without_dx(cuda_lib):
    bl = cuda_lib
    inp = syn.linear_inputs(200, 160, 96, seed=6)
    layer = Layer(inp, with_dx=False)
    bl.tern_materialize(layer.q, layer.scale, layer.tiles, 2, 7)
    bl.tern_linear_bwd(layer.X, layer.dY, layer.tiles, layer.scale, None, layer.gq, layer.sgrad, layer.ws)
    torch.cuda.synchronize()
    gq, gqa, sg, sga = oracle.dw(inp.X, inp.dY, inp.q, inp.scale)
    check_close("gq", layer.gq.cpu().numpy(), gq, gqa)
    check_close("sgrad", layer.sgrad.cpu().numpy(), sg, sga)


# ----------------------------------------------------------------- full sizes, sampled

@pytest.mark.parametrize("name", ["wide_up", "wide_down", "large"])
def test_full_size_sampled(cuda_lib, name):
    if name == "large":
        c = syn.LARGE
        M, K, N = c["M"], c["K"], c["N"]
        inp = syn.linear_inputs(M, K, N, seed=0, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"])
    else:
        c = syn.WIDE
        M, K, N = c["M"], c["K"], c["N"]
        if name == "wide_down":
            K, N = N, K
        inp = syn.linear_inputs(M, K, N, seed=0 if name == "wide_up" else 1, scale_lo=c["scale_lo"],
                                scale_hi=c["scale_hi"], zero_prob=c["zero_prob"])
    layer = Layer(inp).run()
    sampled_oracle_check(layer, n=4096, ncols=64)


# ----------------------------------------------------------------- AdamW

def _adam_close(got, ref, w_old, rel=1e-6):
    got = np.asarray(got, np.float64)
    w_old = np.asarray(w_old, np.float64)
    bound = rel * (np.abs(w_old) + np.abs(ref - w_old)) + 1e-30
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"AdamW: worst |err|/bound = {(err / bound).max():.3g}"


@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, 4099, 1 << 20])
@pytest.mark.parametrize("decoupled", [True, False])
def test_adamw_matches_oracle(cuda_lib, n, decoupled):
    bl = cuda_lib
    w0 = syn.normal_f32(7, syn.TID_W, n, 0.0, 0.02)
    g = syn.normal_f32(7, syn.TID_G, n, 0.0, 1e-3)
    m0 = syn.normal_f32(7, 21, n, 0.0, 1e-4)
    v0 = np.abs(syn.normal_f32(7, 22, n, 0.0, 1e-6))
    w, gd, m, v = dev(w0), dev(g), dev(m0), dev(v0)
    bl.adamw_step(w, gd, m, v, 3, 1e-3, 0.9, 0.95, 1e-8, 0.1, gmul=0.5, decoupled=decoupled)
    torch.cuda.synchronize()
    wo, mo, vo = oracle.adamw(w0, g, m0, v0, 3, 1e-3, 0.9, 0.95, 1e-8, 0.1, gmul=0.5, decoupled=decoupled)
    _adam_close(w.cpu().numpy(), wo, w0)
    _moments_close(m.cpu().numpy(), v.cpu().numpy(), mo, vo, m0, v0, g, 0.5, w0, decoupled)


def _moments_close(m, v, mo, vo, m0, v0, g, gmul, w0, decoupled, b1=0.9, b2=0.95, wd=0.1, rel=1e-6):
    """m and v within 1e-6 of the sum of the magnitudes of their two terms (m cancels)."""
    f = lambda x: float(np.float32(x))  # noqa: E731
    gp = f(gmul) * np.asarray(g, np.float64)
    if not decoupled:
        gp = gp + f(wd) * np.asarray(w0, np.float64)
    mden = f(b1) * np.abs(np.asarray(m0, np.float64)) + (1 - f(b1)) * np.abs(gp)
    vden = f(b2) * np.abs(np.asarray(v0, np.float64)) + (1 - f(b2)) * gp * gp
    assert np.all(np.abs(np.asarray(m, np.float64) - mo) <= rel * mden + 1e-38)
    assert np.all(np.abs(np.asarray(v, np.float64) - vo) <= rel * vden + 1e-38)


def test_adamw_ten_steps_same_gradient(cuda_lib):
    bl = cuda_lib
    n = 100003
    w0 = syn.normal_f32(0, syn.TID_W, n, 0.0, 0.02)
    g = syn.normal_f32(0, syn.TID_G, n, 0.0, 1e-3)
    w, gd = dev(w0), dev(g)
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    wh, mh, vh = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 11):
        bl.adamw_step(w, gd, m, v, t, 1e-3, 0.9, 0.95, 1e-8, 0.1)
        wo, mo, vo = oracle.adamw(wh, g, mh, vh, t, 1e-3, 0.9, 0.95, 1e-8, 0.1)
        torch.cuda.synchronize()
        wg = w.cpu().numpy()
        _adam_close(wg, wo, wh)
        # next step starts from the GPU state on both sides
        wh, mh, vh = wg, m.cpu().numpy(), v.cpu().numpy()


# ----------------------------------------------------------------- error statuses on a GPU

def test_misaligned_and_bad_arguments_are_rejected(cuda_lib):
    bl = cuda_lib
    inp = syn.linear_inputs(64, 64, 64, seed=8)
    layer = Layer(inp)
    layer.run()
    buf = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    Xmis = buf[1:1 + 64 * 64].view(64, 64)            # 2-byte offset
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_fwd(Xmis, layer.tiles, layer.scale, layer.Y)
    assert e.value.status == bl.TERN_ERR_ALIGN
    small_ws = torch.empty(1, dtype=torch.float32, device="cuda")
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd(layer.X, layer.dY, layer.tiles, layer.scale, layer.dX, layer.gq, layer.sgrad,
                           small_ws)
    assert e.value.status == bl.TERN_ERR_WORKSPACE
    with pytest.raises(bl.TernError) as e:
        bl.tern_materialize(layer.q, layer.scale, layer.tiles, theta=3, q_clamp=2)
    assert e.value.status == bl.TERN_ERR_ARG
    assert bl.tern_device_status() == bl.TERN_OK


@pytest.mark.parametrize("theta,clamp", [(1, 7), (3, 7), (5, 127)])
def test_layer_other_thresholds(cuda_lib, theta, clamp):
    inp = syn.linear_inputs(300, 272, 400, seed=theta * 10 + clamp)
    inp.q = syn.int8_uniform(theta, syn.TID_Q, 272 * 400, -128, 127).reshape(272, 400)   # full int8 range
    layer = Layer(inp, theta=theta, q_clamp=clamp).run()
    full_oracle_check(layer)


def test_layer_with_negative_and_zero_scales(cuda_lib):
    inp = syn.linear_inputs(257, 400, 304, seed=77)
    sc = syn.uniform_f32(77, syn.TID_SCALE, 304, -0.1, 0.1)
    sc[::13] = 0.0
    sc[5::17] = -1.0             # exact in bf16: s_lo = 0
    inp.scale = sc
    layer = Layer(inp).run()
    full_oracle_check(layer)


# ----------------------------------------------------------------- forward from the 2-bit codes

@pytest.mark.parametrize("M,K,N", [(64, 128, 128), (130, 144, 320), (300, 528, 64), (257, 64, 768), (1000, 512, 2048),
                                   (8, 80, 192), (513, 1040, 448)])
def test_forward_from_packed_codes(cuda_lib, M, K, N):
    """tern_linear_fwd with t_bf16 = NULL reads T as the 2-bit codes, expanded to bf16 in
    the GEMM: the same Y bits as the bf16-plane forward, and within the oracle tolerance.
    (This operand needs N % 64 == 0: its rows are copied by TMA in 16-byte multiples.)"""
    bl = cuda_lib
    inp = syn.linear_inputs(M, K, N, seed=M + 3 * K + N)
    layer = Layer(inp).run()
    packed_only = bl.Tiles(K, N, packed=layer.tiles.packed)
    Y = torch.full((M, N), float("nan"), device="cuda")
    bl.tern_linear_fwd(layer.X, packed_only, layer.scale, Y)
    assert bl.tern_device_status() == bl.TERN_OK
    assert torch.equal(Y, layer.Y)
    Yr, Ya = oracle.fwd(inp.X, inp.q, inp.scale)
    check_close("Y (2-bit T)", Y.cpu().numpy(), Yr, Ya)


def test_grouped_forward_mixes_packed_and_bf16_layers(cuda_lib):
    bl = cuda_lib
    shapes = [(300, 256, 384), (64, 144, 272), (1000, 512, 512), (257, 128, 1008), (8, 64, 64)]
    layers = [Layer(syn.linear_inputs(M, K, N, seed=900 + i)).run() for i, (M, K, N) in enumerate(shapes)]
    outs = [torch.full_like(L.Y, float("nan")) for L in layers]
    Yb = [torch.empty(L.Y.shape, dtype=torch.bfloat16, device="cuda") for L in layers]
    dicts = []
    for i, (L, Y, B) in enumerate(zip(layers, outs, Yb)):
        tiles = bl.Tiles(L.K, L.N, packed=L.tiles.packed) if i % 2 == 0 else L.tiles
        dicts.append(dict(X=L.X, tiles=tiles, scale=L.scale, Y=Y, Y_bf16=B))
    bl.tern_linear_fwd_grouped(dicts)
    assert bl.tern_device_status() == bl.TERN_OK
    for L, Y, B in zip(layers, outs, Yb):
        assert torch.equal(Y, L.Y)
        assert torch.equal(B, L.Y.to(torch.bfloat16))


def test_forward_from_packed_codes_needs_n_multiple_of_64(cuda_lib):
    bl = cuda_lib
    inp = syn.linear_inputs(64, 64, 48, seed=5)
    layer = Layer(inp)
    bl.tern_materialize(layer.q, layer.scale, layer.tiles, 2, 7)
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_fwd(layer.X, bl.Tiles(64, 48, packed=layer.tiles.packed), layer.scale, layer.Y)
    assert e.value.status == bl.TERN_ERR_ALIGN


def test_grouped_materialize_matches_single_calls(cuda_lib):
    """Several weights in one tern_materialize_grouped call, with different sets of
    encodings (all planes; packed only; packed and hi/lo with the clamp written back):
    every output bit-equal to the oracle."""
    bl = cuda_lib
    shapes = [(512, 512), (129, 4112), (40, 80), (2048, 512), (1, 16)]
    ws, refs = [], []
    for i, (K, N) in enumerate(shapes):
        q = syn.int8_uniform(40 + i, 3, K * N, -128, 127).reshape(K, N)
        scale = syn.uniform_f32(40 + i, 4, N, -0.1, 0.1)
        refs.append((oracle.materialize(q, scale, 2, 7), q))
        if i % 3 == 0:
            tiles = bl.Tiles.empty(K, N)
        elif i % 3 == 1:
            tiles = bl.Tiles(K, N, packed=torch.zeros((K, N // 16), dtype=torch.int32, device="cuda"))
        else:
            tiles = bl.Tiles.empty(K, N, t=False)
        w = dict(q=dev(q), scale=dev(scale), tiles=tiles)
        if i % 3 == 2:
            w["q_clamped"] = torch.full((K, N), 99, dtype=torch.int8, device="cuda")
        ws.append(w)
    bl.tern_materialize_grouped(ws, 2, 7)
    torch.cuda.synchronize()
    for (ref, q), w in zip(refs, ws):
        t = w["tiles"]
        np.testing.assert_array_equal(t.packed.cpu().numpy().view(np.uint32), ref["packed"])
        if t.t_bf16 is not None:
            np.testing.assert_array_equal(host_bits(t.t_bf16), ref["t"])
        if t.whi_bf16 is not None:
            np.testing.assert_array_equal(host_bits(t.whi_bf16), ref["whi"])
            np.testing.assert_array_equal(host_bits(t.wlo_bf16), ref["wlo"])
        if "q_clamped" in w:
            np.testing.assert_array_equal(w["q_clamped"].cpu().numpy(), ref["qc"])
