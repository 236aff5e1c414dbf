"""dX with W_hi / W_lo expanded from the 2-bit codes inside the GEMM (tiles without the
hi/lo planes): the converter warps write the bits tern_materialize would have written,
so dX is bit-equal to the call that reads the planes, and within the oracle's tolerance."""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import check_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def _dx_both(bl, inp, theta=2, clamp=7, with_dw=True):
    M, K, N = inp.M, inp.K, inp.N
    X, dY, q, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.q), dev(inp.scale)
    planes = bl.Tiles.empty(K, N, t=False)
    bl.tern_materialize(q, scale, planes, theta, clamp)
    codes = bl.Tiles(K, N, packed=planes.packed)   # the same 2-bit tiles, no hi/lo planes
    nan = float("nan")
    out = []
    for tiles in (planes, codes):
        dX = torch.full((M, K), nan, device="cuda")
        gq = torch.full((K, N), nan, device="cuda") if with_dw else None
        sg = torch.full((N,), nan, device="cuda") if with_dw else None
        ws = torch.full((max(bl.tern_linear_bwd_workspace(M, K, N) // 4, N),), nan, device="cuda")
        bl.tern_linear_bwd(X, dY, tiles, scale, dX, gq, sg, ws)
        torch.cuda.synchronize()
        assert bl.tern_device_status() == bl.TERN_OK
        out.append((dX, gq, sg))
    return out


@pytest.mark.parametrize("M,K,N", [(64, 128, 128), (130, 144, 320), (300, 528, 64), (257, 64, 768),
                                   (100, 272, 1024), (1000, 512, 2048), (8192, 2048, 512)])
def test_dx_from_codes_equals_the_planes(cuda_lib, M, K, N):
    inp = syn.linear_inputs(M, K, N, seed=M + K + 3 * N)
    (dX0, gq0, sg0), (dX1, gq1, sg1) = _dx_both(cuda_lib, inp)
    assert torch.equal(dX0, dX1)
    assert torch.equal(gq0, gq1) and torch.equal(sg0, sg1)   # G shares the workspace with the s_hi/s_lo table
    if M * K * N <= 1 << 28:
        ref, refa = oracle.dx(inp.dY, inp.q, inp.scale)
        check_close("dX(codes)", dX1.cpu().numpy(), ref, refa)


def test_dx_from_codes_negative_zero_and_exact_scales(cuda_lib):
    inp = syn.linear_inputs(200, 160, 384, seed=31, scale_lo=-0.1, scale_hi=0.1)
    s = inp.scale.copy()
    s[::7] = 0.0
    s[1::7] = 1.0          # exact in bf16: s_lo = 0 (a -1 weight gives -0)
    s[2::7] = -2.0 ** -140
    inp.scale = s
    (dX0, _, _), (dX1, _, _) = _dx_both(cuda_lib, inp, with_dw=False)
    assert torch.equal(dX0.view(torch.int32), dX1.view(torch.int32))


def test_dx_from_codes_large_shape_sampled(cuda_lib):
    c = syn.LARGE
    inp = syn.linear_inputs(c["M"], c["K"], c["N"], seed=0, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"])
    (dX0, _, _), (dX1, _, _) = _dx_both(cuda_lib, inp, with_dw=False)
    assert torch.equal(dX0, dX1)


def test_dx_from_codes_needs_n_multiple_of_64_and_a_workspace(cuda_lib):
    bl = cuda_lib
    M, K, N = 64, 64, 48
    inp = syn.linear_inputs(M, K, N, seed=32)
    X, dY, q, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.q), dev(inp.scale)
    codes = bl.Tiles(K, N, packed=torch.empty((K, N // 16), dtype=torch.int32, device="cuda"))
    bl.tern_materialize(q, scale, codes, 2, 7)
    dX = torch.empty((M, K), device="cuda")
    ws = torch.empty((1024,), device="cuda")
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd(X, dY, codes, scale, dX, None, None, ws)
    assert e.value.status == bl.TERN_ERR_ALIGN
    N = 64
    inp = syn.linear_inputs(M, K, N, seed=33)
    X, dY, q, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.q), dev(inp.scale)
    codes = bl.Tiles(K, N, packed=torch.empty((K, N // 16), dtype=torch.int32, device="cuda"))
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd(X, dY, codes, scale, dX, None, None, None)
    assert e.value.status == bl.TERN_ERR_WORKSPACE
