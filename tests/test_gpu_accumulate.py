"""Micro-batch gradient accumulation (TERN_BWD_ACCUMULATE): gq and sgrad summed
over B backward calls equal the oracle's gq and sgrad of the concatenated
batch (G is a sum over tokens)."""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import check_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Ms,K,N", [((100, 77, 200), 256, 384), ((64, 64), 144, 272), ((1, 2, 3, 300), 512, 128)])
def test_accumulated_backward_equals_the_whole_batch(cuda_lib, Ms, K, N):
    bl = cuda_lib
    parts = [syn.linear_inputs(m, K, N, seed=100 + i) for i, m in enumerate(Ms)]
    q, scale = parts[0].q, parts[0].scale           # one weight for every micro-batch
    tiles = bl.Tiles.empty(K, N)
    bl.tern_materialize(dev(q), dev(scale), tiles, 2, 7)
    gq = torch.full((K, N), float("nan"), device="cuda")
    sgrad = torch.full((N,), float("nan"), device="cuda")
    for i, p in enumerate(parts):
        ws = bl.workspace_for(p.M, K, N)
        dX = torch.empty(p.M, K, device="cuda")
        bl.tern_linear_bwd(dev_bf16(p.X), dev_bf16(p.dY), tiles, dev(scale), dX, gq, sgrad, ws,
                           accumulate=i > 0)
    torch.cuda.synchronize()
    X = np.concatenate([p.X for p in parts])
    dY = np.concatenate([p.dY for p in parts])
    g_ref, g_abs, s_ref, s_abs = oracle.dw(X, dY, q, scale)
    check_close("gq", gq.cpu().numpy(), g_ref, g_abs)
    check_close("sgrad", sgrad.cpu().numpy(), s_ref, s_abs)


def test_unknown_flags_are_rejected(cuda_lib):
    import ctypes
    bl = cuda_lib
    p = syn.linear_inputs(64, 64, 64, seed=1)
    tiles = bl.Tiles.empty(64, 64)
    ct = tiles._c()
    X, dY = dev_bf16(p.X), dev_bf16(p.dY)
    sc = dev(p.scale)
    gq = torch.empty(64, 64, device="cuda")
    st = bl.lib.tern_linear_bwd_ex(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(dY.data_ptr()),
                                   ctypes.byref(ct), ctypes.c_void_p(sc.data_ptr()), None,
                                   ctypes.c_void_p(gq.data_ptr()), None, None, 0, 64, 64, 64, 6, None)
    assert st == bl.TERN_ERR_ARG
