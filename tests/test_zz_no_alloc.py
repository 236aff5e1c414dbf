"""tern_linear_bwd_noalloc: the backward for callers that cannot allocate
device memory (a plugin whose host program owns every device allocation, a
loop that must not pay cudaMalloc's synchronisation).  Its sgrad partials live
in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against tern_linear_bwd (which takes a workspace)
on two calls in a row with different shapes, so the second call runs over the
scratch the first one left behind; and the size limit is checked.  This file
is collected last so a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import REL, Layer

pytestmark = pytest.mark.gpu


def _within(name, a, b, ab):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    err = np.abs(a - b)
    assert np.all(err <= REL * ab), f"{name}: worst |noalloc - workspace| / sum|term| = {(err / ab).max():.3e}"


@pytest.mark.parametrize("first,second", [((300, 528, 400), (130, 144, 272))])
def test_noalloc_matches_workspace_entry_point(cuda_lib, first, second):
    bl = cuda_lib
    for M, K, N in (first, second):
        inp = syn.linear_inputs(M, K, N, seed=M * 7 + K + N)
        ref = Layer(inp).run()                  # tern_linear_bwd with a caller workspace
        nan = float("nan")
        dX = torch.full((M, K), nan, device="cuda")
        gq = torch.full((K, N), nan, device="cuda")
        sgrad = torch.full((N,), nan, device="cuda")
        bl.tern_linear_bwd_noalloc(ref.X, ref.dY, ref.tiles, ref.scale, dX, gq, sgrad)
        assert bl.tern_device_status() == bl.TERN_OK
        _, dXa = oracle.dx(inp.dY, inp.q, inp.scale)
        _, gqa, _, sga = oracle.dw(inp.X, inp.dY, inp.q, inp.scale)
        _within("dX", dX, ref.dX, dXa)
        _within("gq", gq, ref.gq, gqa)
        _within("sgrad", sgrad, ref.sgrad, sga)


def test_noalloc_calls_back_to_back_on_one_stream(cuda_lib):
    """Two no-workspace calls of different shapes enqueued on one stream with no
    synchronisation between them (the second reuses the built-in scratch while the
    first call's kernels may still be finishing), then both compared with the
    workspace entry point."""
    bl = cuda_lib
    shapes = [(300, 528, 400), (517, 400, 528)]
    inps = [syn.linear_inputs(M, K, N, seed=M * 5 + K + N) for M, K, N in shapes]
    refs = [Layer(inp).run() for inp in inps]     # tern_linear_bwd with a caller workspace
    nan = float("nan")
    outs = []
    for (M, K, N), ref in zip(shapes, refs):
        o = (torch.full((M, K), nan, device="cuda"), torch.full((K, N), nan, device="cuda"),
             torch.full((N,), nan, device="cuda"))
        outs.append(o)
    torch.cuda.synchronize()
    for ref, (dX, gq, sgrad) in zip(refs, outs):
        bl.tern_linear_bwd_noalloc(ref.X, ref.dY, ref.tiles, ref.scale, dX, gq, sgrad)
    assert bl.tern_device_status() == bl.TERN_OK
    for inp, ref, (dX, gq, sgrad) in zip(inps, refs, outs):
        _, dXa = oracle.dx(inp.dY, inp.q, inp.scale)
        _, gqa, _, sga = oracle.dw(inp.X, inp.dY, inp.q, inp.scale)
        _within("dX", dX, ref.dX, dXa)
        _within("gq", gq, ref.gq, gqa)
        _within("sgrad", sgrad, ref.sgrad, sga)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    bl = cuda_lib
    K, N = 4096, 16400          # ceil(K/128) * 4 * N = 2,099,200 partials > 2^21
    assert bl.tern_linear_bwd_workspace(1, K, N) > bl.TERN_NOALLOC_SCRATCH_BYTES
    X = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    dY = torch.zeros((1, N), dtype=torch.bfloat16, device="cuda")
    tiles = bl.Tiles(K, N, packed=torch.zeros((K, N // 16), dtype=torch.int32, device="cuda"))
    scale = torch.ones(N, device="cuda")
    sgrad = torch.full((N,), 7.0, device="cuda")
    with pytest.raises(bl.TernError) as e:
        bl.tern_linear_bwd_noalloc(X, dY, tiles, scale, None, None, sgrad)
    assert e.value.status == bl.TERN_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(sgrad == 7.0)      # nothing was enqueued
