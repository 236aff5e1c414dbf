"""SR4 q-update on the GPU against the oracle's reading (parity unpinned: the
page does not print the update's body; see the oracle).

The step scalar s must agree to 1 ulp (both sides sum in fp64 and round the
mean to fp32; only the summation order differs).  Every element whose value
y = x + u lies clear of an integer must take the oracle's step exactly; an
element within 1e-6 of an integer may round either way, and its result must
then be one of the two valid steps.
"""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import dev

pytestmark = pytest.mark.gpu


def _check(q0, gq, q_gpu, s_gpu, inv_bs, target, seed, idx_base, counter, clamp, dither):
    s_ref = oracle.sr4_scale(gq, inv_bs, target)
    assert np.float32(s_gpu) == np.float32(s_ref) or \
        abs(s_gpu - s_ref) <= np.spacing(np.float32(s_ref)), (s_gpu, s_ref)
    q_ref, y = oracle.sr4_update(q0, gq, s_ref, inv_bs, seed, idx_base, counter, clamp, dither)
    near = np.abs(y - np.round(y)) <= 1e-6 * np.maximum(1.0, np.abs(y))
    far = ~near
    np.testing.assert_array_equal(q_gpu[far], q_ref[far])
    if near.any():
        lo = np.clip(q0[near].astype(int) - np.floor(y[near]).astype(int), -clamp, clamp)
        hi = np.clip(q0[near].astype(int) - np.floor(y[near]).astype(int) + 1, -clamp, clamp)
        lo2 = np.clip(q0[near].astype(int) - np.floor(y[near]).astype(int) - 1, -clamp, clamp)
        got = q_gpu[near].astype(int)
        assert np.all((got == lo) | (got == hi) | (got == lo2))


@pytest.mark.parametrize("n", [1, 15, 16, 17, 4099, 1 << 20])
@pytest.mark.parametrize("dither", [True, False])
def test_sr4_matches_oracle(cuda_lib, n, dither):
    bl = cuda_lib
    q0 = syn.int8_uniform(3, syn.TID_Q, n, -7, 7)
    gq = syn.normal_f32(3, syn.TID_G, n, 0.0, 1e-3)
    q = dev(q0)
    s = torch.zeros(1, device="cuda")
    ws = torch.empty(bl.tern_sr4_workspace(n) // 4 + 4, dtype=torch.float32, device="cuda")
    bl.tern_sr4_step(q, dev(gq), ws, inv_bs=0.5, target_step=0.05, seed=42, idx_base=1000, counter=7,
                     q_clamp=7, use_dither=dither, s_out=s)
    torch.cuda.synchronize()
    _check(q0, gq, q.cpu().numpy(), float(s.item()), 0.5, 0.05, 42, 1000, 7, 7, dither)


def test_sr4_on_a_layer_gradient_over_steps(cuda_lib):
    """gq from the G GEMM of a layer, then several SR4 steps (counter = step)."""
    from _parity import Layer
    bl = cuda_lib
    inp = syn.linear_inputs(512, 256, 384, seed=11)
    layer = Layer(inp).run()
    gq = layer.gq.cpu().numpy().ravel()
    q = layer.q.clone()
    ws = torch.empty(bl.tern_sr4_workspace(q.numel()) // 4 + 4, dtype=torch.float32, device="cuda")
    s = torch.zeros(1, device="cuda")
    q_host = inp.q.ravel().copy()
    for step in range(4):
        bl.tern_sr4_step(q, layer.gq, ws, inv_bs=1.0, target_step=0.5, seed=42, idx_base=77, counter=step,
                         q_clamp=7, use_dither=True, s_out=s)
        torch.cuda.synchronize()
        q_gpu = q.cpu().numpy().ravel()
        _check(q_host, gq, q_gpu, float(s.item()), 1.0, 0.5, 42, 77, step, 7, True)
        q_host = q_gpu.copy()
    assert np.abs(q_host.astype(int)).max() <= 7


def test_sr4_zero_gradient_leaves_q(cuda_lib):
    bl = cuda_lib
    n = 10000
    q0 = syn.int8_uniform(4, syn.TID_Q, n, -7, 7)
    q = dev(q0)
    ws = torch.empty(bl.tern_sr4_workspace(n) // 4 + 4, dtype=torch.float32, device="cuda")
    s = torch.full((1,), 7.0, device="cuda")
    bl.tern_sr4_step(q, torch.zeros(n, device="cuda"), ws, s_out=s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), q0)
    assert s.item() == 0.0


@pytest.mark.parametrize("K,N,theta,clamp", [(64, 48, 2, 7), (1000, 1008, 2, 7), (300, 512, 3, 127)])
def test_panel_matches_oracle(cuda_lib, K, N, theta, clamp):
    bl = cuda_lib
    q_prev = syn.int8_uniform(12, syn.TID_Q, K * N, -128, 127).reshape(K, N)
    q = syn.int8_uniform(13, syn.TID_Q, K * N, -128, 127).reshape(K, N)
    q[: K // 2] = q_prev[: K // 2]                     # half the rows unchanged
    scale = syn.uniform_f32(12, syn.TID_SCALE, N, -0.05, 0.1)
    prev_tiles = bl.Tiles(K, N, packed=torch.empty((K, N // 16), dtype=torch.int32, device="cuda"))
    bl.tern_materialize(dev(q_prev), None, prev_tiles, theta, clamp)
    counts = torch.full((6,), -1, dtype=torch.int64, device="cuda")
    stats = torch.zeros(3, dtype=torch.float64, device="cuda")
    bl.tern_sr4_panel(dev(q), dev(scale), counts, stats, packed_prev=prev_tiles.packed, theta=theta, q_clamp=clamp)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.sr4_panel(q, scale, q_prev, theta, clamp)
    np.testing.assert_array_equal(counts.cpu().numpy().astype(np.uint64), ref_c)
    got = stats.cpu().numpy()
    assert got[0] == ref_s[0] and got[2] == ref_s[2]
    assert abs(got[1] - ref_s[1]) <= 1e-12 * abs(ref_s[1]) + 1e-18
    bl.tern_sr4_panel(dev(q), dev(scale), counts, stats, theta=theta, q_clamp=clamp)   # no previous tiles
    torch.cuda.synchronize()
    assert counts[5].item() == 0
