"""Helpers shared by the GPU parity tests: host <-> device marshalling of the
seeded inputs and the element-wise tolerance check against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tern_synth as syn

# |gpu - oracle| <= REL * sum|term| of that output's dot product
REL = 1e-4


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_close(name, got, ref, ref_abs, rel=REL):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output (unwritten or overflow)"
    err = np.abs(got - ref)
    bound = rel * ref_abs
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} outside {rel}*sum|term|; worst at {i}: "
            f"gpu {got[i]!r} oracle {ref[i]!r} |err| {err[i]:.3e} bound {bound[i]:.3e}")
    return float((err / np.maximum(ref_abs, 1e-300)).max())


class Layer:
    """One layer's device buffers, filled from host inputs (seeded)."""

    def __init__(self, inp: syn.LinearInputs, theta=2, q_clamp=7, with_dx=True):
        import bit_linear_gb300 as bl
        self.bl = bl
        self.inp = inp
        M, K, N = inp.M, inp.K, inp.N
        self.M, self.K, self.N = M, K, N
        self.theta, self.q_clamp = theta, q_clamp
        self.X = dev_bf16(inp.X)
        self.dY = dev_bf16(inp.dY)
        self.q = dev(inp.q)
        self.scale = dev(inp.scale)
        self.tiles = bl.Tiles.empty(K, N, hi_lo=with_dx)
        nan = float("nan")
        self.Y = torch.full((M, N), nan, device="cuda")
        self.dX = torch.full((M, K), nan, device="cuda") if with_dx else None
        self.gq = torch.full((K, N), nan, device="cuda")
        self.sgrad = torch.full((N,), nan, device="cuda")
        self.ws = bl.workspace_for(M, K, N)
        self.ws.fill_(nan)

    def run(self):
        bl = self.bl
        bl.tern_materialize(self.q, self.scale, self.tiles, self.theta, self.q_clamp)
        bl.tern_linear_fwd(self.X, self.tiles, self.scale, self.Y)
        bl.tern_linear_bwd(self.X, self.dY, self.tiles, self.scale, self.dX, self.gq, self.sgrad, self.ws)
        assert bl.tern_device_status() == bl.TERN_OK
        return self


def full_oracle_check(layer: Layer, nthreads=0):
    inp = layer.inp
    Y, Ya = oracle.fwd(inp.X, inp.q, inp.scale, layer.theta, nthreads)
    worst = {"Y": check_close("Y", layer.Y.cpu().numpy(), Y, Ya)}
    if layer.dX is not None:
        dX, dXa = oracle.dx(inp.dY, inp.q, inp.scale, layer.theta, nthreads)
        worst["dX"] = check_close("dX", layer.dX.cpu().numpy(), dX, dXa)
    gq, gqa, sg, sga = oracle.dw(inp.X, inp.dY, inp.q, inp.scale, layer.theta, nthreads)
    worst["gq"] = check_close("gq", layer.gq.cpu().numpy(), gq, gqa)
    worst["sgrad"] = check_close("sgrad", layer.sgrad.cpu().numpy(), sg, sga)
    return worst


def sampled_oracle_check(layer: Layer, n=4096, ncols=64, seed=1234):
    """Entries the oracle can compute one by one, at any size."""
    inp = layer.inp
    M, K, N = inp.M, inp.K, inp.N
    rng = np.random.default_rng(seed)
    Yd, gqd, sgd = layer.Y.cpu().numpy(), layer.gq.cpu().numpy(), layer.sgrad.cpu().numpy()
    # Y[m,c]: always include the corners and the ragged edges
    ms = np.concatenate([[0, M - 1, 0, M - 1], rng.integers(0, M, n)])
    cs = np.concatenate([[0, 0, N - 1, N - 1], rng.integers(0, N, n)])
    ref = np.array([oracle.fwd_at(inp.X[m], inp.q[:, c], inp.scale[c], layer.theta) for m, c in zip(ms, cs)])
    check_close("Y(sampled)", Yd[ms, cs], ref[:, 0], ref[:, 1])
    if layer.dX is not None:
        dXd = layer.dX.cpu().numpy()
        rs = np.concatenate([[0, K - 1, 0, K - 1], rng.integers(0, K, n)])
        ref = np.array([oracle.dx_at(inp.dY[m], inp.q[r], inp.scale, layer.theta) for m, r in zip(ms, rs)])
        check_close("dX(sampled)", dXd[ms, rs], ref[:, 0], ref[:, 1])
    rs = np.concatenate([[0, K - 1, 0, K - 1], rng.integers(0, K, n)])
    Xt = np.ascontiguousarray(inp.X[:, np.unique(rs)].T)
    col_of = {r: i for i, r in enumerate(np.unique(rs))}
    dyc = {}
    for c in np.unique(cs):
        dyc[c] = np.ascontiguousarray(inp.dY[:, c])
    ref = np.array([oracle.gq_at(Xt[col_of[r]], dyc[c], inp.scale[c]) for r, c in zip(rs, cs)])
    check_close("gq(sampled)", gqd[rs, cs], ref[:, 0], ref[:, 1])
    cols = np.concatenate([[0, N - 1], rng.integers(0, N, ncols)])
    ref = np.array([oracle.sgrad_at(inp.X, np.ascontiguousarray(inp.dY[:, c]),
                                    np.ascontiguousarray(inp.q[:, c]), layer.theta) for c in cols])
    check_close("sgrad(sampled)", sgd[cols], ref[:, 0], ref[:, 1])
