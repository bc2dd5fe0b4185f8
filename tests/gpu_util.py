"""Helpers of the GPU tests: device copies of synthetic inputs, one read
through the C ABI, and the parity bar."""

from __future__ import annotations

import numpy as np

import synth

TOL = 1e-4  # max|gpu - oracle| <= TOL * max|oracle|, per output tensor
EPS = 1e-6


def dev_weights(ws: synth.WeightSet, dev):
    import torch
    return dict(
        w_norm=torch.from_numpy(ws.w_norm).to(dev),
        gate=torch.from_numpy(ws.gate).to(dev),
        W_down=torch.from_numpy(ws.W_down.view(np.int16)).to(dev),
        W_up=torch.from_numpy(ws.W_up.view(np.int16)).to(dev),
    )


def dev_act(act: synth.Activations, dev):
    import torch
    return dict(R=torch.from_numpy(act.R).to(dev),
                P=None if act.P is None else torch.from_numpy(act.P).to(dev))


def outputs(g: synth.Geometry, T: int, dev):
    import torch
    return dict(out=torch.empty(T, g.N, device=dev), mean=torch.empty(T, g.d, device=dev),
                lo=torch.empty(T, g.K, device=dev), r_out=torch.empty(T, g.N, device=dev),
                rs=torch.empty(T, g.n, device=dev))


def run(rd, w, a, T, o, stream=None, r_out=True):
    rd(a["R"], w["w_norm"], w["W_down"], w["W_up"], w["gate"], a["P"], T,
       o["out"], o["mean"], o["lo"], r_out=o["r_out"] if r_out else None, rs=o["rs"],
       stream=stream)


def assert_parity(o, ref, T, what=""):
    """lo, out, mean within TOL of the largest oracle value; R' bit for bit."""
    for name, want in (("lo", ref.lo), ("out", ref.out), ("mean", ref.mean), ("rs", ref.rs)):
        got = o[name][:T].double().cpu().numpy()
        want = want[:T]
        err = float(np.max(np.abs(got - want)))
        bound = TOL * float(np.max(np.abs(want)))
        assert err <= bound, f"{what} {name}: max err {err:.3e} > {bound:.3e}"
    got_r = o["r_out"][:T].cpu().numpy()
    assert np.array_equal(got_r.view(np.uint32), ref.r_out[:T].view(np.uint32)), f"{what} R' bits"


def bits(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32).copy()
