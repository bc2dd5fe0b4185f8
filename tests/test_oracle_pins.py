"""The FP64 oracle against its pins (no GPU)."""

import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_numpy_cross_check(orc):
    """Supplementary: the same formulas through NumPy float64 matmuls agree at
    the real geometry.  (Not a pin: it restates the definition.)"""
    import synth
    g = synth.G1
    ws = synth.weight_set(g, 0)
    act = synth.activations(g, 2, True)
    res = orc.read(g.n, g.d, g.K, R=act.R, P=act.P, w_norm=ws.w_norm, W_down=ws.W_down,
                   W_up=ws.W_up, gate=ws.gate, eps=1e-6)
    rp = (act.R + act.P).astype(np.float64)
    ss = (rp.reshape(2, g.n, g.d) ** 2).sum(-1)
    rs = 1.0 / np.sqrt(ss / g.d + 1e-6)
    x = rp * ws.w_norm.astype(np.float64)
    Wd = synth.bf16_to_f32(ws.W_down).astype(np.float64)
    Wu = synth.bf16_to_f32(ws.W_up).astype(np.float64)
    lo = sum(rs[:, s:s + 1] * (x[:, s * g.d:(s + 1) * g.d] @ Wd[:, s * g.d:(s + 1) * g.d].T)
             for s in range(g.n))
    u = lo @ Wu.T
    out = rp + u / (1.0 + np.exp(-ws.gate.astype(np.float64)))
    mean = out.reshape(2, g.n, g.d).mean(1)
    for name, want in (("lo", lo), ("u", u), ("out", out), ("mean", mean), ("rs", rs)):
        got = getattr(res, name)
        assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want)), name


def test_q2_numpy_cross_check(orc):
    """Supplementary: the Q2_0 product through a dense NumPy float64 matrix
    (codes unpacked with np.unpackbits) agrees with the oracle.  (Not a pin:
    it restates the definition.)"""
    import synth
    rows, cols, ncols = 1024, 2560, 4
    m = synth.q2_0_matrix(rows, cols, j=3)
    x = synth.q2_0_columns(cols, ncols, j=3)
    bits = np.unpackbits(m.Wq[..., None], axis=-1, bitorder="little").reshape(rows, cols, 2)
    codes = bits[..., 0].astype(np.int64) + 2 * bits[..., 1]
    scale = m.Wscale.view(np.float16).astype(np.float64)
    W = (codes - 2) * np.repeat(scale, 64, axis=1)
    want = x.astype(np.float64) @ W.T
    got = orc.q2_0_matvec(m.Wq, m.Wscale, x)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))
