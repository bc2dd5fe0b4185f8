"""The read without a handle or any device allocation (hc_read_noalloc).

Some callers cannot call cudaMalloc when they run the read: an engine that
reserved nearly all of HBM for weights and KV cache at start-up, code running
inside another framework's allocator, or a path that cannot pay for
cudaMalloc's device-wide synchronisation.  hc_read_noalloc serves them with a
fixed scratch array built into the library.  This test calls it through the C
ABI twice in a row and checks each result against the handle-based hc_read on
the same inputs, within the parity tolerance of the other GPU tests.  The file
name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest

import synth
from gpu_util import EPS, TOL, dev_act, dev_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

hc = pytest.importorskip("hyper_connection_residual_gb300")


def _outs(g, T, dev):
    return (torch.full((T, g.N), float("nan"), device=dev),
            torch.full((T, g.d), float("nan"), device=dev),
            torch.full((T, g.K), float("nan"), device=dev))


def _close(got, want, name):
    got = got.double().cpu().numpy()
    want = want.double().cpu().numpy()
    err = float(np.max(np.abs(got - want)))
    bound = TOL * float(np.max(np.abs(want)))
    assert err <= bound, f"{name}: max err {err:.3e} > {bound:.3e}"


def test_noalloc_matches_handle_read_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib = hc.load()
    g = synth.G1
    cases = [(synth.weight_set(g, 3), 4, True, 41), (synth.weight_set(g, 4), 8, False, 42)]
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
        for ws, T, pending, seed in cases:  # two calls in a row
            w = dev_weights(ws, dev)
            a = dev_act(synth.activations(g, T, pending, s0=seed), dev)
            ref = _outs(g, T, dev)
            rd(a["R"], w["w_norm"], w["W_down"], w["W_up"], w["gate"], a["P"], T, *ref)
            got = _outs(g, T, dev)
            p = [a["R"].data_ptr(), w["w_norm"].data_ptr(), w["W_down"].data_ptr(),
                 w["W_up"].data_ptr(), w["gate"].data_ptr(),
                 a["P"].data_ptr() if a["P"] is not None else None]
            status = lib.hc_read_noalloc(g.n, g.d, g.K, ctypes.c_float(EPS), *p, T,
                                         *[t.data_ptr() for t in got],
                                         torch.cuda.current_stream().cuda_stream or None)
            assert status == hc.HC_OK, hc.status_str(status)
            torch.cuda.synchronize()
            for name, x, y in zip(("out", "mean", "lo"), got, ref):
                _close(x, y, f"T={T} {name}")


NOALLOC_CASES = [(synth.G1, 1), (synth.G1, 4), (synth.G1, 8), (synth.G2, 1), (synth.G2, 5), (synth.G2, 8)]


@pytest.mark.parametrize("g,T", NOALLOC_CASES, ids=[f"d{g.d}_T{T}" for g, T in NOALLOC_CASES])
def test_noalloc_matches_oracle_twice(g, T):
    """Two calls in a row (the second over other inputs, pending write on),
    each against the FP64 oracle at the parity bar: the CUDA-core kernels at
    T = 1, the tensor-core ones above, and d = 4096, K = 512, whose partial
    sums fill the whole fixed array at T = 8.  The first call goes through the
    Python wrapper, the second through the C ABI.  hc_read_noalloc_check then
    reports that no bounded wait ran out."""
    import oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib = hc.load()
    for call, (j, pending) in enumerate(((5, False), (6, True))):
        ws = synth.weight_set(g, j)
        act = synth.activations(g, T, pending, s0=60 + 7 * j + T)
        w = dev_weights(ws, dev)
        a = dev_act(act, dev)
        got = _outs(g, T, dev)
        if call == 0:
            hc.hc_read_noalloc((g.n, g.d, g.K), EPS, a["R"], w["w_norm"], w["W_down"], w["W_up"], w["gate"],
                               a["P"], T, *got)
        else:
            p = [a["R"].data_ptr(), w["w_norm"].data_ptr(), w["W_down"].data_ptr(), w["W_up"].data_ptr(),
                 w["gate"].data_ptr(), a["P"].data_ptr() if a["P"] is not None else None]
            status = lib.hc_read_noalloc(g.n, g.d, g.K, ctypes.c_float(EPS), *p, T,
                                         *[t.data_ptr() for t in got],
                                         torch.cuda.current_stream().cuda_stream or None)
            assert status == hc.HC_OK, hc.status_str(status)
        torch.cuda.synchronize()
        ref = oracle.default().read(g.n, g.d, g.K, R=act.R, P=act.P, w_norm=ws.w_norm, W_down=ws.W_down,
                                    W_up=ws.W_up, gate=ws.gate, eps=EPS)
        for name, x, want in zip(("out", "mean", "lo"), got, (ref.out, ref.mean, ref.lo)):
            err = float(np.max(np.abs(x.double().cpu().numpy() - want)))
            bound = TOL * float(np.max(np.abs(want)))
            assert err <= bound, f"d={g.d} T={T} call {call} {name}: max err {err:.3e} > {bound:.3e}"
    assert hc.hc_read_noalloc_check() == hc.HC_OK


def test_noalloc_rejects_t_above_its_maximum():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = hc.load()
    T = hc.HC_NOALLOC_MAX_T + 1
    status = lib.hc_read_noalloc(4, 2560, 320, ctypes.c_float(EPS), *([16] * 5), None, T,
                                 16, 16, 16, None)
    assert status == hc.HC_ERR_TOO_LARGE
    assert "maximum" in hc.status_str(status)
