"""GPU parity of the Q8_0 read (hc_read_q8) against the FP64 oracle.

Weights: the synthetic weight sets' float32 draws quantized to Q8_0 (blocks of
32 along the dot-product axis, one binary16 scale each).  Bar as for the BF16
read: max|gpu - oracle| <= 1e-4 * max|oracle| for lo, out and mean, R' bit for
bit, graph replays bit for bit equal to the direct call."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import EPS, TOL, bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

hc = pytest.importorskip("hyper_connection_residual_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def dev_q8(ws, dev):
    return dict(
        w_norm=torch.from_numpy(ws.w_norm).to(dev), gate=torch.from_numpy(ws.gate).to(dev),
        Wd_q=torch.from_numpy(ws.Wd_q).to(dev), Wd_scale=torch.from_numpy(ws.Wd_scale.view(np.int16)).to(dev),
        Wu_q=torch.from_numpy(ws.Wu_q).to(dev), Wu_scale=torch.from_numpy(ws.Wu_scale.view(np.int16)).to(dev))


@pytest.fixture(scope="module")
def g1(dev):
    g = synth.G1
    host = [synth.q8_weight_set(g, j) for j in range(2)]
    return g, host, [dev_q8(ws, dev) for ws in host]


@pytest.fixture(scope="module")
def rd(dev):
    r = hc.Read(4, 2560, 320, T_max=64, eps=EPS)
    yield r
    r.close()


def _outs(g, T, dev):
    return dict(out=torch.full((T, g.N), float("nan"), device=dev),
                mean=torch.full((T, g.d), float("nan"), device=dev),
                lo=torch.full((T, g.K), float("nan"), device=dev),
                r_out=torch.full((T, g.N), float("nan"), device=dev))


def _run(r, w, R, P, T, o, stream=None):
    r.q8(R, w["w_norm"], w["Wd_q"], w["Wd_scale"], w["Wu_q"], w["Wu_scale"], w["gate"], P, T,
         o["out"], o["mean"], o["lo"], r_out=o["r_out"], stream=stream)


def _oracle(orc, g, ws, R, P):
    return orc.read_q8(g.n, g.d, g.K, R=R, P=P, w_norm=ws.w_norm, Wd_q=ws.Wd_q, Wd_scale=ws.Wd_scale,
                       Wu_q=ws.Wu_q, Wu_scale=ws.Wu_scale, gate=ws.gate, eps=EPS)


def _check(o, ref, what):
    for name in ("lo", "out", "mean"):
        got = o[name].double().cpu().numpy()
        want = getattr(ref, name)
        err = float(np.max(np.abs(got - want)))
        bound = TOL * float(np.max(np.abs(want)))
        assert err <= bound, f"{what} {name}: max err {err:.3e} > {bound:.3e}"
    assert np.array_equal(o["r_out"].cpu().numpy().view(np.uint32), ref.r_out.view(np.uint32)), f"{what} R'"


@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 8])
def test_q8_parity(dev, orc, g1, rd, T, pending):
    g, host, w = g1
    for j in range(2):
        a = synth.activations(g, T, pending, s0=6000 + 10 * T + j)
        R = torch.from_numpy(a.R).to(dev)
        P = None if a.P is None else torch.from_numpy(a.P).to(dev)
        o = _outs(g, T, dev)
        _run(rd, w[j], R, P, T, o)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
        _check(o, _oracle(orc, g, host[j], a.R, a.P), f"T={T} set {j}")


@pytest.mark.parametrize("T", [9, 16])
def test_q8_eight_token_groups(dev, orc, g1, rd, T):
    g, host, w = g1
    a = synth.activations(g, T, True, s0=6100 + T)
    o = _outs(g, T, dev)
    _run(rd, w[0], torch.from_numpy(a.R).to(dev), torch.from_numpy(a.P).to(dev), T, o)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    _check(o, _oracle(orc, g, host[0], a.R, a.P), f"T={T}")


@pytest.mark.parametrize("T", [1, 4, 5, 8])
def test_q8_wide_geometry(dev, orc, T):
    g = synth.G2
    ws = synth.q8_weight_set(g, 0)
    w = dev_q8(ws, dev)
    a = synth.activations(g, T, True, s0=6200 + T)
    with hc.Read(4, 4096, 512, T_max=8, eps=EPS) as r:
        o = _outs(g, T, dev)
        _run(r, w, torch.from_numpy(a.R).to(dev), torch.from_numpy(a.P).to(dev), T, o)
        torch.cuda.synchronize()
        assert r.check() == hc.HC_OK
    _check(o, _oracle(orc, g, ws, a.R, a.P), f"d=4096 T={T}")


def test_q8_in_place_and_graph_replay(dev, g1, rd):
    """out = R (the residual updated in place) equals separate buffers; a captured
    graph replayed twice equals the direct call bit for bit."""
    g, _, w = g1
    T = 4
    a = synth.activations(g, T, True, s0=6300)
    R = torch.from_numpy(a.R).to(dev)
    P = torch.from_numpy(a.P).to(dev)
    o = _outs(g, T, dev)
    _run(rd, w[1], R, P, T, o)
    torch.cuda.synchronize()
    resid = R.clone()
    oi = _outs(g, T, dev)
    oi["out"] = resid
    _run(rd, w[1], resid, P, T, oi)
    torch.cuda.synchronize()
    assert np.array_equal(bits(resid), bits(o["out"]))
    assert np.array_equal(bits(oi["mean"]), bits(o["mean"])) and np.array_equal(bits(oi["lo"]), bits(o["lo"]))
    first = [bits(o[k]) for k in ("out", "mean", "lo")]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        _run(rd, w[1], R, P, T, o, stream=s)
        graph = hc.hc_graph_end(s)
    try:
        for _ in range(2):
            for t in o.values():
                t.fill_(float("nan"))
            torch.cuda.synchronize()
            hc.hc_graph_launch(graph, s)
            s.synchronize()
            assert all(np.array_equal(x, bits(o[k])) for x, k in zip(first, ("out", "mean", "lo")))
    finally:
        hc.hc_graph_destroy(graph)
    assert rd.check() == hc.HC_OK


def test_q8_argument_errors(dev, g1, rd):
    g, _, ws = g1
    w = ws[0]
    T = 1
    R = torch.zeros(T, g.N, device=dev)
    o = _outs(g, T, dev)
    lib = hc.load()

    def status(**over):
        args = dict(R=R.data_ptr(), w_norm=w["w_norm"].data_ptr(), Wd_q=w["Wd_q"].data_ptr(),
                    Wd_scale=w["Wd_scale"].data_ptr(), Wu_q=w["Wu_q"].data_ptr(),
                    Wu_scale=w["Wu_scale"].data_ptr(), gate=w["gate"].data_ptr(), P=None, T=T,
                    out=o["out"].data_ptr(), mean=o["mean"].data_ptr(), lo=o["lo"].data_ptr())
        args.update(over)
        return lib.hc_read_q8(rd.h, args["R"], args["w_norm"], args["Wd_q"], args["Wd_scale"], args["Wu_q"],
                              args["Wu_scale"], args["gate"], args["P"], args["T"], args["out"], args["mean"],
                              args["lo"], None, None, None)

    assert status() == hc.HC_OK
    assert status(Wd_q=w["Wd_q"].data_ptr() + 8) == hc.HC_ERR_ALIGN
    assert status(Wu_scale=w["Wu_scale"].data_ptr() + 1) == hc.HC_ERR_ALIGN
    assert status(Wd_scale=w["Wd_scale"].data_ptr() + 8) == hc.HC_ERR_ALIGN  # copied in 16-byte pieces
    assert status(Wd_scale=None) == hc.HC_ERR_ARG
    assert status(T=0) == hc.HC_ERR_ARG
    assert lib.hc_read_q8(None, *([None] * 8), 1, *([None] * 6)) == hc.HC_ERR_ARG
    torch.cuda.synchronize()


def _q8_read(w, R, P, o):
    return dict(R=R, P=P, out=o["out"], mean=o["mean"], lo=o["lo"], **w)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_q8_batch_on_lanes_equals_single_reads(dev, g1, rd, T):
    """Twelve independent Q8_0 reads as one batch run on the internal streams;
    every read's outputs equal hc_read_q8's bit for bit."""
    g, _, w = g1
    a = synth.activations(g, T, True, s0=6400 + T)
    R = torch.from_numpy(a.R).to(dev)
    P = torch.from_numpy(a.P).to(dev)
    outs = [_outs(g, T, dev) for _ in range(12)]
    reads = [_q8_read(w[j % 2], R, P if j % 3 else None, outs[j]) for j in range(12)]
    assert rd.batch_q8_plan(reads, T) >= 2
    rd.batch_q8(reads, T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j, r in enumerate(reads):
        o = _outs(g, T, dev)
        _run(rd, w[j % 2], R, r["P"], T, o)
        torch.cuda.synchronize()
        for k in ("out", "mean", "lo"):
            assert np.array_equal(bits(outs[j][k]), bits(o[k])), f"read {j} {k}"


def test_q8_chained_batch_runs_read_by_read(dev, orc, g1, rd):
    """Six chained Q8_0 reads (out of one is R of the next) are one group: the
    plan is read by read, and the last read matches the oracle's chain."""
    g, host, w = g1
    T = 3
    a = synth.activations(g, T, True, s0=6500)
    P = torch.from_numpy(a.P).to(dev)
    R0 = torch.from_numpy(a.R).to(dev)
    bufs = [_outs(g, T, dev) for _ in range(6)]
    reads, R = [], R0
    for j in range(6):
        reads.append(_q8_read(w[j % 2], R, P if j == 0 else None, bufs[j]))
        R = bufs[j]["out"]
    assert rd.batch_q8_plan(reads, T) == 0
    rd.batch_q8(reads, T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    x, p = a.R, a.P
    for j in range(6):
        ref = _oracle(orc, g, host[j % 2], x, p)
        got = bufs[j]["out"].double().cpu().numpy()
        assert np.max(np.abs(got - ref.out)) <= TOL * np.max(np.abs(ref.out)), f"read {j}"
        # the next read takes this read's GPU output as R (what it really read)
        x, p = bufs[j]["out"].cpu().numpy(), None


def test_q8_batch_graph_replay_and_mixed_weights(dev, g1, rd):
    g, _, w = g1
    T = 2
    a = synth.activations(g, T, False, s0=6600)
    R = torch.from_numpy(a.R).to(dev)
    outs = [_outs(g, T, dev) for _ in range(8)]
    reads = [_q8_read(w[j % 2], R, None, outs[j]) for j in range(8)]
    rd.batch_q8(reads, T)
    torch.cuda.synchronize()
    first = [bits(o["out"]) for o in outs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        rd.batch_q8(reads, T, stream=s)
        graph = hc.hc_graph_end(s)
    try:
        for _ in range(2):
            for o in outs:
                o["out"].fill_(float("nan"))
            torch.cuda.synchronize()
            hc.hc_graph_launch(graph, s)
            s.synchronize()
            assert all(np.array_equal(f, bits(o["out"])) for f, o in zip(first, outs))
    finally:
        hc.hc_graph_destroy(graph)
    # a descriptor without quants is rejected before anything is enqueued
    arr = hc._binding._q8_descs(rd.geometry, reads, T)
    arr[3].Wd_q = None
    assert hc.load().hc_read_batch_q8(rd.h, arr, 8, T, None) == hc.HC_ERR_ARG
    assert rd.check() == hc.HC_OK
