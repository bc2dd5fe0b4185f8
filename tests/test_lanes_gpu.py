"""GPU checks of hc_read_batch on the handle's internal streams (batches
whose reads fall into two or more groups that share no memory).

The reads there are the two kernels of hc_read with the same arguments, so
every read's out, mean and lo must equal a direct hc_read of the same inputs
bit for bit; sampled reads are also held to the oracle bar (max|gpu -
oracle| <= 1e-4 * max|oracle|).  Covered: independent reads at T = 1..8 with
the pending write off and on, two chains in one batch, reads in place, the
scaled-up geometry, graph capture and replay, and the order against work on
the caller's stream before and after the batch."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import EPS, TOL, bits, dev_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

hc = pytest.importorskip("hyper_connection_residual_gb300")

NREADS = 24


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


@pytest.fixture(scope="module")
def sets(dev):
    g = synth.G1
    host = [synth.weight_set(g, 30 + j) for j in range(4)]
    return g, host, [dev_weights(ws, dev) for ws in host]


@pytest.fixture(scope="module")
def rd(dev):
    r = hc.Read(4, 2560, 320, T_max=8, eps=EPS)
    yield r
    r.close()


@pytest.fixture(scope="module")
def ref(dev):
    """A second handle for the direct reads the batches are compared with."""
    r = hc.Read(4, 2560, 320, T_max=8, eps=EPS)
    yield r
    r.close()


def _outs(g, T, dev):
    return dict(out=torch.full((T, g.N), float("nan"), device=dev),
                mean=torch.full((T, g.d), float("nan"), device=dev),
                lo=torch.full((T, g.K), float("nan"), device=dev))


def _desc(w, R, P, o):
    return dict(R=R, P=P, w_norm=w["w_norm"], W_down=w["W_down"], W_up=w["W_up"], gate=w["gate"],
                out=o["out"], mean=o["mean"], lo=o["lo"])


def _direct(r, d, T):
    o = {k: torch.full_like(d[k], float("nan")) for k in ("out", "mean", "lo")}
    r(d["R"], d["w_norm"], d["W_down"], d["W_up"], d["gate"], d["P"], T, o["out"], o["mean"], o["lo"])
    return o


def _same_bits(got, want, what):
    for k in ("out", "mean", "lo"):
        assert np.array_equal(bits(got[k]), bits(want[k])), f"{what} {k}"


def _close(o, res, what):
    for name, want in (("lo", res.lo), ("out", res.out), ("mean", res.mean)):
        got = o[name].double().cpu().numpy()
        err = float(np.max(np.abs(got - want)))
        bound = TOL * float(np.max(np.abs(want)))
        assert err <= bound, f"{what} {name}: max err {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 8])
def test_independent_reads_on_lanes(dev, orc, sets, rd, ref, T, pending):
    g, host, w = sets
    acts = [synth.activations(g, T, pending, s0=3000 + 50 * T + j) for j in range(NREADS)]
    R = [torch.from_numpy(a.R).to(dev) for a in acts]
    P = [None if a.P is None else torch.from_numpy(a.P).to(dev) for a in acts]
    o = [_outs(g, T, dev) for _ in range(NREADS)]
    descs = [_desc(w[j % 4], R[j], P[j], o[j]) for j in range(NREADS)]
    assert rd.batch_plan(descs, T) == 6
    rd.batch(descs, T)
    want = [_direct(ref, d, T) for d in descs]
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK and ref.check() == hc.HC_OK
    for j in range(NREADS):
        _same_bits(o[j], want[j], f"T={T} read {j}")
    for j in (0, NREADS - 1):
        res = orc.read(g.n, g.d, g.K, R=acts[j].R, P=acts[j].P, w_norm=host[j % 4].w_norm,
                       W_down=host[j % 4].W_down, W_up=host[j % 4].W_up, gate=host[j % 4].gate, eps=EPS)
        _close(o[j], res, f"T={T} read {j}")


def test_two_chains(dev, sets, rd, ref):
    """Reads 0..5 chain one residual, reads 6..11 another: two groups, each
    run in order on its own stream."""
    g, _, w = sets
    T, L = 4, 6
    a = [synth.activations(g, T, c == 1, s0=3500 + c) for c in range(2)]
    R0 = [torch.from_numpy(x.R).to(dev) for x in a]
    P1 = torch.from_numpy(a[1].P).to(dev)
    o = [_outs(g, T, dev) for _ in range(2 * L)]
    descs = []
    for c in range(2):
        for i in range(L):
            j = c * L + i
            R = R0[c] if i == 0 else o[j - 1]["out"]
            descs.append(_desc(w[j % 4], R, P1 if c == 1 else None, o[j]))
    assert hc.hc_read_batch_groups((4, 2560, 320), descs, T) == [0] * L + [1] * L
    assert rd.batch_plan(descs, T) == 2
    rd.batch(descs, T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in range(2 * L):
        x = _direct(ref, descs[j], T)
        torch.cuda.synchronize()
        _same_bits(o[j], x, f"read {j}")


def test_reads_in_place(dev, sets, rd, ref):
    """out = R for every read (one residual buffer per read, updated in place)."""
    g, _, w = sets
    T = 3
    acts = [synth.activations(g, T, True, s0=3600 + j) for j in range(8)]
    R = [torch.from_numpy(x.R).to(dev) for x in acts]
    P = [torch.from_numpy(x.P).to(dev) for x in acts]
    want = [_direct(ref, _desc(w[j % 4], R[j], P[j], _outs(g, T, dev)), T) for j in range(8)]
    o = [_outs(g, T, dev) for _ in range(8)]
    descs = [_desc(w[j % 4], R[j], P[j], dict(o[j], out=R[j])) for j in range(8)]
    assert rd.batch_plan(descs, T) == 6
    rd.batch(descs, T)
    torch.cuda.synchronize()
    for j in range(8):
        _same_bits(dict(o[j], out=R[j]), want[j], f"in place read {j}")


def test_order_against_the_callers_stream(dev, sets, rd, ref):
    """A read on the caller's stream before the batch feeds one of its reads;
    a read after the batch takes another's output."""
    g, _, w = sets
    T = 2
    acts = [synth.activations(g, T, False, s0=3700 + j) for j in range(7)]
    R = [torch.from_numpy(x.R).to(dev) for x in acts]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    first = _outs(g, T, dev)
    o = [_outs(g, T, dev) for _ in range(6)]
    after = _outs(g, T, dev)
    with torch.cuda.stream(s):
        rd(R[0], w[0]["w_norm"], w[0]["W_down"], w[0]["W_up"], w[0]["gate"], None, T,
           first["out"], first["mean"], first["lo"], stream=s)
        descs = [_desc(w[(j + 1) % 4], first["out"] if j == 3 else R[j + 1], None, o[j]) for j in range(6)]
        rd.batch(descs, T, stream=s)
        rd(o[5]["out"], w[2]["w_norm"], w[2]["W_down"], w[2]["W_up"], w[2]["gate"], None, T,
           after["out"], after["mean"], after["lo"], stream=s)
    s.synchronize()
    w_first = _direct(ref, _desc(w[0], R[0], None, _outs(g, T, dev)), T)
    torch.cuda.synchronize()
    _same_bits(first, w_first, "before")
    for j in range(6):
        x = _direct(ref, descs[j], T)
        torch.cuda.synchronize()
        _same_bits(o[j], x, f"batch read {j}")
    x = _direct(ref, _desc(w[2], o[5]["out"], None, after), T)
    torch.cuda.synchronize()
    _same_bits(after, x, "after")


def test_graph_capture_and_replay_bitwise(dev, sets, rd):
    g, _, w = sets
    T = 4
    acts = [synth.activations(g, T, True, s0=3800 + j) for j in range(NREADS)]
    R = [torch.from_numpy(x.R).to(dev) for x in acts]
    P = [torch.from_numpy(x.P).to(dev) for x in acts]
    o = [_outs(g, T, dev) for _ in range(NREADS)]
    descs = [_desc(w[j % 4], R[j], P[j], o[j]) for j in range(NREADS)]

    def snap():
        return [bits(o[j][k]) for j in range(NREADS) for k in ("out", "mean", "lo")]

    def clear():
        for x in o:
            for t in x.values():
                t.fill_(float("nan"))

    rd.batch(descs, T)
    torch.cuda.synchronize()
    first = snap()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        rd.batch(descs, T, stream=s)
        graph = hc.hc_graph_end(s)
    try:
        for _ in range(3):
            clear()
            torch.cuda.synchronize()
            hc.hc_graph_launch(graph, s)
            s.synchronize()
            assert all(np.array_equal(x, y) for x, y in zip(first, snap())), "graph replay"
    finally:
        hc.hc_graph_destroy(graph)
    assert rd.check() == hc.HC_OK


def test_scaled_geometry_on_lanes(dev, orc):
    g = synth.G2
    host = [synth.weight_set(g, j) for j in range(2)]
    w = [dev_weights(x, dev) for x in host]
    T = 3
    acts = [synth.activations(g, T, True, s0=3900 + j) for j in range(6)]
    R = [torch.from_numpy(x.R).to(dev) for x in acts]
    P = [torch.from_numpy(x.P).to(dev) for x in acts]
    with hc.Read(4, 4096, 512, T_max=4, eps=EPS) as r, hc.Read(4, 4096, 512, T_max=4, eps=EPS) as r2:
        o = [_outs(g, T, dev) for _ in range(6)]
        descs = [_desc(w[j % 2], R[j], P[j], o[j]) for j in range(6)]
        assert r.batch_plan(descs, T) == 6
        r.batch(descs, T)
        want = [_direct(r2, d, T) for d in descs]
        torch.cuda.synchronize()
        assert r.check() == hc.HC_OK
        for j in range(6):
            _same_bits(o[j], want[j], f"G2 read {j}")
    res = orc.read(g.n, g.d, g.K, R=acts[5].R, P=acts[5].P, w_norm=host[1].w_norm, W_down=host[1].W_down,
                   W_up=host[1].W_up, gate=host[1].gate, eps=EPS)
    _close(o[5], res, "G2 read 5")


def test_lane_limit(dev, sets, rd):
    g, _, w = sets
    T = 1
    R = torch.zeros(T, g.N, device=dev)
    o = [_outs(g, T, dev) for _ in range(10)]
    descs = [_desc(w[0], R, None, o[j]) for j in range(10)]
    assert rd.batch_plan(descs, T) == 6
    assert rd.batch_plan(descs[:3], T) == 3
    prev = rd.set_batch_lanes(2)
    try:
        assert rd.batch_plan(descs, T) == 2
        rd.set_batch_lanes(1)
        assert rd.batch_plan(descs, T) == 1  # the persistent kernel, T <= 4
        with pytest.raises(Exception):
            rd.set_batch_lanes(-1)
    finally:
        rd.set_batch_lanes(prev)
    assert rd.batch_plan(descs, T) == 6


def test_bench_sized_batch(dev, orc, sets, rd, ref):
    """The timed configuration of the benchmark: 300 independent reads at T=4
    with the pending write, own outputs each, one batch on the six streams;
    every read bit for bit against a direct read, three against the oracle."""
    g, host, w = sets
    T, L = 4, 300
    acts = [synth.activations(g, T, True, s0=5000 + j) for j in range(8)]
    R = [torch.from_numpy(x.R).to(dev) for x in acts]
    P = [torch.from_numpy(x.P).to(dev) for x in acts]
    o = [_outs(g, T, dev) for _ in range(L)]
    descs = [_desc(w[j % 4], R[j % 8], P[j % 8], o[j]) for j in range(L)]
    assert rd.batch_plan(descs, T) == 6
    rd.batch(descs, T)
    want = _outs(g, T, dev)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in range(L):
        d = descs[j]
        ref(d["R"], d["w_norm"], d["W_down"], d["W_up"], d["gate"], d["P"], T, want["out"], want["mean"], want["lo"])
        _same_bits(o[j], want, f"read {j}")
    for j in (0, 151, L - 1):
        a = acts[j % 8]
        res = orc.read(g.n, g.d, g.K, R=a.R, P=a.P, w_norm=host[j % 4].w_norm, W_down=host[j % 4].W_down,
                       W_up=host[j % 4].W_up, gate=host[j % 4].gate, eps=EPS)
        _close(o[j], res, f"read {j}")
