"""GPU parity of hc_read_batch (a list of reads in one call) against the FP64
oracle, through the C ABI.

At d = 2560, K = 320, T <= 4 the batch runs as the persistent multi-read
kernel; other shapes run read by read.  Bar as for single reads: max|gpu -
oracle| <= 1e-4 * max|oracle| for lo, out and mean of every read; repeated
batches and graph replays bit for bit equal.  Chained reads (R of read j is
read j-1's out) are checked against the oracle fed with the GPU's own input
of that read, so errors cannot hide in the chain.
"""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import EPS, TOL, bits, dev_act, dev_weights

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


@pytest.fixture(scope="module")
def sets(dev):
    g = synth.G1
    host = [synth.weight_set(g, j) for j in range(4)]
    return g, host, [dev_weights(ws, dev) for ws in host]


@pytest.fixture(scope="module")
def rd(dev):
    r = hc.Read(4, 2560, 320, T_max=8, eps=EPS)
    # Batches stay on the caller's stream: these tests are about the
    # persistent kernel (the internal streams: test_lanes_gpu.py).
    r.set_batch_lanes(1)
    yield r
    r.close()


def test_persistent_kernel_is_used(dev, rd):
    """On GB300 the real geometry's batches of up to 4 tokens run as the
    persistent kernel (the other tests would also pass read by read)."""
    assert all(rd.batch_persistent(T) for T in (1, 2, 3, 4))
    assert not any(rd.batch_persistent(T) for T in (5, 8))
    g = synth.G1
    o = [_outs(g, 2, dev) for _ in range(3)]
    w = dev_weights(synth.weight_set(g, 0), dev)
    R = torch.zeros(2, g.N, device=dev)
    assert rd.batch_plan([_desc(w, R, None, o[j]) for j in range(3)], 2) == 1


def _outs(g, T, dev):
    return dict(out=torch.full((T, g.N), float("nan"), device=dev),
                mean=torch.full((T, g.d), float("nan"), device=dev),
                lo=torch.full((T, g.K), float("nan"), device=dev))


def _desc(w, R, P, o):
    return dict(R=R, P=P, w_norm=w["w_norm"], W_down=w["W_down"], W_up=w["W_up"], gate=w["gate"],
                out=o["out"], mean=o["mean"], lo=o["lo"])


def _close(o, ref, T, what):
    for name, want in (("lo", ref.lo), ("out", ref.out), ("mean", ref.mean)):
        got = o[name][:T].double().cpu().numpy()
        err = float(np.max(np.abs(got - want[:T])))
        bound = TOL * float(np.max(np.abs(want[:T])))
        assert err <= bound, f"{what} {name}: max err {err:.3e} > {bound:.3e}"


def _oracle(orc, g, ws, R, P):
    return orc.read(g.n, g.d, g.K, R=R, P=P, w_norm=ws.w_norm, W_down=ws.W_down, W_up=ws.W_up,
                    gate=ws.gate, eps=EPS)


@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 6])
def test_batch_independent_reads(dev, orc, sets, rd, T, pending):
    """Three reads, three weight sets, own inputs and outputs."""
    g, host, w = sets
    acts = [synth.activations(g, T, pending, s0=300 + 10 * T + j) for j in range(3)]
    a = [dev_act(x, dev) for x in acts]
    o = [_outs(g, T, dev) for _ in range(3)]
    rd.batch([_desc(w[j], a[j]["R"], a[j]["P"], o[j]) for j in range(3)], T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in range(3):
        _close(o[j], _oracle(orc, g, host[j], acts[j].R, acts[j].P), T, f"T={T} read {j}")


def test_batch_varying_T_on_one_handle(dev, orc, sets, rd):
    """Batches of different T on one handle: exchange slots of token rows a
    smaller batch did not use must never pass for fresh data later."""
    g, host, w = sets
    for n, T in enumerate((4, 1, 1, 1, 2, 3, 4, 1, 4)):
        acts = [synth.activations(g, T, n % 2 == 1, s0=1000 + 10 * n + j) for j in range(3)]
        a = [dev_act(x, dev) for x in acts]
        o = [_outs(g, T, dev) for _ in range(3)]
        rd.batch([_desc(w[(j + n) % 4], a[j]["R"], a[j]["P"], o[j]) for j in range(3)], T)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
        for j in range(3):
            _close(o[j], _oracle(orc, g, host[(j + n) % 4], acts[j].R, acts[j].P), T, f"batch {n} T={T} read {j}")


@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [1, 4])
def test_batch_chained_reads(dev, orc, sets, rd, T, pending):
    """Six chained reads (R of read j = out of read j-1) over four weight sets."""
    g, host, w = sets
    L = 6
    a0 = synth.activations(g, T, False, s0=400 + T)
    R0 = torch.from_numpy(a0.R).to(dev)
    Ps = [synth.activations(g, T, True, s0=410 + j).P if pending else None for j in range(L)]
    Pd = [None if p is None else torch.from_numpy(p).to(dev) for p in Ps]
    o = [_outs(g, T, dev) for _ in range(L)]
    descs = []
    for j in range(L):
        R = R0 if j == 0 else o[j - 1]["out"]
        descs.append(_desc(w[j % 4], R, Pd[j], o[j]))
    rd.batch(descs, T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in range(L):
        R_in = a0.R if j == 0 else o[j - 1]["out"].cpu().numpy()
        _close(o[j], _oracle(orc, g, host[j % 4], R_in, Ps[j]), T, f"T={T} chained read {j}")


def test_batch_in_place_chain_matches_separate_buffers(dev, sets, rd):
    """One residual buffer updated in place by every read gives the same bits
    as separate output buffers."""
    g, _, w = sets
    T, L = 4, 5
    a0 = synth.activations(g, T, False, s0=500)
    R0 = torch.from_numpy(a0.R).to(dev)
    o = [_outs(g, T, dev) for _ in range(L)]
    rd.batch([_desc(w[j % 4], R0 if j == 0 else o[j - 1]["out"], None, o[j]) for j in range(L)], T)
    resid = R0.clone()
    oi = [_outs(g, T, dev) for _ in range(L)]
    for j in range(L):
        oi[j]["out"] = resid
    rd.batch([_desc(w[j % 4], resid, None, oi[j]) for j in range(L)], T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    assert np.array_equal(bits(resid), bits(o[L - 1]["out"]))
    for j in range(L):
        assert np.array_equal(bits(oi[j]["mean"]), bits(o[j]["mean"])), j
        assert np.array_equal(bits(oi[j]["lo"]), bits(o[j]["lo"])), j


def test_batch_repeat_and_graph_replay_bitwise(dev, sets, rd):
    g, _, w = sets
    T, L = 3, 8
    a0 = synth.activations(g, T, True, s0=600)
    R0 = torch.from_numpy(a0.R).to(dev)
    P0 = torch.from_numpy(a0.P).to(dev)
    o = [_outs(g, T, dev) for _ in range(L)]
    descs = [_desc(w[j % 4], R0 if j == 0 else o[j - 1]["out"], P0, o[j]) for j in range(L)]

    def snap():
        return [bits(o[j][k]) for j in range(L) for k in ("out", "mean", "lo")]

    rd.batch(descs, T)
    torch.cuda.synchronize()
    first = snap()
    for x in o:
        for t in x.values():
            t.fill_(float("nan"))
    rd.batch(descs, T)
    torch.cuda.synchronize()
    assert all(np.array_equal(x, y) for x, y in zip(first, snap())), "repeat"

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        rd.batch(descs, T, stream=s)
        graph = hc.hc_graph_end(s)
    try:
        for _ in range(2):
            for x in o:
                for t in x.values():
                    t.fill_(float("nan"))
            torch.cuda.synchronize()
            hc.hc_graph_launch(graph, s)
            s.synchronize()
            assert all(np.array_equal(x, y) for x, y in zip(first, snap())), "graph replay"
    finally:
        hc.hc_graph_destroy(graph)
    assert rd.check() == hc.HC_OK


def test_batch_matches_single_reads(dev, sets, rd):
    """The persistent kernel and the two-kernel reads agree within the bar."""
    g, _, w = sets
    T, L = 2, 4
    a0 = synth.activations(g, T, False, s0=700)
    R0 = torch.from_numpy(a0.R).to(dev)
    ob = [_outs(g, T, dev) for _ in range(L)]
    rd.batch([_desc(w[j], R0 if j == 0 else ob[j - 1]["out"], None, ob[j]) for j in range(L)], T)
    os_ = [_outs(g, T, dev) for _ in range(L)]
    for j in range(L):
        R = R0 if j == 0 else os_[j - 1]["out"]
        rd(R, w[j]["w_norm"], w[j]["W_down"], w[j]["W_up"], w[j]["gate"], None, T,
           os_[j]["out"], os_[j]["mean"], os_[j]["lo"])
    torch.cuda.synchronize()
    for j in range(L):
        for k in ("out", "mean", "lo"):
            x = ob[j][k].double().cpu().numpy()
            y = os_[j][k].double().cpu().numpy()
            err = float(np.max(np.abs(x - y)))
            assert err <= 2 * TOL * float(np.max(np.abs(y))), (j, k, err)


def test_batch_long_window(dev, orc, sets, rd):
    """A 96-read chained window (the pages' reads per verify window), T = 4:
    sampled reads against the oracle on their GPU inputs."""
    g, host, w = sets
    T, L = 4, 96
    a0 = synth.activations(g, T, False, s0=800)
    R0 = torch.from_numpy(a0.R).to(dev)
    o = [_outs(g, T, dev) for _ in range(L)]
    rd.batch([_desc(w[j % 4], R0 if j == 0 else o[j - 1]["out"], None, o[j]) for j in range(L)], T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in (0, 1, 47, 95):
        R_in = a0.R if j == 0 else o[j - 1]["out"].cpu().numpy()
        _close(o[j], _oracle(orc, g, host[j % 4], R_in, None), T, f"window read {j}")


def test_batch_more_reads_than_one_launch(dev, orc, sets, rd):
    """230 chained reads span two launches of the persistent kernel."""
    g, host, w = sets
    T, L = 1, 230
    a0 = synth.activations(g, T, False, s0=900)
    R0 = torch.from_numpy(a0.R).to(dev)
    o = [_outs(g, T, dev) for _ in range(L)]
    rd.batch([_desc(w[j % 4], R0 if j == 0 else o[j - 1]["out"], None, o[j]) for j in range(L)], T)
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
    for j in (223, 224, 229):
        _close(o[j], _oracle(orc, g, host[j % 4], o[j - 1]["out"].cpu().numpy(), None), T, f"read {j}")


def test_batch_scaled_geometry_runs_read_by_read(dev, orc):
    g = synth.G2
    ws = [synth.weight_set(g, j) for j in range(2)]
    w = [dev_weights(x, dev) for x in ws]
    T = 2
    act = synth.activations(g, T, True, s0=950)
    a = dev_act(act, dev)
    with hc.Read(4, 4096, 512, T_max=4, eps=EPS) as r:
        o = [_outs(g, T, dev) for _ in range(2)]
        r.batch([_desc(w[0], a["R"], a["P"], o[0]), _desc(w[1], o[0]["out"], None, o[1])], T)
        torch.cuda.synchronize()
        assert r.check() == hc.HC_OK
    _close(o[0], _oracle(orc, g, ws[0], act.R, act.P), T, "G2 read 0")
    _close(o[1], _oracle(orc, g, ws[1], o[0]["out"].cpu().numpy(), None), T, "G2 read 1")


def test_batch_argument_errors(dev, sets, rd):
    g, _, w = sets
    T = 2
    a = dev_act(synth.activations(g, T, True, s0=990), dev)
    o = [_outs(g, T, dev) for _ in range(2)]
    ok = [_desc(w[0], a["R"], a["P"], o[0]), _desc(w[1], o[0]["out"], None, o[1])]

    def status(descs, TT=T):
        arr = (hc.hc_read_desc * len(descs))()
        for i, d in enumerate(descs):
            arr[i] = hc.hc_read_desc(*[None if d[k] is None else (d[k] if isinstance(d[k], int) else d[k].data_ptr())
                                       for k in ("R", "w_norm", "W_down", "W_up", "gate", "P", "out", "mean", "lo")])
        return hc.load().hc_read_batch(rd.h, arr, len(descs), TT, None)

    assert status(ok) == hc.HC_OK
    # pending of a later read taken from an earlier read's output
    assert status([ok[0], dict(ok[1], P=o[0]["out"])]) == hc.HC_ERR_ARG
    # R of a later read overlapping an earlier read's mean
    assert status([ok[0], dict(ok[1], R=o[0]["mean"])]) == hc.HC_ERR_ARG
    # pending overlapping the read's own out
    assert status([dict(ok[0], out=a["P"])]) == hc.HC_ERR_ARG
    # misaligned pointer
    assert status([dict(ok[0], lo=o[0]["lo"].data_ptr() + 4)]) == hc.HC_ERR_ALIGN
    assert status(ok, TT=0) == hc.HC_ERR_ARG
    assert status(ok, TT=9) == hc.HC_ERR_ARG
    assert hc.load().hc_read_batch(rd.h, None, 1, T, None) == hc.HC_ERR_ARG
    torch.cuda.synchronize()
    assert rd.check() == hc.HC_OK
