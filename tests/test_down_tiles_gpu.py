"""GPU checks of W_down in tile order (hc_read_register_down_tiles).

A registered tile-ordered copy changes where the down kernels of 32-row
tiles fetch their weights, not what they compute: every read with it must
equal the same read without it bit for bit (direct calls, batches on the
internal streams, graph replays), at d = 2560 (T = 1..4 take the tiles,
larger T ignore them) and at d = 4096 (every T takes them).  That the
kernels really read the tiles is shown by zeroing them: the down projection
then sees zero weights, so lo = 0 and out = R + P exactly, until the
registration is dropped."""

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


def _outs(g, T, dev):
    return dict(out=torch.full((T, g.N), float("nan"), device=dev),
                mean=torch.full((T, g.d), float("nan"), device=dev),
                lo=torch.full((T, g.K), float("nan"), device=dev))


def _read(r, w, a, T, o, stream=None):
    r(a["R"], w["w_norm"], w["W_down"], w["W_up"], w["gate"], a["P"], T, o["out"], o["mean"], o["lo"],
      stream=stream)


def _same(x, y, what):
    for k in ("out", "mean", "lo"):
        assert np.array_equal(bits(x[k]), bits(y[k])), f"{what} {k}"


@pytest.mark.parametrize("geom,T,pending", [
    (synth.G1, 1, False), (synth.G1, 2, True), (synth.G1, 3, False), (synth.G1, 4, True),
    (synth.G1, 6, True), (synth.G2, 1, True), (synth.G2, 5, True), (synth.G2, 8, False)],
    ids=lambda v: f"d{v.d}" if isinstance(v, synth.Geometry) else str(v))
def test_tiles_bit_identical(dev, orc, geom, T, pending):
    g = geom
    ws = synth.weight_set(g, 60 + T)
    w = dev_weights(ws, dev)
    act = synth.activations(g, T, pending, s0=6000 + T)
    a = dev_act(act, dev)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as plain, hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as tiled:
        tiles = tiled.down_tiles(w["W_down"])
        assert tiles.numel() * 2 == hc.hc_read_down_tiles_bytes(tiled.h)
        o1, o2 = _outs(g, T, dev), _outs(g, T, dev)
        _read(plain, w, a, T, o1)
        _read(tiled, w, a, T, o2)
        torch.cuda.synchronize()
        assert plain.check() == hc.HC_OK and tiled.check() == hc.HC_OK
        _same(o2, o1, f"d={g.d} T={T}")
    res = orc.read(g.n, g.d, g.K, R=act.R, P=act.P, w_norm=ws.w_norm, W_down=ws.W_down, W_up=ws.W_up,
                   gate=ws.gate, eps=EPS)
    for name, want in (("lo", res.lo), ("out", res.out), ("mean", res.mean)):
        got = o2[name].double().cpu().numpy()
        assert float(np.max(np.abs(got - want))) <= TOL * float(np.max(np.abs(want))), name


@pytest.mark.parametrize("T,used", [(1, True), (4, True), (5, False)])
def test_tiles_are_what_the_kernels_read(dev, T, used):
    g = synth.G1
    w = dev_weights(synth.weight_set(g, 70), dev)
    a = dev_act(synth.activations(g, T, True, s0=6100 + T), dev)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as r, hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as ref:
        tiles = r.down_tiles(w["W_down"])
        tiles.zero_()
        o, want = _outs(g, T, dev), _outs(g, T, dev)
        _read(r, w, a, T, o)
        _read(ref, w, a, T, want)
        torch.cuda.synchronize()
        if used:
            assert torch.count_nonzero(o["lo"]).item() == 0
            assert np.array_equal(bits(o["out"]), bits(a["R"] + a["P"]))
        else:
            _same(o, want, f"T={T} (tiles not taken)")
        r.forget_down_tiles(w["W_down"])
        o2 = _outs(g, T, dev)
        _read(r, w, a, T, o2)
        torch.cuda.synchronize()
        _same(o2, want, f"T={T} after forget")


def test_tiles_on_lanes_and_in_graphs(dev):
    g, T, n = synth.G1, 4, 24
    wsd = [dev_weights(synth.weight_set(g, 80 + j), dev) for j in range(4)]
    acts = [dev_act(synth.activations(g, T, j % 2 == 0, s0=6200 + j), dev) for j in range(n)]
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as r, hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as ref:
        keep = [r.down_tiles(w["W_down"]) for w in wsd]
        o = [_outs(g, T, dev) for _ in range(n)]
        descs = [dict(R=acts[j]["R"], P=acts[j]["P"], out=o[j]["out"], mean=o[j]["mean"], lo=o[j]["lo"],
                      **{k: wsd[j % 4][k] for k in ("w_norm", "W_down", "W_up", "gate")}) for j in range(n)]
        assert r.batch_plan(descs, T) == 6
        r.batch(descs, T)
        want = [_outs(g, T, dev) for _ in range(n)]
        for j in range(n):
            _read(ref, wsd[j % 4], acts[j], T, want[j])
        torch.cuda.synchronize()
        assert r.check() == hc.HC_OK
        for j in range(n):
            _same(o[j], want[j], f"batch read {j}")
        # A captured read replays the tiles it was captured with.
        s = torch.cuda.Stream(device=dev)
        og = _outs(g, T, dev)
        with torch.cuda.stream(s):
            hc.hc_graph_begin(s)
            _read(r, wsd[1], acts[1], T, og, stream=s)
            graph = hc.hc_graph_end(s)
        hc.hc_graph_launch(graph, s)
        s.synchronize()
        hc.hc_graph_destroy(graph)
        _same(og, want[1], "graph replay")
        del keep


def test_tiles_argument_errors(dev):
    g = synth.G1
    w = dev_weights(synth.weight_set(g, 90), dev)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as r:
        nb = hc.hc_read_down_tiles_bytes(r.h)
        assert nb == 6635520
        buf = torch.empty(nb // 2 + 16, dtype=torch.int16, device=dev)
        lib = hc._binding.load()
        assert lib.hc_read_register_down_tiles(r.h, w["W_down"].data_ptr(), buf.data_ptr() + 2, None) == hc.HC_ERR_ALIGN
        assert lib.hc_read_register_down_tiles(r.h, w["W_down"].data_ptr(), w["W_down"].data_ptr(), None) == hc.HC_ERR_ARG
        assert lib.hc_read_register_down_tiles(r.h, None, buf.data_ptr(), None) == hc.HC_ERR_ARG
        # Not during capture (the copy is waited for); the capture goes on.
        a = dev_act(synth.activations(g, 2, False, s0=6300), dev)
        o = _outs(g, 2, dev)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            hc.hc_graph_begin(s)
            st = lib.hc_read_register_down_tiles(r.h, w["W_down"].data_ptr(), buf.data_ptr(), s.cuda_stream)
            _read(r, w, a, 2, o, stream=s)
            graph = hc.hc_graph_end(s)
        hc.hc_graph_destroy(graph)
        assert st == hc.HC_ERR_ARG
        assert lib.hc_read_forget_down_tiles(r.h, None) == hc.HC_OK
