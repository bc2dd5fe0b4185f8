"""GPU checks of weights in tile order (hc_read_register_down_tiles,
hc_read_register_up_tiles).

A registered tile-ordered copy changes where the kernels fetch their weight
tiles, not what they compute: every read with it must equal the same read
without it bit for bit (direct calls, batches on the internal streams, graph
replays), at d = 2560 (the down tiles serve T = 2..4 with their 32-row
tiles and T >= 5 with their swizzled 64-row tiles, T = 1 reads W_down in
8-row stream-wide tiles of its own; the up tiles serve T >= 9) and at
d = 4096 (down tiles, every T).  That the kernels really read the tiles is
shown by zeroing them: zero down weights give lo = 0 and out = R + P
exactly, zero up weights out = R + P with lo unchanged, until the
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
    (synth.G1, 5, False), (synth.G1, 6, True), (synth.G1, 8, False), (synth.G1, 9, True),
    (synth.G1, 16, False), (synth.G1, 17, True), (synth.G1, 33, False), (synth.G1, 64, True),
    (synth.G2, 1, True), (synth.G2, 5, True), (synth.G2, 8, False)],
    ids=lambda v: f"d{v.d}" if isinstance(v, synth.Geometry) else str(v))
def test_tiles_bit_identical(dev, orc, geom, T, pending):
    g = geom
    ws = synth.weight_set(g, 60 + T)
    w = dev_weights(ws, dev)
    act = synth.activations(g, T, pending, s0=6000 + T)
    a = dev_act(act, dev)
    with hc.Read(g.n, g.d, g.K, T_max=64, eps=EPS) as plain, hc.Read(g.n, g.d, g.K, T_max=64, eps=EPS) as tiled:
        tiles = tiled.down_tiles(w["W_down"])
        up = tiled.up_tiles(w["W_up"])
        assert tiles.numel() * 2 == hc.hc_read_down_tiles_bytes(tiled.h)
        assert (up is None) == (g.d != 2560)
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


@pytest.mark.parametrize("T,which,used", [(1, "down", False), (2, "down", True), (4, "down", True), (5, "down", True),
                                          (16, "down", True), (4, "up", False), (16, "up", True)])
def test_tiles_are_what_the_kernels_read(dev, T, which, used):
    g = synth.G1
    w = dev_weights(synth.weight_set(g, 70), dev)
    a = dev_act(synth.activations(g, T, True, s0=6100 + T), dev)
    with hc.Read(g.n, g.d, g.K, T_max=64, eps=EPS) as r, hc.Read(g.n, g.d, g.K, T_max=64, eps=EPS) as ref:
        tiles = r.down_tiles(w["W_down"]) if which == "down" else r.up_tiles(w["W_up"])
        tiles.zero_()
        o, want = _outs(g, T, dev), _outs(g, T, dev)
        _read(r, w, a, T, o)
        _read(ref, w, a, T, want)
        torch.cuda.synchronize()
        if not used:
            _same(o, want, f"T={T} ({which} tiles not taken)")
        elif which == "down":
            assert torch.count_nonzero(o["lo"]).item() == 0
            assert np.array_equal(bits(o["out"]), bits(a["R"] + a["P"]))
        else:
            assert np.array_equal(bits(o["lo"]), bits(want["lo"]))
            assert np.array_equal(bits(o["out"]), bits(a["R"] + a["P"]))
        (r.forget_down_tiles if which == "down" else r.forget_up_tiles)()
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
        assert nb == 6635520 + 6553600 and hc.hc_read_up_tiles_bytes(r.h) == 6553600
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
    g2 = synth.G2
    with hc.Read(g2.n, g2.d, g2.K, T_max=8, eps=EPS) as r2:
        w2 = dev_weights(synth.weight_set(g2, 91), dev)
        assert hc.hc_read_up_tiles_bytes(r2.h) == 0
        assert lib.hc_read_register_up_tiles(r2.h, w2["W_up"].data_ptr(), buf.data_ptr(), None) == hc.HC_ERR_SHAPE
