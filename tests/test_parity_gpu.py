"""GPU parity of the CUDA read against the FP64 oracle, through the C ABI.

Bar: max|gpu - oracle| <= 1e-4 * max|oracle| for lo, out, mean (and rs);
R' (r_out) bit for bit; graph replays and repeated calls bit for bit equal to
a direct call.
"""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import EPS, assert_parity, bits, dev_act, dev_weights, outputs, run

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
def g1(dev):
    g = synth.G1
    ws = synth.weight_set(g, 0)
    return g, ws, dev_weights(ws, dev)


@pytest.fixture(scope="module")
def rd1(dev):
    r = hc.Read(4, 2560, 320, T_max=64, eps=EPS)
    yield r
    r.close()


def oracle_read(orc, g, ws, act):
    return orc.read(g.n, g.d, g.K, R=act.R, P=act.P, w_norm=ws.w_norm, W_down=ws.W_down,
                    W_up=ws.W_up, gate=ws.gate, eps=EPS)


@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_parity_real_geometry(dev, orc, g1, rd1, T, pending):
    g, ws, w = g1
    act = synth.activations(g, T, pending, s0=100 + T)
    a = dev_act(act, dev)
    o = outputs(g, T, dev)
    run(rd1, w, a, T, o)
    torch.cuda.synchronize()
    assert rd1.check() == hc.HC_OK
    assert_parity(o, oracle_read(orc, g, ws, act), T, f"T={T} pending={pending}")


# Route boundaries of the wide pair: 16/17 (single pass / K-slice ring), 32/33
# (tokens per staging thread), 44/45 (partials' own region / over the weight
# tile), 48/49 (16- / 32-token up passes).
# Pending off and on take different down kernels above 16 tokens.
@pytest.mark.parametrize("pending", [False, True], ids=["pend_off", "pend_on"])
@pytest.mark.parametrize("T", [9, 13, 16, 17, 32, 33, 44, 45, 48, 49, 64])
def test_parity_token_groups(dev, orc, g1, rd1, T, pending):
    """T >= 9: the wide tensor-memory pair, tokens in passes with a ragged last one."""
    g, ws, w = g1
    act = synth.activations(g, T, pending, s0=200 + T)
    a = dev_act(act, dev)
    o = outputs(g, T, dev)
    run(rd1, w, a, T, o)
    torch.cuda.synchronize()
    assert_parity(o, oracle_read(orc, g, ws, act), T, f"T={T} pending={pending}")


@pytest.mark.parametrize("T", [1, 5, 8, 12])
def test_parity_scaled_geometry(dev, orc, T):
    g = synth.G2
    ws = synth.weight_set(g, 0)
    w = dev_weights(ws, dev)
    act = synth.activations(g, T, True, s0=300 + T)
    a = dev_act(act, dev)
    o = outputs(g, T, dev)
    with hc.Read(4, 4096, 512, T_max=16, eps=EPS) as rd:
        run(rd, w, a, T, o)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
    assert_parity(o, oracle_read(orc, g, ws, act), T, f"G2 T={T}")


def test_zero_weights_give_committed_residual(dev, rd1):
    """Invariant: zero projections give out = R' bit for bit."""
    g = synth.G1
    T = 3
    ws = synth.weight_set(g, 1)
    ws.W_down[:] = 0
    ws.W_up[:] = 0
    w = dev_weights(ws, dev)
    act = synth.activations(g, T, True, s0=7)
    a = dev_act(act, dev)
    o = outputs(g, T, dev)
    run(rd1, w, a, T, o)
    torch.cuda.synchronize()
    rp = (act.R + act.P).astype(np.float32)
    assert np.array_equal(bits(o["out"]), rp.view(np.uint32))
    assert np.array_equal(bits(o["r_out"]), rp.view(np.uint32))
    assert float(o["lo"].abs().max()) == 0.0


@pytest.mark.parametrize("T", [4, 8], ids=["T4_mma_sync", "T8_tensor_memory"])
def test_repeat_and_graph_replay_bitwise(dev, g1, rd1, T):
    g, ws, w = g1
    act = synth.activations(g, T, True, s0=11)
    a = dev_act(act, dev)
    o1 = outputs(g, T, dev)
    run(rd1, w, a, T, o1)
    torch.cuda.synchronize()
    ref = {k: bits(v) for k, v in o1.items()}
    # a second direct call on the same handle
    o2 = outputs(g, T, dev)
    run(rd1, w, a, T, o2)
    torch.cuda.synchronize()
    for k in ref:
        assert np.array_equal(bits(o2[k]), ref[k]), f"repeat {k}"
    # captured once, replayed twice
    s = torch.cuda.Stream()
    o3 = outputs(g, T, dev)
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        run(rd1, w, a, T, o3, stream=s)
        graph = hc.hc_graph_end(s)
    try:
        for rep in range(2):
            for v in o3.values():
                v.fill_(float("nan"))
            torch.cuda.synchronize()
            hc.hc_graph_launch(graph, s)
            s.synchronize()
            for k in ref:
                assert np.array_equal(bits(o3[k]), ref[k]), f"replay {rep} {k}"
    finally:
        hc.hc_graph_destroy(graph)


def test_in_place_update(dev, g1, rd1):
    """out may alias R: the residual is updated in place."""
    g, ws, w = g1
    T = 2
    act = synth.activations(g, T, True, s0=12)
    a = dev_act(act, dev)
    o = outputs(g, T, dev)
    run(rd1, w, a, T, o)
    a2 = dev_act(act, dev)
    o2 = outputs(g, T, dev)
    rd1(a2["R"], w["w_norm"], w["W_down"], w["W_up"], w["gate"], a2["P"], T,
        a2["R"], o2["mean"], o2["lo"])
    torch.cuda.synchronize()
    assert np.array_equal(bits(a2["R"]), bits(o["out"]))
    assert np.array_equal(bits(o2["mean"]), bits(o["mean"]))


def test_repeated_rows_agree(dev, g1, rd1):
    """A T=8 call whose 8 tokens are copies of one token gives the same bits on
    every row (tokens are independent), and those rows agree with a T=1 call
    within the parity bar (T=1 runs the CUDA-core kernels, T=8 the tensor-core
    kernels, so the two summation orders differ); R' is bitwise in both."""
    g, ws, w = g1
    act1 = synth.activations(g, 1, True, s0=13)
    a1 = dev_act(act1, dev)
    o1 = outputs(g, 1, dev)
    run(rd1, w, a1, 1, o1)
    a8 = {k: v.repeat(8, 1) for k, v in a1.items()}
    o8 = outputs(g, 8, dev)
    run(rd1, w, a8, 8, o8)
    torch.cuda.synchronize()
    for k in ("out", "mean", "lo", "r_out", "rs"):
        b8 = bits(o8[k])
        for t in range(1, 8):
            assert np.array_equal(b8[t], b8[0]), f"{k} row {t}"
        one = o1[k][0].double().cpu().numpy()
        eight = o8[k][0].double().cpu().numpy()
        assert np.max(np.abs(one - eight)) <= 2e-4 * np.max(np.abs(one)), k
    assert np.array_equal(bits(o8["r_out"])[0], bits(o1["r_out"])[0])


def test_argument_errors(dev, g1, rd1):
    g, ws, w = g1
    act = synth.activations(g, 2, False)
    a = dev_act(act, dev)
    o = outputs(g, 2, dev)
    lib = hc.load()
    ptrs = [a["R"].data_ptr(), w["w_norm"].data_ptr(), w["W_down"].data_ptr(),
            w["W_up"].data_ptr(), w["gate"].data_ptr(), None]
    outs = [o["out"].data_ptr(), o["mean"].data_ptr(), o["lo"].data_ptr()]
    assert lib.hc_read(rd1.h, *ptrs, 0, *outs, None) == hc.HC_ERR_ARG
    assert lib.hc_read(rd1.h, *ptrs, 65, *outs, None) == hc.HC_ERR_ARG
    bad = list(ptrs)
    bad[0] += 4
    assert lib.hc_read(rd1.h, *bad, 1, *outs, None) == hc.HC_ERR_ALIGN
    bad = list(ptrs)
    bad[2] = None
    assert lib.hc_read(rd1.h, *bad, 1, *outs, None) == hc.HC_ERR_ARG
    with pytest.raises(ValueError):
        rd1(a["R"].cpu(), w["w_norm"], w["W_down"], w["W_up"], w["gate"], None, 1,
            o["out"], o["mean"], o["lo"])
    with pytest.raises(hc.HcError):
        hc.Read(4, 2560, 320, T_max=0)
    assert rd1.check() == hc.HC_OK


def _oracle_from_gpu_inputs(orc, g, ws, R, P):
    return orc.read(g.n, g.d, g.K, R=R, P=P, w_norm=ws.w_norm, W_down=ws.W_down,
                    W_up=ws.W_up, gate=ws.gate, eps=EPS)


@pytest.mark.parametrize("T", [4, 6])
@pytest.mark.parametrize("use_graph", [False, True], ids=["direct", "graph"])
def test_chained_reads(dev, orc, rd1, use_graph, T):
    """Read i's out is read i+1's R (the window's chaining): each read is
    checked against the oracle fed with that read's GPU input."""
    g = synth.G1
    n_reads = 5
    sets = [synth.weight_set(g, 20 + i) for i in range(n_reads)]
    w = [dev_weights(ws, dev) for ws in sets]
    act = synth.activations(g, T, True, s0=31)
    P = torch.from_numpy(act.P).to(dev)
    bufs = [torch.from_numpy(act.R).to(dev)] + [torch.empty(T, g.N, device=dev) for _ in range(n_reads)]
    outs = [outputs(g, T, dev) for _ in range(n_reads)]
    s = torch.cuda.Stream()

    def enqueue():
        for i in range(n_reads):
            rd1(bufs[i], w[i]["w_norm"], w[i]["W_down"], w[i]["W_up"], w[i]["gate"], P, T,
                bufs[i + 1], outs[i]["mean"], outs[i]["lo"], r_out=outs[i]["r_out"],
                rs=outs[i]["rs"], stream=s)

    if use_graph:
        with torch.cuda.stream(s):
            hc.hc_graph_begin(s)
            enqueue()
            graph = hc.hc_graph_end(s)
        try:
            hc.hc_graph_launch(graph, s)
            s.synchronize()
        finally:
            hc.hc_graph_destroy(graph)
    else:
        with torch.cuda.stream(s):
            enqueue()
        s.synchronize()
    assert rd1.check() == hc.HC_OK
    for i in range(n_reads):
        R_in = bufs[i].cpu().numpy()
        ref = _oracle_from_gpu_inputs(orc, g, sets[i], R_in, act.P)
        o = dict(outs[i])
        o["out"] = bufs[i + 1]
        assert_parity(o, ref, T, f"chained read {i}")


@pytest.mark.parametrize("same_out", [False, True], ids=["own_outputs", "shared_outputs"])
def test_back_to_back_independent_reads(dev, orc, rd1, same_out):
    """Reads that do not consume each other's outputs overlap on the GPU; each
    still matches the oracle, and with shared output buffers the last read's
    results are what remains."""
    g = synth.G1
    T, n_reads = 3, 6
    sets = [synth.weight_set(g, 40 + i) for i in range(n_reads)]
    w = [dev_weights(ws, dev) for ws in sets]
    act = synth.activations(g, T, True, s0=51)
    a = dev_act(act, dev)
    shared = outputs(g, T, dev)
    outs = [shared if same_out else outputs(g, T, dev) for _ in range(n_reads)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(n_reads):
            run(rd1, w[i], a, T, outs[i], stream=s)
    s.synchronize()
    check = [n_reads - 1] if same_out else range(n_reads)
    for i in check:
        assert_parity(outs[i], oracle_read(orc, g, sets[i], act), T, f"read {i}")


def test_in_place_chain(dev, orc, rd1):
    """out = R in place, three times in a row: each read consumes the previous one."""
    g = synth.G1
    T = 2
    sets = [synth.weight_set(g, 60 + i) for i in range(3)]
    act = synth.activations(g, T, False, s0=61)
    R = torch.from_numpy(act.R).to(dev)
    o = outputs(g, T, dev)
    R_host = act.R.copy()
    for i in range(3):
        w = dev_weights(sets[i], dev)
        rd1(R, w["w_norm"], w["W_down"], w["W_up"], w["gate"], None, T, R, o["mean"], o["lo"])
        ref = _oracle_from_gpu_inputs(orc, g, sets[i], R_host, None)
        torch.cuda.synchronize()
        got = R.double().cpu().numpy()
        err = float(np.max(np.abs(got - ref.out)))
        assert err <= 1e-4 * float(np.max(np.abs(ref.out))), f"in-place read {i}: {err}"
        R_host = R.cpu().numpy()


def test_mixed_dependent_and_independent_sequence(dev, orc, rd1):
    """One stream, one handle: reads that consume the previous read's output
    (which must wait for it) interleaved with reads that do not (which may
    overlap it), different T on both kernel families, a shared output buffer.
    Every read matches the oracle fed with that read's GPU inputs."""
    g = synth.G1
    sets = [synth.weight_set(g, 70 + i) for i in range(5)]
    w = [dev_weights(ws, dev) for ws in sets]
    act = synth.activations(g, 8, True, s0=71)
    R0 = torch.from_numpy(act.R).to(dev)
    P0 = torch.from_numpy(act.P).to(dev)
    bufs = [torch.zeros(8, g.N, device=dev) for _ in range(4)]
    # (weights, T, input, output, pending): B ignores A, C consumes B,
    # D ignores C but rewrites A's output, E consumes D.
    plan = [(0, 1, R0, bufs[0], None), (1, 4, R0, bufs[1], P0), (2, 4, bufs[1], bufs[2], None),
            (3, 8, R0, bufs[0], P0), (4, 2, bufs[0], bufs[3], None)]
    s = torch.cuda.Stream()
    inputs, outs = [], []
    with torch.cuda.stream(s):
        for (j, T, rin, rout, p) in plan:
            o = outputs(g, T, dev)
            rd1(rin, w[j]["w_norm"], w[j]["W_down"], w[j]["W_up"], w[j]["gate"], p, T,
                rout, o["mean"], o["lo"], r_out=o["r_out"], rs=o["rs"], stream=s)
            outs.append(o)
            inputs.append(rin)
    s.synchronize()
    host_in = {0: act.R, 1: act.R, 3: act.R}
    host_in[2] = bufs[1].cpu().numpy()
    host_in[4] = bufs[0].cpu().numpy()
    for k, (j, T, rin, rout, p) in enumerate(plan):
        Rk = host_in[k][:T]
        Pk = act.P[:T] if p is not None else None
        ref = orc.read(g.n, g.d, g.K, R=Rk, P=Pk, w_norm=sets[j].w_norm, W_down=sets[j].W_down,
                       W_up=sets[j].W_up, gate=sets[j].gate, eps=EPS)
        o = dict(outs[k])
        if k in (1, 2, 4):
            o["out"] = rout
        if k == 3:
            o["out"] = bufs[0]
        if k == 0:
            continue  # its output buffer was rewritten by read 3
        assert_parity(o, ref, T, f"read {k} (T={T})")


@pytest.mark.parametrize("T", [1, 4, 8])
def test_overlap_switched_off_gives_the_same_bits(dev, orc, T):
    """hc_read_set_overlap(0): every read waits for its predecessor in full
    instead of computing before the wait; the results are the same bits as
    with the overlap on (the kernels and their summation order do not change),
    and match the oracle."""
    g = synth.G1
    n_reads = 3
    sets = [synth.weight_set(g, 80 + i) for i in range(n_reads)]
    w = [dev_weights(ws, dev) for ws in sets]
    act = synth.activations(g, T, True, s0=81)
    a = dev_act(act, dev)
    got = {}
    for overlap in (True, False):
        with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
            assert rd.set_overlap(overlap) is True  # the default is on
            outs = [outputs(g, T, dev) for _ in range(n_reads)]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for i in range(n_reads):
                    run(rd, w[i], a, T, outs[i], stream=s)
            s.synchronize()
            assert rd.check() == hc.HC_OK
            got[overlap] = outs
    for i in range(n_reads):
        for name in ("out", "mean", "lo", "r_out", "rs"):
            assert np.array_equal(bits(got[True][i][name]), bits(got[False][i][name])), f"read {i} {name}"
        assert_parity(got[False][i], oracle_read(orc, g, sets[i], act), T, f"read {i}")
