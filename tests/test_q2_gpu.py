"""GPU parity of the Q2_0 matrix-vector product (hc_q2_0_matvec) against the
FP64 oracle.

Weights: N(0, 0.02) float32 draws quantized to Q2_0 (64-value blocks, one
binary16 scale each, codes four to a byte); inputs N(0, 1).  Bar: for every
column, max|gpu - oracle| <= 1e-4 * max|oracle| (the read's bar); repeated
calls and graph replays bit for bit equal to the first call; nothing written
outside y."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL, bits

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


def to_dev(m: synth.Q2Matrix, dev):
    return torch.from_numpy(m.Wq).to(dev), torch.from_numpy(m.Wscale.view(np.int16)).to(dev)


def matvec(Wq, Ws, x, rows, guard=0, stream=None):
    """y (with `guard` sentinel floats before and after it) = W x on the GPU."""
    ncols = x.shape[0]
    buf = torch.full((ncols * rows + 2 * guard,), float("nan"), device=x.device)
    y = buf[guard:guard + ncols * rows].view(ncols, rows)
    hc.hc_q2_0_matvec(Wq, Ws, x, y, stream=stream)
    return y, buf


def assert_parity(y, want, what):
    got = y.double().cpu().numpy()
    for c in range(want.shape[0]):
        err = float(np.max(np.abs(got[c] - want[c])))
        bound = TOL * float(np.max(np.abs(want[c])))
        assert err <= bound, f"{what} column {c}: max err {err:.3e} > {bound:.3e}"


@pytest.fixture(scope="module")
def attn_q(dev):
    """The pages' shape: 2560 inputs, 12288 outputs."""
    m = synth.q2_0_matrix(12288, 2560, j=0)
    return m, to_dev(m, dev)


@pytest.mark.parametrize("ncols", [1, 2, 3, 4])
def test_attn_q_parity(dev, orc, attn_q, ncols):
    m, (Wq, Ws) = attn_q
    xh = synth.q2_0_columns(2560, ncols, j=ncols)
    y, _ = matvec(Wq, Ws, torch.from_numpy(xh).to(dev), 12288)
    torch.cuda.synchronize()
    assert_parity(y, orc.q2_0_matvec(m.Wq, m.Wscale, xh), f"attn_q ncols={ncols}")


@pytest.mark.parametrize("rows,cols,ncols", [
    (1, 512, 1), (63, 512, 2), (65, 1024, 3), (200, 2560, 4), (1000, 4096, 4),
    (4097, 3072, 2), (130, 4096, 1), (12289, 2560, 1),
])
def test_ragged_and_wide(dev, orc, rows, cols, ncols):
    m = synth.q2_0_matrix(rows, cols, j=rows)
    xh = synth.q2_0_columns(cols, ncols, j=cols)
    Wq, Ws = to_dev(m, dev)
    guard = 64
    y, buf = matvec(Wq, Ws, torch.from_numpy(xh).to(dev), rows, guard=guard)
    torch.cuda.synchronize()
    assert_parity(y, orc.q2_0_matvec(m.Wq, m.Wscale, xh), f"{rows}x{cols} ncols={ncols}")
    edge = torch.cat([buf[:guard], buf[-guard:]])
    assert torch.isnan(edge).all(), "write outside y"


def test_repeat_and_graph_replay_bitwise(dev, attn_q):
    m, (Wq, Ws) = attn_q
    x = torch.from_numpy(synth.q2_0_columns(2560, 3, j=7)).to(dev)
    y0, _ = matvec(Wq, Ws, x, 12288)
    torch.cuda.synchronize()
    ref = bits(y0)
    for _ in range(3):
        y1, _ = matvec(Wq, Ws, x, 12288)
        torch.cuda.synchronize()
        assert np.array_equal(bits(y1), ref), "repeated call"
    s = torch.cuda.Stream()
    ys = [torch.full((3, 12288), float("nan"), device=dev) for _ in range(2)]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        for y in ys:
            hc.hc_q2_0_matvec(Wq, Ws, x, y, stream=s)
        ge = hc.hc_graph_end(s)
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        hc.hc_graph_launch(ge, s)
        s.synchronize()
        for y in ys:
            assert np.array_equal(bits(y), ref), "graph replay"
    hc.hc_graph_destroy(ge)


def test_chained_square(dev, orc):
    """x of each call is y of the previous one (2560 x 2560): the kernel reads
    x only after the preceding kernel in the stream has completed.  Each step
    is checked against the oracle on the GPU's own input."""
    n, steps = 2560, 6
    mats = [synth.q2_0_matrix(n, n, j=100 + i) for i in range(steps)]
    devm = [to_dev(mm, dev) for mm in mats]
    xs = [torch.from_numpy(synth.q2_0_columns(n, 2, j=9)).to(dev)]
    for i in range(steps):
        y = torch.empty(2, n, device=dev)
        hc.hc_q2_0_matvec(*devm[i], xs[-1], y)
        xs.append(y)  # N(0, 0.02) weights over 2560 inputs keep the values of order one
    torch.cuda.synchronize()
    for i in range(steps):
        xin = xs[i].cpu().numpy()
        assert_parity(xs[i + 1], orc.q2_0_matvec(mats[i].Wq, mats[i].Wscale, xin), f"step {i}")


def test_special_scales(dev, orc):
    """Zero scales give y = 0 exactly; large, tiny (subnormal) and negative
    binary16 scales stay within the bar."""
    rows, cols = 128, 512
    m = synth.q2_0_matrix(rows, cols, j=3)
    xh = synth.q2_0_columns(cols, 2, j=3)
    x = torch.from_numpy(xh).to(dev)
    Wq = torch.from_numpy(m.Wq).to(dev)
    zero = torch.zeros(rows, cols // 64, dtype=torch.int16, device=dev)
    y, _ = matvec(Wq, zero, x, rows)
    torch.cuda.synchronize()
    assert not torch.any(y != 0) and not torch.isnan(y).any()
    rng = np.random.default_rng(5)
    for lo_e, hi_e in ((10, 15), (-24, -15), (-3, 3)):
        s = np.ldexp(1.0, rng.integers(lo_e, hi_e + 1, size=(rows, cols // 64)))
        s *= rng.choice([-1.0, 1.0], size=s.shape) * rng.uniform(1.0, 1.9, size=s.shape)
        sh = s.astype(np.float16).view(np.uint16)
        y, _ = matvec(Wq, torch.from_numpy(sh.view(np.int16)).to(dev), x, rows)
        torch.cuda.synchronize()
        assert_parity(y, orc.q2_0_matvec(m.Wq, sh, xh), f"scales 2^[{lo_e},{hi_e}]")


def test_side_stream(dev, orc):
    m = synth.q2_0_matrix(300, 1024, j=11)
    xh = synth.q2_0_columns(1024, 4, j=11)
    Wq, Ws = to_dev(m, dev)
    s = torch.cuda.Stream()
    x = torch.from_numpy(xh).to(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y, _ = matvec(Wq, Ws, x, 300, stream=s)
    s.synchronize()
    assert_parity(y, orc.q2_0_matvec(m.Wq, m.Wscale, xh), "side stream")


def test_device_argument_errors(dev, attn_q):
    m, (Wq, Ws) = attn_q
    x = torch.zeros(2, 2560, device=dev)
    y = torch.empty(2, 12288, device=dev)
    with pytest.raises(hc.HcError) as e:
        hc.hc_q2_0_matvec(Wq, Ws, x, y, cols=2560 - 64)
    assert e.value.status == hc.HC_ERR_SHAPE
    big = torch.empty(4 * 12288 + 4, device=dev)
    with pytest.raises(hc.HcError) as e:
        hc.hc_q2_0_matvec(Wq, Ws, x, big[1:1 + 2 * 12288].view(2, 12288))
    assert e.value.status == hc.HC_ERR_ALIGN


def test_batch_matches_single_calls_bitwise(dev, orc):
    """Eight independent products (own weights, one x, own y) as one batch:
    each y equals the single call's bits and meets the bar."""
    rows, cols, ncols = 1024, 2560, 3
    mats = [synth.q2_0_matrix(rows, cols, j=40 + i) for i in range(8)]
    dm = [to_dev(mm, dev) for mm in mats]
    xh = synth.q2_0_columns(cols, ncols, j=40)
    x = torch.from_numpy(xh).to(dev)
    ys = [torch.full((ncols, rows), float("nan"), device=dev) for _ in mats]
    hc.hc_q2_0_matvec_batch([(*dm[i], x, ys[i]) for i in range(8)], rows, cols, ncols)
    torch.cuda.synchronize()
    for i in range(8):
        y1, _ = matvec(*dm[i], x, rows)
        torch.cuda.synchronize()
        assert np.array_equal(bits(ys[i]), bits(y1)), f"product {i}"
        assert_parity(ys[i], orc.q2_0_matvec(mats[i].Wq, mats[i].Wscale, xh), f"batch product {i}")


def test_batch_with_dependencies(dev, orc):
    """Products that read an earlier product's y, or reuse its output buffer,
    wait for it; the others overlap.  Square 2560 x 2560 so a y can be an x."""
    n, ncols = 2560, 2
    mats = [synth.q2_0_matrix(n, n, j=60 + i) for i in range(6)]
    dm = [to_dev(mm, dev) for mm in mats]
    x0 = torch.from_numpy(synth.q2_0_columns(n, ncols, j=60)).to(dev)
    x1 = torch.from_numpy(synth.q2_0_columns(n, ncols, j=61)).to(dev)
    y = [torch.full((ncols, n), float("nan"), device=dev) for _ in range(5)]
    plan = [  # (matrix, input, output)
        (0, x0, y[0]), (1, x1, y[1]), (2, y[0], y[2]), (3, x1, y[3]), (4, y[2], y[4]),
        (5, y[3], y[1]),  # reads an earlier y and writes over another earlier y
    ]
    hc.hc_q2_0_matvec_batch([(*dm[m], xi, yo) for (m, xi, yo) in plan], n, n, ncols)
    torch.cuda.synchronize()
    host = {id(x0): x0.cpu().numpy(), id(x1): x1.cpu().numpy()}
    # replay on the host in order with the oracle, feeding the GPU's own inputs
    got = {}
    for k, (m, xi, yo) in enumerate(plan):
        xin = host[id(xi)] if id(xi) in host else got[id(xi)]
        want = orc.q2_0_matvec(mats[m].Wq, mats[m].Wscale, xin)
        got[id(yo)] = want.astype(np.float32)
        if k == 1:
            continue  # y[1] is overwritten by the last product
        assert_parity(yo, want, f"product {k}")


def test_batch_graph_replay_bitwise(dev, attn_q):
    m, (Wq, Ws) = attn_q
    x = torch.from_numpy(synth.q2_0_columns(2560, 4, j=8)).to(dev)
    copies = [(Wq, Ws), (Wq.clone(), Ws.clone())]
    ys = [torch.full((4, 12288), float("nan"), device=dev) for _ in range(4)]
    prods = [(*copies[i % 2], x, ys[i]) for i in range(4)]
    hc.hc_q2_0_matvec_batch(prods, 12288, 2560, 4)
    torch.cuda.synchronize()
    ref = [bits(y) for y in ys]
    assert all(np.array_equal(r, ref[0]) for r in ref), "same weights, same bits"
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        hc.hc_graph_begin(s)
        hc.hc_q2_0_matvec_batch(prods, 12288, 2560, 4, stream=s)
        ge = hc.hc_graph_end(s)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        hc.hc_graph_launch(ge, s)
        s.synchronize()
        for y, r in zip(ys, ref):
            assert np.array_equal(bits(y), r), "batch graph replay"
    hc.hc_graph_destroy(ge)


def test_batch_distinct_inputs(dev, orc):
    """Nine products over five distinct inputs in one batch: every product
    meets the bar and equals its single call bit for bit (the kernel prepares
    x again whenever a tile's input changes)."""
    rows, cols, ncols = 700, 1536, 2
    mats = [synth.q2_0_matrix(rows, cols, j=80 + i) for i in range(9)]
    dm = [to_dev(mm, dev) for mm in mats]
    xh = [synth.q2_0_columns(cols, ncols, j=80 + k) for k in range(5)]
    xd = [torch.from_numpy(v).to(dev) for v in xh]
    which = [0, 1, 0, 2, 3, 3, 4, 1, 2]
    ys = [torch.full((ncols, rows), float("nan"), device=dev) for _ in range(9)]
    hc.hc_q2_0_matvec_batch([(*dm[i], xd[which[i]], ys[i]) for i in range(9)], rows, cols, ncols)
    torch.cuda.synchronize()
    for i in range(9):
        assert_parity(ys[i], orc.q2_0_matvec(mats[i].Wq, mats[i].Wscale, xh[which[i]]), f"product {i}")
        y1, _ = matvec(*dm[i], xd[which[i]], rows)
        torch.cuda.synchronize()
        assert np.array_equal(bits(ys[i]), bits(y1)), f"product {i} batch vs single"


def test_input_range(dev, orc):
    """x far from order one (1e-30, 1e30 and mixed magnitudes) keeps the bar:
    the per-column power-of-two scaling."""
    rows, cols = 256, 1024
    m = synth.q2_0_matrix(rows, cols, j=90)
    Wq, Ws = to_dev(m, dev)
    base = synth.q2_0_columns(cols, 3, j=90)
    xh = np.stack([base[0] * np.float32(1e-30), base[1] * np.float32(1e30),
                   base[2] * np.exp2((np.arange(cols) % 37) - 18.0)]).astype(np.float32)
    y, _ = matvec(Wq, Ws, torch.from_numpy(xh).to(dev), rows)
    torch.cuda.synchronize()
    assert_parity(y, orc.q2_0_matvec(m.Wq, m.Wscale, xh), "input range")
