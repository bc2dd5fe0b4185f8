"""Pins of the FP64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:

* the hand-expanded tiny reads under ``tests/golden/`` (exact rationals);
* closed forms (constant streams, one-hot weight rows, sigmoid(0) = 1/2,
  sigmoid(+-ln 3) = 3/4, 1/4);
* invariants of the definition (zero weights give out = R'; a stream
  permutation permutes out and leaves lo, m unchanged; lo is invariant to a
  positive rescale of R' when eps = 0; tokens are independent);
* IEEE binary32 addition as done by NumPy for R' = fl32(R + P);
* brute-force probing on a tiny read (lo rebuilt from one-hot probes).

``tests/test_oracle_mutants.py`` plants plausible mistakes in a copy of the
oracle's source and checks that at least one pin fails for each.
"""

from __future__ import annotations

import math

import numpy as np

import golden_io

REL = 1e-12


def _close(got, want, what, rel=REL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    scale = max(1.0, float(np.max(np.abs(want))) if want.size else 1.0)
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    assert err <= rel * scale, f"{what}: max abs err {err:.3e} (scale {scale:.3e})"


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(rng, shape, scale=1.0):
    """Random BF16 bit patterns of N(0, scale) values (truncated to BF16)."""
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _bf16_value(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _random_read(seed, n, d, K, T, pending):
    rng = _rng(seed)
    N = n * d
    return dict(
        R=rng.standard_normal((T, N)).astype(np.float32),
        P=(rng.standard_normal((T, N)) * 0.1).astype(np.float32) if pending else None,
        w_norm=(1.0 + 0.05 * rng.standard_normal(N)).astype(np.float32),
        gate=rng.standard_normal(N).astype(np.float32),
        W_down=_bf16(rng, (K, N), 0.05),
        W_up=_bf16(rng, (N, K), 0.05),
    )


# ---------------------------------------------------------------- hand-expanded

def pin_hand_fixtures(orc):
    files = golden_io.fixtures()
    assert len(files) >= 3
    for path in files:
        fx = golden_io.load(path)
        n, d, K, T = fx["n"], fx["d"], fx["K"], fx["T"]
        res = orc.read(
            n, d, K,
            R=fx["R"].astype(np.float32).reshape(T, n * d),
            P=fx["P"].astype(np.float32).reshape(T, n * d) if "P" in fx else None,
            w_norm=fx["w_norm"].astype(np.float32),
            W_down=golden_io.to_bf16_exact(fx["W_down"]).reshape(K, n * d),
            W_up=golden_io.to_bf16_exact(fx["W_up"]).reshape(n * d, K),
            gate=fx["gate"].astype(np.float32),
            eps=float(fx["eps"][0]),
        )
        name = path.rsplit("/", 1)[-1]
        assert np.array_equal(res.r_out.ravel(), fx["r_out"].astype(np.float32)), f"{name}: r_out"
        for key in ("ss", "rs", "lo", "u", "out", "mean"):
            _close(getattr(res, key).ravel(), fx[key], f"{name}: {key}")


# ---------------------------------------------------------------- closed forms

def pin_constant_streams(orc):
    """R'[s, :] = a_s gives ss = d a_s^2 and rs = 1/sqrt(a_s^2 + eps)."""
    n, d, K, T, eps = 4, 40, 3, 2, 0.25
    a = np.array([[0.5, -2.0, 3.0, 0.0], [1.5, 0.25, -1.0, 4.0]], np.float32)
    R = np.repeat(a, d, axis=1).astype(np.float32)
    rd = _random_read(1, n, d, K, T, False)
    res = orc.read(n, d, K, R=R, w_norm=rd["w_norm"], W_down=rd["W_down"], W_up=rd["W_up"],
                   gate=rd["gate"], eps=eps)
    a64 = a.astype(np.float64)
    _close(res.ss, d * a64 ** 2, "ss of constant streams")
    _close(res.rs, 1.0 / np.sqrt(a64 ** 2 + eps), "rs of constant streams")


def pin_one_hot_down(orc):
    """A single 1 at W_down[k, j] gives lo[t, k] = rs[t, s(j)] * R'[t, j] * w_norm[j]."""
    n, d, K, T = 3, 5, 4, 2
    rd = _random_read(2, n, d, K, T, True)
    N = n * d
    for (k, j) in [(0, 0), (3, N - 1), (2, 7), (1, 11)]:
        W = np.zeros((K, N), np.uint16)
        W[k, j] = 0x3F80  # 1.0
        res = orc.read(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], W_down=W,
                       W_up=rd["W_up"], gate=rd["gate"], eps=1e-3)
        s = j // d
        want = np.zeros((T, K))
        want[:, k] = res.rs[:, s] * res.r_out[:, j].astype(np.float64) * np.float64(rd["w_norm"][j])
        _close(res.lo, want, f"lo for one-hot W_down[{k},{j}]")


def pin_one_hot_up(orc):
    """A single 1 at W_up[i, k] gives out[t, i] = R'[t, i] + sigmoid(g_i) lo[t, k] and out = R' elsewhere."""
    n, d, K, T = 2, 6, 3, 3
    rd = _random_read(3, n, d, K, T, True)
    N = n * d
    for (i, k) in [(0, 0), (N - 1, K - 1), (7, 1)]:
        W = np.zeros((N, K), np.uint16)
        W[i, k] = 0x3F80
        gate = rd["gate"].copy()
        gate[i] = 0.0  # sigmoid(0) = 1/2 exactly
        res = orc.read(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], W_down=rd["W_down"],
                       W_up=W, gate=gate, eps=1e-3)
        want = res.r_out.astype(np.float64).copy()
        want[:, i] += 0.5 * res.lo[:, k]
        _close(res.out, want, f"out for one-hot W_up[{i},{k}]")


def pin_sigmoid_values(orc):
    """sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 (up to the rounding of ln 3 to float32)."""
    n, d, K, T = 1, 2, 1, 1
    R = np.zeros((T, 2), np.float32)
    W_down = np.zeros((K, 2), np.uint16)
    W_down[0, 0] = 0x3F80
    R[0, 0] = 2.0  # rs = 1/sqrt(4/2) -> lo = rs * 2 * 1 = sqrt(2)
    W_up = np.full((2, 1), 0x3F80, np.uint16)
    g = np.array([math.log(3.0), -math.log(3.0)], np.float32)
    res = orc.read(n, d, K, R=R, w_norm=np.ones(2, np.float32), W_down=W_down, W_up=W_up,
                   gate=g, eps=0.0)
    lo = math.sqrt(2.0)
    _close(res.lo.ravel(), [lo], "lo", rel=1e-15)
    # d sigmoid / dg <= 1/4, and |float32(ln 3) - ln 3| < 6e-8.
    _close(res.out.ravel(), [2.0 + 0.75 * lo, 0.0 + 0.25 * lo], "sigmoid(+-ln 3)", rel=3e-8)


# ---------------------------------------------------------------- invariants

def pin_zero_weights(orc):
    """Zero projections give out = R' (= fl32(R + P)) exactly and m = stream mean of R'."""
    n, d, K, T = 4, 8, 5, 3
    rd = _random_read(4, n, d, K, T, True)
    N = n * d
    res = orc.read(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"],
                   W_down=np.zeros((K, N), np.uint16), W_up=np.zeros((N, K), np.uint16),
                   gate=rd["gate"], eps=1e-6)
    rp = (rd["R"] + rd["P"]).astype(np.float32)  # NumPy float32 add: IEEE round to nearest
    assert np.array_equal(res.r_out, rp), "r_out != fl32(R + P)"
    assert np.array_equal(res.out, rp.astype(np.float64)), "out != R' with zero weights"
    assert np.all(res.lo == 0.0)
    streams = rp.astype(np.float64).reshape(T, n, d)
    _close(res.mean, streams.sum(axis=1) / n, "mean of R'", rel=1e-15)


def pin_commit_bits(orc):
    """R' is one binary32 round-to-nearest add, bit for bit, including hard cases."""
    N = 8
    R = np.array([[1.0, 1e-30, 3.0, -0.0, 16777216.0, 1.0, 0.1, -5e-39]], np.float32)
    P = np.array([[2 ** -24, 1.0, -3.0, 0.0, 1.0, 1e38, 0.2, 5e-39]], np.float32)
    with np.errstate(over="ignore"):
        want = (R + P).astype(np.float32)
    res = orc.read(1, N, 1, R=R, P=P, w_norm=np.ones(N, np.float32),
                   W_down=np.zeros((1, N), np.uint16), W_up=np.zeros((N, 1), np.uint16),
                   gate=np.zeros(N, np.float32), eps=1.0)
    assert np.array_equal(res.r_out.view(np.uint32), want.view(np.uint32)), "R' bits"


def pin_stream_permutation(orc):
    """Permuting the streams permutes out's streams and leaves lo and m unchanged."""
    n, d, K, T = 4, 6, 5, 2
    rd = _random_read(5, n, d, K, T, True)
    perm = [2, 0, 3, 1]
    cols = np.concatenate([np.arange(s * d, (s + 1) * d) for s in perm])
    base = orc.read(n, d, K, eps=1e-4, **rd)
    prd = dict(
        R=np.ascontiguousarray(rd["R"][:, cols]), P=np.ascontiguousarray(rd["P"][:, cols]),
        w_norm=np.ascontiguousarray(rd["w_norm"][cols]), gate=np.ascontiguousarray(rd["gate"][cols]),
        W_down=np.ascontiguousarray(rd["W_down"][:, cols]), W_up=np.ascontiguousarray(rd["W_up"][cols, :]),
    )
    res = orc.read(n, d, K, eps=1e-4, **prd)
    _close(res.lo, base.lo, "lo under stream permutation")
    _close(res.mean, base.mean, "mean under stream permutation")
    _close(res.out, base.out[:, cols], "out under stream permutation")
    _close(res.rs, base.rs[:, perm], "rs under stream permutation")


def pin_scale_invariance(orc):
    """With eps = 0, scaling R by beta > 0 leaves lo unchanged (rs absorbs the scale)."""
    n, d, K, T = 3, 7, 4, 2
    rd = _random_read(6, n, d, K, T, False)
    base = orc.read(n, d, K, eps=0.0, **rd)
    scaled = dict(rd)
    scaled["R"] = (rd["R"] * np.float32(4.0)).astype(np.float32)  # exact power-of-two scale
    res = orc.read(n, d, K, eps=0.0, **scaled)
    _close(res.lo, base.lo, "lo under R -> 4R")
    _close(res.rs, base.rs / 4.0, "rs under R -> 4R")


def pin_token_independence(orc):
    """Each token's outputs depend only on that token's R and P."""
    n, d, K, T = 2, 5, 3, 3
    rd = _random_read(7, n, d, K, T, True)
    full = orc.read(n, d, K, eps=1e-5, **rd)
    for t in range(T):
        one = dict(rd)
        one["R"] = np.ascontiguousarray(rd["R"][t:t + 1])
        one["P"] = np.ascontiguousarray(rd["P"][t:t + 1])
        r1 = orc.read(n, d, K, eps=1e-5, **one)
        for key in ("ss", "rs", "lo", "u", "out", "mean"):
            _close(getattr(r1, key), getattr(full, key)[t:t + 1], f"token {t} {key}")
        assert np.array_equal(r1.r_out, full.r_out[t:t + 1])


def pin_pending_is_committed_first(orc):
    """The read sees R and P only through R' = fl32(R + P): a read of (R, P) equals
    a read of (R', no pending write) in every output."""
    n, d, K, T = 3, 4, 2, 2
    rd = _random_read(9, n, d, K, T, True)
    rd["P"] = (rd["P"] * np.float32(20.0)).astype(np.float32)  # make P matter in the norm
    a = orc.read(n, d, K, eps=1e-3, **rd)
    committed = dict(rd)
    committed["R"] = (rd["R"] + rd["P"]).astype(np.float32)
    committed["P"] = None
    b = orc.read(n, d, K, eps=1e-3, **committed)
    assert np.array_equal(a.r_out, b.r_out)
    for key in ("ss", "rs", "lo", "u", "out", "mean"):
        _close(getattr(a, key), getattr(b, key), f"{key} of (R, P) vs (R', none)")


# ---------------------------------------------------------------- brute force

def pin_probe_linearity(orc):
    """lo is linear in W_down: rebuild a_i = d lo / d W_down[k, i] from one-hot probes,
    then a random W_down must give lo[k] = sum_i W_down[k, i] a_i; likewise u in W_up."""
    n, d, K, T = 2, 3, 2, 2
    rd = _random_read(8, n, d, K, T, True)
    N = n * d
    a = np.zeros((T, N))
    for i in range(N):
        W = np.zeros((K, N), np.uint16)
        W[0, i] = 0x3F80
        a[:, i] = orc.read(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], W_down=W,
                           W_up=rd["W_up"], gate=rd["gate"], eps=0.01).lo[:, 0]
    res = orc.read(n, d, K, eps=0.01, **rd)
    Wd = _bf16_value(rd["W_down"])
    want_lo = np.array([[sum(Wd[k, i] * a[t, i] for i in range(N)) for k in range(K)]
                        for t in range(T)])
    _close(res.lo, want_lo, "lo from probes")
    Wu = _bf16_value(rd["W_up"])
    want_u = np.array([[sum(Wu[i, k] * res.lo[t, k] for k in range(K)) for i in range(N)]
                       for t in range(T)])
    _close(res.u, want_u, "u from lo")


# ---------------------------------------------------------------- Q8_0 read

def pin_half_decoding(orc):
    """Every binary16 bit pattern decodes to the value NumPy's IEEE binary16 gives
    (NaN patterns to NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    for h in range(1 << 16):
        got = orc.half(h)
        w = want[h]
        assert (math.isnan(got) and math.isnan(w)) or got == w, f"binary16 {h:#06x}: {got!r} != {w!r}"


def _q8_exact_bf16(seed, rows, cols):
    """Q8_0 weights whose values are exact BF16 numbers: int8 quants (7
    significant bits at most) times power-of-two binary16 scales that differ
    from block to block and row to row.  Returns (q, scale bits, BF16 bits)."""
    rng = _rng(seed)
    q = rng.integers(-127, 128, size=(rows, cols), dtype=np.int64).astype(np.int8)
    r = np.arange(rows)[:, None]
    b = np.arange(cols // 32)[None, :]
    e = -(4 + (r * 7 + b * 3 + seed) % 6)               # 2^-4 ... 2^-9
    scale = np.ldexp(np.ones((rows, cols // 32)), e).astype(np.float16)
    w = q.astype(np.float64) * np.repeat(scale.astype(np.float64), 32, axis=1)
    bf = (w.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_bf16_value(bf), w), "test weights must be exact in BF16"
    return q, scale.view(np.uint16), bf


def pin_q8_equals_bf16_read(orc):
    """With Q8_0 values that are exact BF16 numbers, the Q8_0 read equals the BF16
    read of the same values bit for bit (same formulas, same weights)."""
    n, d, K, T = 4, 16, 64, 3
    N = n * d
    rd = _random_read(11, n, d, K, T, True)
    qd, sd, bd = _q8_exact_bf16(12, K, N)
    qu, su, bu = _q8_exact_bf16(13, N, K)
    a = orc.read_q8(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], Wd_q=qd, Wd_scale=sd,
                    Wu_q=qu, Wu_scale=su, gate=rd["gate"], eps=1e-6)
    b = orc.read(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], W_down=bd, W_up=bu,
                 gate=rd["gate"], eps=1e-6)
    for key in ("r_out", "ss", "rs", "lo", "u", "out", "mean"):
        assert np.array_equal(getattr(a, key), getattr(b, key)), f"Q8_0 vs BF16 read: {key}"


def pin_q8_one_block(orc):
    """W_up with a single quant q at row i, column k (scale s of its block) gives
    u[t, i] = s * q * lo[t, k] exactly; all-zero scales give out = R' bit for bit."""
    n, d, K, T = 2, 32, 64, 2
    N = n * d
    rd = _random_read(14, n, d, K, T, True)
    qd, sd, _ = _q8_exact_bf16(15, K, N)
    for (i, k, q, s) in [(0, 0, 3, 0.125), (N - 1, K - 1, -127, 2.0 ** -10), (37, 33, 64, 0.5)]:
        qu = np.zeros((N, K), np.int8)
        su = np.full((N, K // 32), np.float16(7.0)).view(np.uint16)   # every other block: scale 7
        qu[i, k] = q
        su_v = su.view(np.float16).copy()
        su_v[i, k // 32] = np.float16(s)
        res = orc.read_q8(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], Wd_q=qd, Wd_scale=sd,
                          Wu_q=qu, Wu_scale=su_v.view(np.uint16), gate=rd["gate"], eps=1e-6)
        want = np.zeros((T, N))
        want[:, i] = s * q * res.lo[:, k]
        assert np.array_equal(res.u, want), f"one quant at ({i}, {k})"
    zero = np.zeros((K, N // 32), np.uint16)
    res = orc.read_q8(n, d, K, R=rd["R"], P=rd["P"], w_norm=rd["w_norm"], Wd_q=qd, Wd_scale=zero,
                      Wu_q=np.ones((N, K), np.int8), Wu_scale=np.zeros((N, K // 32), np.uint16),
                      gate=rd["gate"], eps=1e-6)
    assert np.array_equal(res.out, res.r_out.astype(np.float64)), "zero scales: out = R'"
    assert not np.any(res.lo), "zero scales: lo = 0"



# ---------------------------------------------------------------- Q2_0 matvec

def _half_bits(values):
    return np.asarray(values, np.float16).view(np.uint16)


def pin_q2_hand_packing(orc):
    """Hand-built bytes: one row of two 64-value blocks (scales 1/2 and -1/4).
    Byte 0 = 0b11100100 holds codes 0, 1, 2, 3 for values 0..3 (least
    significant bits first), byte 17 = 0b00011011 codes 3, 2, 1, 0 for values
    68..71, every other byte 0b10101010 (code 2: weight 0).  Weight =
    scale * (code - 2), so probing with unit columns gives exactly
    -1, -1/2, 0, 1/2 at values 0..3 and -1/4, 0, 1/4, 1/2 at values 68..71."""
    Wq = np.full((1, 32), 0xAA, np.uint8)
    Wq[0, 0] = 0xE4
    Wq[0, 17] = 0x1B
    Wscale = _half_bits([[0.5, -0.25]])
    y = orc.q2_0_matvec(Wq, Wscale, np.eye(128, dtype=np.float32))
    want = np.zeros(128)
    want[0:4] = [-1.0, -0.5, 0.0, 0.5]
    want[68:72] = [-0.25, 0.0, 0.25, 0.5]
    assert np.array_equal(y[:, 0], want), f"hand packing: {y[:8, 0]} ... {y[64:72, 0]}"


def pin_q2_block_sums(orc):
    """All codes 3 (weight = +scale) and all codes 0 (weight = -2 scale): y is
    the scale-weighted sum of each block's inputs, here summed exactly
    (math.fsum) from the inputs; scales differ by row and block."""
    rows, cols, ncols = 3, 192, 2
    rng = _rng(21)
    x = rng.standard_normal((ncols, cols)).astype(np.float32)
    scale = np.ldexp(1.0, -(1 + (np.arange(rows)[:, None] * 5 + np.arange(3)[None, :] * 2) % 7))
    for byte, factor in ((0xFF, 1.0), (0x00, -2.0)):
        y = orc.q2_0_matvec(np.full((rows, cols // 4), byte, np.uint8), _half_bits(scale), x)
        for c in range(ncols):
            for r in range(rows):
                want = math.fsum(factor * scale[r, b] * float(v)
                                 for b in range(3) for v in x[c, 64 * b:64 * (b + 1)])
                assert abs(y[c, r] - want) <= 1e-14 * max(1.0, abs(want)), f"block sums ({c}, {r})"


def pin_q2_probes(orc):
    """Brute force: codes drawn as an array of 0..3, packed by the input
    generator, scales random powers of two; probing with every unit column
    gives back each weight scale * (code - 2) exactly."""
    import synth
    rows, cols = 5, 128
    rng = _rng(22)
    codes = rng.integers(0, 4, size=(rows, cols))
    scale = np.ldexp(1.0, rng.integers(-12, 4, size=(rows, cols // 64))) * \
        rng.choice([-1.0, 1.0], size=(rows, cols // 64))
    y = orc.q2_0_matvec(synth.pack_q2(codes), _half_bits(scale), np.eye(cols, dtype=np.float32))
    want = (codes - 2) * np.repeat(scale, 64, axis=1)
    assert np.array_equal(y, want.T), "probed weights"


def pin_q2_invariants(orc):
    """Linear in x (a power-of-two factor scales y exactly), negating the scales
    negates y, zero scales and zero inputs give y = 0."""
    import synth
    rows, cols, ncols = 7, 256, 3
    m = synth.quantize_q2((_rng(23).standard_normal((rows, cols)) * 0.02).astype(np.float32))
    x = _rng(24).standard_normal((ncols, cols)).astype(np.float32)
    y = orc.q2_0_matvec(m.Wq, m.Wscale, x)
    assert np.array_equal(orc.q2_0_matvec(m.Wq, m.Wscale, x * np.float32(4.0)), 4.0 * y), "4 x"
    neg = (m.Wscale ^ np.uint16(0x8000)).astype(np.uint16)
    assert np.array_equal(orc.q2_0_matvec(m.Wq, neg, x), -y), "negated scales"
    assert not np.any(orc.q2_0_matvec(m.Wq, np.zeros_like(m.Wscale), x)), "zero scales"
    assert not np.any(orc.q2_0_matvec(m.Wq, m.Wscale, np.zeros_like(x))), "zero inputs"
    for c in range(ncols):
        assert np.array_equal(orc.q2_0_matvec(m.Wq, m.Wscale, x[c:c + 1])[0], y[c]), "columns independent"


ALL_PINS = [
    pin_hand_fixtures,
    pin_constant_streams,
    pin_one_hot_down,
    pin_one_hot_up,
    pin_sigmoid_values,
    pin_zero_weights,
    pin_commit_bits,
    pin_stream_permutation,
    pin_scale_invariance,
    pin_token_independence,
    pin_pending_is_committed_first,
    pin_probe_linearity,
    pin_half_decoding,
    pin_q8_equals_bf16_read,
    pin_q8_one_block,
    pin_q2_hand_packing,
    pin_q2_block_sums,
    pin_q2_probes,
    pin_q2_invariants,
]


def failing_pins(orc) -> list[str]:
    """Names of the pins the given oracle fails (used by the mutation test)."""
    bad = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except Exception:  # noqa: BLE001 - any failure counts
            bad.append(pin.__name__)
    return bad
