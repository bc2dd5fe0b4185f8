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
