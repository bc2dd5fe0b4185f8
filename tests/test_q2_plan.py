"""The Q2_0 batch's split into launches (host logic, no GPU), against a
plain restatement over random layouts of a few buffers."""

import random

import pytest

import hyper_connection_residual_gb300 as hc
from hyper_connection_residual_gb300 import build as hcbuild

ROWS, COLS, NCOLS = 128, 512, 2
WQ, WS, X, Y = ROWS * COLS // 4, ROWS * (COLS // 64) * 2, NCOLS * COLS * 4, NCOLS * ROWS * 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    hcbuild.build()
    return hc.load()


def overlap(a, an, b, bn):
    return a < b + bn and b < a + an


def shares(d, e):
    """d (later) reads e's y, or writes its y over any operand of e."""
    return (overlap(d[2], X, e[3], Y) or overlap(d[0], WQ, e[3], Y) or overlap(d[1], WS, e[3], Y)
            or overlap(d[3], Y, e[3], Y) or overlap(d[3], Y, e[2], X) or overlap(d[3], Y, e[0], WQ)
            or overlap(d[3], Y, e[1], WS))


def plan(products):
    out, first, size = [], 0, 0
    for j, d in enumerate(products):
        new = j == 0 or size == 120 or any(shares(d, products[i]) for i in range(first, j))
        if new:
            first, size = j, 0
            out.append(out[-1] + 1 if out else 0)
        else:
            out.append(out[-1])
        size += 1
    return out


def test_independent_products_share_a_launch():
    base = 1 << 40
    prods = [(base + i * (1 << 24), base + i * (1 << 24) + (1 << 22), 7 << 40, base + i * (1 << 24) + (1 << 23))
             for i in range(300)]
    got = hc.hc_q2_0_matvec_batch_plan(prods, ROWS, COLS, NCOLS)
    assert got == [j // 120 for j in range(300)]


def test_random_layouts_match_restatement():
    rng = random.Random(3)
    pool = [(1 << 40) + k * 4096 for k in range(24)]  # 16-byte-aligned slots, some ranges overlap
    for _ in range(300):
        n = rng.randint(1, 12)
        prods = []
        for _ in range(n):
            wq, ws, x, y = (rng.choice(pool) for _ in range(4))
            prods.append((wq, ws + 8192 * 64, x + 8192 * 128, y + 8192 * 192))
        got = hc.hc_q2_0_matvec_batch_plan(prods, ROWS, COLS, NCOLS)
        assert got == plan(prods), prods


def test_chain_splits_every_product():
    a, b = 1 << 40, 2 << 40
    # y of each product is the x of the next (square shape so sizes match)
    n = 512
    xs = [(3 << 40) + k * (1 << 20) for k in range(6)]
    prods = [(a + k * (1 << 22), b + k * (1 << 22), xs[k], xs[k + 1]) for k in range(5)]
    assert hc.hc_q2_0_matvec_batch_plan(prods, n, n, 1) == [0, 1, 2, 3, 4]


def test_plan_argument_errors():
    one = [(1 << 40, 2 << 40, 3 << 40, 4 << 40)]
    with pytest.raises(hc.HcError):
        hc.hc_q2_0_matvec_batch_plan([], ROWS, COLS, NCOLS)
    with pytest.raises(hc.HcError) as e:
        hc.hc_q2_0_matvec_batch_plan(one, ROWS, COLS + 64, NCOLS)
    assert e.value.status == hc.HC_ERR_SHAPE
    with pytest.raises(hc.HcError):
        hc.hc_q2_0_matvec_batch_plan(one, ROWS, COLS, 5)
