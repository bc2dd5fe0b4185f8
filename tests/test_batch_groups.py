"""Host logic of hc_read_batch: which reads of a batch must run in order
(hc_read_batch_groups), checked on the CPU with made-up addresses that are
compared but never dereferenced, against a brute-force partition written
from the rule itself: reads j and k are linked when a byte range of one's
outputs overlaps any range (input or output) of the other, and groups are the
connected components of that relation."""

import ctypes
import random

import pytest

hc = pytest.importorskip("hyper_connection_residual_gb300")

G = (4, 2560, 320)  # n, d, K
N = G[0] * G[1]
ORDER_IN = ("R", "pending", "w_norm", "gate", "W_down", "W_up")
ORDER_OUT = ("out", "mean", "lo")


def sizes(T):
    n, d, K = G
    return {"R": T * N * 4, "pending": T * N * 4, "w_norm": N * 4, "gate": N * 4,
            "W_down": N * K * 2, "W_up": N * K * 2,
            "out": T * N * 4, "mean": T * d * 4, "lo": T * K * 4}


class Arena:
    """Disjoint 256-byte aligned address ranges."""

    def __init__(self, base=1 << 40):
        self.next = base

    def take(self, nbytes):
        a = self.next
        self.next += (nbytes + 255) // 256 * 256 + 4096
        return a


def read(arena, T, weights, **over):
    sz = sizes(T)
    r = {"R": arena.take(sz["R"]), "pending": None, **weights,
         "out": arena.take(sz["out"]), "mean": arena.take(sz["mean"]), "lo": arena.take(sz["lo"])}
    r.update(over)
    return r


def weights(arena):
    sz = sizes(1)
    return {k: arena.take(sz[k]) for k in ("w_norm", "gate", "W_down", "W_up")}


def brute_partition(reads, T):
    sz = sizes(T)

    def rng(r, k):
        a = r.get(k)
        return None if a is None else (a, a + sz[k])

    def hit(a, b):
        return a is not None and b is not None and a[0] < b[1] and b[0] < a[1]

    m = len(reads)
    parent = list(range(m))

    def find(x):
        while parent[x] != x:
            x = parent[x]
        return x

    for j in range(m):
        for k in range(m):
            if j == k:
                continue
            outs_j = [rng(reads[j], o) for o in ORDER_OUT]
            all_k = [rng(reads[k], o) for o in ORDER_IN + ORDER_OUT]
            if any(hit(a, b) for a in outs_j for b in all_k):
                parent[find(j)] = find(k)
    ids, out = {}, []
    for j in range(m):
        out.append(ids.setdefault(find(j), len(ids)))
    return out


def groups(reads, T):
    return hc.hc_read_batch_groups(G, reads, T)


def test_independent_reads_sharing_inputs_are_separate_groups():
    a = Arena()
    w = weights(a)
    R = a.take(sizes(4)["R"])
    P = a.take(sizes(4)["pending"])
    reads = [read(a, 4, w, R=R, pending=P) for _ in range(10)]
    assert groups(reads, 4) == list(range(10))


def test_chain_is_one_group():
    a = Arena()
    w = weights(a)
    reads = [read(a, 2, w)]
    for _ in range(5):
        reads.append(read(a, 2, w, R=reads[-1]["out"]))
    assert groups(reads, 2) == [0] * 6


def test_shared_output_buffers_are_one_group():
    a = Arena()
    w = weights(a)
    first = read(a, 1, w)
    reads = [first] + [read(a, 1, w, out=first["out"]) for _ in range(3)]
    assert groups(reads, 1) == [0, 0, 0, 0]
    # only the mean shared: still ordered
    reads = [first, read(a, 1, w, mean=first["mean"])]
    assert groups(reads, 1) == [0, 0]


def test_write_after_read_links_reads():
    a = Arena()
    w = weights(a)
    r0 = read(a, 3, w)
    r1 = read(a, 3, w, out=r0["R"])  # writes what read 0 takes as R
    r2 = read(a, 3, w)
    assert groups([r0, r1, r2], 3) == [0, 0, 1]


def test_in_place_read_is_its_own_group():
    a = Arena()
    w = weights(a)
    reads = []
    for _ in range(4):
        r = read(a, 4, w)
        r["out"] = r["R"]
        reads.append(r)
    assert groups(reads, 4) == [0, 1, 2, 3]


def test_transitive_links_and_first_appearance_numbering():
    a = Arena()
    w = weights(a)
    r = [read(a, 1, w) for _ in range(6)]
    r[4]["R"] = r[1]["out"]   # 1 - 4
    r[5]["pending"] = r[4]["out"]  # 4 - 5
    r[2]["pending"] = r[0]["out"]  # 0 - 2
    assert groups(r, 1) == [0, 1, 0, 2, 1, 1]
    assert groups(r, 1) == brute_partition(r, 1)


def test_weight_pointer_into_another_reads_output_links_them():
    a = Arena()
    w = weights(a)
    r0 = read(a, 1, w)
    far = Arena(base=1 << 44)
    r1 = read(far, 1, weights(far))
    r1["w_norm"] = r0["out"]
    assert groups([r0, r1], 1) == [0, 0]


def test_overlap_by_one_byte_and_adjacent_ranges():
    a = Arena()
    w = weights(a)
    T = 1
    r0 = read(a, T, w)
    lo_end = r0["lo"] + sizes(T)["lo"]
    r1 = read(a, T, w, mean=lo_end)          # starts where r0's lo ends: disjoint
    r2 = read(a, T, w, mean=lo_end - 4)      # overlaps r0's lo by 4 bytes
    assert groups([r0, r1], T) == [0, 1]
    assert groups([r0, r2], T) == [0, 0]


def test_weights_shared_by_every_read_do_not_link_them():
    a = Arena()
    w = weights(a)
    reads = [read(a, 8, w) for _ in range(5)]
    assert groups(reads, 8) == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("seed", range(12))
def test_random_layouts_match_brute_force(seed):
    rnd = random.Random(seed)
    T = rnd.choice((1, 2, 4, 8))
    sz = sizes(T)
    a = Arena()
    pool = [a.take(sz["R"]) for _ in range(6)]  # buffers big enough for any role
    wsets = [weights(a) for _ in range(3)]
    reads = []
    for _ in range(rnd.randint(1, 24)):
        r = read(a, T, rnd.choice(wsets))
        for k in ("R", "pending", "out", "mean", "lo"):
            if rnd.random() < 0.25:
                r[k] = rnd.choice(pool) + 256 * rnd.randint(0, 3)
        if rnd.random() < 0.1:
            r["W_down"] = rnd.choice(pool)
        reads.append(r)
    assert groups(reads, T) == brute_partition(reads, T)


def test_group_count_return_and_argument_errors():
    lib = hc.load()
    a = Arena()
    w = weights(a)
    reads = [read(a, 1, w) for _ in range(3)]
    arr = hc._binding._descs(G, reads, 1)
    out = (ctypes.c_int * 3)()
    assert lib.hc_read_batch_groups(arr, 3, *G, 1, out) == 3
    assert lib.hc_read_batch_groups(None, 3, *G, 1, out) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_groups(arr, 0, *G, 1, out) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_groups(arr, 3, *G, 0, out) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_groups(arr, 3, *G, 1, None) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_plan(None, arr, 3, 1) == hc.HC_ERR_ARG


# ---- Q8_0 reads: quants one byte per weight, scales as further inputs

ORDER_IN_Q8 = ("R", "pending", "w_norm", "gate", "Wd_q", "Wd_scale", "Wu_q", "Wu_scale")


def sizes_q8(T):
    n, d, K = G
    sz = sizes(T)
    return {**{k: sz[k] for k in ("R", "pending", "w_norm", "gate", "out", "mean", "lo")},
            "Wd_q": N * K, "Wu_q": N * K, "Wd_scale": N * K // 32 * 2, "Wu_scale": N * K // 32 * 2}


def q8_weights(arena):
    sz = sizes_q8(1)
    return {k: arena.take(sz[k]) for k in ("w_norm", "gate", "Wd_q", "Wd_scale", "Wu_q", "Wu_scale")}


def brute_partition_q8(reads, T):
    sz = sizes_q8(T)

    def rng(r, k):
        a = r.get(k)
        return None if a is None else (a, a + sz[k])

    m = len(reads)
    parent = list(range(m))

    def find(x):
        while parent[x] != x:
            x = parent[x]
        return x

    for j in range(m):
        for k in range(m):
            if j != k and any(a and b and a[0] < b[1] and b[0] < a[1]
                              for a in (rng(reads[j], o) for o in ORDER_OUT)
                              for b in (rng(reads[k], o) for o in ORDER_IN_Q8 + ORDER_OUT)):
                parent[find(j)] = find(k)
    ids = {}
    return [ids.setdefault(find(j), len(ids)) for j in range(m)]


def q8_groups(reads, T):
    return hc.hc_read_batch_q8_groups(G, reads, T)


def test_q8_output_into_a_scale_array_links_reads():
    a = Arena()
    w = q8_weights(a)
    r0 = read(a, 1, w)
    far = Arena(base=1 << 44)
    r1 = read(far, 1, q8_weights(far))
    r1["Wu_scale"] = r0["lo"]  # scales are inputs: written by read 0
    assert q8_groups([r0, r1], 1) == [0, 0]
    # the byte just past read 1's Wd_scale array is not part of it
    r2 = read(far, 1, q8_weights(far))
    r0b = read(a, 1, w, lo=r2["Wd_scale"] + sizes_q8(1)["Wd_scale"])  # 1280 bytes, inside the gap
    assert q8_groups([r0b, r2], 1) == [0, 1]


def test_q8_quant_range_is_one_byte_per_weight():
    a = Arena()
    w = q8_weights(a)
    r0 = read(a, 1, w)
    r1 = read(a, 1, w)
    # an output placed right after r0's Wd_q bytes (N*K, not N*K*2) stays apart
    r1["lo"] = w["Wd_q"] + N * G[2]
    assert q8_groups([r0, r1], 1) == [0, 1]
    r1["lo"] = w["Wd_q"] + N * G[2] - 4
    assert q8_groups([r0, r1], 1) == [0, 0]


@pytest.mark.parametrize("seed", range(8))
def test_q8_random_layouts_match_brute_force(seed):
    rnd = random.Random(100 + seed)
    T = rnd.choice((1, 2, 4, 8))
    sz = sizes_q8(T)
    a = Arena()
    pool = [a.take(sz["R"]) for _ in range(6)]
    wsets = [q8_weights(a) for _ in range(3)]
    reads = []
    for _ in range(rnd.randint(1, 24)):
        r = read(a, T, rnd.choice(wsets))
        for k in ("R", "pending", "out", "mean", "lo"):
            if rnd.random() < 0.25:
                r[k] = rnd.choice(pool) + 256 * rnd.randint(0, 3)
        for k in ("Wd_scale", "Wu_scale"):
            if rnd.random() < 0.1:
                r[k] = rnd.choice(pool) + 2 * rnd.randint(0, 7)
        reads.append(r)
    assert q8_groups(reads, T) == brute_partition_q8(reads, T)


def test_q8_group_argument_errors():
    lib = hc.load()
    a = Arena()
    w = q8_weights(a)
    reads = [read(a, 1, w) for _ in range(2)]
    arr = hc._binding._q8_descs(G, reads, 1)
    out = (ctypes.c_int * 2)()
    assert lib.hc_read_batch_q8_groups(arr, 2, *G, 1, out) == 2
    assert lib.hc_read_batch_q8_groups(arr, 2, 4, 2560, 300, 1, out) == hc.HC_ERR_ARG  # K not a multiple of 32
    assert lib.hc_read_batch_q8_groups(None, 2, *G, 1, out) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_q8_plan(None, arr, 2, 1) == hc.HC_ERR_ARG
    assert lib.hc_read_batch_q8(None, arr, 2, 1, None) == hc.HC_ERR_ARG
