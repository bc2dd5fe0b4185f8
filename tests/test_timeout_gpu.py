"""The timeout path of the read's bounded waits, exercised on purpose.

A kernel's bounded wait that runs out records a bit in the handle's error
word, carries on with what is in shared memory (its results are void), and
drains its copies before it exits; hc_read_check then reports
HC_ERR_TIMEOUT until hc_read_reset.  hc_read_set_wait_limit shortens the
first bulk-copy wait of the down kernel (counted from the kernel's start) to
a few nanoseconds, so that wait gives up whether or not its copy has landed.
Nothing here faults or hangs: the copy lands, the drain waits for it with its
full bound, and the GPU context stays usable (the next read passes parity).
"""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import EPS, assert_parity, dev_act, dev_weights, outputs, run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

hc = pytest.importorskip("hyper_connection_residual_gb300")

# The down kernel's first bulk-copy wait and its error bit: w_norm (bit 1) in
# the CUDA-core kernel of T = 1, the weight tile (bit 2) in the others.
CASES = [(synth.G1, 1, 1), (synth.G1, 4, 2), (synth.G1, 8, 2), (synth.G2, 4, 2), (synth.G2, 8, 2)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    hc.load()
    return d


@pytest.mark.parametrize("g,T,bit", CASES, ids=[f"d{g.d}_T{T}" for g, T, _ in CASES])
def test_first_wait_runs_out_and_reports(dev, g, T, bit):
    ws = synth.weight_set(g, 7)
    w = dev_weights(ws, dev)
    act = synth.activations(g, T, True, s0=70 + T)
    a = dev_act(act, dev)
    ref = oracle.default().read(g.n, g.d, g.K, R=act.R, P=act.P, w_norm=ws.w_norm, W_down=ws.W_down,
                                W_up=ws.W_up, gate=ws.gate, eps=EPS)
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
        o = outputs(g, T, dev)
        rd.set_wait_limit(2)  # ns from the kernel's start: over before the first wait
        run(rd, w, a, T, o)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_ERR_TIMEOUT
        word = rd.error_word()
        assert word & bit, f"error word {word:#x} lacks bit {bit}"
        assert word & ~3 == 0, f"error word {word:#x}: only the down kernel's copy waits may run out"
        # The record stays until reset; a read with the default limit is whole again.
        rd.reset()
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
        rd.set_wait_limit(0)
        o = outputs(g, T, dev)
        run(rd, w, a, T, o)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
        assert_parity(o, ref, T, f"after the timeout, d={g.d} T={T}")


def test_timeout_on_the_batch_lanes(dev):
    """Reads of a batch on the internal streams take the handle's limit too;
    after a reset the same batch is whole."""
    g, T = synth.G1, 2
    sets = [synth.weight_set(g, j) for j in range(3)]
    acts = [synth.activations(g, T, False, s0=90 + j) for j in range(3)]
    ws = [dev_weights(s, dev) for s in sets]
    av = [dev_act(a, dev) for a in acts]
    with hc.Read(g.n, g.d, g.K, T_max=8, eps=EPS) as rd:
        outs = [outputs(g, T, dev) for _ in range(3)]
        reads = [dict(R=av[j]["R"], P=None, out=outs[j]["out"], mean=outs[j]["mean"], lo=outs[j]["lo"],
                      **ws[j]) for j in range(3)]
        assert rd.batch_plan(reads, T) >= 2
        rd.set_wait_limit(2)
        rd.batch(reads, T)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_ERR_TIMEOUT
        rd.reset()
        rd.set_wait_limit(0)
        rd.batch(reads, T)
        torch.cuda.synchronize()
        assert rd.check() == hc.HC_OK
        for j in range(3):
            ref = oracle.default().read(g.n, g.d, g.K, R=acts[j].R, P=None, w_norm=sets[j].w_norm,
                                        W_down=sets[j].W_down, W_up=sets[j].W_up, gate=sets[j].gate, eps=EPS)
            for name, want in (("lo", ref.lo), ("out", ref.out), ("mean", ref.mean)):
                got = outs[j][name].double().cpu().numpy()
                err = float(np.max(np.abs(got - want)))
                assert err <= 1e-4 * float(np.max(np.abs(want))), f"batch read {j} {name}"
