"""Fixed-budget decode on the GPU against the oracle's decode simulation:
slot sets and evicted positions bit-exact at every step, O / LSE within
tolerance (O max-abs 2e-2, LSE max-abs 2e-3)."""
import math

import numpy as np
import pytest

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def run_decode(wl, steps, check_seqs, float_seqs, check_every=1):
    inp = synth.make_decode(wl, steps=steps)
    f = synth.bf16_bits_to_f32
    cache = kvpop.Cache(wl.n, wl.H, wl.G, wl.D, wl.s, wl.w, wl.k)
    kp, vp = dev_bf16(inp.k_prefix), dev_bf16(inp.v_prefix)
    pp = dev(inp.prio_prefix)
    _, _, ev, _ = kvpop.mask(pp, wl.s, wl.w, wl.k, lists=False)
    cache.prefill(kp, vp, pp, ev)
    assert cache.position() == wl.P
    scale = 1 / math.sqrt(wl.D)
    # slot sets need only the priorities; floats are simulated for a subset of sequences
    ref = oracle.decode_sim(inp.k_prefix, inp.v_prefix, inp.prio_prefix, inp.q_steps, inp.k_steps,
                            inp.v_steps, inp.prio_steps, wl.s, wl.w, wl.k, scale, seqs=list(check_seqs),
                            want_floats=False)
    fs = list(float_seqs)
    if fs:
        reff = oracle.decode_sim(f(inp.k_prefix[fs]), f(inp.v_prefix[fs]), inp.prio_prefix[fs],
                                 f(inp.q_steps[:, fs]), f(inp.k_steps[:, fs]), f(inp.v_steps[:, fs]),
                                 inp.prio_steps[:, fs], wl.s, wl.w, wl.k, scale, seqs=range(len(fs)))
        for i, n in enumerate(fs):
            ref.setdefault(n, {}).update(O=reff[i]["O"], lse=reff[i]["lse"])
    qs, ks, vs = dev_bf16(inp.q_steps), dev_bf16(inp.k_steps), dev_bf16(inp.v_steps)
    ps = dev(inp.prio_steps)
    worst_o = worst_l = 0.0
    for i in range(steps):
        O, lse, evicted = cache.step(qs[i], ks[i], vs[i], ps[i])
        ev_h = host(evicted)
        if i % check_every == 0 or i == steps - 1:
            slots = host(cache.slots())
            for n in check_seqs:
                for h in range(wl.H):
                    got = np.sort(slots[n, h][slots[n, h] >= 0])
                    assert np.array_equal(got, ref[n]["slots"][i][h]), f"slots step {i} seq {n} head {h}"
                    assert ev_h[n, h] == ref[n]["evicted"][i, h], f"evicted step {i} seq {n} head {h}"
        O, lse = host(O), host(lse)
        for n in float_seqs:
            worst_l = max(worst_l, assert_close_log(lse[n], ref[n]["lse"][i], TOL_LSE, f"lse step {i}"))
            err = float(np.abs(O[n] - ref[n]["O"][i]).max())
            worst_o = max(worst_o, err)
            assert err <= TOL_O, f"O step {i} seq {n}: {err}"
    assert cache.position() == wl.P + steps
    cache.close()
    return worst_o, worst_l


@pytest.mark.parametrize("budget", [(4, 16, 24), (0, 0, 10), (3, 0, 0), (2, 7, 1), (1, 30, 500)],
                         ids=lambda b: "s{}w{}k{}".format(*b))
@pytest.mark.parametrize("D,G", [(128, 4), (64, 2)])
def test_decode_small(budget, D, G):
    s, w, k = budget
    wl = synth.DecodeWorkload("small", n=3, H=2, G=G, D=D, s=s, w=w, k=k, P=100, steps=70, seed=s + w + k)
    run_decode(wl, 70, check_seqs=range(3), float_seqs=range(3))


def test_decode_prefix_shorter_than_budget():
    wl = synth.DecodeWorkload("short", n=2, H=2, G=4, D=128, s=4, w=16, k=24, P=5, steps=60, seed=9)
    run_decode(wl, 60, check_seqs=range(2), float_seqs=range(2))


def test_decode_full_workload_sampled():
    """The decode workload's shape (64 sequences, B = 2048, 8192-token prefix):
    slot sets of every sequence, floats of sequences 0-3, for a few steps."""
    wl = synth.DECODE
    run_decode(wl, 6, check_seqs=range(wl.n), float_seqs=range(4), check_every=1)
