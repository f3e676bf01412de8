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


def _decode_inputs(wl, steps):
    """Step tokens and priorities on the host; the prefix K/V on the device.  Large
    prefixes are generated on the device and the oracle regenerates only the
    sequences whose floats it checks (element i of a tensor is draw i)."""
    n, P, H, D, Hq = wl.n, wl.P, wl.H, wl.D, wl.Hq
    shp = (n, P, H, D)
    pp = synth.priorities("uniform", wl.seed, (n, H, P))
    qs = synth.bf16_block(wl.seed, synth.QN, (steps, n, Hq, D), 0)
    ks = synth.bf16_block(wl.seed, synth.KN, (steps, n, H, D), 0)
    vs = synth.bf16_block(wl.seed, synth.VN, (steps, n, H, D), 0)
    ps = synth.priorities("uniform", wl.seed, (steps, n, H), stream=synth.PRION)
    if n * P * H * D > (1 << 26):
        kp = synth.normal_bf16_torch(wl.seed, synth.K, shp, "cuda")
        vp = synth.normal_bf16_torch(wl.seed, synth.V, shp, "cuda")
    else:
        kp = dev_bf16(synth.bf16_block(wl.seed, synth.K, shp, 0))
        vp = dev_bf16(synth.bf16_block(wl.seed, synth.V, shp, 0))

    def prefix_f32(seqs, stream):
        blocks = [synth.bf16_block(wl.seed, stream, (P, H, D), i * P * H * D) for i in seqs]
        return synth.bf16_bits_to_f32(np.stack(blocks)) if blocks else np.zeros((0, P, H, D), np.float32)

    return kp, vp, pp, qs, ks, vs, ps, prefix_f32


def run_decode(wl, steps, check_seqs, float_seqs, check_every=1):
    kp, vp, prio_prefix, q_steps, k_steps, v_steps, prio_steps, prefix_f32 = _decode_inputs(wl, steps)
    f = synth.bf16_bits_to_f32
    cache = kvpop.Cache(wl.n, wl.H, wl.G, wl.D, wl.s, wl.w, wl.k)
    pp = dev(prio_prefix)
    _, _, ev, _ = kvpop.mask(pp, wl.s, wl.w, wl.k, lists=False)
    cache.prefill(kp, vp, pp, ev)
    assert cache.position() == wl.P
    scale = 1 / math.sqrt(wl.D)
    # slot sets need only the priorities and shapes; floats are simulated for a subset
    shape_only = np.empty((wl.n, wl.P, wl.H, wl.D), np.uint16)
    ref = oracle.decode_sim(shape_only, shape_only, prio_prefix, q_steps, k_steps, v_steps, prio_steps,
                            wl.s, wl.w, wl.k, scale, seqs=list(check_seqs), want_floats=False)
    fs = list(float_seqs)
    if fs:
        reff = oracle.decode_sim(prefix_f32(fs, synth.K), prefix_f32(fs, synth.V), prio_prefix[fs],
                                 f(q_steps[:, fs]), f(k_steps[:, fs]), f(v_steps[:, fs]),
                                 prio_steps[:, fs], wl.s, wl.w, wl.k, scale, seqs=range(len(fs)))
        for i, n in enumerate(fs):
            ref.setdefault(n, {}).update(O=reff[i]["O"], lse=reff[i]["lse"])
    qs, ks, vs = dev_bf16(q_steps), dev_bf16(k_steps), dev_bf16(v_steps)
    ps = dev(prio_steps)
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
    slot sets and evicted positions of all 64 sequences at each of 64 steps (every
    step evicts: the prefix is longer than the budget), floats of sequences 0-3."""
    wl = synth.DECODE
    run_decode(wl, 64, check_seqs=range(wl.n), float_seqs=range(4), check_every=1)
