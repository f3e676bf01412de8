"""kvpop_mask on the GPU against the fp64 oracle: bit-exact rank, tau,
evict_at and long-range lists, from tiny inputs to the full workloads."""
import numpy as np
import pytest

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def expected_lists(ev, s, w, k, S):
    """list i = {t in [s, 64 i - w] : evict_at[t] > 64 i} (from the oracle's evict_at): first
    the keys still held at row 64 i + 63, then those dropped inside the block, each sorted."""
    out = []
    for i in range((S + 63) // 64):
        q0 = 64 * i
        t = np.arange(s, max(s, q0 - w + 1))
        held = t[ev[t] > q0]
        order = np.concatenate([held[ev[held] > q0 + 63], held[ev[held] <= q0 + 63]])
        out.append(np.stack([order, ev[order]], axis=1) if order.size else np.zeros((0, 2), np.int64))
    return out


def check(prio, s, w, k, lists=True, full_lists=True):
    b, H, S = prio.shape
    r, tau, ev, lst = kvpop.mask(dev(prio), s, w, k, lists=lists)
    r, tau, ev = host(r), host(tau), host(ev)
    ro = oracle.rank(prio)
    to = oracle.tau_fenwick(ro, s, w, k)
    eo = oracle.evict_at_sweep(ro, to, s, w, k)
    assert np.array_equal(r, ro), "rank"
    assert np.array_equal(tau, to), "tau"
    assert np.array_equal(ev, eo), "evict_at"
    if lists and k > 0:
        lh = host(lst)
        for bi in range(b):
            for h in range(H) if full_lists else [0, H - 1]:
                exp = expected_lists(eo[bi, h], s, w, k, S)
                for i, e in enumerate(exp):
                    assert e.shape[0] == min(k, max(0, 64 * i - w - s + 1))
                    assert np.array_equal(lh[bi, h, i, :e.shape[0]], e), f"list {bi},{h},{i}"
    return r, tau, ev


def _prio(rng, shape, kind):
    if kind == "uniform":
        return rng.random(shape).astype(np.float32)
    if kind == "ties":
        return rng.choice(np.array([0.0, 0.5, 1.0], np.float32), size=shape)
    p = rng.standard_normal(shape).astype(np.float32)
    p[rng.random(shape) < 0.03] = np.nan
    p[rng.random(shape) < 0.03] = -0.0
    p[rng.random(shape) < 0.03] = 0.0
    p[rng.random(shape) < 0.01] = -np.inf
    p[rng.random(shape) < 0.01] = np.inf
    return p


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 1000, 2048, 2049, 5000])
@pytest.mark.parametrize("kind", ["uniform", "ties", "special"])
def test_mask_small(S, kind):
    rng = np.random.default_rng(S * 7 + len(kind))
    prio = _prio(rng, (2, 3, S), kind)
    for s, w, k in [(4, 32, 32), (0, 0, 5), (2, 0, 7), (0, 3, 0), (1, 1, 1), (16, 64, 200), (3, 5, S + 10)]:
        check(prio, s, w, k)


def test_mask_hand_example():
    prio = np.array([[[9, 0.3, 0.9, 0.1, 0.5, 0.7, 0.2, 0.4]]], np.float32)
    r, tau, ev = check(prio, 1, 2, 2)
    assert ev[0, 0].tolist() == [8, 6, 8, 5, 7, 8, 8, 8]


@pytest.mark.parametrize("S", [8191, 8193, 16384, 40000])
def test_mask_cluster_sizes(S):
    """S above 8192 builds the wavelet matrix across a cluster of CTAs."""
    rng = np.random.default_rng(S)
    prio = _prio(rng, (1, 2, S), "uniform")
    check(prio, 16, 512, 1520, full_lists=False)
    prio = _prio(rng, (1, 1, S), "ties")
    check(prio, 3, 100, 700, full_lists=False)


def test_mask_tiny_workload():
    wl = synth.TINY
    prio = synth.priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))
    check(prio, wl.s, wl.w, wl.k)


@pytest.mark.parametrize("wl", [synth.QWEN3_4B, synth.QWEN3_8B, synth.LONG], ids=lambda w: w.name)
def test_mask_full_workloads(wl):
    prio = synth.priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))
    check(prio, wl.s, wl.w, wl.k, full_lists=False)


def test_mask_row_invariants_full():
    """Every row holds min(q+1, B) keys and each key is held on one interval."""
    wl = synth.QWEN3_8B
    prio = synth.priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))
    _, _, ev = kvpop.mask(dev(prio), wl.s, wl.w, wl.k, lists=False)[:3]
    ev = host(ev)
    S, B = wl.S, wl.B
    t = np.arange(S)
    for bi in range(wl.b):
        for h in range(wl.H):
            e = ev[bi, h]
            assert (e >= np.minimum(t + wl.w, S))[wl.s:].all() and (e[:wl.s] == S).all()
            # row sizes from the interval form: #{t <= q < e_t}
            diff = np.zeros(S + 1, np.int64)
            np.add.at(diff, t, 1)
            np.add.at(diff, e, -1)
            assert (np.cumsum(diff)[:S] == np.minimum(t + 1, B)).all()
