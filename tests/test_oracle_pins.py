"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a hand-worked example, a closed form, an
invariant the pages imply, a brute-force route or a library routine, so that a
dropped term, a wrong sign or index, or a transposed operand fails somewhere.
"""
import collections
import math
import os

import numpy as np
import pytest
import scipy.special

from fixed_budget_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TAU_ALL = np.iinfo(np.int32).max


def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def _prio_cases(rng, S):
    yield rng.random(S).astype(np.float32)
    yield rng.choice(np.array([0.0, 0.5, 1.0], np.float32), size=S)     # heavy ties
    p = rng.standard_normal(S).astype(np.float32)
    p[rng.random(S) < 0.05] = np.nan
    p[rng.random(S) < 0.05] = -0.0
    p[rng.random(S) < 0.05] = 0.0
    p[rng.random(S) < 0.02] = -np.inf
    p[rng.random(S) < 0.02] = np.inf
    yield p


# ----------------------------------------------------------------------------
# rank
# ----------------------------------------------------------------------------

def test_rank_hand_example(oracle_mod):
    fx = _read_fixture("hand_mask_example.txt")
    prio = np.array([float(x) for x in fx["prio"]], np.float32)
    assert oracle_mod.rank(prio).tolist() == [int(x) for x in fx["rank"]]


def test_rank_special_values(oracle_mod):
    # 1.0 first; the two 0.5 by index; -0.0 == +0.0 by index; NaN ties with -inf, by index
    prio = np.array([0.5, np.nan, 0.5, -np.inf, 1.0, -0.0, 0.0], np.float32)
    assert oracle_mod.rank(prio).tolist() == [1, 5, 2, 6, 0, 3, 4]


def test_rank_matches_library_sort(oracle_mod):
    rng = np.random.default_rng(1)
    for S in (1, 2, 17, 1000, 4099):
        for p in _prio_cases(rng, S):
            v = np.where(np.isnan(p), -np.inf, p.astype(np.float64))
            order = np.lexsort((np.arange(S), -v))     # primary: -v asc, then index asc
            expect = np.empty(S, np.int64)
            expect[order] = np.arange(S)
            assert (oracle_mod.rank(p) == expect).all()


# ----------------------------------------------------------------------------
# tau / mask
# ----------------------------------------------------------------------------

def test_mask_hand_example(oracle_mod):
    fx = _read_fixture("hand_mask_example.txt")
    S, s, w, k = (int(fx[x][0]) for x in ("S", "s", "w", "k"))
    prio = np.array([float(x) for x in fx["prio"]], np.float32)
    r, tau, ev = oracle_mod.mask(prio, s, w, k)
    assert tau.tolist() == [int(x) for x in fx["tau"]]
    assert ev.tolist() == [int(x) for x in fx["evict_at"]]
    assert oracle_mod.evict_at_scan(r, tau, s, w).tolist() == [int(x) for x in fx["evict_at"]]
    M = oracle_mod.mask_dense(r, tau, s, w)
    for q in range(S):
        assert np.nonzero(M[q])[0].tolist() == [int(x) for x in fx[f"row{q}"]]


BUDGETS = [(4, 32, 32), (0, 0, 5), (0, 3, 0), (2, 0, 7), (1, 1, 1), (16, 64, 200), (3, 5, 10000),
           (0, 0, 0), (5, 0, 0), (0, 100, 3)]


@pytest.mark.parametrize("s,w,k", BUDGETS)
def test_tau_fenwick_equals_bruteforce(oracle_mod, s, w, k):
    rng = np.random.default_rng(s * 1000 + w * 10 + k)
    for S in (1, 7, 300, 1500):
        for p in _prio_cases(rng, S):
            r = oracle_mod.rank(p)
            assert (oracle_mod.tau_fenwick(r, s, w, k) == oracle_mod.tau_bruteforce(r, s, w, k)).all()


@pytest.mark.parametrize("s,w,k", BUDGETS)
def test_evict_scan_equals_sweep(oracle_mod, s, w, k):
    rng = np.random.default_rng(7 + s + w + k)
    for S in (1, 9, 400, 2000):
        for p in _prio_cases(rng, S):
            r = oracle_mod.rank(p)
            tau = oracle_mod.tau_fenwick(r, s, w, k)
            assert (oracle_mod.evict_at_scan(r, tau, s, w) ==
                    oracle_mod.evict_at_sweep(r, tau, s, w, k)).all()


@pytest.mark.parametrize("s,w,k", BUDGETS)
def test_row_size_is_min_q1_B(oracle_mod, s, w, k):
    rng = np.random.default_rng(3)
    S = 600
    B = s + w + k
    for p in _prio_cases(rng, S):
        r, tau, _ = oracle_mod.mask(p, s, w, k)
        M = oracle_mod.mask_dense(r, tau, s, w)
        counts = M.sum(axis=1)
        assert (counts == np.minimum(np.arange(S) + 1, B)).all()
        assert not np.triu(M, 1).any()           # causal


@pytest.mark.parametrize("s,w,k", BUDGETS)
def test_evicted_never_returns(oracle_mod, s, w, k):
    rng = np.random.default_rng(5)
    S = 500
    for p in _prio_cases(rng, S):
        r, tau, ev = oracle_mod.mask(p, s, w, k)
        M = oracle_mod.mask_dense(r, tau, s, w)
        for q in range(S - 1):
            new = np.nonzero(M[q + 1] & ~M[q])[0]
            assert new.tolist() in ([], [q + 1])            # only the new token arrives
            assert (M[q] & ~M[q + 1]).sum() <= 1             # at most one key leaves
        # each key is retained on one contiguous interval [t, evict_at[t])
        for t in range(S):
            rows = np.nonzero(M[:, t])[0]
            assert rows.size == 0 or (rows[0] == t and rows[-1] == rows[0] + rows.size - 1)
            assert ev[t] == (rows[-1] + 1 if rows.size else t)


def test_budget_covers_sequence_is_dense(oracle_mod):
    rng = np.random.default_rng(11)
    S = 300
    for s, w, k in ((4, 32, S), (0, 0, S), (10, S, 0), (S, 0, 0)):
        for p in _prio_cases(rng, S):
            r, tau, _ = oracle_mod.mask(p, s, w, k)
            M = oracle_mod.mask_dense(r, tau, s, w)
            assert (M == np.tril(np.ones((S, S), bool))).all()


def test_k0_is_streaming_llm(oracle_mod):
    """k = 0: sinks plus window only (StreamingLLM, the pages' structural baseline)."""
    rng = np.random.default_rng(12)
    S = 400
    q = np.arange(S)[:, None]
    t = np.arange(S)[None, :]
    for s, w in ((4, 32), (0, 16), (16, 0), (0, 1)):
        p = rng.random(S).astype(np.float32)
        r, tau, _ = oracle_mod.mask(p, s, w, 0)
        M = oracle_mod.mask_dense(r, tau, s, w)
        expect = (t <= q) & ((t < s) | (q - t < w))
        assert (M == expect).all()
        assert (tau == -1).all()


def test_monotone_priorities_closed_forms(oracle_mod):
    S, k = 300, 37
    q = np.arange(S)[:, None]
    t = np.arange(S)[None, :]
    # s = w = 0, later tokens better: a sliding window of the last k tokens
    r, tau, _ = oracle_mod.mask(np.arange(S, dtype=np.float32), 0, 0, k)
    M = oracle_mod.mask_dense(r, tau, 0, 0)
    assert (M == ((t <= q) & (q - t < k))).all()
    # s = w = 0, earlier tokens better: the first k tokens forever
    r, tau, _ = oracle_mod.mask(-np.arange(S, dtype=np.float32), 0, 0, k)
    M = oracle_mod.mask_dense(r, tau, 0, 0)
    assert (M == ((t <= q) & (t < k))).all()


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def _tiny_inputs(S=96, H=2, G=2, D=16, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, S, H * G, D)).astype(np.float32)
    k = rng.standard_normal((1, S, H, D)).astype(np.float32)
    v = rng.standard_normal((1, S, H, D)).astype(np.float32)
    p = rng.random((1, H, S)).astype(np.float32)
    return q, k, v, p


def test_attn_matches_library_softmax(oracle_mod):
    S, H, G, D = 96, 2, 2, 16
    s, w, kk = 3, 8, 10
    q, k, v, p = _tiny_inputs(S, H, G, D)
    scale = 1 / math.sqrt(D)
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    O, lse = oracle_mod.attn(q, k, v, scale, r, tau, s, w)
    for j in range(H * G):
        h = j // G
        M = oracle_mod.mask_dense(r[0, h], tau[0, h], s, w)
        logits = scale * (q[0, :, j, :].astype(np.float64) @ k[0, :, h, :].astype(np.float64).T)
        logits = np.where(M, logits, -np.inf)
        ref_lse = scipy.special.logsumexp(logits, axis=1)
        ref_o = scipy.special.softmax(logits, axis=1) @ v[0, :, h, :].astype(np.float64)
        assert np.allclose(lse[0, j], ref_lse, atol=1e-12, rtol=0)
        assert np.allclose(O[0, :, j, :], ref_o, atol=1e-12, rtol=0)
    # dense causal mode
    O, lse = oracle_mod.attn(q, k, v, scale)
    for j in range(H * G):
        h = j // G
        logits = scale * (q[0, :, j, :].astype(np.float64) @ k[0, :, h, :].astype(np.float64).T)
        logits = np.where(np.tril(np.ones((S, S), bool)), logits, -np.inf)
        assert np.allclose(lse[0, j], scipy.special.logsumexp(logits, axis=1), atol=1e-12, rtol=0)
        assert np.allclose(O[0, :, j, :], scipy.special.softmax(logits, axis=1) @
                           v[0, :, h, :].astype(np.float64), atol=1e-12, rtol=0)


def test_attn_zero_queries_uniform(oracle_mod):
    S, H, G, D = 120, 2, 3, 8
    s, w, kk = 2, 10, 20
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=4)
    q[:] = 0
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    O, lse = oracle_mod.attn(q, k, v, 0.3, r, tau, s, w)
    B = s + w + kk
    for j in range(H * G):
        h = j // G
        assert np.allclose(lse[0, j], np.log(np.minimum(np.arange(S) + 1, B)), atol=1e-13)
        M = oracle_mod.mask_dense(r[0, h], tau[0, h], s, w)
        for qq in range(0, S, 7):
            sel = np.nonzero(M[qq])[0]
            assert np.allclose(O[0, qq, j], v[0, sel, h].astype(np.float64).mean(axis=0), atol=1e-13)


def test_attn_sparse_equals_dense_when_budget_covers(oracle_mod):
    S, H, G, D = 80, 1, 4, 16
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=9)
    r, tau, _ = oracle_mod.mask(p, 2, 5, S)
    Os, ls = oracle_mod.attn(q, k, v, 0.25, r, tau, 2, 5)
    Od, ld = oracle_mod.attn(q, k, v, 0.25)
    assert np.array_equal(ls, ld) and np.array_equal(Os, Od)


def test_attn_head_group_mapping(oracle_mod):
    """Query head j reads KV head j // G (contiguous groups)."""
    S, H, G, D = 40, 3, 2, 8
    q, k, v, _ = _tiny_inputs(S, H, G, D, seed=21)
    O, lse = oracle_mod.attn(q, k, v, 0.5)
    for j in range(H * G):
        O1, l1 = oracle_mod.attn(q[:, :, j:j + 1], k[:, :, j // G:j // G + 1], v[:, :, j // G:j // G + 1], 0.5)
        assert np.array_equal(O1[0, :, 0], O[0, :, j]) and np.array_equal(l1[0, 0], lse[0, j])


# ----------------------------------------------------------------------------
# future-attention target
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("w", [0, 1, 7, 40])
def test_target_routes_agree(oracle_mod, w):
    S, H, G, D = 90, 2, 2, 16
    q, k, _, _ = _tiny_inputs(S, H, G, D, seed=w)
    scale = 1 / math.sqrt(D)
    _, lse = oracle_mod.attn(q, k, k, scale, want_o=False)
    tb = oracle_mod.target_lse(q, k, lse, w, scale)
    ta = oracle_mod.target_colsum(q, k, w, scale)
    fin = np.isfinite(ta)
    assert (fin == np.isfinite(tb)).all()
    assert np.allclose(ta[fin], tb[fin], atol=1e-11, rtol=0)
    # empty future: t + w > S - 1 gives -inf, everything else finite
    t = np.arange(S)
    assert (np.isneginf(ta[..., t + w > S - 1])).all() and fin[..., t + w <= S - 1].all()


def test_target_mass_conservation_w0(oracle_mod):
    """w = 0: every query row's probabilities sum to 1, so sum_t exp(target) = S * G."""
    S, H, G, D = 100, 2, 4, 16
    q, k, _, _ = _tiny_inputs(S, H, G, D, seed=31)
    scale = 1 / math.sqrt(D)
    _, lse = oracle_mod.attn(q, k, k, scale, want_o=False)
    tb = oracle_mod.target_lse(q, k, lse, 0, scale)
    assert np.allclose(np.exp(tb).sum(axis=-1), S * G, rtol=1e-12)


def test_target_zero_queries_harmonic(oracle_mod):
    """q = 0: A_{d,t} = 1/(d+1), so target_t = log(G * sum_{d=t+w}^{S-1} 1/(d+1))."""
    S, H, G, D, w = 70, 1, 3, 8, 5
    q, k, _, _ = _tiny_inputs(S, H, G, D, seed=2)
    q[:] = 0
    _, lse = oracle_mod.attn(q, k, k, 1.0, want_o=False)
    tb = oracle_mod.target_lse(q, k, lse, w, 1.0)
    for t in range(S):
        if t + w > S - 1:
            assert np.isneginf(tb[0, 0, t])
        else:
            ref = math.log(G * sum(1.0 / (d + 1) for d in range(t + w, S)))
            assert abs(tb[0, 0, t] - ref) < 1e-12


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

def _cache_simulation(prio, s, w, k):
    """Step-by-step fixed-budget cache, written from the inference description:
    sinks stay, the newest w tokens are protected, and the token leaving the
    window competes with the worst held long-range token by priority."""
    S = prio.shape[0]
    val = lambda t: -np.inf if np.isnan(prio[t]) else float(prio[t])
    sinks, window, topk = [], collections.deque(), []
    sets, evicted = [], []
    for qq in range(S):
        ev = -1
        if qq < s:
            sinks.append(qq)
        else:
            window.append(qq)
            if len(window) > w:
                u = window.popleft()
                if len(topk) < k:
                    topk.append(u)
                elif k == 0:
                    ev = u
                else:
                    m = min(topk, key=lambda t: (val(t), -t))      # worst: lowest prio, later index
                    if val(u) > val(m):
                        topk[topk.index(m)] = u
                        ev = m
                    else:
                        ev = u
        sets.append(sorted(sinks + list(window) + topk))
        evicted.append(ev)
    return sets, evicted


@pytest.mark.parametrize("s,w,k", [(2, 5, 6), (0, 0, 4), (3, 0, 0), (1, 8, 1), (4, 3, 50)])
def test_decode_sim_matches_cache_simulation(oracle_mod, s, w, k):
    rng = np.random.default_rng(s + 10 * w + 100 * k)
    n, H, G, D, P, T = 2, 2, 2, 8, 30, 40
    kp = rng.standard_normal((n, P, H, D)).astype(np.float32)
    vp = rng.standard_normal((n, P, H, D)).astype(np.float32)
    pp = rng.choice(np.array([0.1, 0.2, 0.3, 0.5], np.float32), size=(n, H, P))
    qs = rng.standard_normal((T, n, H * G, D)).astype(np.float32)
    ks = rng.standard_normal((T, n, H, D)).astype(np.float32)
    vs = rng.standard_normal((T, n, H, D)).astype(np.float32)
    ps = rng.choice(np.array([0.1, 0.2, 0.3, 0.5], np.float32), size=(T, n, H))
    res = oracle_mod.decode_sim(kp, vp, pp, qs, ks, vs, ps, s, w, k, 0.4, seqs=[0, 1])
    for nn in (0, 1):
        for h in range(H):
            prio = np.concatenate([pp[nn, h], ps[:, nn, h]])
            sets, evicted = _cache_simulation(prio, s, w, k)
            for i in range(T):
                assert res[nn]["slots"][i][h].tolist() == sets[P + i]
                assert res[nn]["evicted"][i, h] == evicted[P + i]
        # floats: attention over the held set, via the library softmax
        for i in range(0, T, 9):
            for j in range(H * G):
                h = j // G
                sel = res[nn]["slots"][i][h]
                kh = np.concatenate([kp[nn, :, h], ks[:, nn, h]])[sel].astype(np.float64)
                vh = np.concatenate([vp[nn, :, h], vs[:, nn, h]])[sel].astype(np.float64)
                lg = 0.4 * kh @ qs[i, nn, j].astype(np.float64)
                assert abs(res[nn]["lse"][i, j] - scipy.special.logsumexp(lg)) < 1e-12
                assert np.allclose(res[nn]["O"][i, j], scipy.special.softmax(lg) @ vh, atol=1e-12)


# ----------------------------------------------------------------------------
# generator
# ----------------------------------------------------------------------------

def test_generator_matches_scalar_definition():
    """The vectorised draws equal a scalar restatement of the stated generator."""
    M64 = (1 << 64) - 1

    def mix(z):
        z ^= z >> 30
        z = (z * 0xBF58476D1CE4E5B9) & M64
        z ^= z >> 27
        z = (z * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)

    seed, stream = 3, synth.K
    key = mix(((seed * 0x9E3779B97F4A7C15) & M64) ^ ((stream * 0xD1B54A32D192ED03) & M64))
    draws = [mix((key + (i + 1) * 0x9E3779B97F4A7C15) & M64) for i in range(10)]
    assert synth.raw_draws(seed, stream, 0, 10).tolist() == draws
    u = synth.uniform24(seed, stream, 10)
    assert u.tolist() == [np.float32((z >> 40) * 2.0 ** -24) for z in draws]
    nrm = synth.normal(seed, stream, 5)
    for i in range(5):
        u1 = ((draws[2 * i] >> 11) + 1) * 2.0 ** -53
        u2 = (draws[2 * i + 1] >> 11) * 2.0 ** -53
        assert nrm[i] == np.float32(math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2))
    # bf16 round-to-nearest-even
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], np.float32)
    b = synth.f32_to_bf16_bits(x)
    assert synth.bf16_bits_to_f32(b).tolist() == [1.0, 1.0, 1.015625, -2.5, np.float32(0.0030059814453125)]
