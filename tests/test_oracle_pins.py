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
# attention backward
# ----------------------------------------------------------------------------

_BWD_BUDGETS = [(3, 8, 10), (0, 0, 12), (2, 6, 0), (1, 0, 5), (4, 200, 200)]


@pytest.mark.parametrize("s,w,kk", _BWD_BUDGETS)
def test_attn_bwd_matches_autograd(oracle_mod, s, w, kk):
    """The hand-written chain rule against torch autograd (fp64, CPU) of the
    masked softmax attention written with an explicit mask matrix."""
    torch = pytest.importorskip("torch")
    S, H, G, D = 72, 2, 3, 8
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=31 + kk)
    p[..., ::7] = p[..., 3:4]                      # ties in the priority order
    dO = np.random.default_rng(5 + w).standard_normal(q.shape).astype(np.float32)
    scale = 1 / math.sqrt(D)
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, dO, scale, r, tau, s, w)
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    loss = 0
    for j in range(H * G):
        h = j // G
        M = torch.tensor(oracle_mod.mask_dense(r[0, h], tau[0, h], s, w))
        logits = scale * tq[0, :, j, :] @ tk[0, :, h, :].T
        logits = logits.masked_fill(~M, float("-inf"))
        O = torch.softmax(logits, dim=1) @ tv[0, :, h, :]
        loss = loss + (O * torch.tensor(dO[0, :, j, :], dtype=torch.float64)).sum()
    loss.backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-12, rtol=0)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-12, rtol=0)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-12, rtol=0)


def test_attn_bwd_finite_differences(oracle_mod):
    """Central differences of L = sum(dO * O) through the oracle's forward pass
    (itself pinned to the library softmax) at sampled input entries."""
    S, H, G, D = 40, 1, 2, 8
    s, w, kk = 2, 5, 6
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=13)
    dO = np.random.default_rng(3).standard_normal(q.shape).astype(np.float32)
    scale = 0.4
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    grads = dict(zip("qkv", oracle_mod.attn_bwd(q, k, v, dO, scale, r, tau, s, w)))
    dO64 = dO.astype(np.float64)

    def loss(qq, kk_, vv):
        O, _ = oracle_mod.attn(qq, kk_, vv, scale, r, tau, s, w)
        return float((O * dO64).sum())

    rng = np.random.default_rng(8)
    for name in "qkv":
        for _ in range(6):
            arrs = {"q": q, "k": k, "v": v}
            idx = tuple(int(rng.integers(0, n)) for n in arrs[name].shape)
            if name != "q":                        # a key that some row retains
                idx = (0, int(rng.integers(0, 12)), 0, idx[3])
            hi = {n: a.copy() for n, a in arrs.items()}
            lo = {n: a.copy() for n, a in arrs.items()}
            hi[name][idx] = np.float32(arrs[name][idx] + np.float32(2.0 ** -9))
            lo[name][idx] = np.float32(arrs[name][idx] - np.float32(2.0 ** -9))
            step = float(hi[name][idx]) - float(lo[name][idx])
            fd = (loss(hi["q"], hi["k"], hi["v"]) - loss(lo["q"], lo["k"], lo["v"])) / step
            assert abs(fd - grads[name][idx]) <= 1e-5 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


def test_attn_bwd_invariants(oracle_mod):
    """Each softmax row's logit gradients sum to zero, so sum_t dk_t = 0 per KV
    head; each row's probabilities sum to one, so sum_t dv_t = sum over rows of dO."""
    S, H, G, D = 90, 2, 4, 8
    s, w, kk = 3, 9, 14
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=41)
    dO = np.random.default_rng(6).standard_normal(q.shape).astype(np.float32)
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    _, dk, dv = oracle_mod.attn_bwd(q, k, v, dO, 0.3, r, tau, s, w)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12
    ref = dO.astype(np.float64).reshape(1, S, H, G, D).sum(axis=(1, 3))
    assert np.allclose(dv.sum(axis=1), ref, atol=1e-11, rtol=0)


def test_attn_bwd_rows_and_keys_equal_full(oracle_mod):
    S, H, G, D = 64, 2, 2, 8
    s, w, kk = 2, 6, 9
    q, k, v, p = _tiny_inputs(S, H, G, D, seed=2)
    dO = np.random.default_rng(1).standard_normal(q.shape).astype(np.float32)
    r, tau, _ = oracle_mod.mask(p, s, w, kk)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, dO, 0.5, r, tau, s, w)
    rows = np.array([[0, j, t] for j in range(H * G) for t in (0, 1, 7, 30, S - 1)], np.int32)
    got = oracle_mod.attn_bwd_rows(q[0, rows[:, 2], rows[:, 1]], dO[0, rows[:, 2], rows[:, 1]], k, v, G, 0.5,
                                   rows, r, tau, s, w)
    assert np.allclose(got, dq[0, rows[:, 2], rows[:, 1]], atol=1e-13, rtol=0)
    keys = np.array([[0, h, t] for h in range(H) for t in (0, 1, 5, 20, S - 1)], np.int32)
    gk, gv = oracle_mod.attn_bwd_keys(q, k, v, dO, 0.5, keys, r, tau, s, w)
    assert np.allclose(gk, dk[0, keys[:, 2], keys[:, 1]], atol=1e-13, rtol=0)
    assert np.allclose(gv, dv[0, keys[:, 2], keys[:, 1]], atol=1e-13, rtol=0)


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


# ----------------------------------------------------------------------------
# normalised target, teacher boundary labels, pairwise boundary loss
# ("KVpop ... 精读笔记", section 2.2)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_target_normalize_zero_queries_closed_form(oracle_mod, eps):
    """q = 0: A_{d,t} = 1/(d+1) for every head, so (1/G) sum_g m_t = (1/N_t) sum_{d=t+w}^{S-1} 1/(d+1)
    with N_t = S - t - w; no future query -> log(eps)."""
    S, H, G, D, w = 60, 1, 3, 8, 4
    q, k, _, _ = _tiny_inputs(S, H, G, D, seed=5)
    q[:] = 0
    _, lse = oracle_mod.attn(q, k, k, 1.0, want_o=False)
    r = oracle_mod.target_normalize(oracle_mod.target_lse(q, k, lse, w, 1.0), G, w, eps)
    for t in range(S):
        nt = S - t - w
        if nt <= 0:
            assert (np.isneginf(r[0, 0, t]) if eps == 0 else r[0, 0, t] == math.log(eps))
        else:
            ref = math.log(eps + sum(1.0 / (d + 1) for d in range(t + w, S)) / nt)
            assert abs(r[0, 0, t] - ref) < 1e-12


def test_teacher_labels_hand_example(oracle_mod):
    f = _read_fixture("hand_labels_example.txt")
    S, s, w, k, n = (int(f[x][0]) for x in ("S", "s", "w", "k", "n"))
    r = np.array([float(v) for v in f["r"]], np.float32).reshape(1, 1, S)
    tb, y = oracle_mod.teacher_labels(r, s, w, k, n, [float(f["log_gamma"][0])])
    assert tb.ravel().tolist() == [int(v) for v in f["t_bnd"]]
    assert y.ravel().tolist() == [int(v) for v in f["y"]]


@pytest.mark.parametrize("s,w,k", [(2, 3, 4), (0, 0, 5), (3, 7, 1), (1, 2, 0), (0, 5, 200)])
def test_teacher_labels_without_decay_follow_the_mask(oracle_mod, s, w, k):
    """No decay (log_gamma = 0, or a step n beyond S): the teacher keeps the mask's
    retained set, so t_new = q - w is kept at row q exactly when q < evict_at[t_new];
    a dropped t_new faces the token of rank tau_q, and a kept one displaces the token
    evicted at row q (evict_at == q), if any."""
    rng = np.random.default_rng(11 + s + w + k)
    S = 300
    for prio in _prio_cases(rng, S):
        rk, tau, ev = oracle_mod.mask(prio.reshape(1, 1, S), s, w, k)
        for lg, n in ((0.0, 1), (-0.5, S + 1)):
            tb, y = oracle_mod.teacher_labels(prio.reshape(1, 1, S), s, w, k, n, [lg])
            tb, y = tb[0, 0], y[0, 0]
            for q in range(S):
                tn = q - w
                if tn < s:
                    assert y[q] == 0 and tb[q] == -1
                    continue
                kept = q < ev[0, 0, tn]
                assert y[q] == (1 if kept else -1), (q, lg)
                if k == 0:
                    assert tb[q] == -1
                elif not kept:
                    assert rk[0, 0, tb[q]] == tau[0, 0, q]
                elif tb[q] >= 0:
                    assert ev[0, 0, tb[q]] == q
                else:
                    assert tn - s < k            # fewer than k other eligible tokens


def test_teacher_labels_strong_decay_keeps_the_youngest(oracle_mod):
    """n = 1 and a decay far larger than the spread of r: younger always wins, so the
    leaving token is kept and the cutoff is the k-th youngest other token, q - w - k."""
    S, s, w, k = 200, 3, 5, 7
    r = np.random.default_rng(4).standard_normal((1, 2, S)).astype(np.float32)
    tb, y = oracle_mod.teacher_labels(r, s, w, k, 1, [-1e6, -2e6])
    for h in range(2):
        for q in range(S):
            tn = q - w
            if tn < s:
                assert y[0, h, q] == 0
            else:
                assert y[0, h, q] == 1
                assert tb[0, h, q] == (q - w - k if tn - s >= k else -1)


def _label_case(oracle_mod, seed, b=2, H=2, S=160, s=2, w=6, k=9, n=4):
    rng = np.random.default_rng(seed)
    r = rng.standard_normal((b, H, S)).astype(np.float32)
    lg = np.log(np.array([0.9, 0.7][:H], np.float32)).astype(np.float32)
    tb, y = oracle_mod.teacher_labels(r, s, w, k, n, lg)
    return rng, tb, y, lg


def test_boundary_loss_gradient_is_the_derivative(oracle_mod):
    """Central differences of the loss match the returned gradient."""
    rng, tb, y, lg = _label_case(oracle_mod, 8)
    b, H, S = tb.shape
    rh = rng.standard_normal((b, H, S)).astype(np.float32)
    om = rng.random((b, H, S)).astype(np.float32) + 0.5
    loss, grad, pairs = oracle_mod.boundary_loss(rh, tb, y, 6, 4, lg, 0.7, om)
    assert pairs == int(((y != 0) & (tb >= 0)).sum()) and pairs > 100
    h = 2.0 ** -10                     # exact in fp32 near |r| ~ 1
    for idx in list(zip(*np.nonzero(np.abs(grad) > 1e-6)))[:40]:
        up, dn = rh.copy(), rh.copy()
        up[idx] += h
        dn[idx] -= h
        fd = (oracle_mod.boundary_loss(up, tb, y, 6, 4, lg, 0.7, om)[0]
              - oracle_mod.boundary_loss(dn, tb, y, 6, 4, lg, 0.7, om)[0]) / (float(up[idx]) - float(dn[idx]))
        assert abs(fd - grad[idx]) < 1e-6 + 1e-4 * abs(grad[idx])


def test_boundary_loss_closed_forms(oracle_mod):
    """Equal decayed scores give softplus(0) = log 2 per pair (weighted mean); a wide
    margin on the labelled side gives ~0, on the wrong side ~margin / tau."""
    rng, tb, y, _ = _label_case(oracle_mod, 9)
    b, H, S = tb.shape
    zero = np.zeros(H, np.float32)
    om = rng.random((b, H, S)).astype(np.float32)
    valid = (y != 0) & (tb >= 0)
    loss, _, _ = oracle_mod.boundary_loss(np.zeros((b, H, S), np.float32), tb, y, 6, 4, zero, 1.3, om)
    assert abs(loss - math.log(2) * om[valid].astype(np.float64).mean()) < 1e-12
    # rhat = +/- 40 * position order: t_new (the later token) is far above / below t_bnd
    pos = np.broadcast_to(np.arange(S, dtype=np.float32), (b, H, S)).copy()
    for sign in (1.0, -1.0):
        rh = (sign * 40.0 * pos).astype(np.float32)
        loss, _, _ = oracle_mod.boundary_loss(rh, tb, y, 6, 4, zero, 2.0)
        qs = np.nonzero(valid)
        margins = sign * 40.0 * ((qs[2] - 6) - tb[valid]) * y[valid]     # y * (rhat_new - rhat_bnd)
        ref = np.mean([max(0.0, -m / 2.0) for m in margins])
        assert abs(loss - ref) < 1e-6 * max(1.0, ref)


def test_boundary_loss_hand_example(oracle_mod):
    """The decayed predictions of the worked example (all rhat = 0, n = 1)."""
    f = _read_fixture("hand_labels_example.txt")
    S = int(f["S"][0])
    tb = np.array([int(v) for v in f["t_bnd"]], np.int32).reshape(1, 1, S)
    y = np.array([int(v) for v in f["y"]], np.int32).reshape(1, 1, S)
    loss, grad, pairs = oracle_mod.boundary_loss(np.zeros((1, 1, S), np.float32), tb, y, int(f["w"][0]),
                                                 int(f["loss_n"][0]), [float(f["log_gamma"][0])],
                                                 float(f["loss_tau"][0]))
    assert pairs == 8
    assert abs(loss - float(f["loss_mean"][0])) < 1e-9


def test_teacher_labels_rows_equal_full(oracle_mod):
    """The sampled-row entry gives the full sweep's values on the rows it is asked for."""
    rng = np.random.default_rng(21)
    r = rng.standard_normal((1, 1, 400)).astype(np.float32)
    tb, y = oracle_mod.teacher_labels(r, 3, 9, 11, 5, [-0.2])
    rows = rng.choice(400, size=60, replace=False).astype(np.int32)
    tbr, yr = oracle_mod.teacher_labels_rows(r[0, 0], 3, 9, 11, 5, -0.2, rows)
    assert (tbr == tb[0, 0, rows]).all() and (yr == y[0, 0, rows]).all()
