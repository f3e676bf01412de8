"""kvpop_attn_fwd (sparse and dense) and kvpop_future_target on the GPU against
the fp64 oracle.  Tolerances: O max-abs 2e-2, LSE max-abs 2e-3, targets 2e-2
in the log domain (-inf must match)."""
import math

import numpy as np
import pytest

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_T = 2e-2, 2e-3, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def small_case(b, H, G, D, S, s, w, k, seed, prio="uniform"):
    wl = synth.Workload("case", b=b, H=H, G=G, D=D, S=S, s=s, w=w, k=k, prio=prio, seed=seed)
    return synth.make_prefill(wl)


def run_sparse(inp, want_o=True):
    wl = inp.wl
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    rank, tau, ev, lists = kvpop.mask(dev(inp.prio), wl.s, wl.w, wl.k)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, (wl.s, wl.w, wl.k))
    return host(O), host(lse)


CASES = [
    # b, H, G, D, S, s, w, k
    (1, 1, 2, 64, 256, 4, 32, 32),        # the tiny workload's shape
    (1, 2, 4, 128, 300, 4, 32, 32),
    (2, 2, 4, 128, 777, 16, 64, 100),     # ragged tail, several tiles
    (1, 1, 4, 128, 1000, 0, 0, 50),       # w = 0, s = 0
    (1, 2, 4, 64, 513, 3, 100, 0),        # k = 0 (sinks + window)
    (1, 1, 8, 128, 400, 2, 17, 33),       # G = 8
    (1, 1, 1, 128, 300, 1, 40, 60),       # G = 1
    (1, 1, 4, 128, 600, 8, 16, 2000),     # budget covers the sequence
    (1, 1, 16, 128, 350, 3, 24, 40),      # G = 16: 8 positions per query tile
    (2, 3, 2, 128, 520, 5, 40, 70),       # G = 2, three KV heads, two sequences
    (1, 2, 4, 128, 3000, 16, 256, 700),   # full lists (gathered tiles) and window spans over many blocks
    (1, 1, 64, 128, 50, 2, 8, 10),        # G = 64
    (1, 1, 128, 64, 40, 2, 5, 6),         # G = 128, D = 64: one position per query tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}H{}G{}D{}S{}_s{}w{}k{}".format(*c))
def test_sparse_attention_small(case):
    b, H, G, D, S, s, w, k = case
    inp = small_case(*case, seed=sum(case))
    O, lse = run_sparse(inp)
    scale = 1 / math.sqrt(D)
    r, tau, _ = oracle.mask(inp.prio, s, w, k)
    Or, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("v"), scale, r, tau, s, w)
    assert_close_log(lse.ravel(), lr.ravel(), TOL_LSE, "lse")
    assert np.abs(O - Or).max() <= TOL_O, f"O max err {np.abs(O - Or).max()}"


@pytest.mark.parametrize("case", [(1, 1, 2, 64, 256), (1, 2, 4, 128, 300), (2, 1, 4, 128, 1100),
                                  (1, 1, 8, 64, 333), (1, 1, 1, 128, 257)],
                         ids=lambda c: "b{}H{}G{}D{}S{}".format(*c))
def test_dense_attention_small(case):
    b, H, G, D, S = case
    inp = small_case(b, H, G, D, S, 0, 0, 1, seed=S)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    scale = 1 / math.sqrt(D)
    Or, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("v"), scale)
    _, lse_only = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    assert_close_log(host(lse_only).ravel(), lr.ravel(), TOL_LSE, "lse (LSE-only)")
    O, lse = kvpop.attn_fwd(q, k, v, 0.0)
    assert_close_log(host(lse).ravel(), lr.ravel(), TOL_LSE, "lse (with O)")
    assert np.abs(host(O) - Or).max() <= TOL_O


@pytest.mark.parametrize("case", [(1, 1, 2, 64, 256, 32), (1, 2, 4, 128, 700, 64), (2, 1, 4, 128, 900, 0),
                                  (1, 1, 8, 128, 333, 5), (1, 1, 1, 64, 300, 299), (1, 1, 4, 128, 260, 300)],
                         ids=lambda c: "b{}H{}G{}D{}S{}w{}".format(*c))
def test_future_target_small(case):
    b, H, G, D, S, w = case
    inp = small_case(b, H, G, D, S, 0, 0, 1, seed=S + w)
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    scale = 1 / math.sqrt(D)
    _, lse = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, lse, w))
    _, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("k"), scale, want_o=False)
    tr = oracle.target_lse(inp.f32("q"), inp.f32("k"), lr, w, scale)
    assert_close_log(tgt.ravel(), tr.ravel(), TOL_T, "target")


def test_tiny_workload_pipeline():
    """The tiny workload end to end: mask, sparse attention, dense LSE, targets."""
    inp = synth.make_prefill(synth.TINY)
    wl = inp.wl
    scale = 1 / math.sqrt(wl.D)
    O, lse = run_sparse(inp)
    r, tau, _ = oracle.mask(inp.prio, wl.s, wl.w, wl.k)
    Or, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("v"), scale, r, tau, wl.s, wl.w)
    assert_close_log(lse.ravel(), lr.ravel(), TOL_LSE, "sparse lse")
    assert np.abs(O - Or).max() <= TOL_O
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    _, dlr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("k"), scale, want_o=False)
    assert_close_log(host(dl).ravel(), dlr.ravel(), TOL_LSE, "dense lse")
    tgt = host(kvpop.future_target(q, k, dl, wl.w))
    tr = oracle.target_lse(inp.f32("q"), inp.f32("k"), dlr, wl.w, scale)
    assert_close_log(tgt.ravel(), tr.ravel(), TOL_T, "target")


# ----------------------------------------------------------------------------
# full-size workloads: sampled outputs and properties
# ----------------------------------------------------------------------------

@pytest.fixture(scope="module")
def w4b():
    return synth.make_prefill(synth.QWEN3_4B)


def _sample_rows(rng, wl, n):
    bi = rng.integers(0, wl.b, n)
    j = rng.integers(0, wl.Hq, n)
    qp = np.concatenate([rng.integers(0, wl.S, n - 8), [0, 1, wl.S - 1, wl.S - 2, 63, 64, 2047, 2048]])
    return np.stack([bi, j, qp[:n]], axis=1).astype(np.int32)


@pytest.mark.parametrize("wlname", ["qwen3-4b-layer-prefill", "qwen3-8b-layer-prefill"])
def test_full_workload_sampled(wlname, w4b):
    wl = synth.PREFILL_WORKLOADS[wlname]
    inp = w4b if wl is synth.QWEN3_4B else synth.make_prefill(wl)
    scale = 1 / math.sqrt(wl.D)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    prio = dev(inp.prio)
    rank, tau, ev, lists = kvpop.mask(prio, wl.s, wl.w, wl.k)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, (wl.s, wl.w, wl.k))
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    O, lse, dl = host(O), host(lse), host(dl)
    rng = np.random.default_rng(5)
    rows = _sample_rows(rng, wl, 256)
    qf = inp.f32("q")
    kf, vf = inp.f32("k"), inp.f32("v")
    qv = qf[rows[:, 0], rows[:, 2], rows[:, 1]]
    r, ta, _ = oracle.mask(inp.prio, wl.s, wl.w, wl.k)
    Or, lr = oracle.attn_rows(qv, kf, vf, wl.G, scale, rows, r, ta, wl.s, wl.w)
    got_l = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    got_o = O[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_close_log(got_l, lr, TOL_LSE, "sparse lse")
    assert np.abs(got_o - Or).max() <= TOL_O
    _, dlr = oracle.attn_rows(qv, kf, vf, wl.G, scale, rows, want_o=False)
    assert_close_log(dl[rows[:, 0], rows[:, 1], rows[:, 2]], dlr, TOL_LSE, "dense lse")


def test_full_workload_target_late_keys(w4b):
    """Targets of the last keys of one KV head against the oracle, which needs the
    dense LSE only for the query rows those keys can see."""
    inp = w4b
    wl = inp.wl
    scale = 1 / math.sqrt(wl.D)
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, dl, wl.w))
    h = 3
    t_lo = wl.S - wl.w - 1024
    d_rows = np.arange(t_lo + wl.w, wl.S)
    qf, kf = inp.f32("q"), inp.f32("k")
    rows = np.array([[0, h * wl.G + g, d] for g in range(wl.G) for d in d_rows], np.int32)
    qv = qf[0, rows[:, 2], rows[:, 1]]
    _, lr = oracle.attn_rows(qv, kf, kf, wl.G, scale, rows, want_o=False)
    lse_full = np.full((wl.b, wl.Hq, wl.S), np.nan)
    lse_full[0, rows[:, 1], rows[:, 2]] = lr
    keys = np.array([[0, h, t] for t in range(t_lo, wl.S, 7)] + [[0, h, wl.S - 1]], np.int32)
    tr = oracle.target_lse(qf, kf, lse_full, wl.w, scale, keys)
    assert_close_log(tgt[0, h, keys[:, 2]], tr, TOL_T, "target")


def test_full_workload_target_mass_conservation(w4b):
    """w = 0: each query row's probabilities sum to 1, so sum_t exp(target) = S * G."""
    inp = w4b
    wl = inp.wl
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, dl, 0)).astype(np.float64)
    tot = np.exp(tgt).sum(axis=-1)
    assert np.allclose(tot, wl.S * wl.G, rtol=2e-3), tot
