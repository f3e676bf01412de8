"""Training-side passes on the GPU against the fp64 oracle ("KVpop ... 精读笔记",
section 2.2): the normalised target (1e-5 in the log domain), the teacher boundary
labels (bit-exact: integers decided by fp32 scores computed the same way on both
sides) and the pairwise boundary loss with its gradient (fp32 atomics: relative
1e-5 on the loss, 1e-6 + 1e-4 relative on each gradient entry)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_R = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def _targets(rng, b, H, S, kind):
    r = rng.standard_normal((b, H, S)).astype(np.float32)
    if kind == "ties":      # few distinct values: ties in the decayed score
        r = np.round(r * 2) / 2
    elif kind == "special":
        r[rng.random((b, H, S)) < 0.03] = np.nan
        r[rng.random((b, H, S)) < 0.03] = -np.inf
        r[rng.random((b, H, S)) < 0.05] = -0.0
        r[rng.random((b, H, S)) < 0.05] = 0.0
    return r


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_target_normalize_matches_oracle(eps):
    rng = np.random.default_rng(3)
    b, H, S, G, w = 2, 3, 500, 4, 37
    t = (rng.standard_normal((b, H, S)) * 3).astype(np.float32)
    t[:, :, S - w:] = -np.inf                  # no future query
    t[0, 0, 5] = -np.inf                       # an underflowed key
    got = host(kvpop.target_normalize(dev(t), G, w, eps))
    ref = oracle.target_normalize(t.astype(np.float64), G, w, eps)
    if eps > 0:
        assert np.isfinite(got).all()
    assert_close_log(got.ravel(), ref.ravel(), TOL_R, "r_tgt")


CASES = [
    # b, H, S, s, w, k, n, gammas, kind
    (1, 1, 300, 2, 5, 7, 4, [0.9], "normal"),
    (2, 2, 700, 3, 20, 40, 16, [0.95, 0.6], "ties"),
    (1, 2, 513, 0, 0, 25, 1, [0.99, 0.5], "special"),
    (1, 1, 400, 4, 9, 0, 3, [0.8], "normal"),              # k = 0
    (1, 1, 400, 1, 3, 500, 2, [0.8], "normal"),            # budget above every row
    (1, 3, 900, 16, 64, 100, 32, [1.0, 0.97, 0.9], "ties"),  # gamma = 1: no decay
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}H{}S{}_s{}w{}k{}n{}_{}".format(*c[:7], c[8]))
def test_teacher_labels_bit_exact(case):
    b, H, S, s, w, k, n, gammas, kind = case
    rng = np.random.default_rng(S + k)
    r = _targets(rng, b, H, S, kind)
    lg = np.log(np.array(gammas, np.float32)).astype(np.float32)
    tb, y = kvpop.teacher_labels(dev(r), s, w, k, n, dev(lg))
    tbr, yr = oracle.teacher_labels(r, s, w, k, n, lg)
    assert (host(y) == yr).all(), np.argwhere(host(y) != yr)[:5]
    assert (host(tb) == tbr).all(), np.argwhere(host(tb) != tbr)[:5]


def test_teacher_labels_long_rows_uncached():
    """S beyond the shared-memory cache (targets read from global memory); only the
    last rows have a leaving token, so the oracle stays small."""
    rng = np.random.default_rng(77)
    S, s, w, k, n = 40000, 5, 39000, 60, 8
    r = _targets(rng, 1, 1, S, "ties")
    lg = np.array([math.log(0.9)], np.float32)
    tb, y = kvpop.teacher_labels(dev(r), s, w, k, n, dev(lg))
    rows = np.arange(w + s - 2, S, 3, dtype=np.int32)
    tbr, yr = oracle.teacher_labels_rows(r[0, 0], s, w, k, n, float(lg[0]), rows)
    assert (host(y)[0, 0, rows] == yr).all() and (host(tb)[0, 0, rows] == tbr).all()


@pytest.mark.parametrize("S,kind,gammas", [(20000, "ties", [0.93, 0.99]),      # targets cached in shared memory
                                            (40000, "ties", [0.93, 0.99]),      # targets read from global memory
                                            (24000, "special", [1.0, 0.95])])   # NaN/-inf/-0, no decay
def test_teacher_labels_long_rows(S, kind, gammas):
    """Rows of tens of thousands of candidates (a band of scores carried from row
    to row, the previous cutoff as pivot, radix select when the cutoff leaves the
    band); whole CTA chunks and scattered rows against the oracle, bit-exact."""
    rng = np.random.default_rng(S)
    s, w, k, n = 5, 100, 3000, 8
    r = _targets(rng, 1, 2, S, kind)
    lg = np.log(np.array(gammas, np.float32)).astype(np.float32)
    tb, y = kvpop.teacher_labels(dev(r), s, w, k, n, dev(lg))
    tb, y = host(tb), host(y)
    rows = np.concatenate([np.arange(S - 192, S), np.arange(3136, 3200),
                           np.random.default_rng(1).integers(w + s, S, 40)]).astype(np.int32)
    for h in range(2):
        tbr, yr = oracle.teacher_labels_rows(r[0, h], s, w, k, n, float(lg[h]), rows)
        assert (y[0, h, rows] == yr).all() and (tb[0, h, rows] == tbr).all(), h


def test_teacher_labels_long_context_rows():
    """The long-context shape (S = 131072, budget s16 w1024 k3056, n = 64): rows of up
    to 130 000 candidates, where each CTA carries a band of scores around its cutoff
    from row to row.  Whole CTA chunks (64 consecutive rows, so every row after the
    first works from the band and the previous cutoff) and scattered rows against
    the oracle, bit-exact, for a slow and a fast decay."""
    rng = np.random.default_rng(131072)
    S, s, w, k, n = 131072, 16, 1024, 3056, 64
    r = _targets(rng, 1, 2, S, "normal")
    lg = np.log(np.array([0.90, 0.99], np.float32)).astype(np.float32)
    tb, y = kvpop.teacher_labels(dev(r), s, w, k, n, dev(lg))
    tb, y = host(tb), host(y)
    rows = np.concatenate([np.arange(S - 128, S), np.arange(65536, 65600), np.arange(w + s + k, w + s + k + 64),
                           np.random.default_rng(2).integers(w + s, S, 48)]).astype(np.int32)
    for h in range(2):
        tbr, yr = oracle.teacher_labels_rows(r[0, h], s, w, k, n, float(lg[h]), rows)
        assert (y[0, h, rows] == yr).all() and (tb[0, h, rows] == tbr).all(), h


def test_teacher_labels_full_size_follow_the_mask():
    """4B-like size (b1 H8 S16384, k 1520, w 512) without decay: the labels are the
    mask's decisions (property at any size, checked against the GPU mask, itself
    parity-tested); with decay, sampled rows against the oracle."""
    wl = synth.QWEN3_4B
    prio = torch.from_numpy(synth.priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))).cuda()
    rk, tau, ev, _ = kvpop.mask(prio, wl.s, wl.w, wl.k, lists=False)
    zero = torch.zeros(wl.H, dtype=torch.float32, device="cuda")
    tb, y = kvpop.teacher_labels(prio, wl.s, wl.w, wl.k, 64, zero)
    tb, y, rk, tau, ev = host(tb), host(y), host(rk), host(tau), host(ev)
    q = np.arange(wl.S)
    tn = q - wl.w
    for h in range(wl.H):
        lab = tn >= wl.s
        assert (y[0, h, ~lab] == 0).all()
        kept = ev[0, h, tn[lab]] > q[lab]
        assert (y[0, h, lab] == np.where(kept, 1, -1)).all()
        drop = lab & (y[0, h] == -1)
        assert (rk[0, h, tb[0, h, drop]] == tau[0, h, drop]).all()
        kb = lab & (y[0, h] == 1) & (tb[0, h] >= 0)
        assert (ev[0, h, tb[0, h, kb]] == q[kb]).all()
    lg = np.log(np.linspace(0.9, 0.99, wl.H)).astype(np.float32)
    tb, y = kvpop.teacher_labels(prio, wl.s, wl.w, wl.k, 64, dev(lg))
    tb, y = host(tb), host(y)
    p = host(prio)
    rows = np.random.default_rng(5).choice(np.arange(wl.w + wl.s, wl.S), size=48, replace=False).astype(np.int32)
    for h in (0, wl.H - 1):
        tbr, yr = oracle.teacher_labels_rows(p[0, h], wl.s, wl.w, wl.k, 64, float(lg[h]), rows)
        assert (y[0, h, rows] == yr).all() and (tb[0, h, rows] == tbr).all()


@pytest.mark.parametrize("with_omega", [False, True])
def test_boundary_loss_matches_oracle(with_omega):
    rng = np.random.default_rng(12)
    b, H, S, s, w, k, n = 2, 2, 600, 2, 11, 30, 8
    r = _targets(rng, b, H, S, "normal")
    lg = np.log(np.array([0.93, 0.7], np.float32)).astype(np.float32)
    tbr, yr = oracle.teacher_labels(r, s, w, k, n, lg)
    rh = rng.standard_normal((b, H, S)).astype(np.float32)
    om = (rng.random((b, H, S)) + 0.25).astype(np.float32) if with_omega else None
    loss_r, grad_r, pairs = oracle.boundary_loss(rh, tbr, yr, w, n, lg, 0.8, om)
    for _ in range(2):             # twice: the call clears its own accumulators
        loss, grad = kvpop.boundary_loss(dev(rh), dev(tbr), dev(yr), w, n, dev(lg), 0.8,
                                         None if om is None else dev(om))
        loss, grad = host(loss), host(grad)
        assert loss[1] == pairs and pairs > 500
        assert abs(loss[0] - loss_r) <= 1e-5 * abs(loss_r)
        assert (np.abs(grad - grad_r) <= 1e-6 + 1e-4 * np.abs(grad_r)).all()


def test_boundary_loss_no_pairs():
    """k = 0 and no leaving token leave no pairs: loss 0, count 0, zero gradient."""
    S = 50
    tb = np.full((1, 1, S), -1, np.int32)
    y = np.zeros((1, 1, S), np.int32)
    loss, grad = kvpop.boundary_loss(dev(np.ones((1, 1, S), np.float32)), dev(tb), dev(y), 3, 2,
                                     dev(np.zeros(1, np.float32)), 1.0)
    assert host(loss).tolist() == [0.0, 0.0] and (host(grad) == 0).all()


def test_sparse_lse_target_variant():
    """The target pass fed with the sparse-attention LSE ("KVpop ... 精读笔记",
    section 2.3: the sparse normaliser stands in for the dense one) against the
    oracle's Eq. (8) with the oracle's sparse LSE; and it is never below the
    dense-LSE target (the sparse normaliser sums fewer terms)."""
    wl = synth.Workload("case", b=1, H=2, G=4, D=128, S=700, s=4, w=48, k=64, prio="uniform", seed=9)
    inp = synth.make_prefill(wl)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    _, _, ev, lists = kvpop.mask(dev(inp.prio), wl.s, wl.w, wl.k)
    _, lse_s = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, (wl.s, wl.w, wl.k))
    _, lse_d = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    t_s = host(kvpop.future_target(q, k, lse_s, wl.w))
    t_d = host(kvpop.future_target(q, k, lse_d, wl.w))
    scale = 1 / math.sqrt(wl.D)
    rank, tau, _ = oracle.mask(inp.prio, wl.s, wl.w, wl.k)
    _, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("v"), scale, rank, tau, wl.s, wl.w)
    tr = oracle.target_lse(inp.f32("q"), inp.f32("k"), lr, wl.w, scale)
    assert_close_log(t_s.ravel(), tr.ravel(), 2e-2, "target (sparse LSE)")
    fin = np.isfinite(t_d)
    assert (t_s[fin] >= t_d[fin] - 2e-2).all()
