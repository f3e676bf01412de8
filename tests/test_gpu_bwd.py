"""kvpop_attn_bwd on the GPU against the fp64 oracle's gradient of the sparse
attention ("KVpop ... 精读笔记", section 2.1, Figure 1: the student is trained
through the sparse attention).

The GPU path runs mask -> sparse forward -> backward on the same seeded bf16
inputs the oracle reads (q, k, v, the upstream gradient dO); the oracle
recomputes everything in fp64 from those inputs.  Tolerance per tensor:
max |gpu - oracle| <= 1e-2 * max |oracle|.  Derivation: the kernels round the
softmax probabilities P and the logit gradients dS to bf16 (relative error up
to 2^-9, about 1.1e-3 RMS for round-to-nearest) before the products whose
fp32 sums give dv, dq and dk; each output is a random-sign sum of such terms,
so its error is about that relative RMS of the sum's own scale, and the bound
leaves a factor of about ten for the largest of many elements.  dO . O with
the bf16 forward output stands in for sum_t P dP, an error of the same order.
A gradient that vanishes exactly (a row with one retained key has P = 1 and
dS = 0) leaves only that fp32 rounding, so 1e-5 is allowed on top.

Each row of dq (and each key's row of dk, dv) is also held to its own scale, so
that rows far smaller than the tensor's largest (rarely attended keys) cannot
hide a large relative error under the global bound:
||gpu - oracle|| <= 5e-2 ||oracle|| + floor over the D entries of the row, and the
whole tensor's RMS error <= 5e-3 of its RMS.  The expected relative error of a row
is about the 1e-3 RMS rounding above.  The floor is for rows whose terms cancel:
in a row whose softmax is peaked on one of few keys, dS = P (dP - dO.O) is a small
difference, and the bf16 rounding of the forward's O (at most 2^-9 relative per
entry) moves dO.O by at most 2^-9 ||dO|| ||O||, hence that row's dq by at most
scale 2^-9 ||dO|| ||O|| ||sum_t P_t k_t||; twice that bound is the floor of a dq
row where the oracle's O and sum_t P_t k_t are at hand, 3e-2 of the median row
norm elsewhere (dk, dv and sampled rows)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-2
ATOL_GRAD = 1e-5
TOL_ROW = 5e-2
ROW_FLOOR = 3e-2  # of the median row norm, where no bound from the inputs is at hand
TOL_RMS = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def gpu_grads(wl, inp, dO_bits):
    bud = (wl.s, wl.w, wl.k)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    dO = dev_bf16(dO_bits)
    _, _, ev, lists = kvpop.mask(dev(inp.prio), *bud)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, bud)
    dq, dk, dv = kvpop.attn_bwd(q, k, v, O, dO, lse, ev, lists, bud)
    return host(dq), host(dk), host(dv)


def check(got, ref, what, row_floor=None):
    scale = float(np.abs(ref).max())
    err = float(np.abs(got - ref).max())
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err <= TOL_GRAD * scale + ATOL_GRAD, f"{what}: max abs error {err:.3e} > {TOL_GRAD:.0e} * {scale:.3e}"
    # per row (last axis = the head dimension), relative to the row's own norm
    g = np.asarray(got, np.float64).reshape(-1, got.shape[-1])
    r = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    row_err = np.linalg.norm(g - r, axis=1)
    row_ref = np.linalg.norm(r, axis=1)
    if row_floor is None:
        floor = ROW_FLOOR * float(np.median(row_ref)) + ATOL_GRAD * math.sqrt(r.shape[1])
    else:
        floor = np.asarray(row_floor, np.float64).reshape(-1) + ATOL_GRAD * math.sqrt(r.shape[1])
    bound = TOL_ROW * row_ref + floor
    bad = np.nonzero(row_err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows above the per-row bound, worst excess "
                           f"{float((row_err / bound)[bad].max()):.3f}x at row {bad[0]}")
    rms_err = math.sqrt(float(np.mean((g - r) ** 2)))
    rms_ref = math.sqrt(float(np.mean(r ** 2)))
    assert rms_err <= TOL_RMS * rms_ref + ATOL_GRAD, f"{what}: RMS error {rms_err:.3e} > {TOL_RMS} x {rms_ref:.3e}"
    return err / max(scale, ATOL_GRAD)


CASES = [
    # b, H, G, D, S, s, w, k
    (1, 1, 2, 64, 256, 4, 32, 32),        # the tiny workload's shape
    (1, 2, 4, 128, 700, 4, 48, 64),       # several tiles, ragged tail
    (2, 2, 4, 128, 1000, 16, 100, 200),
    (1, 1, 4, 128, 1000, 0, 0, 50),       # w = 0, s = 0: no band pass
    (1, 2, 4, 64, 513, 3, 100, 0),        # k = 0 (sinks + window, no lists)
    (1, 1, 8, 128, 400, 2, 17, 33),       # G = 8
    (1, 2, 1, 64, 400, 2, 30, 60),        # G = 1: 128 positions per query tile
    (1, 1, 4, 128, 600, 8, 16, 2000),     # budget covers the sequence
    (1, 1, 16, 128, 350, 3, 24, 40),      # G = 16: 8 positions per query tile
    (2, 3, 2, 128, 520, 5, 40, 70),       # G = 2, three KV heads, two sequences
    (1, 1, 4, 128, 2100, 600, 300, 400),  # more sinks than a key tile, blocks of sinks only
    (1, 1, 2, 64, 1, 1, 1, 1),            # one token
    (1, 2, 4, 64, 20, 2, 3, 4),           # shorter than one query tile
    (1, 1, 4, 128, 300, 0, 400, 8),       # the window covers the sequence: band pairs only
    (1, 1, 128, 64, 40, 2, 5, 6),         # G = 128: one position per query tile
    # D = 128 runs the CTA-pair dQ kernel (256-row query tiles): its edge shapes
    (1, 2, 1, 128, 400, 2, 30, 60),       # G = 1: 256 positions per pair of CTAs
    (1, 1, 32, 128, 100, 2, 10, 12),      # G = 32: one position per warp
    (1, 1, 128, 128, 40, 2, 5, 6),        # G = 128: one position per CTA
    (1, 1, 2, 128, 1, 1, 1, 1),           # one token: the second CTA of the pair has no rows
    (1, 2, 4, 128, 20, 2, 3, 4),          # shorter than one query tile
    # long pairs: an odd key-chunk count and a last block inside one query tile (one-tile items)
    (1, 2, 4, 128, 1040, 8, 64, 300),
    (1, 1, 64, 128, 30, 2, 4, 6),         # G = 64: two positions per query tile
    (2, 2, 4, 64, 1100, 8, 64, 300),      # D = 64: two sequences, several long-pair blocks
    (1, 1, 1, 128, 1300, 4, 100, 300),    # G = 1 across several 512-row blocks
    (1, 2, 8, 128, 1500, 0, 200, 500),    # s = 0, G = 8, several blocks
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}H{}G{}D{}S{}_s{}w{}k{}".format(*c))
def test_attn_bwd_matches_oracle(case):
    b, H, G, D, S, s, w, k = case
    wl = synth.Workload("case", b=b, H=H, G=G, D=D, S=S, s=s, w=w, k=k, prio="uniform", seed=sum(case) + 7)
    inp = synth.make_prefill(wl)
    dO_bits = synth.upstream_grad(wl)
    dq, dk, dv = gpu_grads(wl, inp, dO_bits)
    rank, tau, _ = oracle.mask(inp.prio, s, w, k)
    qf, kf, vf, dOf = inp.f32("q"), inp.f32("k"), inp.f32("v"), synth.bf16_bits_to_f32(dO_bits)
    scale = 1 / math.sqrt(D)
    rq, rk, rv = oracle.attn_bwd(qf, kf, vf, dOf, scale, rank, tau, s, w)
    # the dq floor: what the bf16 rounding of O can move dO.O by, carried through sum_t P_t k_t
    Or, _ = oracle.attn(qf, kf, vf, scale, rank, tau, s, w)
    Kbar, _ = oracle.attn(qf, kf, kf, scale, rank, tau, s, w)
    nrm = lambda a: np.linalg.norm(np.asarray(a, np.float64), axis=-1)
    dq_floor = 2.0 * scale * 2.0 ** -9 * nrm(dOf) * nrm(Or) * nrm(Kbar)
    check(dq, rq, "dq", row_floor=dq_floor)
    check(dk, rk, "dk")
    check(dv, rv, "dv")


def test_attn_bwd_repeatable_and_workspace_reuse():
    """A second call with the same workspace gives the same dq bit for bit (dq
    has one writer per element) and dk/dv equal up to the atomics' order."""
    wl = synth.Workload("case", b=1, H=2, G=4, D=128, S=900, s=4, w=64, k=96, prio="normal", seed=3)
    inp = synth.make_prefill(wl)
    bud = (wl.s, wl.w, wl.k)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    dO = dev_bf16(synth.upstream_grad(wl))
    _, _, ev, lists = kvpop.mask(dev(inp.prio), *bud)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, bud)
    ws = torch.empty(kvpop.attn_bwd_workspace_size(1, wl.S, wl.Hq, wl.H, bud), dtype=torch.uint8, device="cuda")
    a = [host(t) for t in kvpop.attn_bwd(q, k, v, O, dO, lse, ev, lists, bud, workspace=ws)]
    c = [host(t) for t in kvpop.attn_bwd(q, k, v, O, dO, lse, ev, lists, bud, workspace=ws)]
    assert np.array_equal(a[0], c[0])
    for x, y in zip(a[1:], c[1:]):
        assert np.abs(x - y).max() <= 1e-5 * np.abs(x).max()


def test_attn_bwd_full_size_sampled():
    """The 4B-like layer (b1 H8 G4 D128 S16384, s16 w512 k1520) in the launch the
    benchmark times: dq of sampled rows and dk/dv of sampled keys (keys whose
    rows the oracle can afford: window-only keys and keys held up to ~1500 rows
    past the window) against the oracle; over all keys, the softmax-row
    invariants sum_t dk_t = 0 and sum_t dv_t = sum over rows of dO."""
    wl = synth.QWEN3_4B
    bud = (wl.s, wl.w, wl.k)
    q, k, v, prio = synth.make_prefill_device(wl, "cuda")
    dO = synth.normal_bf16_torch(wl.seed, synth.DO, (wl.b, wl.S, wl.Hq, wl.D), "cuda")
    _, _, ev, lists = kvpop.mask(prio, *bud)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, bud)
    dq, dk, dv = kvpop.attn_bwd(q, k, v, O, dO, lse, ev, lists, bud)
    torch.cuda.synchronize()
    # invariants over all keys of every head
    dkh, dvh, dOh = host(dk).astype(np.float64), host(dv).astype(np.float64), host(dO).astype(np.float64)
    assert np.abs(dkh.sum(axis=1)).max() <= 1e-3 * np.abs(dkh).sum(axis=1).max()
    ref_v = dOh.reshape(wl.b, wl.S, wl.H, wl.G, wl.D).sum(axis=(1, 3))
    assert np.abs(dvh.sum(axis=1) - ref_v).max() <= 1e-2 * np.abs(ref_v).max() + 1e-2
    # sampled rows and keys against the oracle
    qf, kf, vf, dOf = host(q), host(k), host(v), dOh.astype(np.float32)
    rank, tau, _ = oracle.mask(host(prio), *bud)
    evh = host(ev)
    rng = np.random.default_rng(17)
    pos = np.concatenate([rng.integers(0, wl.S, 40), [0, 1, 600, 4095, wl.S - 1]])
    rows = np.stack([np.zeros_like(pos), rng.integers(0, wl.Hq, len(pos)), pos], axis=1).astype(np.int32)
    rq = oracle.attn_bwd_rows(qf[0, rows[:, 2], rows[:, 1]], dOf[0, rows[:, 2], rows[:, 1]], kf, vf, wl.G,
                              1 / math.sqrt(wl.D), rows, rank, tau, wl.s, wl.w)
    check(host(dq)[0, rows[:, 2], rows[:, 1]], rq, "dq rows")
    keys = []
    for h in (0, 5):
        life = evh[0, h] - np.arange(wl.S)
        short = np.nonzero((life == wl.w) & (np.arange(wl.S) >= wl.s))[0]
        mid = np.nonzero((life > wl.w + 200) & (life < wl.w + 1500))[0]
        keys += [[0, h, t] for t in rng.choice(short, 3, replace=False)]
        keys += [[0, h, t] for t in rng.choice(mid, 2, replace=False)]
    keys = np.array(keys, np.int32)
    rk, rv = oracle.attn_bwd_keys(qf, kf, vf, dOf, 1 / math.sqrt(wl.D), keys, rank, tau, wl.s, wl.w)
    check(dkh[0, keys[:, 2], keys[:, 1]], rk, "dk keys")
    check(dvh[0, keys[:, 2], keys[:, 1]], rv, "dv keys")


def test_attn_bwd_long_context_sampled():
    """The long-context workload (b1 H8 G4 D128 S131072, s16 w1024 k3056): dq of sampled
    rows and dk/dv of window-only keys against the oracle; the softmax-row invariants
    over all keys."""
    wl = synth.LONG
    bud = (wl.s, wl.w, wl.k)
    q, k, v, prio = synth.make_prefill_device(wl, "cuda")
    dO = synth.normal_bf16_torch(wl.seed, synth.DO, (wl.b, wl.S, wl.Hq, wl.D), "cuda")
    _, _, ev, lists = kvpop.mask(prio, *bud)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, bud)
    dq, dk, dv = kvpop.attn_bwd(q, k, v, O, dO, lse, ev, lists, bud)
    torch.cuda.synchronize()
    # invariants, summed on the device in fp64
    dks = dk.double().sum(dim=1)
    assert float(dks.abs().max()) <= 1e-3 * float(dk.double().abs().sum(dim=1).max())
    ref_v = dO.double().view(wl.b, wl.S, wl.H, wl.G, wl.D).sum(dim=(1, 3))
    assert float((dv.double().sum(dim=1) - ref_v).abs().max()) <= 1e-2 * float(ref_v.abs().max()) + 1e-2
    qf, kf, vf = host(q), host(k), host(v)
    rank, tau, _ = oracle.mask(host(prio), *bud)
    evh = host(ev)
    rng = np.random.default_rng(23)
    pos = np.concatenate([rng.integers(0, wl.S, 24), [0, 4095, 65536, wl.S - 1]])
    rows = np.stack([np.zeros_like(pos), rng.integers(0, wl.Hq, len(pos)), pos], axis=1).astype(np.int32)
    qi, ji = torch.from_numpy(rows[:, 2]).long().cuda(), torch.from_numpy(rows[:, 1]).long().cuda()
    rq = oracle.attn_bwd_rows(host(q[0, qi, ji]), host(dO[0, qi, ji]), kf, vf, wl.G, 1 / math.sqrt(wl.D), rows,
                              rank, tau, wl.s, wl.w)
    check(host(dq[0, qi, ji]), rq, "dq rows")
    h = 3
    life = evh[0, h] - np.arange(wl.S)
    short = np.nonzero((life == wl.w) & (np.arange(wl.S) >= wl.s) & (np.arange(wl.S) < wl.S - wl.w))[0]
    keys = np.array([[0, h, t] for t in rng.choice(short, 3, replace=False)], np.int32)
    # the oracle only needs the rows these keys reach: positions [t, t + w) of KV head h
    rk, rv = oracle.attn_bwd_keys(qf, kf, vf, host(dO), 1 / math.sqrt(wl.D), keys, rank, tau, wl.s, wl.w)
    check(host(dk[0, torch.from_numpy(keys[:, 2]).long().cuda(), h]), rk, "dk keys")
    check(host(dv[0, torch.from_numpy(keys[:, 2]).long().cuda(), h]), rv, "dv keys")
