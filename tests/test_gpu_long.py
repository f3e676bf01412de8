"""The long-context workload (b1 H8 G4 D128 S131072, budget s16 w1024 k3056) through
the GPU path against the fp64 oracle: sparse O/LSE and dense LSE on sampled rows,
targets of the last keys of one head.  The inputs are generated on the device by
the counter-based generator and copied back for the oracle.  Tolerances as the
other parity tests: O 2e-2, LSE 2e-3, targets 2e-2 (log domain).  The mask of
this workload is compared bit-exactly in test_gpu_mask.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, host

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


def test_long_context_sampled():
    wl = synth.LONG
    S, H, G, D = wl.S, wl.H, wl.G, wl.D
    bud = (wl.s, wl.w, wl.k)
    scale = 1 / math.sqrt(D)
    q, k, v, prio = synth.make_prefill_device(wl, "cuda")
    _, _, ev, lists = kvpop.mask(prio, *bud)
    O, lse = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, bud)
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, dl, wl.w))
    torch.cuda.synchronize()
    kf, vf = host(k), host(v)
    rank, tau, _ = oracle.mask(host(prio), *bud)
    rng = np.random.default_rng(31)
    pos = np.concatenate([rng.integers(0, S, 120), [0, 1, S - 1, S - 2, 4095, 4096, 65535, 65536]])
    rows = np.stack([np.zeros_like(pos), rng.integers(0, wl.Hq, len(pos)), pos], axis=1).astype(np.int32)
    qv = host(q[0, torch.from_numpy(rows[:, 2]).long().cuda(), torch.from_numpy(rows[:, 1]).long().cuda()])
    Or, lr = oracle.attn_rows(qv, kf, vf, G, scale, rows, rank, tau, wl.s, wl.w)
    got_o = host(O[0, torch.from_numpy(rows[:, 2]).long().cuda(), torch.from_numpy(rows[:, 1]).long().cuda()])
    assert np.abs(got_o - Or).max() <= TOL_O
    assert_close_log(host(lse)[0, rows[:, 1], rows[:, 2]], lr, TOL_LSE, "sparse lse")
    _, dlr = oracle.attn_rows(qv[:64], kf, vf, G, scale, rows[:64], want_o=False)
    dlh = host(dl)
    assert_close_log(dlh[0, rows[:64, 1], rows[:64, 2]], dlr, TOL_LSE, "dense lse")
    # targets of the last keys of head 5.  Their future rows d >= t + w need the
    # dense LSE; Eq. (8) only sees positions through d >= t + w and d < S, so the
    # oracle runs on the tail [t_lo, S) of the sequence with the origin moved.
    h = 5
    t_lo = S - wl.w - 96
    d_rows = np.arange(t_lo + wl.w, S)
    trows = np.array([[0, h * G + g, d] for g in range(G) for d in d_rows], np.int32)
    tq = host(q[0, torch.from_numpy(trows[:, 2]).long().cuda(), torch.from_numpy(trows[:, 1]).long().cuda()])
    _, tlr = oracle.attn_rows(tq, kf, kf, G, scale, trows, want_o=False)
    St = S - t_lo
    lse_t = np.full((1, wl.Hq, St), np.nan)
    lse_t[0, trows[:, 1], trows[:, 2] - t_lo] = tlr
    q_t = np.zeros((1, St, wl.Hq, D), np.float32)
    q_t[0, trows[:, 2] - t_lo, trows[:, 1]] = tq
    keys = np.array([[0, h, t] for t in range(0, St - wl.w, 5)] + [[0, h, St - 1]], np.int32)
    tr = oracle.target_lse(q_t, np.ascontiguousarray(kf[:, t_lo:]), lse_t, wl.w, scale, keys)
    assert_close_log(tgt[0, h, keys[:, 2] + t_lo], tr, TOL_T, "target")
