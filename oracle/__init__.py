"""fp64 CPU oracle for the KVpop hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library; the
heavy loops live in ``oracle.c`` (plain C, fp64, OpenMP over independent rows)
and this module only marshals numpy arrays.

Every function restates a definition from the KVpop pages:
  * budget, eligible set, mask and rank cutoff -- "KVpop ... 精读笔记",
    section 2.1 (B = s + w + k), section 2.2 (E(q)), section 2.3 (M_{q,t}, tau_q);
  * running threshold with a Fenwick tree -- "KVpop — 基于预测性在线剪枝的键值缓存压缩",
    section 2.4;
  * softmax attention and its log-sum-exp -- "KVpop ... 精读笔记", section 2.3;
  * the gradient of that attention (the student is trained through the
    sparse attention) -- "KVpop ... 精读笔记", section 2.1, Figure 1;
  * future-attention mass and Eq. (8) -- "KVpop ... 精读笔记", sections 2.2-2.3;
  * decode-time eviction at the window boundary -- "KVpop ... 精读笔记",
    section 2.4 (token u = q - w leaves the window) and section 2.3;
  * normalised target r_t, decayed scores, teacher boundary labels and the
    pairwise boundary loss -- "KVpop ... 精读笔记", section 2.2.
Readings where the pages are silent are listed in the header of ``oracle.c``.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, invariants, brute force and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
TAU_ALL = np.iinfo(np.int32).max

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (fp64, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-o", _SO, _SRC,
               "-lm"]
        subprocess.check_call(cmd)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        _lib.oracle_rank.argtypes = [P, i32, P]
        _lib.oracle_tau_fenwick.argtypes = [P, i32, i32, i32, i32, P]
        _lib.oracle_tau_bruteforce.argtypes = [P, i32, i32, i32, i32, P]
        _lib.oracle_retained.argtypes = [P, P, i32, i32, i32, i32]
        _lib.oracle_mask_dense.argtypes = [P, P, i32, i32, i32, P]
        _lib.oracle_evict_at_scan.argtypes = [P, P, i32, i32, i32, P]
        _lib.oracle_evict_at_sweep.argtypes = [P, P, i32, i32, i32, i32, P]
        _lib.oracle_attn_rows.argtypes = [P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32, i32,
                                          P, i64, P, P]
        _lib.oracle_attn_bwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32, i32, P, P, P]
        _lib.oracle_attn_bwd_rows.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32, i32,
                                              P, i64, P]
        _lib.oracle_attn_bwd_keys.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32, i32,
                                              P, i64, P, P]
        _lib.oracle_target_lse.argtypes = [P, P, P, i32, i32, i32, i32, i32, f64, i32, P, i64, P]
        _lib.oracle_target_colsum.argtypes = [P, P, i32, i32, i32, i32, i32, f64, i32, P]
        _lib.oracle_target_normalize.argtypes = [P, i64, i32, i32, i32, f64, P]
        _lib.oracle_teacher_labels.argtypes = [P, i32, i32, i32, i32, i32, ctypes.c_float, P, P]
        _lib.oracle_teacher_labels_rows.argtypes = [P, i32, i32, i32, i32, i32, ctypes.c_float, P, i32, P, P]
        _lib.oracle_boundary_loss.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, P, f64, P, P]
        _lib.oracle_boundary_loss.restype = i64
        _lib.oracle_num_threads.restype = i32
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------------------
# mask
# ----------------------------------------------------------------------------

def rank(prio: np.ndarray) -> np.ndarray:
    """rank[..., t] = position of t in (priority desc, index asc) order, 0 = best."""
    lib = _load()
    prio = np.ascontiguousarray(prio, dtype=np.float32)
    S = prio.shape[-1]
    flat = prio.reshape(-1, S)
    out = np.empty(flat.shape, dtype=np.int32)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty(S, dtype=np.int32)
        lib.oracle_rank(_p(row), S, _p(o))
        out[i] = o
    return out.reshape(prio.shape)


def _per_row(fn, rank_: np.ndarray, *args) -> np.ndarray:
    rank_ = np.ascontiguousarray(rank_, dtype=np.int32)
    S = rank_.shape[-1]
    flat = rank_.reshape(-1, S)
    out = np.empty(flat.shape, dtype=np.int32)
    for i in range(flat.shape[0]):
        o = np.empty(S, dtype=np.int32)
        fn(_p(np.ascontiguousarray(flat[i])), S, *args, _p(o))
        out[i] = o
    return out.reshape(rank_.shape)


def tau_fenwick(rank_: np.ndarray, s: int, w: int, k: int) -> np.ndarray:
    """tau[..., q]: rank of the k-th best token of E(q) (Fenwick tree)."""
    return _per_row(_load().oracle_tau_fenwick, rank_, s, w, k)


def tau_bruteforce(rank_: np.ndarray, s: int, w: int, k: int) -> np.ndarray:
    """tau by sorting E(q) for every q (small S only)."""
    return _per_row(_load().oracle_tau_bruteforce, rank_, s, w, k)


def _per_row2(fn, rank_, tau_, *args):
    rank_ = np.ascontiguousarray(rank_, dtype=np.int32)
    tau_ = np.ascontiguousarray(tau_, dtype=np.int32)
    S = rank_.shape[-1]
    fr, ft = rank_.reshape(-1, S), tau_.reshape(-1, S)
    out = np.empty(fr.shape, dtype=np.int32)
    for i in range(fr.shape[0]):
        o = np.empty(S, dtype=np.int32)
        fn(_p(np.ascontiguousarray(fr[i])), _p(np.ascontiguousarray(ft[i])), S, *args, _p(o))
        out[i] = o
    return out.reshape(rank_.shape)


def evict_at_scan(rank_, tau_, s: int, w: int) -> np.ndarray:
    """First row q >= t + w at which t is not retained (S if never; S for sinks)."""
    return _per_row2(_load().oracle_evict_at_scan, rank_, tau_, s, w)


def evict_at_sweep(rank_, tau_, s: int, w: int, k: int) -> np.ndarray:
    """evict_at by the online eviction sweep (one entrant per row)."""
    return _per_row2(_load().oracle_evict_at_sweep, rank_, tau_, s, w, k)


def mask_dense(rank_1d: np.ndarray, tau_1d: np.ndarray, s: int, w: int) -> np.ndarray:
    """Boolean [S,S] mask M_{q,t} (with t <= q) for one (batch, KV head)."""
    S = rank_1d.shape[0]
    M = np.zeros((S, S), dtype=np.uint8)
    _load().oracle_mask_dense(_p(np.ascontiguousarray(rank_1d, np.int32)),
                              _p(np.ascontiguousarray(tau_1d, np.int32)), S, s, w, _p(M))
    return M.astype(bool)


def mask(prio: np.ndarray, s: int, w: int, k: int):
    """rank, tau and evict_at for priorities [..., S]."""
    r = rank(prio)
    t = tau_fenwick(r, s, w, k)
    e = evict_at_sweep(r, t, s, w, k)
    return r, t, e


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def attn_rows(qvecs, k, v, G: int, scale: float, rows, rank_=None, tau_=None, s=0, w=0,
              want_o=True):
    """Attention for explicit rows.

    qvecs [n, D] float (query vectors), k/v [b,S,H,D] float, rows [n,3] int
    (batch, query head, position).  rank/tau [b,H,S] select the sparse mask;
    None gives dense causal attention.  Returns (O [n,D] fp64 or None, lse [n]).
    """
    lib = _load()
    qvecs = np.ascontiguousarray(qvecs, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    b, S, H, D = k.shape
    n = rows.shape[0]
    O = np.zeros((n, D), dtype=np.float64) if want_o else None
    lse = np.empty(n, dtype=np.float64)
    rk = None if rank_ is None else np.ascontiguousarray(rank_, dtype=np.int32)
    tu = None if tau_ is None else np.ascontiguousarray(tau_, dtype=np.int32)
    lib.oracle_attn_rows(_p(qvecs), _p(k), _p(v), b, S, H, G, D, float(scale),
                         None if rk is None else _p(rk), None if tu is None else _p(tu),
                         int(s), int(w), _p(rows), n, None if O is None else _p(O), _p(lse))
    return O, lse


def attn(q, k, v, scale: float, rank_=None, tau_=None, s=0, w=0, want_o=True):
    """Full attention. q [b,S,Hq,D]; returns O [b,S,Hq,D] fp64 and lse [b,Hq,S] fp64."""
    b, S, Hq, D = q.shape
    H = k.shape[2]
    G = Hq // H
    bi, j, qp = np.meshgrid(np.arange(b), np.arange(Hq), np.arange(S), indexing="ij")
    rows = np.stack([bi.ravel(), j.ravel(), qp.ravel()], axis=1).astype(np.int32)
    qvecs = np.ascontiguousarray(np.transpose(q, (0, 2, 1, 3)).reshape(-1, D), dtype=np.float32)
    O, lse = attn_rows(qvecs, k, v, G, scale, rows, rank_, tau_, s, w, want_o)
    lse = lse.reshape(b, Hq, S)
    if O is not None:
        O = np.transpose(O.reshape(b, Hq, S, D), (0, 2, 1, 3))
    return O, lse


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32_or_none(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def attn_bwd(q, k, v, dO, scale: float, rank_=None, tau_=None, s=0, w=0):
    """Gradient of sum(dO * O) through the attention of ``attn`` (sparse when
    rank/tau are given, dense causal otherwise).  q, dO [b,S,Hq,D]; k, v
    [b,S,H,D].  Returns dq [b,S,Hq,D], dk, dv [b,S,H,D], all fp64."""
    lib = _load()
    q, k, v, dO = _f32(q), _f32(k), _f32(v), _f32(dO)
    b, S, Hq, D = q.shape
    H = k.shape[2]
    dq = np.empty((b, S, Hq, D), dtype=np.float64)
    dk = np.empty((b, S, H, D), dtype=np.float64)
    dv = np.empty((b, S, H, D), dtype=np.float64)
    rk, tu = _i32_or_none(rank_), _i32_or_none(tau_)
    lib.oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dO), b, S, H, Hq // H, D, float(scale),
                        None if rk is None else _p(rk), None if tu is None else _p(tu), int(s), int(w),
                        _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def attn_bwd_rows(qvecs, dovecs, k, v, G: int, scale: float, rows, rank_=None, tau_=None, s=0, w=0):
    """dq of explicit rows [n,3] = (batch, query head, position); qvecs/dovecs
    [n,D] are those rows' query and upstream-gradient vectors.  Returns [n,D]."""
    lib = _load()
    qvecs, dovecs, k, v = _f32(qvecs), _f32(dovecs), _f32(k), _f32(v)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    b, S, H, D = k.shape
    out = np.empty((rows.shape[0], D), dtype=np.float64)
    rk, tu = _i32_or_none(rank_), _i32_or_none(tau_)
    lib.oracle_attn_bwd_rows(_p(qvecs), _p(dovecs), _p(k), _p(v), b, S, H, G, D, float(scale),
                             None if rk is None else _p(rk), None if tu is None else _p(tu), int(s), int(w),
                             _p(rows), rows.shape[0], _p(out))
    return out


def attn_bwd_keys(q, k, v, dO, scale: float, keys, rank_=None, tau_=None, s=0, w=0):
    """dk, dv of explicit keys [n,3] = (batch, KV head, position): each row that
    retains the key is solved in full.  Returns two [n,D] arrays."""
    lib = _load()
    q, k, v, dO = _f32(q), _f32(k), _f32(v), _f32(dO)
    keys = np.ascontiguousarray(keys, dtype=np.int32).reshape(-1, 3)
    b, S, Hq, D = q.shape
    H = k.shape[2]
    dk = np.empty((keys.shape[0], D), dtype=np.float64)
    dv = np.empty((keys.shape[0], D), dtype=np.float64)
    rk, tu = _i32_or_none(rank_), _i32_or_none(tau_)
    lib.oracle_attn_bwd_keys(_p(q), _p(k), _p(v), _p(dO), b, S, H, Hq // H, D, float(scale),
                             None if rk is None else _p(rk), None if tu is None else _p(tu), int(s), int(w),
                             _p(keys), keys.shape[0], _p(dk), _p(dv))
    return dk, dv


# ----------------------------------------------------------------------------
# future-attention target
# ----------------------------------------------------------------------------

def target_lse(q, k, lse, w: int, scale: float, keys=None):
    """Route B (Eq. 8): log sum_g sum_{d>=t+w} exp(l(d,t) - LSE_d).

    q [b,S,Hq,D], k [b,S,H,D], lse [b,Hq,S] fp64 (rows d >= t+w must be valid).
    keys [n,3] (batch, KV head, t) or None for all; returns [n] or [b,H,S].
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    b, S, Hq, D = q.shape
    H = k.shape[2]
    full = keys is None
    if full:
        bi, h, t = np.meshgrid(np.arange(b), np.arange(H), np.arange(S), indexing="ij")
        keys = np.stack([bi.ravel(), h.ravel(), t.ravel()], axis=1)
    keys = np.ascontiguousarray(keys, dtype=np.int32).reshape(-1, 3)
    out = np.empty(keys.shape[0], dtype=np.float64)
    lib.oracle_target_lse(_p(q), _p(k), _p(lse), b, S, H, Hq // H, D, float(scale), int(w),
                          _p(keys), keys.shape[0], _p(out))
    return out.reshape(b, H, S) if full else out


def target_colsum(q, k, w: int, scale: float):
    """Route A: log of the column sums of the dense attention map, [b,H,S]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    b, S, Hq, D = q.shape
    H = k.shape[2]
    out = np.empty((b, H, S), dtype=np.float64)
    lib.oracle_target_colsum(_p(q), _p(k), b, S, H, Hq // H, D, float(scale), int(w), _p(out))
    return out


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

def decode_sim(k_prefix, v_prefix, prio_prefix, q_steps, k_steps, v_steps, prio_steps,
               s: int, w: int, kk: int, scale: float, seqs, want_floats=True):
    """Decode with a fixed budget, simulated through the mask over the history.

    Inputs are float arrays: k/v_prefix [n,P,H,D], prio_prefix [n,H,P],
    q_steps [T,n,Hq,D], k/v_steps [T,n,H,D], prio_steps [T,n,H].
    At step i the query sits at position q = P + i; the retained slot set of
    (sequence, head) is {t : M_{q,t}} over the concatenated history, and the
    evicted position is the t whose evict_at equals q (or -1).

    Returns a dict per sequence with 'slots' (list over steps of [H] sorted
    position arrays), 'evicted' [T,H] and, if want_floats, 'O' [T,Hq,D] and
    'lse' [T,Hq].
    """
    T = q_steps.shape[0]
    P = k_prefix.shape[1]
    H = k_prefix.shape[2]
    Hq = q_steps.shape[2]
    D = k_prefix.shape[3]
    G = Hq // H
    S = P + T
    out = {}
    for n in seqs:
        prio = np.concatenate([prio_prefix[n], np.transpose(prio_steps[:, n, :])], axis=1)  # [H,S]
        r, tau, ev = mask(prio[None], s, w, kk)
        slots, evicted = [], np.full((T, H), -1, dtype=np.int32)
        for i in range(T):
            qpos = P + i
            row = []
            for h in range(H):
                sel = _row_positions(r[0, h], tau[0, h], s, w, qpos)
                row.append(np.asarray(sel, dtype=np.int32))
                hit = np.nonzero(ev[0, h] == qpos)[0]
                evicted[i, h] = int(hit[0]) if hit.size else -1
            slots.append(row)
        res = {"slots": slots, "evicted": evicted}
        if want_floats:
            kh = np.concatenate([k_prefix[n], k_steps[:, n]], axis=0)[None]   # [1,S,H,D]
            vh = np.concatenate([v_prefix[n], v_steps[:, n]], axis=0)[None]
            rows = np.array([[0, j, P + i] for i in range(T) for j in range(Hq)], dtype=np.int32)
            qv = q_steps[:, n].reshape(T * Hq, D)
            O, lse = attn_rows(qv, kh, vh, G, scale, rows, r, tau, s, w)
            res["O"] = O.reshape(T, Hq, D)
            res["lse"] = lse.reshape(T, Hq)
        out[n] = res
    return out


def _retained(rank_1d, tau_1d, s, w, q, t) -> bool:
    return bool(_load().oracle_retained(_p(np.ascontiguousarray(rank_1d, np.int32)),
                                        _p(np.ascontiguousarray(tau_1d, np.int32)), s, w, q, t))


def _row_positions(rank_1d, tau_1d, s, w, q):
    """Positions t <= q with M_{q,t}: sinks, window, or eligible with rank <= tau_q."""
    t = np.arange(q + 1)
    keep = (t < s) | (q - t < w) | ((t >= s) & (t <= q - w) & (rank_1d[: q + 1] <= tau_1d[q]))
    return t[keep]


# ----------------------------------------------------------------------------
# normalised target, teacher boundary labels, pairwise boundary loss
# ----------------------------------------------------------------------------

def target_normalize(target: np.ndarray, G: int, w: int, eps: float) -> np.ndarray:
    """r_t = log(eps + (1/G) sum_g (1/N_t) sum_{d>=t+w} A_{d,t}) from the
    unnormalised log target [..., S]; N_t = S - t - w; no future -> log(eps)."""
    t = np.ascontiguousarray(target, dtype=np.float64)
    S = t.shape[-1]
    out = np.empty_like(t)
    _load().oracle_target_normalize(_p(t), t.size // S, S, G, w, float(eps), _p(out))
    return out


def teacher_labels(r_tgt: np.ndarray, s: int, w: int, k: int, n: int, log_gamma):
    """(t_bnd, y) per row q for targets [b, H, S] (fp32) and log_gamma [H] (fp32):
    the teacher's top-k of E(q) under the decayed target, the cutoff t_bnd that the
    leaving token q - w has to beat, and y = +1 kept / -1 dropped / 0 no leaving token."""
    r = np.ascontiguousarray(r_tgt, dtype=np.float32)
    b, H, S = r.shape
    lg = np.asarray(log_gamma, dtype=np.float32).reshape(H)
    tb = np.empty((b, H, S), dtype=np.int32)
    y = np.empty((b, H, S), dtype=np.int32)
    lib = _load()
    for bi in range(b):
        for h in range(H):
            lib.oracle_teacher_labels(_p(r[bi, h]), S, s, w, k, n, ctypes.c_float(lg[h]), _p(tb[bi, h]),
                                      _p(y[bi, h]))
    return tb, y


def boundary_loss(r_hat: np.ndarray, t_bnd: np.ndarray, y: np.ndarray, w: int, n: int, log_gamma,
                  tau: float, omega=None):
    """Mean pairwise logistic loss over the labelled rows and its gradient
    d loss / d r_hat, [b, H, S]; returns (loss, grad, number of pairs)."""
    rh = np.ascontiguousarray(r_hat, dtype=np.float32)
    b, H, S = rh.shape
    tb = np.ascontiguousarray(t_bnd, dtype=np.int32)
    yy = np.ascontiguousarray(y, dtype=np.int32)
    lg = np.ascontiguousarray(np.asarray(log_gamma, dtype=np.float32).reshape(H))
    om = None if omega is None else np.ascontiguousarray(omega, dtype=np.float32)
    grad = np.empty((b, H, S), dtype=np.float64)
    loss = ctypes.c_double()
    pairs = _load().oracle_boundary_loss(_p(rh), _p(tb), _p(yy), None if om is None else _p(om), b * H, S, H,
                                         w, n, _p(lg), float(tau), ctypes.byref(loss), _p(grad))
    return loss.value, grad, int(pairs)


def teacher_labels_rows(r_1d: np.ndarray, s: int, w: int, k: int, n: int, log_gamma: float, rows):
    """(t_bnd, y) of the listed rows only, for one (batch, head) row of targets."""
    r = np.ascontiguousarray(r_1d, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    tb = np.empty(len(rows), dtype=np.int32)
    y = np.empty(len(rows), dtype=np.int32)
    _load().oracle_teacher_labels_rows(_p(r), r.shape[-1], s, w, k, n, ctypes.c_float(np.float32(log_gamma)),
                                       _p(rows), len(rows), _p(tb), _p(y))
    return tb, y
