"""Python binding of libkvpop (ctypes).

Argument marshalling only: every step of the hot path runs in the CUDA
library.  torch provides device memory and the current stream.  If the shared
library has not been built the import of this module still works, but every
call raises ``KvpopUnavailable`` -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvpop.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvpop.h")
TAU_ALL = 2147483647
LIST_QBLOCK = 64

c_int = ctypes.c_int
c_i32 = ctypes.c_int32
c_size = ctypes.c_size_t
c_float = ctypes.c_float
c_void_p = ctypes.c_void_p


class KvpopError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class KvpopUnavailable(RuntimeError):
    pass


class Budget(ctypes.Structure):
    _fields_ = [("s", c_i32), ("w", c_i32), ("k", c_i32)]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions that include/kvpop.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(kvpop_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise KvpopUnavailable(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P = c_void_p
    sig = {
        "kvpop_status_string": ([c_int], ctypes.c_char_p),
        "kvpop_last_error": ([], ctypes.c_char_p),
        "kvpop_version": ([], c_int),
        "kvpop_device_status": ([P, c_int], c_int),
        "kvpop_mask_workspace_size": ([c_int, c_int, c_int, Budget, P], c_int),
        "kvpop_mask_lists_size": ([c_int, c_int, c_int, Budget, P], c_int),
        "kvpop_mask": ([P, c_int, c_int, c_int, Budget, P, P, P, P, P, c_size, P], c_int),
        "kvpop_attn_fwd": ([P, P, P, c_int, c_int, c_int, c_int, c_int, c_float, P, P, Budget, P, P, P],
                           c_int),
        "kvpop_attn_bwd_workspace_size": ([c_int, c_int, c_int, c_int, Budget, P], c_int),
        "kvpop_attn_bwd": ([P, P, P, P, P, P, c_int, c_int, c_int, c_int, c_int, c_float, P, P, Budget, P, P, P,
                            P, c_size, P], c_int),
        "kvpop_future_target_workspace_size": ([c_int, c_int, c_int, c_int, P], c_int),
        "kvpop_future_target": ([P, P, P, c_int, c_int, c_int, c_int, c_int, c_float, c_int, P, P, c_size,
                                 P], c_int),
        "kvpop_future_target_noalloc": ([P, P, P, c_int, c_int, c_int, c_int, c_int, c_float, c_int, P, P],
                                        c_int),
        "kvpop_target_normalize": ([P, c_int, c_int, c_int, c_int, c_int, c_float, P, P], c_int),
        "kvpop_teacher_labels": ([P, c_int, c_int, c_int, Budget, c_int, P, P, P, P], c_int),
        "kvpop_boundary_loss": ([P, P, P, P, c_int, c_int, c_int, c_int, c_int, P, c_float, P, P, P], c_int),
        "kvpop_cache_create": ([c_int, c_int, c_int, c_int, Budget, P], c_int),
        "kvpop_cache_destroy": ([P], c_int),
        "kvpop_cache_prefill": ([P, P, P, P, c_int, P, P], c_int),
        "kvpop_decode_step": ([P, P, P, P, P, P, P, P, P], c_int),
        "kvpop_cache_slots": ([P, P, P], c_int),
        "kvpop_cache_position": ([P, P], c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def available() -> bool:
    try:
        load()
        return True
    except (KvpopUnavailable, OSError):
        return False


def _check(st: int, what: str):
    if st != 0:
        lib = load()
        msg = lib.kvpop_status_string(st).decode()
        detail = lib.kvpop_last_error().decode()
        raise KvpopError(st, f"{what}: {msg}: {detail}")


def _p(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return c_void_p(s.cuda_stream)


def _need(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def device_status(reset: bool = True):
    out = (c_i32 * 4)()
    st = load().kvpop_device_status(ctypes.cast(out, c_void_p), int(reset))
    return st, list(out)


# ----------------------------------------------------------------------------
# mask
# ----------------------------------------------------------------------------

def mask_workspace_size(b, H, S, s, w, k) -> int:
    n = c_size()
    _check(load().kvpop_mask_workspace_size(b, H, S, Budget(s, w, k), ctypes.byref(n)), "mask_workspace_size")
    return n.value


def mask_lists_size(b, H, S, s, w, k) -> int:
    n = c_size()
    _check(load().kvpop_mask_lists_size(b, H, S, Budget(s, w, k), ctypes.byref(n)), "mask_lists_size")
    return n.value


def mask(prio: torch.Tensor, s: int, w: int, k: int, lists: bool = True, workspace=None, out=None,
         stream=None):
    """rank, tau, evict_at [b,H,S] int32 and the long-range lists [b,H,ceil(S/64),k,2]
    (position, evict_at) for priorities [b,H,S] fp32."""
    _need(prio, torch.float32, "prio")
    b, H, S = prio.shape
    lib = load()
    dev = prio.device
    if out is None:
        rank = torch.empty((b, H, S), dtype=torch.int32, device=dev)
        tau = torch.empty_like(rank)
        ev = torch.empty_like(rank)
        nl = (S + LIST_QBLOCK - 1) // LIST_QBLOCK
        lst = torch.empty((b, H, nl, max(k, 0), 2), dtype=torch.int32, device=dev) if (lists and k > 0) else None
    else:
        rank, tau, ev, lst = out
    if workspace is None:
        workspace = torch.empty(mask_workspace_size(b, H, S, s, w, k), dtype=torch.uint8, device=dev)
    _check(lib.kvpop_mask(_p(prio), b, H, S, Budget(s, w, k), _p(rank), _p(tau), _p(ev), _p(lst),
                          _p(workspace), workspace.numel(), _stream(stream)), "kvpop_mask")
    return rank, tau, ev, lst


# ----------------------------------------------------------------------------
# attention and target
# ----------------------------------------------------------------------------

def attn_fwd(q, k, v, scale: float = 0.0, evict_at=None, lists=None, budget=(0, 0, 0), want_o=True,
             out=None, stream=None):
    """Sparse (evict_at/lists given) or dense causal attention.  Returns (O or None, lse)."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    if v is not None:
        _need(v, torch.bfloat16, "v")
    b, S, Hq, D = q.shape
    H = k.shape[2]
    if out is None:
        O = torch.empty_like(q) if want_o else None
        lse = torch.empty((b, Hq, S), dtype=torch.float32, device=q.device)
    else:
        O, lse = out
    _check(load().kvpop_attn_fwd(_p(q), _p(k), _p(v), b, S, Hq, H, D, float(scale), _p(evict_at),
                                 _p(lists), Budget(*budget), _p(O), _p(lse), _stream(stream)),
           "kvpop_attn_fwd")
    return O, lse


def attn_bwd_workspace_size(b, S, Hq, H, budget) -> int:
    n = c_size()
    _check(load().kvpop_attn_bwd_workspace_size(b, S, Hq, H, Budget(*budget), ctypes.byref(n)),
           "attn_bwd_workspace_size")
    return n.value


def attn_bwd(q, k, v, O, dO, lse, evict_at, lists, budget, scale: float = 0.0, workspace=None, out=None,
             stream=None):
    """Gradient of the sparse attention: (dq [b,S,Hq,D], dk, dv [b,S,H,D]), fp32.

    O and lse are the forward's outputs for the same inputs; dO is the upstream
    gradient (bf16, the shape of q)."""
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (O, "O"), (dO, "dO")):
        _need(t, torch.bfloat16, name)
    _need(lse, torch.float32, "lse")
    b, S, Hq, D = q.shape
    H = k.shape[2]
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(b, S, Hq, H, budget), dtype=torch.uint8, device=q.device)
    if out is None:
        dq = torch.empty((b, S, Hq, D), dtype=torch.float32, device=q.device)
        dk = torch.empty((b, S, H, D), dtype=torch.float32, device=q.device)
        dv = torch.empty_like(dk)
    else:
        dq, dk, dv = out
    _check(load().kvpop_attn_bwd(_p(q), _p(k), _p(v), _p(O), _p(dO), _p(lse), b, S, Hq, H, D, float(scale),
                                 _p(evict_at), _p(lists), Budget(*budget), _p(dq), _p(dk), _p(dv), _p(workspace),
                                 workspace.numel(), _stream(stream)), "kvpop_attn_bwd")
    return dq, dk, dv


def target_workspace_size(b, S, Hq, H) -> int:
    n = c_size()
    _check(load().kvpop_future_target_workspace_size(b, S, Hq, H, ctypes.byref(n)),
           "future_target_workspace_size")
    return n.value


def future_target(q, k, lse, w: int, scale: float = 0.0, workspace=None, out=None, stream=None):
    """log future-attention mass per (batch, KV head, token): [b,H,S] fp32."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(lse, torch.float32, "lse")
    b, S, Hq, D = q.shape
    H = k.shape[2]
    if workspace is None:
        workspace = torch.empty(target_workspace_size(b, S, Hq, H), dtype=torch.uint8, device=q.device)
    target = torch.empty((b, H, S), dtype=torch.float32, device=q.device) if out is None else out
    _check(load().kvpop_future_target(_p(q), _p(k), _p(lse), b, S, Hq, H, D, float(scale), int(w),
                                      _p(target), _p(workspace), workspace.numel(), _stream(stream)),
           "kvpop_future_target")
    return target


def future_target_noalloc(q, k, lse, w: int, scale: float = 0.0, out=None, stream=None):
    """Same result as future_target, for callers that cannot allocate device
    memory: the pass's scratch lives in a fixed 16 MiB array inside the library
    (problems needing more raise KvpopError).  Only the output is allocated here,
    and only when `out` is not given."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(lse, torch.float32, "lse")
    b, S, Hq, D = q.shape
    H = k.shape[2]
    target = torch.empty((b, H, S), dtype=torch.float32, device=q.device) if out is None else out
    _check(load().kvpop_future_target_noalloc(_p(q), _p(k), _p(lse), b, S, Hq, H, D, float(scale), int(w),
                                              _p(target), _stream(stream)), "kvpop_future_target_noalloc")
    return target


# ----------------------------------------------------------------------------
# training-side passes: normalised target, teacher labels, boundary loss
# ----------------------------------------------------------------------------

def target_normalize(target, G: int, w: int, eps: float, out=None, stream=None):
    """r_tgt = log(eps + exp(target) / (G * N_t)), N_t = S - t - w, [b, H, S]."""
    _need(target, torch.float32, "target")
    b, H, S = target.shape
    r = torch.empty_like(target) if out is None else out
    _check(load().kvpop_target_normalize(_p(target), b, H, S, int(G), int(w), float(eps), _p(r), _stream(stream)),
           "kvpop_target_normalize")
    return r


def teacher_labels(r_tgt, s: int, w: int, k: int, n: int, log_gamma, out=None, stream=None):
    """(t_bnd, y) per row, int32 [b, H, S]; log_gamma: fp32 [H] on the device."""
    _need(r_tgt, torch.float32, "r_tgt")
    _need(log_gamma, torch.float32, "log_gamma")
    b, H, S = r_tgt.shape
    if out is None:
        tb = torch.empty((b, H, S), dtype=torch.int32, device=r_tgt.device)
        y = torch.empty_like(tb)
    else:
        tb, y = out
    _check(load().kvpop_teacher_labels(_p(r_tgt), b, H, S, Budget(s, w, k), int(n), _p(log_gamma), _p(tb), _p(y),
                                       _stream(stream)), "kvpop_teacher_labels")
    return tb, y


def boundary_loss(r_hat, t_bnd, y, w: int, n: int, log_gamma, tau: float, omega=None, out=None, stream=None):
    """(loss[2] = (mean loss, pair count), grad [b, H, S]) of the pairwise boundary loss."""
    _need(r_hat, torch.float32, "r_hat")
    b, H, S = r_hat.shape
    if out is None:
        loss = torch.empty(2, dtype=torch.float32, device=r_hat.device)
        grad = torch.empty_like(r_hat)
    else:
        loss, grad = out
    _check(load().kvpop_boundary_loss(_p(r_hat), _p(t_bnd), _p(y), _p(omega), b, H, S, int(w), int(n),
                                      _p(log_gamma), float(tau), _p(loss), _p(grad), _stream(stream)),
           "kvpop_boundary_loss")
    return loss, grad


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

class Cache:
    """Fixed-budget decode cache of B = s + w + k slots per (sequence, KV head)."""

    def __init__(self, n: int, H: int, G: int, D: int, s: int, w: int, k: int):
        self.n, self.H, self.G, self.D = n, H, G, D
        self.s, self.w, self.k = s, w, k
        self.B = s + w + k
        self._h = c_void_p()
        _check(load().kvpop_cache_create(n, H, G, D, Budget(s, w, k), ctypes.byref(self._h)),
               "kvpop_cache_create")

    def close(self):
        if self._h:
            load().kvpop_cache_destroy(self._h)
            self._h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, k, v, prio, evict_at, stream=None):
        _need(k, torch.bfloat16, "k")
        _need(v, torch.bfloat16, "v")
        _need(prio, torch.float32, "prio")
        _need(evict_at, torch.int32, "evict_at")
        P = k.shape[1]
        _check(load().kvpop_cache_prefill(self._h, _p(k), _p(v), _p(prio), P, _p(evict_at), _stream(stream)),
               "kvpop_cache_prefill")

    def step(self, q_new, k_new, v_new, prio_new, out=None, stream=None):
        if out is None:
            O = torch.empty_like(q_new)
            lse = torch.empty(q_new.shape[:2], dtype=torch.float32, device=q_new.device)
            ev = torch.empty((self.n, self.H), dtype=torch.int32, device=q_new.device)
        else:
            O, lse, ev = out
        _check(load().kvpop_decode_step(self._h, _p(q_new), _p(k_new), _p(v_new), _p(prio_new), _p(O),
                                        _p(lse), _p(ev), _stream(stream)), "kvpop_decode_step")
        return O, lse, ev

    def slots(self, stream=None):
        out = torch.empty((self.n, self.H, self.B), dtype=torch.int32, device="cuda")
        _check(load().kvpop_cache_slots(self._h, _p(out), _stream(stream)), "kvpop_cache_slots")
        return out

    def position(self) -> int:
        q = c_i32()
        _check(load().kvpop_cache_position(self._h, ctypes.byref(q)), "kvpop_cache_position")
        return q.value
