"""Seeded synthetic inputs for the KVpop hot path.

This module is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle's tests.  It holds no arithmetic of the method itself: it only draws
numbers (counter-based, platform independent) and names the workload shapes.

Generator (stated here so that any other implementation can reproduce it):

* ``mix64(z)`` is the splitmix64 finaliser
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
  z ^= z >> 31`` on unsigned 64-bit integers (wrapping multiply).
* A stream is keyed by ``key = mix64(seed * 0x9E3779B97F4A7C15 ^ stream * 0xD1B54A32D192ED03)``.
* Draw number ``i`` of a stream is ``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``.
* ``uniform24``: ``(z >> 40) * 2**-24`` -- an exact fp32 value in [0, 1).
* ``normal``: Box-Muller (cosine branch) from draws ``2i`` and ``2i+1``:
  ``u1 = ((z0 >> 11) + 1) * 2**-53``, ``u2 = (z1 >> 11) * 2**-53``,
  ``n = sqrt(-2 ln u1) * cos(2 pi u2)`` in fp64, then rounded to fp32.
* bf16 values are the round-to-nearest-even of the fp32 draw.

Element ``i`` of a tensor is draw ``i`` of that tensor's stream in its natural
row-major layout, so a sub-block can be regenerated without the rest.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21

# stream ids
Q, K, V, PRIO, SPIKE = 1, 2, 3, 4, 5
DO = 6  # upstream gradient dL/dO of the attention output (training path)
QN, KN, VN, PRION = 11, 12, 13, 14


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = (np.uint64(seed) * _GOLDEN) ^ (np.uint64(stream) * _STREAM_MUL)
        return _mix64(np.array([z], dtype=np.uint64))[0]


def raw_draws(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of a stream as uint64."""
    key = stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GOLDEN)


def _chunked(n: int, fill) -> np.ndarray:
    """Fill an fp32 array chunk by chunk; chunks are independent (counter-based
    draws), so they run on a thread pool (numpy releases the GIL)."""
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for c0 in starts:
            fill(out, c0, min(n, c0 + _CHUNK))
        return out
    workers = min(len(starts), os.cpu_count() or 1, 32)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda c0: fill(out, c0, min(n, c0 + _CHUNK)), starts))
    return out


def uniform24(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    def fill(out, c0, c1):
        z = raw_draws(seed, stream, start + c0, c1 - c0)
        out[c0:c1] = (z >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    return _chunked(n, fill)


def normal(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    def fill(out, c0, c1):
        z = raw_draws(seed, stream, 2 * (start + c0), 2 * (c1 - c0))
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        out[c0:c1] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(np.float32)
    return _chunked(n, fill)


def normal_at(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """Normal draws number ``idx`` (any integer array) of a stream, fp32: the same
    values as ``normal`` at those positions, without drawing the rest."""
    idx = np.asarray(idx, dtype=np.uint64)
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        z0 = _mix64(key + (np.uint64(2) * idx + np.uint64(1)) * _GOLDEN)
        z1 = _mix64(key + (np.uint64(2) * idx + np.uint64(2)) * _GOLDEN)
    u1 = ((z0 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (z1 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rnd = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rnd) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic prefill workload (shapes plus value recipe)."""
    name: str
    b: int
    H: int          # KV heads
    G: int          # query heads per KV head
    D: int
    S: int
    s: int          # sink tokens
    w: int          # protected window
    k: int          # long-range top-k slots
    k_scale: float = 1.0
    prio: str = "uniform"     # "uniform" | "normal" | "normal_spikes"
    seed: int = 0

    @property
    def Hq(self) -> int:
        return self.H * self.G

    @property
    def B(self) -> int:
        return self.s + self.w + self.k

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    n: int
    H: int
    G: int
    D: int
    s: int
    w: int
    k: int
    P: int          # prefix length
    steps: int
    seed: int = 0

    @property
    def Hq(self) -> int:
        return self.H * self.G

    @property
    def B(self) -> int:
        return self.s + self.w + self.k

    def replace(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny", b=1, H=1, G=2, D=64, S=256, s=4, w=32, k=32, prio="uniform")
QWEN3_4B = Workload("qwen3-4b-layer-prefill", b=1, H=8, G=4, D=128, S=16384, s=16, w=512, k=1520,
                    k_scale=0.5, prio="normal")
QWEN3_8B = Workload("qwen3-8b-layer-prefill", b=2, H=8, G=4, D=128, S=16384, s=16, w=1024, k=3056,
                    prio="normal_spikes")
LONG = Workload("long-context-prefill", b=1, H=8, G=4, D=128, S=131072, s=16, w=1024, k=3056,
                prio="uniform")
DECODE = DecodeWorkload("fixed-budget-decode", n=64, H=8, G=4, D=128, s=16, w=512, k=1520,
                        P=8192, steps=4096)

PREFILL_WORKLOADS = {w.name: w for w in (TINY, QWEN3_4B, QWEN3_8B, LONG)}


@dataclasses.dataclass
class PrefillInputs:
    """Host arrays: q/k/v as bf16 bit patterns [b,S,heads,D]; prio fp32 [b,H,S]."""
    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    prio: np.ndarray

    def f32(self, name: str) -> np.ndarray:
        return bf16_bits_to_f32(getattr(self, name))


def _bf16_tensor(seed, stream, shape, scale=1.0):
    n = int(np.prod(shape))
    x = normal(seed, stream, n)
    if scale != 1.0:
        x = x * np.float32(scale)
    return f32_to_bf16_bits(x).reshape(shape)


def priorities(kind: str, seed: int, shape, stream: int = PRIO) -> np.ndarray:
    n = int(np.prod(shape))
    if kind == "uniform":
        p = uniform24(seed, stream, n)
    elif kind == "normal":
        p = normal(seed, stream, n)
    elif kind == "normal_spikes":
        p = normal(seed, stream, n)
        spike = uniform24(seed, SPIKE, n) < np.float32(0.01)
        p = p + np.where(spike, np.float32(5.0), np.float32(0.0)).astype(np.float32)
    else:
        raise ValueError(kind)
    return p.reshape(shape).astype(np.float32)


def make_prefill(wl: Workload) -> PrefillInputs:
    q = _bf16_tensor(wl.seed, Q, (wl.b, wl.S, wl.Hq, wl.D))
    k = _bf16_tensor(wl.seed, K, (wl.b, wl.S, wl.H, wl.D), wl.k_scale)
    v = _bf16_tensor(wl.seed, V, (wl.b, wl.S, wl.H, wl.D))
    prio = priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))
    return PrefillInputs(wl, q, k, v, prio)


@dataclasses.dataclass
class DecodeInputs:
    """Prefix (k/v [n,P,H,D] bf16 bits, prio [n,H,P]) and per-step tokens
    (q [steps,n,Hq,D], k/v [steps,n,H,D] bf16 bits, prio [steps,n,H])."""
    wl: DecodeWorkload
    k_prefix: np.ndarray
    v_prefix: np.ndarray
    prio_prefix: np.ndarray
    q_steps: np.ndarray
    k_steps: np.ndarray
    v_steps: np.ndarray
    prio_steps: np.ndarray


def make_decode(wl: DecodeWorkload, steps: int | None = None) -> DecodeInputs:
    T = wl.steps if steps is None else steps
    s = wl.seed
    kp = _bf16_tensor(s, K, (wl.n, wl.P, wl.H, wl.D))
    vp = _bf16_tensor(s, V, (wl.n, wl.P, wl.H, wl.D))
    pp = priorities("uniform", s, (wl.n, wl.H, wl.P))
    qn = _bf16_tensor(s, QN, (T, wl.n, wl.Hq, wl.D))
    kn = _bf16_tensor(s, KN, (T, wl.n, wl.H, wl.D))
    vn = _bf16_tensor(s, VN, (T, wl.n, wl.H, wl.D))
    pn = priorities("uniform", s, (T, wl.n, wl.H), stream=PRION)
    return DecodeInputs(wl, kp, vp, pp, qn, kn, vn, pn)


# --------------------------------------------------------------------------
# the same generator on a torch device (for multi-GB workloads)
# --------------------------------------------------------------------------
# uint64 arithmetic is emulated on int64 tensors: + and * wrap modulo 2**64 in
# two's complement, and a logical right shift is an arithmetic shift masked to
# the low 64 - k bits.  uniform24 is exact integer arithmetic, so it matches the
# numpy path bit for bit; normals go through the device's fp64 log/sqrt/cos and
# then fp32 -> bf16 rounding, so an element can differ from the numpy value only
# when the fp64 result sits within an ulp of an fp32 rounding boundary.

def _s64(x: int) -> int:
    x &= (1 << 64) - 1
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(z, k: int):
    import torch
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix64_t(z):
    z = z ^ _lsr(z, 30)
    z = z * _s64(0xBF58476D1CE4E5B9)
    z = z ^ _lsr(z, 27)
    z = z * _s64(0x94D049BB133111EB)
    return z ^ _lsr(z, 31)


def _raw_draws_t(seed, stream, start, count, device):
    import torch
    key = _s64(int(stream_key(seed, stream)))
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix64_t(idx * _s64(0x9E3779B97F4A7C15) + key)


def normal_bf16_torch(seed: int, stream: int, shape, device, scale: float = 1.0, chunk: int = 1 << 26):
    """bf16 tensor of the stated normal draws (times `scale`, in fp32), generated on `device`."""
    import torch
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        z = _raw_draws_t(seed, stream, 2 * c0, 2 * (c1 - c0), device)
        u1 = (_lsr(z[0::2], 11).to(torch.float64) + 1.0) * 2.0 ** -53
        u2 = _lsr(z[1::2], 11).to(torch.float64) * 2.0 ** -53
        x = (torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * np.pi * u2)).to(torch.float32)
        if scale != 1.0:
            x = x * scale
        out[c0:c1] = x.to(torch.bfloat16)
        del z, u1, u2, x
    return out.view(*shape)


def upstream_grad(wl: Workload) -> np.ndarray:
    """dO for the attention backward: bf16 bits [b,S,Hq,D], N(0,1) draws of stream DO."""
    return _bf16_tensor(wl.seed, DO, (wl.b, wl.S, wl.Hq, wl.D))


def make_prefill_device(wl: Workload, device):
    """(q, k, v, prio) on `device`: q/k/v generated there, prio copied from the numpy path."""
    import torch
    q = normal_bf16_torch(wl.seed, Q, (wl.b, wl.S, wl.Hq, wl.D), device)
    k = normal_bf16_torch(wl.seed, K, (wl.b, wl.S, wl.H, wl.D), device, wl.k_scale)
    v = normal_bf16_torch(wl.seed, V, (wl.b, wl.S, wl.H, wl.D), device)
    prio = torch.from_numpy(priorities(wl.prio, wl.seed, (wl.b, wl.H, wl.S))).to(device)
    return q, k, v, prio


def bf16_block(seed: int, stream: int, shape, start_elem: int, scale: float = 1.0) -> np.ndarray:
    """numpy bf16 bits of elements start_elem .. start_elem + prod(shape) of a stream."""
    n = int(np.prod(shape))
    x = normal(seed, stream, n, start=start_elem)
    if scale != 1.0:
        x = x * np.float32(scale)
    return f32_to_bf16_bits(x).reshape(shape)
