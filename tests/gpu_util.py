"""Helpers for the GPU parity tests (host <-> device marshalling, comparisons)."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor (same shape)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a if dtype is None else a.astype(dtype))).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def assert_close_log(got, ref, atol, what=""):
    """Element-wise |got - ref| <= atol; -inf must match -inf exactly."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    bad = np.nonzero(ninf_g != ninf_r)[0] if got.ndim == 1 else np.argwhere(ninf_g != ninf_r)
    assert not (ninf_g != ninf_r).any(), f"{what}: -inf pattern differs at {bad[:5]}"
    fin = ~ninf_r
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite values"
    err = np.abs(got[fin] - ref[fin])
    worst = float(err.max()) if err.size else 0.0
    assert worst <= atol, f"{what}: max abs error {worst:.3e} > {atol:.1e}"
    return worst
