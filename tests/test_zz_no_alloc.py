"""kvpop_future_target_noalloc: the future-target pass for callers that cannot
call cudaMalloc (an engine whose allocator owns all device memory, or a path
where cudaMalloc's implicit synchronisation is not allowed).  Its scratch lives
in a fixed 16 MiB array inside the library, so the caller passes only inputs
and outputs.  Checked through the C ABI against kvpop_future_target (caller
workspace) on two calls in a row with different inputs and sizes, which also
shows that the shared array carries nothing over from one call to the next.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_T = 2e-2
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kvpop.load()


def _inputs(seed, S, H, G, D):
    wl = synth.Workload("noalloc", b=1, H=H, G=G, D=D, S=S, s=0, w=0, k=1, seed=seed)
    inp = synth.make_prefill(wl)
    return dev_bf16(inp.q), dev_bf16(inp.k)


def _noalloc(lib, q, k, lse, w):
    b, S, Hq, D = q.shape
    H = k.shape[2]
    out = torch.full((b, H, S), float("nan"), dtype=torch.float32, device=q.device)
    st = lib.kvpop_future_target_noalloc(P(q.data_ptr()), P(k.data_ptr()), P(lse.data_ptr()), b, S, Hq, H, D,
                                         0.0, w, P(out.data_ptr()),
                                         P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.kvpop_last_error()
    return out


def test_noalloc_matches_workspace_entry_point(lib):
    # two calls in a row, different inputs and sizes, then a full Qwen3-4B-sized one
    for seed, S, H, G, D, w in [(11, 700, 2, 4, 128, 64), (12, 2000, 3, 2, 64, 300), (13, 16384, 8, 4, 128, 512)]:
        q, k = _inputs(seed, S, H, G, D)
        _, lse = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
        ref = kvpop.future_target(q, k, lse, w)
        got = _noalloc(lib, q, k, lse, w)
        torch.cuda.synchronize()
        assert_close_log(host(got).ravel(), host(ref).ravel(), TOL_T, f"noalloc S={S}")
    st, words = kvpop.device_status(reset=True)
    assert st == 0, words


def test_noalloc_rejects_oversized(lib):
    # two long-context rows need 2 x 16 MiB of scratch: refused before any launch
    st = lib.kvpop_future_target_noalloc(P(16), P(16), P(16), 2, 131072, 32, 8, 128, 0.0, 1024, P(16), None)
    assert st == 2
    assert b"scratch" in lib.kvpop_last_error()
