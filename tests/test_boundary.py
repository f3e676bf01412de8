"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before anything is launched."""
import ctypes

import pytest

from fixed_budget_kv_gb300 import kvpop


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kvpop.load()


def test_exports_every_declared_symbol(lib):
    names = kvpop.header_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in range(6):
        assert lib.kvpop_status_string(st)
    assert lib.kvpop_version() >= 1


def test_sizes(lib):
    # mask workspace and lists grow with the problem; lists are [b,H,ceil(S/64),k] int32 pairs
    assert kvpop.mask_lists_size(1, 8, 16384, 16, 512, 1520) == 8 * 256 * 1520 * 8
    assert kvpop.mask_lists_size(2, 1, 100, 0, 0, 3) == 2 * 2 * 3 * 8
    assert kvpop.mask_workspace_size(1, 1, 256, 4, 32, 32) > 0
    assert kvpop.target_workspace_size(1, 16384, 32, 8) == 16384 * 32 * 4


@pytest.mark.parametrize("args,code", [
    ((1, 1, 0, kvpop.Budget(1, 1, 1)), 1),           # S = 0
    ((1, 1, 10, kvpop.Budget(0, 0, 0)), 1),          # B = 0
    ((1, 1, 10, kvpop.Budget(-1, 2, 2)), 1),         # negative budget
    ((1, 1, 131073, kvpop.Budget(1, 1, 1)), 2),      # S above the supported maximum
])
def test_mask_validation(lib, args, code):
    n = ctypes.c_size_t()
    assert lib.kvpop_mask_workspace_size(*args, ctypes.byref(n)) == code
    assert lib.kvpop_last_error()


def test_attn_validation(lib):
    P = ctypes.c_void_p(16)
    bud = kvpop.Budget(0, 0, 0)
    # D = 96 unsupported
    assert lib.kvpop_attn_fwd(P, P, P, 1, 64, 4, 1, 96, 0.0, None, None, bud, None, P, None) == 2
    # Hq not a multiple of H
    assert lib.kvpop_attn_fwd(P, P, P, 1, 64, 5, 2, 64, 0.0, None, None, bud, None, P, None) == 1
    # G = 3 does not divide 128
    assert lib.kvpop_attn_fwd(P, P, P, 1, 64, 3, 1, 64, 0.0, None, None, bud, None, P, None) == 2
    # misaligned pointer
    assert lib.kvpop_attn_fwd(ctypes.c_void_p(18), P, P, 1, 64, 4, 1, 64, 0.0, None, None, bud, None, P,
                              None) == 2
    # sparse mode without lists and O
    assert lib.kvpop_attn_fwd(P, P, P, 1, 64, 4, 1, 64, 0.0, P, None, kvpop.Budget(1, 1, 1), None, P,
                              None) == 1


def test_target_and_cache_validation(lib):
    P = ctypes.c_void_p(16)
    n = ctypes.c_size_t()
    assert lib.kvpop_future_target_workspace_size(1, 64, 3, 1, ctypes.byref(n)) == 2
    assert lib.kvpop_future_target(P, P, P, 1, 64, 4, 1, 64, 0.0, -1, P, P, 1 << 20, None) == 1
    h = ctypes.c_void_p()
    assert lib.kvpop_cache_create(1, 1, 3, 64, kvpop.Budget(1, 1, 1), ctypes.byref(h)) == 2
    assert lib.kvpop_cache_create(1, 1, 4, 64, kvpop.Budget(0, 0, 0), ctypes.byref(h)) == 1
    # at most 65536 slots per head (the split merge holds 256 splits of 256 slots)
    assert lib.kvpop_cache_create(1, 1, 4, 64, kvpop.Budget(16, 1024, 65536 - 1040 + 1), ctypes.byref(h)) == 1
    assert lib.kvpop_decode_step(None, P, P, P, P, P, P, None, None) == 1


def test_training_side_validation(lib):
    """Argument checks of the normalised target, teacher labels and boundary loss
    (host-side: nothing is launched on these paths)."""
    P = ctypes.c_void_p(16)
    bud = kvpop.Budget(1, 2, 3)
    assert lib.kvpop_target_normalize(None, 1, 1, 8, 4, 2, 0.0, P, None) == 1
    assert lib.kvpop_target_normalize(P, 1, 1, 8, 4, 2, -1.0, P, None) == 1        # eps < 0
    assert lib.kvpop_teacher_labels(P, 1, 1, 8, bud, 0, P, P, P, None) == 1          # n = 0
    assert lib.kvpop_teacher_labels(P, 1, 1, 8, kvpop.Budget(-1, 2, 3), 2, P, P, P, None) == 1
    assert lib.kvpop_teacher_labels(P, 300, 300, 8, bud, 2, P, P, P, None) == 2      # b*H > 65535
    assert lib.kvpop_boundary_loss(P, P, P, None, 1, 1, 8, 2, 2, P, 0.0, P, P, None) == 1   # tau = 0
    assert lib.kvpop_boundary_loss(P, P, P, None, 1, 1, 8, 2, 2, None, 1.0, P, P, None) == 1
    assert lib.kvpop_boundary_loss(P, P, P, None, 64, 64, 8192, 2, 2, P, 1.0, P, P, None) == 2  # > 2^24


def test_attn_bwd_sizes_and_validation(lib):
    # workspace: two fp32 row arrays [b,H,S rounded up to 128,G], per 512-row block a key
    # list of s + k + 512 pairs, and one count per block (each part 256-byte aligned)
    def up(x):
        return (x + 255) // 256 * 256
    b, S, Hq, H, bud = 1, 1000, 8, 2, (3, 40, 60)
    nblk = (S + 511) // 512
    want = 2 * up(b * H * 1024 * 4 * 4) + up(b * H * nblk * (3 + 60 + 512) * 8) + up(b * H * nblk * 4)
    assert kvpop.attn_bwd_workspace_size(b, S, Hq, H, bud) == want
    n = ctypes.c_size_t()
    assert lib.kvpop_attn_bwd_workspace_size(1, 0, 8, 2, kvpop.Budget(1, 1, 1), ctypes.byref(n)) == 1
    assert lib.kvpop_attn_bwd_workspace_size(1, 10, 8, 2, kvpop.Budget(0, 0, 0), ctypes.byref(n)) == 1
    assert lib.kvpop_attn_bwd_workspace_size(1, 10, 6, 2, kvpop.Budget(1, 1, 1), ctypes.byref(n)) == 2  # G = 3
    assert lib.kvpop_attn_bwd_workspace_size(1, 10, 8, 2, kvpop.Budget(1, 1, 1), None) == 1
    P = ctypes.c_void_p(256)
    ok = kvpop.Budget(1, 2, 3)
    ws = ctypes.c_size_t(1 << 30)

    def call(q=P, O=P, D=64, ev=P, lists=P, bud=ok, dq=P, wsp=P, wsn=ws, Hq=8, H=2):
        return lib.kvpop_attn_bwd(q, P, P, O, P, P, 1, 100, Hq, H, D, 0.0, ev, lists, bud, dq, P, P, wsp, wsn, None)
    assert call(O=None) == 1                        # O missing
    assert call(ev=None) == 1                       # not sparse
    assert call(lists=None) == 1                    # k > 0 needs lists
    assert call(dq=None) == 1                       # output missing
    assert call(D=96) == 2                          # head dim
    assert call(Hq=6, H=2) == 2                     # G = 3 does not divide 128
    assert call(wsn=ctypes.c_size_t(16)) == 1       # workspace too small
    assert call(wsp=ctypes.c_void_p(272)) == 2      # workspace not 256-byte aligned
    assert call(q=ctypes.c_void_p(264)) == 2        # tensor not 16-byte aligned
    assert lib.kvpop_last_error()
