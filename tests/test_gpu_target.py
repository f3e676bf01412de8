"""kvpop_future_target against the fp64 oracle where a key's future spans several
query chunks of the kernel.

The target of key t ("KVpop ... 精读笔记", sections 2.2-2.3, Eq. (8), Figure 2)
sums over every future query d = t + w .. S - 1 and the G query heads of its KV
head.  The kernel splits that range into chunks of 64 query tiles (2048
positions at G = 4, 8192 at G = 1) run by different CTAs whose partial sums meet
in the output; the cases here make every early key take that path:

* small problems of 2-3 chunks, every key compared (w = 0, w beyond one chunk,
  G = 1, 2, 4, 8, D = 64 and 128, two sequences), and the sparse-LSE variant;
* the 4B-like and 8B-like workloads at full size: ~200 keys per sampled head
  spread over all positions (t = 0, 1, s, the first and last key of every
  512-key block of the kernel, random keys, the last keys with a future and
  the first without), the oracle computing the dense LSE of every row of that
  head's query heads;
* the long-context workload (S = 131072, 64 chunks): the target is a function of
  (q, k, LSE), and the oracle's dense LSE of all 524 288 rows of one head is
  out of reach for a test (O(S^2) in fp64), so both sides take the same seeded
  LSE-shaped input (log(d + 1) + U(0.25, 0.75): the size of a dense causal LSE
  of N(0,1) logits); the dense LSE itself is compared on sampled rows in
  test_gpu_long.py, and the chain dense LSE -> target is checked at this size
  by the w = 0 invariant below.

Tolerance: 2e-2 in the log domain; -inf (no future query) must match."""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_budget_kv_gb300 import kvpop, synth
from gpu_util import assert_close_log, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

TOL_T = 2e-2
CHUNK_TILES = 64  # query tiles per CTA chunk of the kernel (positions: 64 * 128 / G)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    kvpop.device_status(reset=True)
    yield
    st, words = kvpop.device_status(reset=True)
    assert st == 0, f"device status {words}"


def _chunks_spanned(S, G, w):
    """Chunks the key t = 0 sums over."""
    P = 128 // G
    tiles = (S - 1) // P - w // P + 1 if w < S else 0
    return -(-tiles // CHUNK_TILES)


# b, H, G, D, S, w
MULTI_CHUNK = [
    (1, 1, 4, 128, 5000, 64),     # 157 query tiles: three chunks
    (1, 1, 4, 128, 5000, 0),      # w = 0: every key sees every later row
    (1, 1, 4, 128, 5000, 2100),   # w beyond one chunk's 2048 positions
    (1, 1, 1, 128, 9000, 0),      # G = 1: 128 positions per tile, two chunks
    (1, 1, 1, 128, 17000, 8300),  # G = 1, w beyond one chunk's 8192 positions
    (2, 1, 2, 128, 6000, 300),    # G = 2, two sequences
    (1, 2, 8, 128, 3000, 10),     # G = 8: 16 positions per tile, three chunks
    (1, 2, 4, 64, 4500, 0),       # D = 64
]


@pytest.mark.parametrize("case", MULTI_CHUNK, ids=lambda c: "b{}H{}G{}D{}S{}w{}".format(*c))
def test_target_multi_chunk(case):
    b, H, G, D, S, w = case
    assert _chunks_spanned(S, G, w) >= 2
    wl = synth.Workload("case", b=b, H=H, G=G, D=D, S=S, s=0, w=0, k=1, prio="uniform", seed=S + 7 * w + G)
    inp = synth.make_prefill(wl)
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    scale = 1 / math.sqrt(D)
    _, lse = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, lse, w))
    qf, kf = inp.f32("q"), inp.f32("k")
    _, lr = oracle.attn(qf, kf, kf, scale, want_o=False)
    tr = oracle.target_lse(qf, kf, lr, w, scale)
    assert_close_log(tgt.ravel(), tr.ravel(), TOL_T, "target")


def test_sparse_lse_target_multi_chunk():
    """The sparse-LSE variant ("KVpop ... 精读笔记", section 2.3) on a problem of
    three chunks: GPU sparse LSE -> GPU target against oracle sparse LSE ->
    oracle target."""
    wl = synth.Workload("case", b=1, H=1, G=4, D=128, S=5000, s=16, w=64, k=200, prio="uniform", seed=21)
    inp = synth.make_prefill(wl)
    q, k, v = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    _, _, ev, lists = kvpop.mask(dev(inp.prio), wl.s, wl.w, wl.k)
    _, lse_s = kvpop.attn_fwd(q, k, v, 0.0, ev, lists, (wl.s, wl.w, wl.k))
    tgt = host(kvpop.future_target(q, k, lse_s, wl.w))
    scale = 1 / math.sqrt(wl.D)
    rank, tau, _ = oracle.mask(inp.prio, wl.s, wl.w, wl.k)
    _, lr = oracle.attn(inp.f32("q"), inp.f32("k"), inp.f32("v"), scale, rank, tau, wl.s, wl.w)
    tr = oracle.target_lse(inp.f32("q"), inp.f32("k"), lr, wl.w, scale)
    assert_close_log(tgt.ravel(), tr.ravel(), TOL_T, "target (sparse LSE)")


# ----------------------------------------------------------------------------
# full-size workloads: sampled keys over every position
# ----------------------------------------------------------------------------

def _sample_keys(rng, wl, n_random, block=512):
    """Key positions: 0, 1, s, the first and last of every `block` keys, the last
    keys with a future query (S - w - 1), the first without (S - w) and S - 1,
    plus random ones."""
    S, w = wl.S, wl.w
    fixed = [0, 1, wl.s, S - w - 1, S - w, S - 1]
    edges = [t for b0 in range(0, S, block) for t in (b0, min(S, b0 + block) - 1)]
    ts = np.unique(np.concatenate([fixed, edges, rng.integers(0, S, n_random)]))
    return ts[(ts >= 0) & (ts < S)].astype(np.int64)


def _oracle_head_targets(qh, kh, w, scale, ts, lse_h=None):
    """Eq. (8) for keys ts of one KV head.  qh [1,S,G,D] (that head's query heads),
    kh [1,S,1,D]; the dense causal LSE of all S*G rows from the oracle unless given
    ([1,G,S])."""
    if lse_h is None:
        _, lse_h = oracle.attn(qh, kh, kh, scale, want_o=False)
    keys = np.stack([np.zeros_like(ts), np.zeros_like(ts), ts], axis=1).astype(np.int32)
    return oracle.target_lse(qh, kh, lse_h, w, scale, keys)


@pytest.mark.parametrize("wlname,heads", [
    ("qwen3-4b-layer-prefill", [(0, 0), (0, 5)]),
    ("qwen3-8b-layer-prefill", [(0, 2), (1, 6)]),   # both batch rows
])
def test_full_workload_target_sampled_keys(wlname, heads):
    wl = synth.PREFILL_WORKLOADS[wlname]
    inp = synth.make_prefill(wl)
    scale = 1 / math.sqrt(wl.D)
    q, k = dev_bf16(inp.q), dev_bf16(inp.k)
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = host(kvpop.future_target(q, k, dl, wl.w))
    del q, k, dl
    rng = np.random.default_rng(11)
    G = wl.G
    qf, kf = inp.f32("q"), inp.f32("k")
    for bi, h in heads:
        qh = qf[bi:bi + 1, :, h * G:(h + 1) * G]
        kh = kf[bi:bi + 1, :, h:h + 1]
        ts = _sample_keys(rng, wl, 120)
        assert _chunks_spanned(wl.S, G, wl.w) >= 7
        tr = _oracle_head_targets(np.ascontiguousarray(qh), np.ascontiguousarray(kh), wl.w, scale, ts)
        assert_close_log(tgt[bi, h, ts], tr, TOL_T, f"target b{bi} h{h}")


def _lse_shaped_input(S, Hq, seed):
    """[1, Hq, S] fp32: log(d + 1) + U(0.25, 0.75), drawn from the seeded generator."""
    u = synth.uniform24(seed, 40, Hq * S).reshape(1, Hq, S).astype(np.float64)
    return (np.log1p(np.arange(S, dtype=np.float64))[None, None, :] + 0.25 + 0.5 * u).astype(np.float32)


def test_long_context_target_early_keys():
    """The long-context workload (S = 131072: 64 chunks for the key t = 0)."""
    wl = synth.LONG
    S, G, D = wl.S, wl.G, wl.D
    scale = 1 / math.sqrt(D)
    q, k, _, _ = synth.make_prefill_device(wl, "cuda")
    lse_in = _lse_shaped_input(S, wl.Hq, seed=3)
    tgt = host(kvpop.future_target(q, k, dev(lse_in), wl.w))
    rng = np.random.default_rng(17)
    for h in (1, 6):
        qh = host(q[:, :, h * G:(h + 1) * G].contiguous())
        kh = host(k[:, :, h:h + 1].contiguous())
        ts = _sample_keys(rng, wl, 60, block=4096)
        tr = _oracle_head_targets(qh, kh, wl.w, scale, ts, lse_in[:, h * G:(h + 1) * G].astype(np.float64))
        assert_close_log(tgt[0, h, ts], tr, TOL_T, f"target h{h}")
    del q, k
    torch.cuda.empty_cache()


def test_long_context_target_mass_conservation():
    """w = 0 with the dense LSE at S = 131072: the probabilities of every query row
    sum to 1, so sum_t exp(target_t) = S * G for each KV head."""
    wl = synth.LONG
    q, k, _, _ = synth.make_prefill_device(wl, "cuda")
    _, dl = kvpop.attn_fwd(q, k, None, 0.0, want_o=False)
    tgt = kvpop.future_target(q, k, dl, 0).double()
    tot = host(torch.exp(tgt).sum(dim=-1))
    del q, k, dl, tgt
    torch.cuda.empty_cache()
    assert np.allclose(tot, wl.S * wl.G, rtol=2e-3), tot
