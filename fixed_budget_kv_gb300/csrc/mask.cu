// kvpop_mask: rank, running top-k threshold, eviction rows and long-range
// lists for the fixed-budget retained set.
//
// Definitions ("KVpop ... 精读笔记", sections 2.2-2.3; "KVpop — 基于预测性在线剪枝
// 的键值缓存压缩", section 2.4): E(q) = {t : s <= t <= q - w}; tau_q is the rank of
// the k-th best token of E(q) under static priorities; row q retains sinks, the
// protected window and the eligible tokens with rank <= tau_q.
//
// GPU scheme (bit-exact with a sequential Fenwick-tree sweep):
//   1. rank: segmented LSD radix sort (4 x 8-bit digits) of an order-preserving
//      32-bit key, stable in the token index.
//   2. tau: tau_q is the k-th smallest value of rank[s .. q-w], a prefix
//      order statistic.  A wavelet matrix over rank (one stable bit-partition
//      per level, built by a thread-block cluster in distributed shared memory)
//      answers every q independently in log2(S) steps.
//   3. evict_at: tau is non-increasing in q, so the first row that drops t is a
//      binary search for the first q >= t + w with tau_q < rank[t].
//   4. lists: the long-range keys retained at rows 64 i as (position,
//      evict_at) pairs -- those held through the whole 64-row block first --
//      from group base lists (every 16 lists) plus the tokens that became
//      eligible since.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace kvpop {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortItems = 4;
constexpr int kSortTile = kSortThreads * kSortItems;  // 1024
constexpr int kListGroup = 16;                         // lists per group base
constexpr int kWmThreads = 1024;
constexpr int kMaxClusterCtas = 8;
constexpr int kMaxS = 131072;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Order-preserving key: ascending key = (priority descending); NaN == -inf; -0 == +0.
__device__ __forceinline__ uint32_t prio_key(float p) {
  uint32_t b = __float_as_uint(p);
  if (p != p) b = 0xFF800000u;           // NaN -> -inf
  if (b == 0x80000000u) b = 0u;          // -0 -> +0
  uint32_t asc = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ~asc;
}

// ---------------------------------------------------------------------------
// 1. radix sort
// ---------------------------------------------------------------------------

template <bool FIRST>
__global__ void __launch_bounds__(kSortThreads)
    radix_upsweep(const float* __restrict__ prio, const uint32_t* __restrict__ keys, int S,
                  int shift, int nblk, uint32_t* __restrict__ hist) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  __shared__ uint32_t h[256];
  const int seg = blockIdx.y, blk = blockIdx.x, tid = threadIdx.x;
  h[tid] = 0;
  __syncthreads();
  const size_t segoff = (size_t)seg * S;
#pragma unroll
  for (int i = 0; i < kSortItems; ++i) {
    int e = blk * kSortTile + i * kSortThreads + tid;
    if (e < S) {
      uint32_t key = FIRST ? prio_key(prio[segoff + e]) : keys[segoff + e];
      atomicAdd(&h[(key >> shift) & 255u], 1u);
    }
  }
  __syncthreads();
  hist[((size_t)seg * 256 + tid) * nblk + blk] = h[tid];
}

// Exclusive scan of hist[seg][digit][blk] in (digit, blk) order.
__global__ void __launch_bounds__(1024) radix_scan(uint32_t* __restrict__ hist, int nblk) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  __shared__ uint32_t wsum[32];
  const int seg = blockIdx.x, tid = threadIdx.x;
  const int n = 256 * nblk;
  const int per = (n + 1023) / 1024;
  uint32_t* h = hist + (size_t)seg * n;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) {
    int idx = tid * per + i;
    if (idx < n) local += h[idx];
  }
  // block exclusive scan of `local`
  uint32_t x = local;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if ((tid & 31) >= o) x += y;
  }
  if ((tid & 31) == 31) wsum[tid >> 5] = x;
  __syncthreads();
  if (tid < 32) {
    uint32_t v = wsum[tid];
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (tid >= o) v += y;
    }
    wsum[tid] = v;
  }
  __syncthreads();
  uint32_t run = x - local + ((tid >> 5) ? wsum[(tid >> 5) - 1] : 0u);
  for (int i = 0; i < per; ++i) {
    int idx = tid * per + i;
    if (idx < n) {
      uint32_t v = h[idx];
      h[idx] = run;
      run += v;
    }
  }
}

template <bool FIRST, bool LAST>
__global__ void __launch_bounds__(kSortThreads)
    radix_downsweep(const float* __restrict__ prio, const uint32_t* __restrict__ keys_in,
                    const int32_t* __restrict__ idx_in, int S, int shift, int nblk,
                    const uint32_t* __restrict__ hist, uint32_t* __restrict__ keys_out,
                    int32_t* __restrict__ idx_out, int32_t* __restrict__ rank_out, int* status) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  constexpr int W = kSortThreads / 32;
  __shared__ uint32_t wcnt[W][256];
  __shared__ uint32_t wpre[W][256];
  __shared__ uint32_t run[256];
  __shared__ uint32_t base[256];
  __shared__ uint32_t gofs[256];
  const int seg = blockIdx.y, blk = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const size_t segoff = (size_t)seg * S;
  for (int w = 0; w < W; ++w) wcnt[w][tid] = 0;
  run[tid] = 0;
  gofs[tid] = hist[((size_t)seg * 256 + tid) * nblk + blk];
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i = 0; i < kSortItems; ++i) {
    int e = blk * kSortTile + i * kSortThreads + tid;
    bool valid = e < S;
    uint32_t key = 0;
    int32_t idx = 0;
    if (valid) {
      if (FIRST) {
        key = prio_key(prio[segoff + e]);
        idx = e;
      } else {
        key = keys_in[segoff + e];
        idx = idx_in[segoff + e];
      }
    }
    uint32_t digit = valid ? ((key >> shift) & 255u) : 256u;
    uint32_t peers = __match_any_sync(0xffffffffu, digit);
    uint32_t lrank = __popc(peers & lt_mask);
    bool leader = (peers & lt_mask) == 0;
    if (valid && leader) wcnt[warp][digit] = __popc(peers);
    __syncthreads();
    {
      uint32_t acc = 0;
      for (int w = 0; w < W; ++w) {
        wpre[w][tid] = acc;
        acc += wcnt[w][tid];
        wcnt[w][tid] = 0;
      }
      base[tid] = run[tid];
      run[tid] += acc;
    }
    __syncthreads();
    if (valid) {
      uint32_t dst = gofs[digit] + base[digit] + wpre[warp][digit] + lrank;
      if (dst >= (uint32_t)S || idx < 0 || idx >= S) {
        report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 3);
      } else if (LAST) {
        rank_out[segoff + idx] = (int32_t)dst;
      } else {
        keys_out[segoff + dst] = key;
        idx_out[segoff + dst] = idx;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// 2. wavelet matrix (cluster build) and tau queries
// ---------------------------------------------------------------------------

// wm[seg][level][word] = (bits, ones before this word); zeros[seg][level].
__global__ void __launch_bounds__(kWmThreads)
    wavelet_build(const int32_t* __restrict__ rank, int S, int L, int slice, int nwords,
                  uint2* __restrict__ wm, int32_t* __restrict__ zeros, int* status) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  cg::cluster_group cluster = cg::this_cluster();
  const int csize = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  const int seg = blockIdx.x / csize;
  const int tid = threadIdx.x;
  extern __shared__ __align__(16) int32_t wsm[];
  int32_t* buf0 = wsm;
  int32_t* buf1 = wsm + slice;
  __shared__ int32_t cta_zeros, cta_ones;
  __shared__ int32_t wsum[32];

  const int base = crank * slice;
  const size_t segoff = (size_t)seg * S;
  for (int i = tid; i < slice; i += kWmThreads) buf0[i] = (base + i < S) ? rank[segoff + base + i] : 0;
  cluster.sync();

  const int per = slice / kWmThreads;  // 1..16 consecutive elements per thread
  int32_t* cur = buf0;
  int32_t* nxt = buf1;
  for (int lvl = 0; lvl < L; ++lvl) {
    const int bit = L - 1 - lvl;
    // bits and counts of this thread's run
    uint32_t mybits = 0;
    int ones = 0, nvalid = 0;
    for (int i = 0; i < per; ++i) {
      int li = tid * per + i;
      if (base + li < S) {
        uint32_t b = ((uint32_t)cur[li] >> bit) & 1u;
        mybits |= b << i;
        ones += (int)b;
        nvalid += 1;
      }
    }
    // block exclusive scan of ones and valid counts (packed 16|16 would overflow; use two scans)
    int xo = ones, xv = nvalid;
    for (int o = 1; o < 32; o <<= 1) {
      int yo = __shfl_up_sync(0xffffffffu, xo, o);
      int yv = __shfl_up_sync(0xffffffffu, xv, o);
      if ((tid & 31) >= o) {
        xo += yo;
        xv += yv;
      }
    }
    // pack warp totals: ones in low 16 bits is unsafe for large slices, so keep two arrays
    __shared__ int32_t wsum_v[32];
    if ((tid & 31) == 31) {
      wsum[tid >> 5] = xo;
      wsum_v[tid >> 5] = xv;
    }
    __syncthreads();
    if (tid < 32) {
      int vo = wsum[tid], vv = wsum_v[tid];
      for (int o = 1; o < 32; o <<= 1) {
        int yo = __shfl_up_sync(0xffffffffu, vo, o);
        int yv = __shfl_up_sync(0xffffffffu, vv, o);
        if (tid >= o) {
          vo += yo;
          vv += yv;
        }
      }
      wsum[tid] = vo;
      wsum_v[tid] = vv;
    }
    __syncthreads();
    const int ones_before = xo - ones + ((tid >> 5) ? wsum[(tid >> 5) - 1] : 0);
    const int valid_before = xv - nvalid + ((tid >> 5) ? wsum_v[(tid >> 5) - 1] : 0);
    if (tid == kWmThreads - 1) {
      cta_ones = ones_before + ones;
      cta_zeros = (valid_before + nvalid) - (ones_before + ones);
    }
    cluster.sync();
    int Z = 0, zoff = 0, ooff = 0;
    for (int r = 0; r < csize; ++r) {
      int zr = *cluster.map_shared_rank(&cta_zeros, r);
      int orr = *cluster.map_shared_rank(&cta_ones, r);
      Z += zr;
      if (r < crank) {
        zoff += zr;
        ooff += orr;
      }
    }
    // bit-vector words: `per` (1..16, a power of two) bits per thread, 32/per threads per word
    uint2* wml = wm + ((size_t)seg * L + lvl) * nwords;
    {
      const int tpw = 32 / per;
      uint32_t word_bits = mybits << ((tid % tpw) * per);
      for (int o = 1; o < tpw; o <<= 1) word_bits |= __shfl_xor_sync(0xffffffffu, word_bits, o);
      int first_ones = __shfl_sync(0xffffffffu, ones_before, (tid & 31) & ~(tpw - 1));
      if (tid % tpw == 0) {
        int word = (base + tid * per) / 32;
        wml[word] = make_uint2(word_bits, (uint32_t)(ooff + first_ones));
      }
    }
    if (crank == csize - 1 && tid == 0) {
      wml[nwords - 1] = make_uint2(0u, (uint32_t)(S - Z));  // rank1 at position csize*slice
      zeros[(size_t)seg * L + lvl] = Z;
    }
    // stable partition into the cluster's next buffers
    int o_run = ones_before, z_run = valid_before - ones_before;
    for (int i = 0; i < per; ++i) {
      int li = tid * per + i;
      if (base + li >= S) break;
      int32_t val = cur[li];
      int dst;
      if ((mybits >> i) & 1u) {
        dst = Z + ooff + o_run;
        ++o_run;
      } else {
        dst = zoff + z_run;
        ++z_run;
      }
      if (dst < 0 || dst >= S) {
        report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 4);
        continue;
      }
      int32_t* remote = cluster.map_shared_rank(nxt, dst / slice);
      remote[dst % slice] = val;
    }
    cluster.sync();
    int32_t* t = cur;
    cur = nxt;
    nxt = t;
  }
}

__device__ __forceinline__ int wm_rank1(const uint2* lvl, int i) {
  uint2 w = lvl[i >> 5];
  uint32_t m = (1u << (i & 31)) - 1u;
  return (int)w.y + __popc(w.x & m);
}

__global__ void tau_query(const uint2* __restrict__ wm, const int32_t* __restrict__ zeros, int S,
                          int L, int nwords, int s, int w, int k, int nseg,
                          int32_t* __restrict__ tau, int* status) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)nseg * S) return;
  const int seg = (int)(gid / S), q = (int)(gid % S);
  const int x = q - w;
  int32_t out;
  if (k == 0) {
    out = -1;
  } else {
    const int n = x >= s ? x - s + 1 : 0;
    if (n <= k) {
      out = KVPOP_TAU_ALL;
    } else {
      int kk = k - 1, l = s, r = x + 1, val = 0;
      for (int lvl = 0; lvl < L; ++lvl) {
        const uint2* wl = wm + ((size_t)seg * L + lvl) * nwords;
        const int ol = wm_rank1(wl, l), orr = wm_rank1(wl, r);
        const int zc = (r - l) - (orr - ol);
        if (kk < zc) {
          l -= ol;
          r -= orr;
        } else {
          kk -= zc;
          const int Z = zeros[(size_t)seg * L + lvl];
          l = Z + ol;
          r = Z + orr;
          val |= 1 << (L - 1 - lvl);
        }
        if (l < 0 || r < l || r > S) {  // cannot happen for a consistent matrix
          report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 5);
          break;
        }
      }
      out = val;
    }
  }
  tau[gid] = out;
}

// ---------------------------------------------------------------------------
// 3. evict_at
// ---------------------------------------------------------------------------

__global__ void evict_search(const int32_t* __restrict__ rank, const int32_t* __restrict__ tau,
                             int S, int s, int w, int nseg, int32_t* __restrict__ ev) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)nseg * S) return;
  const int seg = (int)(gid / S), t = (int)(gid % S);
  const int32_t* tu = tau + (size_t)seg * S;
  int out = S;
  if (t >= s && (long long)t + w < S) {
    const int r = rank[gid];
    int lo = t + w, hi = S;  // first q in [lo, hi) with tau[q] < r, else S
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (tu[mid] < r) hi = mid;
      else lo = mid + 1;
    }
    out = lo;
  }
  ev[gid] = out;
}

// ---------------------------------------------------------------------------
// 4. long-range lists
// ---------------------------------------------------------------------------

// Ordered compaction of candidates in [0, n) where `cand(i)` gives the
// position: keeps those with lo < evict_at <= hi, calls emit(slot, pos, ev)
// with slots counted from out_start (only below out_cap); returns the end.
// Each thread takes kCompactItems consecutive candidates of a chunk (their
// evict_at loads in flight together); one block-wide exclusive scan of the
// per-thread counts per chunk keeps the order.  All threads of the block call it.
constexpr int kGroupThreads = 1024;  // group bases: long scans (up to S candidates)
constexpr int kListThreads = 256;    // lists: k + 1024 candidates at most, many blocks
constexpr int kCompactItems = 4;

template <int THREADS, typename Cand, typename Emit>
__device__ int compact_alive(Cand cand, int n, int S, const int32_t* __restrict__ ev, int lo, int hi,
                             Emit emit, int out_cap, int out_start) {
  __shared__ int wsum[THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = THREADS / 32;
  int running = out_start;
  for (int c0 = 0; c0 < n; c0 += THREADS * kCompactItems) {
    int pos[kCompactItems], e[kCompactItems];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kCompactItems; ++u) {
      const int i = c0 + tid * kCompactItems + u;
      pos[u] = -1;
      e[u] = 0;
      if (i < n) {
        const int pp = cand(i);
        if (pp >= 0 && pp < S) {
          pos[u] = pp;
          e[u] = ev[pp];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCompactItems; ++u) {
      const bool keep = pos[u] >= 0 && e[u] > lo && e[u] <= hi;
      if (!keep) pos[u] = -1;
      cnt += keep;
    }
    // block exclusive scan of cnt
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll 4
    for (int w2 = 0; w2 < nw; ++w2) {
      const int v = wsum[w2];
      before += w2 < warp ? v : 0;
      total += v;
    }
    int slot = running + before + x - cnt;
#pragma unroll
    for (int u = 0; u < kCompactItems; ++u)
      if (pos[u] >= 0) {
        if (slot < out_cap) emit(slot, pos[u], e[u]);
        ++slot;
      }
    running += total;
    __syncthreads();  // wsum is reused by the next chunk
  }
  return running;
}

__global__ void __launch_bounds__(kGroupThreads)
    lists_group_base(const int32_t* __restrict__ evict_at, int S, int s, int w, int k,
                     int ngroups, int32_t* __restrict__ gbase, int32_t* __restrict__ gcount,
                     int* status) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  const int g = blockIdx.x, seg = blockIdx.y;
  const int q0 = g * kListGroup * KVPOP_LIST_QBLOCK;
  const int x0 = q0 - w;
  const int32_t* ev = evict_at + (size_t)seg * S;
  const int n = x0 >= s ? x0 - s + 1 : 0;
  int32_t* out = gbase + ((size_t)seg * ngroups + g) * k;
  int cnt = compact_alive<kGroupThreads>([=](int i) { return s + i; }, n, S, ev, q0, 0x7fffffff,
                          [=](int slot, int pos, int) { out[slot] = pos; }, k, 0);
  if (threadIdx.x == 0) {
    gcount[(size_t)seg * ngroups + g] = cnt;
    if (cnt > k) report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 1);
  }
}

// List j: keys of E(64 j) held at row 64 j as (position, evict_at) pairs --
// first those held through row 64 j + 63, then those dropped inside the block,
// each group in increasing position.
__global__ void __launch_bounds__(kListThreads)
    lists_build(const int32_t* __restrict__ evict_at, int S, int s, int w, int k, int nL,
                int ngroups, const int32_t* __restrict__ gbase, const int32_t* __restrict__ gcount,
                int2* __restrict__ lists, int* status) {
  grid_dep_wait();  // inputs of earlier kernels of the stream are complete
  grid_dep_launch();
  const int j = blockIdx.x, seg = blockIdx.y;
  const int g = j / kListGroup;
  const int q0 = j * KVPOP_LIST_QBLOCK, x0 = q0 - w;
  const int q1 = q0 + KVPOP_LIST_QBLOCK - 1;
  const int qg = g * kListGroup * KVPOP_LIST_QBLOCK, xg = qg - w;
  const int32_t* ev = evict_at + (size_t)seg * S;
  const int32_t* gb = gbase + ((size_t)seg * ngroups + g) * k;
  const int nb = gcount[(size_t)seg * ngroups + g];
  const int r0 = max(s, xg + 1);
  const int nr = x0 >= r0 ? x0 - r0 + 1 : 0;
  int2* out = lists + ((size_t)seg * nL + j) * k;
  auto cand = [=](int i) { return i < nb ? gb[i] : r0 + (i - nb); };
  auto emit = [=](int slot, int pos, int e) { out[slot] = make_int2(pos, e); };
  const int na = compact_alive<kListThreads>(cand, nb + nr, S, ev, q1, 0x7fffffff, emit, k, 0);
  const int cnt = compact_alive<kListThreads>(cand, nb + nr, S, ev, q0, q1, emit, k, na);
  if (threadIdx.x == 0) {
    const int expect = min(k, x0 >= s ? x0 - s + 1 : 0);
    if (cnt != expect) report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 2);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct MaskPlan {
  int nseg, S, nblk, L, csize, slice, nwords, nL, ngroups;
  size_t off_keys0, off_keys1, off_idx0, off_idx1, off_hist, off_wm, off_zeros, off_gbase,
      off_gcount, total;
};

kvpop_status plan_mask(int b, int H, int S, kvpop_budget bud, MaskPlan* p) {
  if (b <= 0 || H <= 0 || S <= 0) {
    set_last_error("kvpop_mask: b, H, S must be positive (b=%d H=%d S=%d)", b, H, S);
    return KVPOP_ERR_INVALID_ARG;
  }
  if (bud.s < 0 || bud.w < 0 || bud.k < 0 || (long long)bud.s + bud.w + bud.k < 1 ||
      (long long)bud.s + bud.w + bud.k > 0x7fffffff) {
    set_last_error("kvpop_mask: invalid budget s=%d w=%d k=%d", bud.s, bud.w, bud.k);
    return KVPOP_ERR_INVALID_ARG;
  }
  if (S > kMaxS) {
    set_last_error("kvpop_mask: S=%d exceeds the supported maximum %d", S, kMaxS);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if ((long long)b * H > 65535) {
    set_last_error("kvpop_mask: b*H=%lld exceeds 65535", (long long)b * H);
    return KVPOP_ERR_UNSUPPORTED;
  }
  p->nseg = b * H;
  p->S = S;
  p->nblk = (S + kSortTile - 1) / kSortTile;
  int L = 1;
  while ((1 << L) < S) ++L;
  p->L = L;
  // slice: elements per CTA, 1024 * (1, 2, 4, 8 or 16); up to 8 CTAs per cluster
  int slice = 1024;
  while (slice * kMaxClusterCtas < S) slice *= 2;
  p->slice = slice;
  p->csize = (S + slice - 1) / slice;
  p->nwords = p->csize * slice / 32 + 1;
  p->nL = (S + KVPOP_LIST_QBLOCK - 1) / KVPOP_LIST_QBLOCK;
  p->ngroups = (p->nL + kListGroup - 1) / kListGroup;
  size_t n = (size_t)p->nseg * S;
  size_t off = 0;
  p->off_keys0 = off; off = align256(off + n * 4);
  p->off_keys1 = off; off = align256(off + n * 4);
  p->off_idx0 = off; off = align256(off + n * 4);
  p->off_idx1 = off; off = align256(off + n * 4);
  p->off_hist = off; off = align256(off + (size_t)p->nseg * 256 * p->nblk * 4);
  p->off_wm = off; off = align256(off + (size_t)p->nseg * L * p->nwords * 8);
  p->off_zeros = off; off = align256(off + (size_t)p->nseg * L * 4);
  p->off_gbase = off; off = align256(off + (size_t)p->nseg * p->ngroups * (size_t)bud.k * 4);
  p->off_gcount = off; off = align256(off + (size_t)p->nseg * p->ngroups * 4);
  p->total = off;
  return KVPOP_OK;
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_mask_workspace_size(int b, int H, int S, kvpop_budget bud,
                                                  size_t* bytes) {
  if (!bytes) {
    set_last_error("kvpop_mask_workspace_size: bytes is NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  MaskPlan p;
  kvpop_status st = plan_mask(b, H, S, bud, &p);
  if (st != KVPOP_OK) return st;
  *bytes = p.total;
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_mask_lists_size(int b, int H, int S, kvpop_budget bud,
                                              size_t* bytes) {
  if (!bytes) {
    set_last_error("kvpop_mask_lists_size: bytes is NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  MaskPlan p;
  kvpop_status st = plan_mask(b, H, S, bud, &p);
  if (st != KVPOP_OK) return st;
  *bytes = (size_t)p.nseg * p.nL * (size_t)bud.k * 8;
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_mask(const float* prio, int b, int H, int S, kvpop_budget bud,
                                   int32_t* rank, int32_t* tau, int32_t* evict_at, int32_t* lists,
                                   void* workspace, size_t ws_bytes, kvpop_stream stream) {
  MaskPlan p;
  kvpop_status st = plan_mask(b, H, S, bud, &p);
  if (st != KVPOP_OK) return st;
  if (!prio || !rank || !tau || !evict_at || !workspace) {
    set_last_error("kvpop_mask: prio, rank, tau, evict_at and workspace must be non-NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (ws_bytes < p.total) {
    set_last_error("kvpop_mask: workspace has %zu bytes, needs %zu", ws_bytes, p.total);
    return KVPOP_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) {
    set_last_error("kvpop_mask: workspace must be 256-byte aligned");
    return KVPOP_ERR_INVALID_ARG;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(ws + p.off_keys0),
                       reinterpret_cast<uint32_t*>(ws + p.off_keys1)};
  int32_t* idx[2] = {reinterpret_cast<int32_t*>(ws + p.off_idx0),
                     reinterpret_cast<int32_t*>(ws + p.off_idx1)};
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + p.off_hist);
  uint2* wm = reinterpret_cast<uint2*>(ws + p.off_wm);
  int32_t* zeros = reinterpret_cast<int32_t*>(ws + p.off_zeros);
  int32_t* gbase = reinterpret_cast<int32_t*>(ws + p.off_gbase);
  int32_t* gcount = reinterpret_cast<int32_t*>(ws + p.off_gcount);
  int* status = device_status_ptr();

  // 1. rank
  dim3 sgrid(p.nblk, p.nseg);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    const uint32_t* kin = keys[(pass + 1) & 1];
    const int32_t* iin = idx[(pass + 1) & 1];
    uint32_t* kout = keys[pass & 1];
    int32_t* iout = idx[pass & 1];
    if (pass == 0)
      launch_pdl(radix_upsweep<true>, sgrid, dim3(kSortThreads), 0, cs, prio, nullptr, S, shift, p.nblk, hist);
    else
      launch_pdl(radix_upsweep<false>, sgrid, dim3(kSortThreads), 0, cs, nullptr, kin, S, shift, p.nblk, hist);
    launch_pdl(radix_scan, dim3(p.nseg), dim3(1024), 0, cs, hist, p.nblk);
    if (pass == 0)
      launch_pdl(radix_downsweep<true, false>, sgrid, dim3(kSortThreads), 0, cs, prio, nullptr, nullptr, S, shift,
                 p.nblk, hist, kout, iout, nullptr, status);
    else if (pass < 3)
      launch_pdl(radix_downsweep<false, false>, sgrid, dim3(kSortThreads), 0, cs, nullptr, kin, iin, S, shift,
                 p.nblk, hist, kout, iout, nullptr, status);
    else
      launch_pdl(radix_downsweep<false, true>, sgrid, dim3(kSortThreads), 0, cs, nullptr, kin, iin, S, shift,
                 p.nblk, hist, nullptr, nullptr, rank, status);
  }
  st = cuda_check(cudaGetLastError(), "kvpop_mask: rank kernels");
  if (st != KVPOP_OK) return st;

  // 2. wavelet matrix + tau
  {
    const size_t smem = (size_t)2 * p.slice * sizeof(int32_t);
    st = cuda_check(cudaFuncSetAttribute(wavelet_build, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem),
                    "kvpop_mask: wavelet smem attribute");
    if (st != KVPOP_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nseg * p.csize);
    cfg.blockDim = dim3(kWmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = cs;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    st = cuda_check(cudaLaunchKernelEx(&cfg, wavelet_build, (const int32_t*)rank, S, p.L, p.slice,
                                       p.nwords, wm, zeros, status),
                    "kvpop_mask: wavelet build");
    if (st != KVPOP_OK) return st;
  }
  const long long total = (long long)p.nseg * S;
  const int tb = 256;
  const unsigned nb = (unsigned)((total + tb - 1) / tb);
  launch_pdl(tau_query, dim3(nb), dim3(tb), 0, cs, wm, zeros, S, p.L, p.nwords, bud.s, bud.w, bud.k, p.nseg, tau,
             status);
  // 3. evict_at
  launch_pdl(evict_search, dim3(nb), dim3(tb), 0, cs, rank, tau, S, bud.s, bud.w, p.nseg, evict_at);
  // 4. lists
  if (lists != nullptr && bud.k > 0) {
    launch_pdl(lists_group_base, dim3(p.ngroups, p.nseg), dim3(kGroupThreads), 0, cs, evict_at, S, bud.s, bud.w,
               bud.k, p.ngroups, gbase, gcount, status);
    launch_pdl(lists_build, dim3(p.nL, p.nseg), dim3(kListThreads), 0, cs, evict_at, S, bud.s, bud.w, bud.k, p.nL,
               p.ngroups, gbase, gcount, reinterpret_cast<int2*>(lists), status);
  }
  return cuda_check(cudaGetLastError(), "kvpop_mask: launch");
}
