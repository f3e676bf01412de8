// Sparse attention forward on CTA pairs (tcgen05 cta_group::2), head dim 128:
// the retained-set attention of "KVpop ... 精读笔记", sections 2.1 and 2.3, the same
// computation as the single-CTA attn_kernel in attn.cu (which serves D = 64),
// laid out for two SMs.
//
// A cluster of two CTAs on one TPC is persistent and walks work items with a
// stride of the number of clusters.  An item is two 256-row query tiles u of
// one (batch, KV head), rows being (position, query head) pairs; CTA r holds
// the second 128 rows of each tile when r = 1.  Every M = 256 MMA, issued by the
// leader (rank 0), spans both SMs:
//   S_u = Q_u K^T   -- K tile of 128 keys split by keys: CTA r holds keys
//                      [64 r, 64 r + 64) of the tile (all 128 dims);
//   O_u += P_u V    -- P_u from each CTA's tensor memory; V tile split by
//                      columns: CTA r holds dims [64 r, 64 r + 64) of all keys.
// So each SM gathers and stores half of every K and V tile, and the tensor
// cores read half of every B operand from each SM's shared memory; four K/V
// stages fit.  Loads of both CTAs complete on the leader's barriers, MMA
// commits arrive on both CTAs' barriers, and the softmax warps of both CTAs
// hand P and O's columns back to the leader's issuer with remote arrivals.
// Roles per CTA (384 threads): warp 0 key metadata (the whole tile, for the
// masks), warp 1 the MMA issuer (leader), warp 2 query tile 0 and K rows, warp
// 3 query tile 1 and V rows (sinks and long-range keys by TMA gather4, the
// contiguous span by tiled TMA), warps 4-11 softmax (one thread per row).
#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kThreads = 384;
constexpr int kKeys = 128;  // keys per tile (64 per CTA in K)
constexpr int kNS = 4;      // K/V stages
constexpr int kMetaStages = 4;
constexpr int kQBytes = 128 * 128;    // one 64-dim half of a 128-row query tile
constexpr int kKHalf = 64 * 128;      // 64 key rows x 64 dims
constexpr int kVBytes = 128 * 128;    // 128 key rows x 64 dims
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleMax = 256.0f;  // 2^kRescaleLog2
constexpr int kRegsIo = 64;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsNeeded = (128 * kRegsIo + 256 * kRegsSoftmax + kThreads - 1) / kThreads;

struct PairParams {
  CUtensorMap tq;        // Q [b, S, Hq, D]: box 64 x G x P
  CUtensorMap tk64;      // K [b, S, H, D]: box 64 x 1 x 64 (half a tile's keys)
  CUtensorMap tv;        // V [b, S, H, D]: box 64 x 1 x 128
  CUtensorMap tkr, tvr;  // K, V as [b*S*H rows, D], one-row boxes (gather4)
  const int32_t* evict_at;
  const int2* lists;
  __nv_bfloat16* O;
  float* lse;
  int* status;
  int S, Hq, H, G, P, npb, nb, nitems;
  int s, w, kk, nL;
  float scale_log2;
};

struct PBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kNS], k_empty[kNS], v_full[kNS];  // a V stage is freed by a K-stage commit
  uint64_t s_full[2], p_full[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t meta_full[kMetaStages], meta_empty[kMetaStages];
  uint64_t drain;
};

struct PLayout {
  static constexpr int q_off = 0;                                  // [u][dh] 16 KB
  static constexpr int k_off = q_off + 2 * 2 * kQBytes;            // [stage][dh] 8 KB
  static constexpr int v_off = k_off + kNS * 2 * kKHalf;           // [stage] 16 KB
  static constexpr int meta_off = v_off + kNS * kVBytes;
  static constexpr int bar_off = meta_off + kMetaStages * (kKeys + 4) * 8;
  static constexpr int misc_off = bar_off + (int)sizeof(PBars);
  static constexpr int total = misc_off + 64 + 1024;
  static_assert(total <= 232448, "shared memory");
};

// One item: 4P consecutive positions (two 256-row query tiles) of (batch b, KV head h).
struct PItem {
  int b, h, qb0, qb1;
  int NT, NTg, n_sink, n_sl, sp0;
  const int2* list;
};

__device__ __forceinline__ PItem make_pitem(const PairParams& p, int it) {
  PItem x;
  const int nbh = p.H * p.nb;
  const int rank = it / nbh, rem = it - rank * nbh;
  x.h = rem % p.H;
  x.b = rem / p.H;
  const int pblock = p.npb - 1 - rank;  // the short early blocks run last
  x.qb0 = pblock * 4 * p.P;
  x.qb1 = min(x.qb0 + 4 * p.P, p.S) - 1;
  const int jl = x.qb0 / KVPOP_LIST_QBLOCK;
  const int q0l = jl * KVPOP_LIST_QBLOCK;
  x.n_sink = min(p.s, x.qb1 + 1);
  const int n_list = p.kk > 0 ? min(p.kk, max(0, q0l - p.w - p.s + 1)) : 0;
  x.list = p.lists ? p.lists + ((size_t)(x.b * p.H + x.h) * p.nL + jl) * (size_t)p.kk : nullptr;
  x.n_sl = x.n_sink + n_list;
  x.sp0 = max(p.s, q0l - p.w + 1);
  const int n_span = max(0, x.qb1 - x.sp0 + 1);
  x.NTg = (x.n_sl + kKeys - 1) / kKeys;
  x.NT = x.NTg + (n_span + kKeys - 1) / kKeys;
  return x;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_pair_kernel(const __grid_constant__ PairParams p) {
  using L = PLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  PBars* bars = reinterpret_cast<PBars*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off);
  const uint32_t sbase = smem_u32(smem);

  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int S = p.S, G = p.G, P = p.P;
  const int it0 = (int)(blockIdx.x >> 1), dit = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 8);  // 4 softmax warps in each CTA
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 8);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kMetaStages; ++i) {
      mbar_init(&bars->meta_full[i], 1);
      mbar_init(&bars->meta_empty[i], 10);  // 8 softmax warps + 2 loader warps of this CTA
    }
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // the previous kernel of the stream may still be running (programmatic
  // launch): wait for it before any global access; this CTA already holds its
  // tensor memory, so the next kernel may be scheduled
  grid_dep_wait();
  grid_dep_launch();

  auto fail = [&](int site, int detail) {
    report_error(p.status, KVPOP_ERR_TIMEOUT, site, detail);
    *abort_flag = 1;
  };
  auto leader_bar = [&](uint64_t* bar) { return cluster_addr(smem_u32(bar), 0); };
  // this CTA's half of query tile u of item x, once the previous item's last S
  // MMA of that tile has read the buffer; completion counts on the leader
  auto load_q = [&](const PItem& x, int u, int n) -> bool {
    if (!mbar_wait(&bars->q_empty[u], (n & 1) ^ 1, abort_flag)) {
      fail(SITE_ATTN_PRODUCER, 7);
      return false;
    }
    if (leader) mbar_arrive_expect_tx(&bars->q_full[u], 2 * 2 * kQBytes);
    const uint32_t qb = leader_bar(&bars->q_full[u]);
    for (int dh = 0; dh < 2; ++dh)
      tma_load_4d_pair(smem + L::q_off + (u * 2 + dh) * kQBytes, &p.tq, qb, dh * 64, x.h * G,
                       x.qb0 + u * 2 * P + (int)rank * P, x.b);
    return true;
  };

  const uint32_t q_addr = sbase + L::q_off;
  const uint32_t k_addr = sbase + L::k_off;
  const uint32_t v_addr = sbase + L::v_off;

  if (warp < 4) {
    setmaxnreg_dec<kRegsIo>();
    if (warp == 0) {
      // ---------------------------------------------------------- key metadata
      bool ok = true;
      int t = 0;
      for (int it = it0; ok && it < p.nitems; it += dit) {
        const PItem x = make_pitem(p, it);
        const int32_t* ev = p.evict_at + (size_t)(x.b * p.H + x.h) * S;
        auto load_tile = [&](int j, int2 (&e)[4]) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = lane + 32 * c;
            e[c] = make_int2(0x7fffffff, 0);  // padding: never visible
            if (j < x.NTg) {
              const int i = j * kKeys + r;
              if (i < x.n_sink) e[c] = make_int2(i, S);
              else if (i < x.n_sl) e[c] = __ldg(x.list + (i - x.n_sink));
            } else {
              const int pos = x.sp0 + (j - x.NTg) * kKeys + r;
              if (pos <= x.qb1) e[c] = make_int2(pos, __ldg(ev + pos));
            }
          }
        };
        int2 cur_e[4], nxt_e[4];
        load_tile(0, cur_e);
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int ms = t % kMetaStages;
          if (j + 1 < x.NT) load_tile(j + 1, nxt_e);
          if (!warp_wait(&bars->meta_empty[ms], ((t / kMetaStages) & 1) ^ 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 3);
            ok = false;
            break;
          }
          int2* m = meta + ms * (kKeys + 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = lane + 32 * c;
            int2 e = cur_e[c];
            if (e.x != 0x7fffffff && (e.x < 0 || e.x >= S)) {  // a corrupt list entry: never gathered
              report_error(p.status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 10);
              e = make_int2(0x7fffffff, 0);
            }
            m[r] = e;
            int lo = e.x, hi = e.y;  // rows in [lo, hi) see every key of the chunk
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              lo = max(lo, __shfl_xor_sync(0xffffffffu, lo, o));
              hi = min(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            if (lane == 0) m[kKeys + c] = make_int2(lo, hi);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->meta_full[ms]);
#pragma unroll
          for (int c = 0; c < 4; ++c) cur_e[c] = nxt_e[c];
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (leader)
      // TMEM of both CTAs: S/P of tile u at columns 128 u, O of tile u at 256 + 128 u.
      if (lane == 0 && leader && it0 < p.nitems) {
        constexpr uint32_t idesc_qk = idesc_bf16(256, 128, 0);
        constexpr uint32_t idesc_pv = idesc_bf16(256, 128, 1);
        auto issue_s = [&](int u, int st) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int dh = ks >> 2;
            const uint32_t w32 = (uint32_t)(ks & 3) * 32;
            const uint64_t a = smem_desc_sw128(q_addr + (u * 2 + dh) * kQBytes + w32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(k_addr + (st * 2 + dh) * kKHalf + w32, 16, 1024);
            mma_ss_pair(tbase + 128 * u, a, bd, idesc_qk, ks > 0 ? 1u : 0u);
          }
        };
        auto wait_bar = [&](uint64_t* bar, uint32_t ph, int detail) -> bool {
          if (!mbar_wait(bar, ph, abort_flag)) {
            fail(SITE_ATTN_MMA, detail);
            return false;
          }
          tc_fence_after();
          return true;
        };
        PItem x = make_pitem(p, it0);
        int NTn = it0 + dit < p.nitems ? make_pitem(p, it0 + dit).NT : 0;  // next item's tiles, once per item
        bool ok = wait_bar(&bars->k_full[0], 0, 2);
        for (int u = 0; u < 2 && ok; ++u) {
          ok = wait_bar(&bars->q_full[u], 0, 1);
          if (!ok) break;
          issue_s(u, 0);
          mma_commit_pair(&bars->s_full[u]);
          if (x.NT == 1) mma_commit_pair(&bars->q_empty[u]);
          if (u == 1) mma_commit_pair(&bars->k_empty[0]);
        }
        int t = 0, n = 0;
        for (int it = it0; ok;) {
          for (int j = 0; ok && j < x.NT; ++j, ++t) {
            const int st = t % kNS;
            const uint32_t ph = (t / kNS) & 1;
            const bool last = j + 1 == x.NT;
            const bool has_next = !last || it + dit < p.nitems;
            const int NT1 = last ? NTn : x.NT;
            const int j1 = last ? 0 : j + 1;
            const int n1 = last ? n + 1 : n;
            const int st1 = (t + 1) % kNS;
            const uint32_t ph1 = ((t + 1) / kNS) & 1;
            for (int u = 0; u < 2 && ok; ++u) {
              if (!(ok = wait_bar(&bars->p_full[u], t & 1, 3))) break;
              if (u == 0 && !(ok = wait_bar(&bars->v_full[st], ph, 4))) break;
              if (j == 0 && !(ok = wait_bar(&bars->o_empty[u], (n & 1) ^ 1, 6))) break;
#pragma unroll
              for (int ks = 0; ks < kKeys / 16; ++ks) {
                const uint64_t bd = smem_desc_sw128(v_addr + st * kVBytes + ks * 2048, kVBytes, 1024);
                mma_ts_pair(tbase + 256 + 128 * u, tbase + 128 * u + ks * 8, bd, idesc_pv,
                            (j > 0 || ks > 0) ? 1u : 0u);
              }
              if (last) mma_commit_pair(&bars->o_full[u]);
              if (has_next) {
                if (j1 == 0 && !(ok = wait_bar(&bars->q_full[u], n1 & 1, 1))) break;
                if (u == 0 && !(ok = wait_bar(&bars->k_full[st1], ph1, 5))) break;
                issue_s(u, st1);
                mma_commit_pair(&bars->s_full[u]);
                if (j1 == NT1 - 1) mma_commit_pair(&bars->q_empty[u]);
                if (u == 1) mma_commit_pair(&bars->k_empty[st1]);
              }
            }
          }
          if (!ok) break;
          it += dit;
          ++n;
          if (it >= p.nitems) break;
          x = make_pitem(p, it);
          NTn = it + dit < p.nitems ? make_pitem(p, it + dit).NT : 0;
        }
        mma_commit_pair(&bars->drain);
      }
      // both CTAs: every pair MMA is done with this CTA's memory before teardown
      if (lane == 0 && it0 < p.nitems) mbar_wait(&bars->drain, 0, nullptr);
    } else {
      // ---------------------------------------------------------- loaders: warp 2 K, warp 3 V
      const bool is_v = warp == 3;
      uint64_t* full = is_v ? bars->v_full : bars->k_full;
      uint64_t* empty = bars->k_empty;
      const int tile_bytes = 2 * 2 * kKHalf;  // both CTAs: 2 x 8 KB per dim half (K) or 2 x 16 KB (V)
      if (lane == 0 && !is_v) tma_prefetch_desc(&p.tq);
      bool ok = true;
      int t = 0, n = 0;
      for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
        const PItem x = make_pitem(p, it);
        if (lane == 0) ok = load_q(x, is_v ? 1 : 0, n);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int row_base = x.b * S * p.H + x.h;  // row of position t is row_base + t * H
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int st = t % kNS;
          const uint32_t ph = (t / kNS) & 1;
          const int ms = t % kMetaStages;
          if (!warp_wait(&bars->meta_full[ms], (t / kMetaStages) & 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 6);
            ok = false;
            break;
          }
          bool free_ok = true;
          if (!is_v) {
            free_ok = warp_wait(&empty[st], ph ^ 1, abort_flag);
          } else if (t >= kNS) {
            // V stage of tile t - kNS: its PVs ran before tile t - kNS + 1's S, whose
            // K-stage commit therefore frees it too
            const int tn = t - kNS + 1;
            free_ok = warp_wait(&bars->k_empty[tn % kNS], (tn / kNS) & 1, abort_flag);
          }
          if (!free_ok) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 4);
            ok = false;
            break;
          }
          if (lane == 0 && leader) mbar_arrive_expect_tx(&full[st], tile_bytes);
          const uint32_t fb = leader_bar(&full[st]);
          __syncwarp();
          if (j < x.NTg) {
            const int2* km = meta + ms * (kKeys + 4);
            if (!is_v) {
              // K: this CTA's 64 keys (entries 64 r ..), all 128 dims; lanes 0-15
              if (lane < 16) {
                int rows[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const int pos = km[64 * (int)rank + 4 * lane + q4].x;
                  rows[q4] = pos != 0x7fffffff ? row_base + pos * p.H : row_base;  // padding: masked
                }
#pragma unroll
                for (int dh = 0; dh < 2; ++dh)
                  tma_gather4_pair(smem + L::k_off + (st * 2 + dh) * kKHalf + lane * 512, &p.tkr, fb, dh * 64,
                                   rows[0], rows[1], rows[2], rows[3]);
              }
            } else {
              // V: all 128 keys, this CTA's 64 dims; lanes 0-31
              int rows[4];
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const int pos = km[4 * lane + q4].x;
                rows[q4] = pos != 0x7fffffff ? row_base + pos * p.H : row_base;
              }
              tma_gather4_pair(smem + L::v_off + st * kVBytes + lane * 512, &p.tvr, fb, 64 * (int)rank, rows[0],
                               rows[1], rows[2], rows[3]);
            }
          } else if (lane == 0) {
            const int span_row = x.sp0 + (j - x.NTg) * kKeys;
            if (!is_v) {
              for (int dh = 0; dh < 2; ++dh)
                tma_load_4d_pair(smem + L::k_off + (st * 2 + dh) * kKHalf, &p.tk64, fb, dh * 64, x.h,
                                 span_row + 64 * (int)rank, x.b);
            } else {
              tma_load_4d_pair(smem + L::v_off + st * kVBytes, &p.tv, fb, 64 * (int)rank, x.h, span_row, x.b);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->meta_empty[ms]);
        }
      }
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int u = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int p_row = row / G, g = row - p_row * G;
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = 128 * u, o_col = 256 + 128 * u;
    const uint32_t p_bar = leader_bar(&bars->p_full[u]);
    const uint32_t oe_bar = leader_bar(&bars->o_empty[u]);
    const float sl2 = p.scale_log2;
    const uint64_t s2 = pack2(sl2, sl2);
    bool ok = true;
    int t = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
      const PItem x = make_pitem(p, it);
      const int q_first = x.qb0 + u * 2 * P + (int)rank * P;
      const int q = q_first + p_row;
      const int jh = x.h * G + g;
      float m_ref = neg_inf(), l = 0.0f;
      for (int j = 0; j < x.NT; ++j, ++t) {
        if (!warp_wait(&bars->s_full[u], t & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 1);
          ok = false;
          break;
        }
        tc_fence_after();
        const int ms = t % kMetaStages;
        const int2* km = meta + ms * (kKeys + 4);
        if (!warp_wait(&bars->meta_full[ms], (t / kMetaStages) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 2);
          ok = false;
          break;
        }
        // the whole S row of this thread (128 fp32) in registers; invisible keys -> -inf
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(tl + s_col + ch * 32, sr[ch]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_wait_ld_dep(sr[ch]);
        if (G == 4) {
          // the layers this kernel is tuned for: a warp's 32 rows hold 8 positions
          // (4 heads each); lane l tests key 32 ch + l against each of them, one
          // ballot per position, and keeps the word of its own position, whose bit c
          // says whether key 32 ch + c is visible (a bit test per element instead
          // of a metadata load and two compares)
          const int qw = q_first + quarter * 8;  // this warp's first position
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int2 sum = km[kKeys + ch];
            if (__any_sync(0xffffffffu, !(q >= sum.x && q < sum.y))) {
              const int2 e = km[ch * 32 + lane];
              uint32_t mw = 0;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int qi = qw + i;
                const uint32_t w = __ballot_sync(0xffffffffu, e.x <= qi && qi < e.y);
                mw = (lane >> 2) == i ? w : mw;
              }
              if (mw != 0xffffffffu) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                  if (!(mw & (1u << c))) sr[ch][c] = 0xff800000u;
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int2 sum = km[kKeys + ch];
            if (!(q >= sum.x && q < sum.y)) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int2 e = km[ch * 32 + c];
                if (!(e.x <= q && q < e.y)) sr[ch][c] = 0xff800000u;
              }
            }
          }
        }
        // P = exp2(s * scale_log2 - m) as bf16, written over S; returns the row's sum
        auto exps = [&](float nm) -> float {
          const uint64_t n2 = pack2(nm, nm);
          uint64_t lacc[4] = {0, 0, 0, 0};
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const uint64_t xx =
                  fma2(pack2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), s2, n2);
              float e0, e1;
              unpack2(xx, e0, e1);
              const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
              lacc[(c >> 1) & 3] = add2(lacc[(c >> 1) & 3], pack2(p0, p1));
              pk[c >> 1] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tl + s_col + ch * 16, pk);
          }
          float l0, l1;
          unpack2(add2(add2(lacc[0], lacc[1]), add2(lacc[2], lacc[3])), l0, l1);
          return l0 + l1;
        };
        // The running reference m_ref moves only when a row's maximum exceeds it by
        // more than 2^kRescaleLog2 in probability.  Once every row of the warp has a
        // reference, the exponentials are taken against it straight away: if no
        // row's sum exceeds 2^kRescaleLog2, no single term can, and the maximum is
        // never formed.  Otherwise (and on an item's first tile) the exact path runs.
        float ts = 0.0f;
        bool fast = false;
        if (j > 0 && __all_sync(0xffffffffu, m_ref != neg_inf())) {
          ts = exps(-m_ref * sl2);
          fast = __all_sync(0xffffffffu, ts <= kRescaleMax);
        }
        if (!fast) {
          tmem_wait_st();
          float mt = neg_inf();
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) mt = fmaxf(mt, max32(sr[ch]));
          const float m_new = fmaxf(m_ref, mt);
          const bool need = (m_new - m_ref) * sl2 > kRescaleLog2;  // true when m_ref == -inf and mt finite
          float alpha = 1.0f;
          if (need) {
            alpha = ex2_approx((m_ref - m_new) * sl2);
            l *= alpha;
            m_ref = m_new;
          }
          if (__any_sync(0xffffffffu, need) && j > 0) {
            // O of tile j-1 is complete: s_full for tile j was committed after it
#pragma unroll
            for (int cd = 0; cd < 4; ++cd) {
              uint32_t r[32];
              tmem_ld32(tl + o_col + cd * 32, r);
              tmem_wait_ld_dep(r);
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
              tmem_st32(tl + o_col + cd * 32, r);
            }
            tmem_wait_st();
          }
          ts = exps((m_ref == neg_inf()) ? 0.0f : -m_ref * sl2);
        }
        l += ts;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(p_bar);
          mbar_arrive(&bars->meta_empty[ms]);
        }
      }
      if (!ok) break;
      // epilogue: O / l and the LSE; O's TMEM columns are released as soon as read
      if (!warp_wait(&bars->o_full[u], n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_EPILOGUE, 1);
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      __nv_bfloat16* orow = p.O + (((size_t)x.b * S + q) * p.Hq + jh) * 128;
      // all 128 columns in flight at once; O's TMEM goes back before the conversion
      uint32_t orr[4][32];
#pragma unroll
      for (int cd = 0; cd < 4; ++cd) tmem_ld32(tl + o_col + cd * 32, orr[cd]);
#pragma unroll
      for (int cd = 0; cd < 4; ++cd) tmem_wait_ld_dep(orr[cd]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(oe_bar);
      uint32_t pk[64];
#pragma unroll
      for (int cd = 0; cd < 4; ++cd)
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          pk[cd * 16 + (c >> 1)] =
              pack_bf16x2(__uint_as_float(orr[cd][c]) * inv, __uint_as_float(orr[cd][c + 1]) * inv);
      if (q <= x.qb1) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int v4 = 0; v4 < 16; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        p.lse[((size_t)x.b * p.Hq + jh) * S + q] =
            l > 0.0f ? (m_ref * sl2 + __log2f(l)) * 0.69314718055994531f : neg_inf();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // neither CTA releases its tensor or shared memory while the pair still works
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}

}  // namespace

// Called by kvpop_attn_fwd for sparse mode with D = 128 (arguments validated).
kvpop_status launch_sparse_pair(const void* q, const void* k, const void* v, int b, int S, int Hq, int H,
                                float scale_log2, const int32_t* evict_at, const int32_t* lists,
                                kvpop_budget bud, void* O, float* lse, cudaStream_t cs) {
  PairParams prm;
  memset(&prm, 0, sizeof(prm));
  const int G = Hq / H, P = 128 / G, D = 128;
  {
    uint64_t dq[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)S, (uint64_t)b};
    uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)S * Hq * D * 2};
    uint32_t bq[4] = {64, (uint32_t)G, (uint32_t)P, 1};
    uint64_t dk[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)b};
    uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
    uint32_t bk64[4] = {64, 1, 64, 1};
    uint32_t bv[4] = {64, 1, 128, 1};
    if (!make_tmap_4d(&prm.tq, q, dq, sq, bq) || !make_tmap_4d(&prm.tk64, k, dk, sk, bk64) ||
        !make_tmap_4d(&prm.tv, v, dk, sk, bv) ||
        !make_tmap_rows(&prm.tkr, k, (uint64_t)D, (uint64_t)b * S * H, 64) ||
        !make_tmap_rows(&prm.tvr, v, (uint64_t)D, (uint64_t)b * S * H, 64))
      return KVPOP_ERR_CUDA;
  }
  prm.evict_at = evict_at;
  prm.lists = reinterpret_cast<const int2*>(lists);
  prm.O = static_cast<__nv_bfloat16*>(O);
  prm.lse = lse;
  prm.status = device_status_ptr();
  prm.S = S;
  prm.Hq = Hq;
  prm.H = H;
  prm.G = G;
  prm.P = P;
  prm.npb = (S + 4 * P - 1) / (4 * P);
  if ((long long)prm.npb * H * b > (1LL << 30)) {
    set_last_error("kvpop_attn_fwd: too many query blocks");
    return KVPOP_ERR_UNSUPPORTED;
  }
  prm.nb = b;
  prm.nitems = prm.npb * H * b;
  prm.s = bud.s;
  prm.w = bud.w;
  prm.kk = bud.k;
  prm.nL = (S + KVPOP_LIST_QBLOCK - 1) / KVPOP_LIST_QBLOCK;
  prm.scale_log2 = scale_log2;
  auto kern = attn_pair_kernel;
  kvpop_status st = cuda_check(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PLayout::total),
      "kvpop_attn_fwd: smem attribute");
  if (st != KVPOP_OK) return st;
  cudaFuncAttributes fa;
  st = cuda_check(cudaFuncGetAttributes(&fa, kern), "kvpop_attn_fwd: attributes");
  if (st != KVPOP_OK) return st;
  if (((fa.numRegs + 7) / 8) * 8 < kRegsNeeded) {
    set_last_error("kvpop_attn_fwd: kernel built with %d registers per thread, %d needed", fa.numRegs, kRegsNeeded);
    return KVPOP_ERR_INTERNAL;
  }
  // persistent: one cluster per TPC walks the items with a stride of the cluster count
  const int clusters = min(prm.nitems, max(1, num_sms() / 2));
  return cuda_check(launch_pdl(kern, dim3(2 * clusters), dim3(kThreads), PLayout::total, cs, prm),
                    "kvpop_attn_fwd: launch");
}

}  // namespace kvpop
