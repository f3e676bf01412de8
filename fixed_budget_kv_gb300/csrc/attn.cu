// kvpop_attn_fwd: causal GQA attention over the fixed-budget retained set
// (sparse) or over all past tokens (dense), returning O and the log-sum-exp
// ("KVpop ... 精读笔记", sections 2.1 and 2.3).  This file holds the entry point,
// the sparse kernel for D = 64 and the dense kernel with O; the sparse kernel
// for D = 128 (CTA pairs) is in attn_pair.cu and the dense LSE-only teacher pass
// in dense_lse.cu.
//
// Persistent: one CTA per SM walks the work items with a stride of the grid
// size.  An item is two 128-row query tiles of one (batch, KV head); a row is
// one (position, query head) pair: the G query heads of a KV head share every
// K/V tile, so a tile covers 128/G positions.  The K/V and metadata rings run
// on across items, the next item's query tiles load while the current item's
// last tiles are in flight, and its first S tiles are issued before the
// current item's epilogue, so no SM idles between items.  Warp roles (384
// threads):
//   warp 0      dense mode: TMA producer of Q, K and V; sparse mode: the key
//               metadata of each KV tile: (position, eviction row) per key
//               and, per 32-key chunk, the latest position and the earliest
//               eviction row, so that rows inside that range skip masking
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issuer
//   warps 2-3   sparse mode: query tile 0 / 1 of each item, and K (warp 2)
//               and V (warp 3) rows of sinks and long-range keys gathered by
//               TMA (tile::gather4, four rows per instruction) into the
//               128B-swizzled operand layout; the contiguous span (window and
//               recent tokens) by TMA tiles
//   warps 4-7   softmax for query tile 0 (one thread per row / TMEM lane)
//   warps 8-11  softmax for query tile 1
// S = Q K^T lands in TMEM (fp32); the softmax warps turn it into bf16 P in
// place and the MMA warp accumulates O += P V with A read from TMEM.  The two
// query tiles ping-pong so that the tensor core works on one tile while the
// softmax warps work on the other.  Running-max updates are lazy: O and the
// row sum are rescaled only when the max grows by more than 2^8.
//
// Sparse key plan of a CTA covering rows [qb0, qb1] with list i = qb0 / 64
// (taken at row q0 = 64 i <= qb0):
//   [0, s)                          sinks
//   list i                          long-range keys held at row q0
//   [max(s, q0 - w + 1), qb1]       every later token (window + new entries)
// and row q keeps key t exactly when t <= q < evict_at[t].
#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kThreads = 384;
constexpr int kKeys = 128;
constexpr int kMetaStages = 4;
constexpr int kBlockBytes = 128 * 128;  // 128 rows x 128 bytes
constexpr float kRescaleLog2 = 8.0f;
// Register split: warpgroup 0 (producer, MMA, loaders) drops to kRegsIo, the two
// softmax warpgroups (one S row of 128 fp32 per thread) rise to kRegsSoftmax.
constexpr int kRegsIo = 64;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsNeeded = (128 * kRegsIo + 256 * kRegsSoftmax + kThreads - 1) / kThreads;  // per thread at launch

struct AttnParams {
  CUtensorMap tq, tk, tv;
  CUtensorMap tkr, tvr;  // K, V as [b*S*H rows, D] with one-row boxes (gather4)
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* evict_at;
  const int2* lists;
  __nv_bfloat16* O;
  float* lse;
  int* status;
  int S, Hq, H, G, P, nqb, nb, nitems;
  int s, w, kk, nL;
  float scale_log2;
};

template <int NS>
struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], p_full[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t meta_full[kMetaStages], meta_empty[kMetaStages];
  uint64_t drain;
};

template <int D, bool SPARSE>
struct Layout {
  static constexpr int DH = D / 64;
  static constexpr int NS = D == 128 ? 2 : 4;
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + 2 * DH * kBlockBytes;
  static constexpr int v_off = k_off + NS * DH * kBlockBytes;
  static constexpr int meta_off = v_off + NS * DH * kBlockBytes;
  static constexpr int meta_bytes = kMetaStages * (kKeys + 4) * 8;  // entries + chunk summaries
  static constexpr int bar_off = meta_off + (SPARSE ? meta_bytes : 0);
  static constexpr int misc_off = bar_off + (int)sizeof(Bars<NS>);
  static constexpr int total = misc_off + 64 + 1024;  // + alignment slack
};

// One work item: query block `qblock` (rows of 2P positions) of (batch b, KV head h).
struct Item {
  int b, h, qb0, qb1;
  int NT, NTg;  // key tiles; in sparse mode the first NTg are gathered ([sinks][list])
  int n_sink, n_sl, sp0;
  const int2* list;
};

// Items run longest first: in dense mode the late query blocks see the most
// keys; in sparse mode every block past the first few holds the full budget.
template <bool SPARSE>
__device__ __forceinline__ Item make_item(const AttnParams& p, int it) {
  Item x;
  const int nbh = p.H * p.nb;
  const int rank = it / nbh, rem = it - rank * nbh;
  x.h = rem % p.H;
  x.b = rem / p.H;
  const int qblock = p.nqb - 1 - rank;
  x.qb0 = qblock * 2 * p.P;
  x.qb1 = min(x.qb0 + 2 * p.P, p.S) - 1;
  x.n_sink = 0;
  x.n_sl = 0;
  x.sp0 = 0;
  x.NTg = 0;
  x.list = nullptr;
  if (SPARSE) {
    const int jl = x.qb0 / KVPOP_LIST_QBLOCK;
    const int q0l = jl * KVPOP_LIST_QBLOCK;
    x.n_sink = min(p.s, x.qb1 + 1);
    const int n_list = p.kk > 0 ? min(p.kk, max(0, q0l - p.w - p.s + 1)) : 0;
    if (p.lists) x.list = p.lists + ((size_t)(x.b * p.H + x.h) * p.nL + jl) * (size_t)p.kk;
    x.n_sl = x.n_sink + n_list;
    x.sp0 = max(p.s, q0l - p.w + 1);
    const int n_span = max(0, x.qb1 - x.sp0 + 1);
    x.NTg = (x.n_sl + kKeys - 1) / kKeys;
    x.NT = x.NTg + (n_span + kKeys - 1) / kKeys;
  } else {
    x.NT = (x.qb1 + 1 + kKeys - 1) / kKeys;
  }
  return x;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int D, bool SPARSE>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D, SPARSE>;
  constexpr int DH = L::DH;
  constexpr int NS = L::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Bars<NS>* bars = reinterpret_cast<Bars<NS>*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off);  // [stage][128 entries + 4 summaries]
  const uint32_t sbase = smem_u32(smem);

  const int warp = warp_id(), lane = lane_id();
  const int S = p.S, G = p.G, P = p.P;
  const int it0 = blockIdx.x, dit = gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 4);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < kMetaStages; ++i) {
      mbar_init(&bars->meta_full[i], 1);
      mbar_init(&bars->meta_empty[i], 10);  // 8 softmax warps + 2 loader warps
    }
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
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
  // Q tile qt of item x, once the previous item's last S MMA of that tile has read it
  auto load_q = [&](const Item& x, int qt, int n) -> bool {
    if (!mbar_wait(&bars->q_empty[qt], (n & 1) ^ 1, abort_flag)) {
      fail(SITE_ATTN_PRODUCER, 7);
      return false;
    }
    mbar_arrive_expect_tx(&bars->q_full[qt], DH * kBlockBytes);
    for (int dh = 0; dh < DH; ++dh)
      tma_load_4d(smem + L::q_off + (qt * DH + dh) * kBlockBytes, &p.tq, &bars->q_full[qt], dh * 64, x.h * G,
                  x.qb0 + qt * P, x.b);
    return true;
  };

  const uint32_t q_addr = sbase + L::q_off;
  const uint32_t k_addr = sbase + L::k_off;
  const uint32_t v_addr = sbase + L::v_off;

  if (warp < 4) {
    setmaxnreg_dec<kRegsIo>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer / metadata
    if (!SPARSE) {
      if (lane == 0) {
        tma_prefetch_desc(&p.tq);
        bool ok = true;
        int t = 0, n = 0;
        for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
          const Item x = make_item<SPARSE>(p, it);
          ok = load_q(x, 0, n) && load_q(x, 1, n);
          for (int j = 0; ok && j < x.NT; ++j, ++t) {
            const int st = t % NS;
            const uint32_t ph = (t / NS) & 1;
            if (!mbar_wait(&bars->k_empty[st], ph ^ 1, abort_flag)) {
              fail(SITE_ATTN_PRODUCER, 1);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->k_full[st], DH * kBlockBytes);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(smem + L::k_off + (st * DH + dh) * kBlockBytes, &p.tk, &bars->k_full[st], dh * 64, x.h,
                          j * kKeys, x.b);
            if (!mbar_wait(&bars->v_empty[st], ph ^ 1, abort_flag)) {
              fail(SITE_ATTN_PRODUCER, 2);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->v_full[st], DH * kBlockBytes);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(smem + L::v_off + (st * DH + dh) * kBlockBytes, &p.tv, &bars->v_full[st], dh * 64, x.h,
                          j * kKeys, x.b);
          }
        }
      }
    } else {
      // lane owns entries lane + 32 c of a tile: chunk c has one entry per lane.
      // The loads of tile j + 1 are issued before tile j is written out, so
      // one L2 round trip per tile hides behind the previous tile.
      bool ok = true;
      int t = 0;
      for (int it = it0; ok && it < p.nitems; it += dit) {
        const Item x = make_item<SPARSE>(p, it);
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
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile t and query tile qt: O_qt += P_qt V_t, then S_qt = Q_qt K_{t+1}^T
    // for the next tile, which may be the first tile of the CTA's next item.
    // TMEM: S/P tiles at columns 0 / 128, O tiles at 256 / 384.
    if (lane == 0 && it0 < p.nitems) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 1);
      auto issue_s = [&](int qt, int st) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int dh = ks >> 2;
          const uint32_t w32 = (uint32_t)(ks & 3) * 32;
          const uint64_t a = smem_desc_sw128(q_addr + (qt * DH + dh) * kBlockBytes + w32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(k_addr + (st * DH + dh) * kBlockBytes + w32, 16, 1024);
          mma_ss(tbase + 128 * qt, a, bd, idesc_qk, ks > 0 ? 1u : 0u);
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
      Item x = make_item<SPARSE>(p, it0);
      bool ok = wait_bar(&bars->k_full[0], 0, 2);
      for (int qt = 0; qt < 2 && ok; ++qt) {
        ok = wait_bar(&bars->q_full[qt], 0, 1);
        if (!ok) break;
        issue_s(qt, 0);
        mma_commit(&bars->s_full[qt]);
        if (x.NT == 1) mma_commit(&bars->q_empty[qt]);
        if (qt == 1) mma_commit(&bars->k_empty[0]);
      }
      int t = 0, n = 0;
      for (int it = it0; ok;) {
        for (int j = 0; ok && j < x.NT; ++j, ++t) {
          const int st = t % NS;
          const uint32_t ph = (t / NS) & 1;
          const bool last = j + 1 == x.NT;
          const int it1 = last ? it + dit : it;
          const bool has_next = it1 < p.nitems;
          const int NT1 = last ? (has_next ? make_item<SPARSE>(p, it1).NT : 0) : x.NT;
          const int j1 = last ? 0 : j + 1;
          const int n1 = last ? n + 1 : n;
          const int st1 = (t + 1) % NS;
          const uint32_t ph1 = ((t + 1) / NS) & 1;
          for (int qt = 0; qt < 2 && ok; ++qt) {
            if (!(ok = wait_bar(&bars->p_full[qt], t & 1, 3))) break;
            if (qt == 0 && !(ok = wait_bar(&bars->v_full[st], ph, 4))) break;
            if (j == 0 && !(ok = wait_bar(&bars->o_empty[qt], (n & 1) ^ 1, 6))) break;
#pragma unroll
            for (int ks = 0; ks < kKeys / 16; ++ks) {
              const uint64_t bd = smem_desc_sw128(v_addr + st * DH * kBlockBytes + ks * 2048,
                                                  DH > 1 ? kBlockBytes : 16, 1024);
              mma_ts(tbase + 256 + 128 * qt, tbase + 128 * qt + ks * 8, bd, idesc_pv,
                     (j > 0 || ks > 0) ? 1u : 0u);
            }
            if (qt == 1) mma_commit(&bars->v_empty[st]);
            if (last) mma_commit(&bars->o_full[qt]);
            if (has_next) {
              if (j1 == 0 && !(ok = wait_bar(&bars->q_full[qt], n1 & 1, 1))) break;
              if (qt == 0 && !(ok = wait_bar(&bars->k_full[st1], ph1, 5))) break;
              issue_s(qt, st1);
              mma_commit(&bars->s_full[qt]);
              if (j1 == NT1 - 1) mma_commit(&bars->q_empty[qt]);
              if (qt == 1) mma_commit(&bars->k_empty[st1]);
            }
          }
        }
        if (!ok) break;
        it += dit;
        ++n;
        if (it >= p.nitems) break;
        x = make_item<SPARSE>(p, it);
      }
      // drain every issued MMA before teardown
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr);
    }
  } else if (SPARSE) {
    // ------------------------------------------------------------ loaders: warp 2 streams K, warp 3 V
    // Each runs its own sequence of stages, so K tiles run ahead of the V tiles.
    // Warp 2 also loads query tile 0 of each item, warp 3 query tile 1.
    // Sinks and long-range keys: TMA gather4 (four scattered rows per
    // instruction, lane l takes rows 4l..4l+3); the span: one tiled TMA box.
    const bool is_v = warp == 3;
    const CUtensorMap* rmap = is_v ? &p.tvr : &p.tkr;
    const CUtensorMap* tmap = is_v ? &p.tv : &p.tk;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    const int off = is_v ? L::v_off : L::k_off;
    if (lane == 0 && !is_v) tma_prefetch_desc(&p.tq);
    bool ok = true;
    int t = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
      const Item x = make_item<SPARSE>(p, it);
      if (lane == 0) ok = load_q(x, is_v ? 1 : 0, n);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int row_base = x.b * S * p.H + x.h;  // row of position t is row_base + t * H
      for (int j = 0; j < x.NT; ++j, ++t) {
        const int st = t % NS;
        const uint32_t ph = (t / NS) & 1;
        const int ms = t % kMetaStages;
        if (!warp_wait(&bars->meta_full[ms], (t / kMetaStages) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_PRODUCER, 6);
          ok = false;
          break;
        }
        if (!warp_wait(&empty[st], ph ^ 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_PRODUCER, 4);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[st], DH * kBlockBytes);
        __syncwarp();
        if (j < x.NTg) {
          const int2* km = meta + ms * (kKeys + 4);
          int rows[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int pos = km[4 * lane + u].x;
            rows[u] = pos != 0x7fffffff ? row_base + pos * p.H : row_base;  // padding: any row, masked
          }
#pragma unroll
          for (int d2 = 0; d2 < DH; ++d2)
            tma_gather4(smem + off + (st * DH + d2) * kBlockBytes + lane * 512, rmap, &full[st], d2 * 64,
                        rows[0], rows[1], rows[2], rows[3]);
        } else if (lane == 0) {
          const int span_row = x.sp0 + (j - x.NTg) * kKeys;
          for (int d2 = 0; d2 < DH; ++d2)
            tma_load_4d(smem + off + (st * DH + d2) * kBlockBytes, tmap, &full[st], d2 * 64, x.h, span_row, x.b);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->meta_empty[ms]);
      }
    }
  
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int qt = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int p_row = row / G, g = row - p_row * G;
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = 128 * qt, o_col = 256 + 128 * qt;
    const float sl2 = p.scale_log2;
    const uint64_t s2 = pack2(sl2, sl2);
    bool ok = true;
    int t = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
      const Item x = make_item<SPARSE>(p, it);
      const int q = x.qb0 + qt * P + p_row;
      const int q_first = x.qb0 + qt * P;
      const int jh = x.h * G + g;
      float m_ref = neg_inf(), l = 0.0f;
      for (int j = 0; j < x.NT; ++j, ++t) {
        if (!warp_wait(&bars->s_full[qt], t & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 1);
          ok = false;
          break;
        }
        tc_fence_after();
        const int ms = t % kMetaStages;
        const int2* km = meta + ms * (kKeys + 4);
        if (SPARSE) {
          if (!warp_wait(&bars->meta_full[ms], (t / kMetaStages) & 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_SOFTMAX, 2);
            ok = false;
            break;
          }
        }
        const bool diag = !SPARSE && (j * kKeys + kKeys - 1) > q_first;
        // the whole S row of this thread (128 fp32) in registers; invisible keys -> -inf
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(tl + s_col + ch * 32, sr[ch]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_wait_ld_dep(sr[ch]);
        float mt = neg_inf();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          bool fast;
          if (SPARSE) {
            const int2 sum = km[kKeys + ch];
            fast = q >= sum.x && q < sum.y;
          } else {
            fast = !diag || (j * kKeys + ch * 32 + 31) <= q;
          }
          if (!fast) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              bool visible;
              if (SPARSE) {
                const int2 e = km[ch * 32 + c];
                visible = e.x <= q && q < e.y;
              } else {
                visible = j * kKeys + ch * 32 + c <= q;
              }
              if (!visible) sr[ch][c] = 0xff800000u;
            }
          }
          mt = fmaxf(mt, max32(sr[ch]));
        }
        // lazy rescale of the running max
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
          for (int cd = 0; cd < D / 32; ++cd) {
            uint32_t r[32];
            tmem_ld32(tl + o_col + cd * 32, r);
            tmem_wait_ld_dep(r);
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tmem_st32(tl + o_col + cd * 32, r);
          }
          tmem_wait_st();
        }
        // P = exp2(s * scale_log2 - m) as bf16, written over S
        const float nm = (m_ref == neg_inf()) ? 0.0f : -m_ref * sl2;
        const uint64_t n2 = pack2(nm, nm);
        uint64_t lacc = 0;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t xx = fma2(pack2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), s2, n2);
            float e0, e1;
            unpack2(xx, e0, e1);
            const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
            lacc = add2(lacc, pack2(p0, p1));
            pk[c >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tl + s_col + ch * 16, pk);
        }
        {
          float l0, l1;
          unpack2(lacc, l0, l1);
          l += l0 + l1;
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->p_full[qt]);
          if (SPARSE) mbar_arrive(&bars->meta_empty[ms]);
        }
      }
      if (!ok) break;
      // epilogue: O / l and the LSE; O's TMEM columns are released as soon as read
      if (!warp_wait(&bars->o_full[qt], n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_EPILOGUE, 1);
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      __nv_bfloat16* orow = p.O + (((size_t)x.b * S + q) * p.Hq + jh) * D;
      uint32_t pk[D / 2];
#pragma unroll
      for (int cd = 0; cd < D / 32; ++cd) {
        uint32_t r[32];
        tmem_ld32(tl + o_col + cd * 32, r);
        tmem_wait_ld_dep(r);
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          pk[cd * 16 + (c >> 1)] = pack_bf16x2(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty[qt]);
      if (q <= x.qb1) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int u = 0; u < D / 8; ++u)
          dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        p.lse[((size_t)x.b * p.Hq + jh) * S + q] =
            l > 0.0f ? (m_ref * sl2 + __log2f(l)) * 0.69314718055994531f : neg_inf();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool SPARSE>
kvpop_status launch(const AttnParams& prm, cudaStream_t stream) {
  using L = Layout<D, SPARSE>;
  auto kern = attn_kernel<D, SPARSE>;
  kvpop_status st = cuda_check(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total),
      "kvpop_attn_fwd: smem attribute");
  if (st != KVPOP_OK) return st;
  // the register re-split must fit in the launch allocation (granule: 8 per thread)
  cudaFuncAttributes fa;
  st = cuda_check(cudaFuncGetAttributes(&fa, kern), "kvpop_attn_fwd: attributes");
  if (st != KVPOP_OK) return st;
  if (((fa.numRegs + 7) / 8) * 8 < kRegsNeeded) {
    set_last_error("kvpop_attn_fwd: kernel built with %d registers per thread, %d needed", fa.numRegs, kRegsNeeded);
    return KVPOP_ERR_INTERNAL;
  }
  // persistent: one CTA per SM walks the items with a stride of the grid size
  dim3 grid(min(prm.nitems, num_sms()));
  return cuda_check(launch_pdl(kern, grid, dim3(kThreads), L::total, stream, prm), "kvpop_attn_fwd: launch");
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_attn_fwd(const void* q, const void* k, const void* v, int b, int S,
                                       int Hq, int H, int D, float scale, const int32_t* evict_at,
                                       const int32_t* lists, kvpop_budget bud, void* O, float* lse,
                                       kvpop_stream stream) {
  if (!q || !k || !lse || (O && !v)) {
    set_last_error("kvpop_attn_fwd: q, k, lse (and v when O is requested) must be non-NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (b <= 0 || S <= 0 || H <= 0 || Hq <= 0 || Hq % H != 0) {
    set_last_error("kvpop_attn_fwd: bad shape b=%d S=%d Hq=%d H=%d", b, S, Hq, H);
    return KVPOP_ERR_INVALID_ARG;
  }
  const int G = Hq / H;
  if (D != 64 && D != 128) {
    set_last_error("kvpop_attn_fwd: D=%d unsupported (64 or 128)", D);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (128 % G != 0) {
    set_last_error("kvpop_attn_fwd: G=%d must divide 128", G);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (b > 65535 || H > 65535) {
    set_last_error("kvpop_attn_fwd: b and H must be <= 65535");
    return KVPOP_ERR_UNSUPPORTED;
  }
  const bool sparse = evict_at != nullptr || lists != nullptr;
  if (sparse) {
    if (!evict_at || (!lists && bud.k > 0) || !O || !v) {
      set_last_error("kvpop_attn_fwd: sparse mode needs evict_at, lists (k > 0), v and O");
      return KVPOP_ERR_INVALID_ARG;
    }
    if (bud.s < 0 || bud.w < 0 || bud.k < 0 || (long long)bud.s + bud.w + bud.k < 1) {
      set_last_error("kvpop_attn_fwd: invalid budget");
      return KVPOP_ERR_INVALID_ARG;
    }
  }
  const uintptr_t am = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(O);
  if (am & 15) {
    set_last_error("kvpop_attn_fwd: q, k, v, O must be 16-byte aligned");
    return KVPOP_ERR_UNSUPPORTED;
  }
  const float sc = scale > 0.0f ? scale : 1.0f / sqrtf((float)D);
  const float scale_log2 = sc * 1.4426950408889634f;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (!sparse && !O) return launch_dense_lse(q, k, b, S, Hq, H, D, scale_log2, lse, cs);
  if (sparse && D == 128)
    return launch_sparse_pair(q, k, v, b, S, Hq, H, scale_log2, evict_at, lists, bud, O, lse, cs);

  AttnParams prm;
  memset(&prm, 0, sizeof(prm));
  const int P = 128 / G;
  {
    uint64_t dq[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)S, (uint64_t)b};
    uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)S * Hq * D * 2};
    uint32_t bq[4] = {64, (uint32_t)G, (uint32_t)P, 1};
    uint64_t dk[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)b};
    uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
    uint32_t bk[4] = {64, 1, 128, 1};
    if (!make_tmap_4d(&prm.tq, q, dq, sq, bq) || !make_tmap_4d(&prm.tk, k, dk, sk, bk) ||
        !make_tmap_4d(&prm.tv, v, dk, sk, bk) ||
        !make_tmap_rows(&prm.tkr, k, (uint64_t)D, (uint64_t)b * S * H, 64) ||
        !make_tmap_rows(&prm.tvr, v, (uint64_t)D, (uint64_t)b * S * H, 64))
      return KVPOP_ERR_CUDA;
  }
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
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
  prm.nqb = (S + 2 * P - 1) / (2 * P);
  if ((long long)prm.nqb * H * b > (1LL << 30)) {
    set_last_error("kvpop_attn_fwd: too many query blocks (b * H * ceil(S / (256 / G)) > 2^30)");
    return KVPOP_ERR_UNSUPPORTED;
  }
  prm.nb = b;
  prm.nitems = prm.nqb * H * b;
  prm.s = bud.s;
  prm.w = bud.w;
  prm.kk = bud.k;
  prm.nL = (S + KVPOP_LIST_QBLOCK - 1) / KVPOP_LIST_QBLOCK;
  prm.scale_log2 = scale_log2;
  if (sparse) return launch<64, true>(prm, cs);  // D = 128 runs on CTA pairs (attn_pair.cu)
  return D == 128 ? launch<128, false>(prm, cs) : launch<64, false>(prm, cs);
}
