// kvpop_attn_bwd: gradient of the sparse attention of kvpop_attn_fwd with
// respect to q, k and v ("KVpop ... 精读笔记", section 2.1 and Figure 1: the
// student runs attention over the retained set and is trained through it).
//
// Per row (position q, query head j) with P_t = exp(scale q.k_t - LSE_q) over
// the retained set and upstream gradient dO_q:
//   dv_t += P_t dO_q,   dS_t = P_t (dO_q.v_t - dO_q.O_q),
//   dq_q  = scale sum_t dS_t k_t,   dk_t += scale dS_t q_q.
// Row q retains key t exactly when t <= q < evict_at[t].  That set splits
// without overlap into the band pairs t <= q < t + w (the window; sinks
// included) and the long pairs t + w <= q < evict_at[t].
//
// Four kernels:
//   bwd_prep   -Delta_q = -dO_q.O_q and -LSE_q in log2 units, in the order
//              [b, H, Spad, G]: one 128-row query tile (128/G positions x G
//              heads) is 512 contiguous bytes; padded rows get -LSE = -inf.
//              Negated so that the elementwise steps are one packed FMA
//              (scale s - LSE) and one packed add (dP - Delta) per pair.
//   bwd_keys   per block of kRows query positions and KV head, the keys that
//              hold a long pair with a row of the block: sinks, the long-range
//              list at the block's first row, and the keys entering the top-k
//              inside the block (evict_at[t] > t + w).
//   bwd_dq     query-major, the forward's key plan (sinks, long-range list,
//              span): S = Q K^T and dP = dO V^T in TMEM, dS in bf16 written
//              over S, dQ += dS K accumulated in TMEM over the key tiles.
//   bwd_dkdv   key-major: the 128 keys of an item are the TMEM lanes and the
//              query rows stream by in 128-row tiles: S^T = K Q^T and
//              dP^T = V dO^T, P^T and dS^T in bf16 written over them,
//              dV += P^T dO and dK += dS^T Q.  Launched twice: band items (128
//              consecutive keys against rows t <= q < t + w) store dk and dv;
//              long items (128 keys of a block's list against the block's
//              rows, t + w <= q < evict_at[t]) add theirs with fp32 atomics.
#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kThreads = 384;
constexpr int kKeys = 128;
constexpr int kRows = 512;  // query positions per long-pair block (a multiple of the list block)
constexpr int kBlockBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr int kHalfBytes = 64 * 128;    // 64 rows of such a block
constexpr int kRegsIo = 80;
constexpr int kRegsEw = 208;
constexpr int kRegsNeeded = (128 * kRegsIo + 256 * kRegsEw + kThreads - 1) / kThreads;
// The dQ kernel adds a fourth warpgroup of gather issuers: tile::gather4 from one
// warp moves only about 8 B/clk/SM, and its K and V tiles (64 KB per 128 query
// rows) are spread over three issuing warps each.
constexpr int kDqThreads = 512;
constexpr int kDqRegsIo = 64;
constexpr int kDqRegsHelp = 48;
constexpr int kDqRegsEw = 200;
constexpr int kDqRegsNeeded = (128 * kDqRegsIo + 128 * kDqRegsHelp + 256 * kDqRegsEw + kDqThreads - 1) / kDqThreads;
constexpr int kGatherOps = 2 * (kKeys / 4);  // gather4 ops per 128-key tile: two 64-dim halves
constexpr int kOpsPerIssuer = (kGatherOps + 2) / 3;
static_assert(kRows % KVPOP_LIST_QBLOCK == 0 && kRows % 128 == 0, "block of rows");

struct BwdParams {
  CUtensorMap tq, tdo, tk, tv;  // 4-D tiles: q/dO box {64, G, P, 1}; k/v box {64, 1, 128, 1}
  CUtensorMap tk64, tv64;       // k/v box {64, 1, 64, 1} (half a key tile)
  CUtensorMap tkr, tvr;         // K, V as [b*S*H rows, D] with one-row boxes (gather4)
  CUtensorMap tdqs;             // dq fp32 [b, S, Hq, D]: box {8, min(G, 32), 32 / min(G, 32), 1} (stores)
  const int32_t* evict_at;
  const int2* lists;
  const float* nlse2;   // [b, H, Spad, G]: -LSE * log2(e)
  const float* ndelta;  // [b, H, Spad, G]: -dO . O
  const int2* keys;    // [b, H, nblk, cap]
  const int32_t* nkeys;  // [b, H, nblk]
  float* dq;
  float* dk;
  float* dv;
  int* status;
  int S, Spad, Hq, H, G, gshift, P, nb;
  int s, w, kk, nL;
  int nqt, nqt2, nblk, cap, ctiles;  // nqt2: 256-row query tiles (CTA pairs)
  int nitems;
  float scale, scale_log2;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// ---------------------------------------------------------------------------
// bwd_prep: -Delta and -LSE (log2 units) per row, in query-tile order
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_prep(const __nv_bfloat16* __restrict__ O,
                                                const __nv_bfloat16* __restrict__ dO,
                                                const float* __restrict__ lse, int b, int S, int Spad, int H,
                                                int G, float* __restrict__ nlse2, float* __restrict__ ndelta) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int TPR = D / 8;  // threads per row, 8 elements each
  const int Hq = H * G;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  // rows of O and dO in memory order (batch, position, query head); only the
  // lane that writes a row's results splits its index
  const size_t n = (size_t)b * S * Hq * TPR;  // a multiple of TPR
  const size_t n32 = (n + 31) & ~(size_t)31;   // whole warps take part in the row sums
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n32; i += stride) {
    const bool in = i < n;
    float acc = 0.0f;
    if (in) {
      const uint4 a = *reinterpret_cast<const uint4*>(O + i * 8);
      const uint4 c = *reinterpret_cast<const uint4*>(dO + i * 8);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 fa = __bfloat1622float2(a2[u]), fc = __bfloat1622float2(c2[u]);
        acc = fmaf(fa.x, fc.x, acc);
        acc = fmaf(fa.y, fc.y, acc);
      }
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (in && (i & (TPR - 1)) == 0) {
      const size_t r = i / TPR;
      int j, qp, bi;
      if (r < 0xffffffffull) {
        const uint32_t r32 = (uint32_t)r, bq = r32 / (uint32_t)Hq;
        j = (int)(r32 - bq * (uint32_t)Hq);
        bi = (int)(bq / (uint32_t)S);
        qp = (int)(bq - (uint32_t)bi * (uint32_t)S);
      } else {
        const size_t bq = r / Hq;
        j = (int)(r - bq * Hq);
        bi = (int)(bq / S);
        qp = (int)(bq - (size_t)bi * S);
      }
      const int h = j / G, g = j - h * G;
      const size_t o = (((size_t)bi * H + h) * Spad + qp) * G + g;
      const float l = lse[((size_t)bi * Hq + j) * S + qp];
      nlse2[o] = l != neg_inf() ? -l * 1.4426950408889634f : neg_inf();  // empty rows: every probability is 0
      ndelta[o] = -acc;
    }
  }
  // the padding rows [S, Spad) of every (batch, KV head): no probabilities
  const int pad = Spad - S;
  const size_t np = (size_t)b * H * pad * G;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < np; i += stride) {
    const size_t bh = i / ((size_t)pad * G);
    const int rem = (int)(i - bh * pad * G);
    const size_t o = (bh * Spad + S) * G + rem;
    nlse2[o] = neg_inf();
    ndelta[o] = 0.0f;
  }
}

// ---------------------------------------------------------------------------
// bwd_keys: the keys holding a long pair with a row of each block
// ---------------------------------------------------------------------------
// One CTA of kRows threads per (block, batch x KV head): blockIdx.x = bh * nblk + block.  Order inside a list:
// sinks, the long-range list at row r0, then the entering keys by position.
__global__ void __launch_bounds__(kRows) bwd_keys(const int32_t* __restrict__ evict_at, const int2* __restrict__ lists,
                                                  int S, int s, int w, int kk, int nL, int nblk, int cap,
                                                  int2* __restrict__ keys, int32_t* __restrict__ nkeys) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int warp_tot[kRows / 32];
  const int blk = (int)(blockIdx.x % (unsigned)nblk), bh = (int)(blockIdx.x / (unsigned)nblk);
  const int r0 = blk * kRows;
  const int r1 = min(r0 + kRows, S) - 1;
  int2* out = keys + ((size_t)bh * nblk + blk) * cap;
  const int32_t* ev = evict_at + (size_t)bh * S;
  // sinks t with a row q >= t + w inside the block
  const int n_sink = max(0, min(s, r1 - w + 1));
  for (int i = threadIdx.x; i < n_sink; i += blockDim.x) out[i] = make_int2(i, S);
  // keys retained at row r0 from E(r0): the forward's list (r0 is a list-block start)
  const int n_list = kk > 0 ? min(kk, max(0, r0 - w - s + 1)) : 0;
  if (n_list > 0) {
    const int2* lst = lists + ((size_t)bh * nL + r0 / KVPOP_LIST_QBLOCK) * kk;
    for (int i = threadIdx.x; i < n_list; i += blockDim.x) out[n_sink + i] = lst[i];
  }
  // keys entering E at a row of the block (t + w in (r0, r1]) and retained there
  const int e0 = max(s, r0 - w + 1), e1 = r1 - w;  // at most kRows - 1 positions
  const int t = e0 + (int)threadIdx.x;
  int e = 0;
  if (t <= e1) e = __ldg(ev + t);
  const bool enter = t <= e1 && e > t + w;
  const unsigned bal = __ballot_sync(0xffffffffu, enter);
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  if (lane == 0) warp_tot[wp] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int u = 0; u < kRows / 32; ++u) {
    before += u < wp ? warp_tot[u] : 0;
    total += warp_tot[u];
  }
  if (enter) out[n_sink + n_list + before + __popc(bal & ((1u << lane) - 1))] = make_int2(t, e);
  if (threadIdx.x == 0) nkeys[(size_t)bh * nblk + blk] = n_sink + n_list + total;
}

// ---------------------------------------------------------------------------
// bwd_dq: query-major dQ
// ---------------------------------------------------------------------------
constexpr int kDqMetaStages = 2;  // key metadata is read by the elementwise warps only

template <int NSK, int NSV>
struct DqBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2], ds_full[2];
  uint64_t dp_empty;
  uint64_t o_full, o_empty;
  uint64_t meta_full[kDqMetaStages], meta_empty[kDqMetaStages];
  uint64_t drain;
};

// A K stage lives from its gather until dQ of its tile has run (after the next
// tile's S and dP), a V stage only until dP: three K stages and two V stages.
// The layout fills the opt-in maximum exactly, so it assumes (and the kernel
// checks) a 1024-byte aligned dynamic shared-memory base.
template <int D>
struct DqLayout {
  static constexpr int DH = D / 64;
  static constexpr int NSK = D == 128 ? 3 : 4;
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr int q_off = 0;
  static constexpr int do_off = q_off + DH * kBlockBytes;
  static constexpr int k_off = do_off + DH * kBlockBytes;
  static constexpr int v_off = k_off + NSK * DH * kBlockBytes;
  static constexpr int meta_off = v_off + NSV * DH * kBlockBytes;
  static constexpr int meta_bytes = kDqMetaStages * (kKeys + 4) * 8;
  static constexpr int bar_off = meta_off + meta_bytes;
  static constexpr int misc_off = bar_off + (int)sizeof(DqBars<NSK, NSV>);
  static constexpr int total = misc_off + 64;
  static_assert(total <= 232448, "shared memory");
};

// One query tile (P positions x G heads) of (batch b, KV head h) and its key
// plan: [0, s) sinks, the list at row q0l = 64 floor(q0 / 64), then every
// token in [max(s, q0l - w + 1), q1].
struct DqItem {
  int b, h, q0, q1;
  int NT, NTg;
  int n_sink, n_sl, sp0;
  const int2* list;
};

// pair: a 256-row query tile (2P positions) of the CTA-pair kernel
__device__ __forceinline__ DqItem make_dq_item(const BwdParams& p, int it, bool pair = false) {
  DqItem x;
  const int nbh = p.H * p.nb;
  const int rank = it / nbh, rem = it - rank * nbh;
  x.h = rem % p.H;
  x.b = rem / p.H;
  const int span = pair ? 2 * p.P : p.P;
  const int qt = (pair ? p.nqt2 : p.nqt) - 1 - rank;  // latest tiles first: they hold the full budget
  x.q0 = qt * span;
  x.q1 = min(x.q0 + span, p.S) - 1;
  const int jl = x.q0 / KVPOP_LIST_QBLOCK;
  const int q0l = jl * KVPOP_LIST_QBLOCK;
  x.n_sink = min(p.s, x.q1 + 1);
  const int n_list = p.kk > 0 ? min(p.kk, max(0, q0l - p.w - p.s + 1)) : 0;
  x.list = p.lists ? p.lists + ((size_t)(x.b * p.H + x.h) * p.nL + jl) * (size_t)p.kk : nullptr;
  x.n_sl = x.n_sink + n_list;
  x.sp0 = max(p.s, q0l - p.w + 1);
  const int n_span = max(0, x.q1 - x.sp0 + 1);
  x.NTg = (x.n_sl + kKeys - 1) / kKeys;
  x.NT = x.NTg + (n_span + kKeys - 1) / kKeys;
  return x;
}

// Position of key i of an item's gathered part (sinks, then the list), or -1
// for padding and for a list entry outside [0, S) (the metadata warp reports those).
__device__ __forceinline__ int dq_gather_pos(const DqItem& x, int i, int S) {
  int pos = -1;
  if (i < x.n_sink) pos = i;
  else if (i < x.n_sl) pos = __ldg(&x.list[i - x.n_sink].x);
  return pos >= 0 && pos < S ? pos : -1;
}

// Warp roles (512 threads):
//   warp 0      key metadata of each K/V tile: (position, eviction row) per key
//               and per 32-key chunk the latest position and earliest
//               eviction row (rows inside that range skip masking)
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issuer
//   warp 2      Q tile of each item and the K tiles (gather4 for sinks and
//               long-range keys, one TMA box per span tile)
//   warp 3      dO tile of each item and the V tiles
//   warps 4-11  elementwise: warpgroup 0 takes keys 0-63 of each tile,
//               warpgroup 1 keys 64-127, one query row per thread; then the
//               dQ epilogue (warpgroup 0 the low half of the columns)
//   warps 12-15 gather helpers: 12 and 13 issue two thirds of each gathered K
//               tile's ops with warp 2, 14 and 15 of each V tile's with warp 3
// TMEM columns: S of key tile t at 128 (t & 1) (two buffers), dP at 256, dQ at
// 384.  Each warpgroup packs its 64 dS values (bf16 pairs) over the first 32
// of its own 64 S columns, so neither overwrites S the other has not read.
// MMA order: S_{t+1}, dP_{t+1} (once dP_t has been read), then dQ += dS_t K_t,
// so the tensor core computes the next tile while the elementwise warps work.
template <int D>
__global__ void __launch_bounds__(kDqThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = DqLayout<D>;
  constexpr int DH = L::DH;
  constexpr int NSK = L::NSK, NSV = L::NSV;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the 128-byte swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) report_error(p.status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 12);
    return;
  }
  uint8_t* smem = smem_raw;
  DqBars<NSK, NSV>* bars = reinterpret_cast<DqBars<NSK, NSV>*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off);
  const uint32_t sbase = smem_u32(smem);
  const int warp = warp_id(), lane = lane_id();
  const int S = p.S, G = p.G;
  const int it0 = blockIdx.x, dit = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 2);  // Q (warp 2) and dO (warp 3)
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->ds_full[i], 8);
    }
    mbar_init(&bars->dp_empty, 8);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 8);
    for (int i = 0; i < kDqMetaStages; ++i) {
      mbar_init(&bars->meta_full[i], 1);
      mbar_init(&bars->meta_empty[i], 8);  // the elementwise warps
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
  grid_dep_wait();
  grid_dep_launch();

  auto fail = [&](int site, int detail) {
    report_error(p.status, KVPOP_ERR_TIMEOUT, site, detail);
    *abort_flag = 1;
  };
  const uint32_t q_addr = sbase + L::q_off;
  const uint32_t do_addr = sbase + L::do_off;
  const uint32_t k_addr = sbase + L::k_off;
  const uint32_t v_addr = sbase + L::v_off;
  // gather4 op `o` of a gathered tile (o < kGatherOps): keys 4 (o % 32) .. + 3, dims 64 (o / 32) ..;
  // the rows are read from the item's list before the stage is free, so the
  // list loads overlap the wait
  auto gather_rows = [&](int first, int count, const DqItem& x, int j, int row_base, int (&rows)[4]) {
    if (lane < count) {
      const int q4 = (first + lane) & 31;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = dq_gather_pos(x, j * kKeys + 4 * q4 + u, S);
        rows[u] = pos >= 0 ? row_base + pos * p.H : row_base;  // padding: any row, masked
      }
    }
  };
  auto issue_gather_ops = [&](int first, int count, const int (&rows)[4], int off, int st, const CUtensorMap* rmap,
                              uint64_t* bar) {
    if (lane < count) {
      const int o = first + lane;
      const int q4 = o & 31, d2 = o >> 5;
      tma_gather4(smem + off + (st * DH + d2) * kBlockBytes + q4 * 512, rmap, bar, d2 * 64, rows[0], rows[1],
                  rows[2], rows[3]);
    }
  };

  if (warp >= 12) {
    setmaxnreg_dec<kDqRegsHelp>();
    // ---------------------------------------------------------- gather helpers
    const bool is_v = warp >= 14;
    const int part = 1 + (warp & 1);  // issuer 0 is the loader warp itself
    const CUtensorMap* rmap = is_v ? &p.tvr : &p.tkr;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    const int off = is_v ? L::v_off : L::k_off;
    const int ns = is_v ? NSV : NSK;
    const int first = part * kOpsPerIssuer;
    const int count = min(kOpsPerIssuer, (DH * kKeys / 4) - first);
    bool ok = true;
    int t = 0;
    for (int it = it0; ok && it < p.nitems; it += dit) {
      const DqItem x = make_dq_item(p, it);
      const int row_base = x.b * S * p.H + x.h;
      for (int j = 0; j < x.NT; ++j, ++t) {
        const int st = t % ns;
        int rows[4];
        if (j < x.NTg) gather_rows(first, count, x, j, row_base, rows);
        // every tile, gathered or not: a parity wait is only exact while the
        // waiter is at most one phase ahead of the barrier
        if (!warp_wait(&empty[st], ((t / ns) & 1) ^ 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_PRODUCER, 43);
          ok = false;
          break;
        }
        if (j < x.NTg) issue_gather_ops(first, count, rows, off, st, rmap, &full[st]);
        __syncwarp();
      }
    }
  } else if (warp < 4) {
    setmaxnreg_dec<kDqRegsIo>();
    if (warp == 0) {
      // ---------------------------------------------------------- key metadata
      bool ok = true;
      int t = 0;
      for (int it = it0; ok && it < p.nitems; it += dit) {
        const DqItem x = make_dq_item(p, it);
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
              if (pos <= x.q1) e[c] = make_int2(pos, __ldg(ev + pos));
            }
          }
        };
        int2 cur_e[4], nxt_e[4];
        load_tile(0, cur_e);
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int ms = t % kDqMetaStages;
          if (j + 1 < x.NT) load_tile(j + 1, nxt_e);
          if (!warp_wait(&bars->meta_empty[ms], ((t / kDqMetaStages) & 1) ^ 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 31);
            ok = false;
            break;
          }
          int2* m = meta + ms * (kKeys + 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = lane + 32 * c;
            int2 e = cur_e[c];
            if (e.x != 0x7fffffff && (e.x < 0 || e.x >= S)) {  // a corrupt list entry: never gathered
              report_error(p.status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 11);
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
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && it0 < p.nitems) {
        constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0);
        constexpr uint32_t idesc_dq = idesc_bf16(128, D, 1);
        // the issuing thread shares its SMSP with busy elementwise warps, so each
        // MMA is issued with as few instructions as possible: descriptor low
        // words stepped by constants
        auto issue_nt = [&](uint32_t a_lo, uint32_t b_lo, uint32_t d) {  // A B^T over D
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (uint32_t)(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
            mma_ss_lo(d, a_lo + off, b_lo + off, idesc_s, ks > 0 ? 1u : 0u);
          }
        };
        const uint32_t q_lo = desc_lo(q_addr, 16), do_lo = desc_lo(do_addr, 16);
        const uint32_t k_lo = desc_lo(k_addr, 16), v_lo = desc_lo(v_addr, 16);
        const uint32_t kq_lo = desc_lo(k_addr, DH > 1 ? kBlockBytes : 16);  // K as the MN-major B of dQ
        auto wait_bar = [&](uint64_t* bar, uint32_t ph, int detail) -> bool {
          if (!mbar_wait(bar, ph, abort_flag)) {
            fail(SITE_ATTN_MMA, detail);
            return false;
          }
          tc_fence_after();
          return true;
        };
        // S_t and dP_t of global tile t; item counter n
        auto issue_sdp = [&](int t, bool first_of_item, int n) -> bool {
          const int kst = t % NSK, vst = t % NSV;
          if (first_of_item && !wait_bar(&bars->q_full, n & 1, 31)) return false;
          if (!wait_bar(&bars->k_full[kst], (t / NSK) & 1, 32)) return false;
          issue_nt(q_lo, k_lo + (uint32_t)(kst * DH * kBlockBytes >> 4), tbase + 128u * (uint32_t)(t & 1));
          if (t > 0 && !wait_bar(&bars->dp_empty, (t - 1) & 1, 33)) return false;
          if (!wait_bar(&bars->v_full[vst], (t / NSV) & 1, 34)) return false;
          issue_nt(do_lo, v_lo + (uint32_t)(vst * DH * kBlockBytes >> 4), tbase + 256u);
          mma_commit(&bars->s_full[t & 1]);
          mma_commit(&bars->v_empty[vst]);
          return true;
        };
        DqItem x = make_dq_item(p, it0);
        // the next item's tile count, worked out once per item (its index
        // arithmetic stays off the per-tile path)
        int NTn = it0 + dit < p.nitems ? make_dq_item(p, it0 + dit).NT : 0;
        bool ok = issue_sdp(0, true, 0);
        if (ok && x.NT == 1) mma_commit(&bars->q_empty);
        int t = 0, n = 0;
        for (int it = it0; ok;) {
          for (int j = 0; ok && j < x.NT; ++j, ++t) {
            const int st = t % NSK;
            const bool last = j + 1 == x.NT;
            if (!last || NTn > 0) {
              const int NT1 = last ? NTn : x.NT;
              const int j1 = last ? 0 : j + 1;
              if (!(ok = issue_sdp(t + 1, j1 == 0, last ? n + 1 : n))) break;
              if (j1 == NT1 - 1) mma_commit(&bars->q_empty);  // every S and dP of that item issued
            }
            if (!(ok = wait_bar(&bars->ds_full[t & 1], (t >> 1) & 1, 35))) break;
            if (j == 0 && !(ok = wait_bar(&bars->o_empty, (n & 1) ^ 1, 36))) break;
            const uint32_t b0 = kq_lo + (uint32_t)(st * DH * kBlockBytes >> 4);
            const uint32_t a0 = tbase + 128u * (uint32_t)(t & 1);
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int ks = 0; ks < kKeys / 16; ++ks) {
              // dS of keys 16 ks .. 16 ks + 15: warpgroup ks / 4 packed them over its own S columns
              mma_ts_lo(tbase + 384, a0 + (uint32_t)(64 * (ks >> 2) + 8 * (ks & 3)), b0 + (uint32_t)(ks * 2048 >> 4),
                        idesc_dq, ks > 0 ? 1u : acc0);
            }
            mma_commit(&bars->k_empty[st]);
            if (last) mma_commit(&bars->o_full);
          }
          if (!ok) break;
          it += dit;
          ++n;
          if (it >= p.nitems) break;
          x = make_dq_item(p, it);
          NTn = it + dit < p.nitems ? make_dq_item(p, it + dit).NT : 0;
        }
        mma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, nullptr);
      }
    } else {
      // ---------------------------------------------------------- loaders: warp 2 Q and K, warp 3 dO and V
      const bool is_v = warp == 3;
      const CUtensorMap* rmap = is_v ? &p.tvr : &p.tkr;
      const CUtensorMap* tmap = is_v ? &p.tv : &p.tk;
      const CUtensorMap* qmap = is_v ? &p.tdo : &p.tq;
      uint64_t* full = is_v ? bars->v_full : bars->k_full;
      uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
      const int off = is_v ? L::v_off : L::k_off;
      const int qoff = is_v ? L::do_off : L::q_off;
      const int ns = is_v ? NSV : NSK;
      if (lane == 0) tma_prefetch_desc(qmap);
      bool ok = true;
      int t = 0, n = 0;
      for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
        const DqItem x = make_dq_item(p, it);
        if (lane == 0) {
          ok = mbar_wait(&bars->q_empty, (n & 1) ^ 1, abort_flag);
          if (!ok) {
            fail(SITE_ATTN_PRODUCER, 37);
          } else {
            mbar_arrive_expect_tx(&bars->q_full, DH * kBlockBytes);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(smem + qoff + dh * kBlockBytes, qmap, &bars->q_full, dh * 64, x.h * G, x.q0, x.b);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int row_base = x.b * S * p.H + x.h;  // row of position t is row_base + t * H
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int st = t % ns;
          const uint32_t ph = (t / ns) & 1;
          int rows[4];
          if (j < x.NTg) gather_rows(0, min(kOpsPerIssuer, DH * kKeys / 4), x, j, row_base, rows);
          if (!warp_wait(&empty[st], ph ^ 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 39);
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&full[st], DH * kBlockBytes);
          __syncwarp();
          if (j < x.NTg) {
            // the first third of the tile's gather4 ops; warps 12-15 issue the rest
            issue_gather_ops(0, min(kOpsPerIssuer, DH * kKeys / 4), rows, off, st, rmap, &full[st]);
          } else if (lane == 0) {
            const int span_row = x.sp0 + (j - x.NTg) * kKeys;
            for (int d2 = 0; d2 < DH; ++d2)
              tma_load_4d(smem + off + (st * DH + d2) * kBlockBytes, tmap, &full[st], d2 * 64, x.h, span_row, x.b);
          }
          __syncwarp();
        }
      }
    }
  } else {
    setmaxnreg_inc<kDqRegsEw>();
    // ------------------------------------------------------------ elementwise
    const int wg = (warp - 4) >> 2;  // key half of each tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int p_row = row >> p.gshift, g = row - (p_row << p.gshift);
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int t = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
      const DqItem x = make_dq_item(p, it);
      const int q = x.q0 + p_row;
      const size_t ro = ((size_t)(x.b * p.H + x.h) * p.Spad + x.q0) * G + row;
      const float nl2 = __ldg(p.nlse2 + ro);
      const float nd = __ldg(p.ndelta + ro);
      const uint64_t s2 = pack2(sl2, sl2), n2 = pack2(nl2, nl2), nd2 = pack2(nd, nd), zero2 = pack2(0.0f, 0.0f);
      for (int j = 0; j < x.NT; ++j, ++t) {
        const int sb = t & 1;
        if (!warp_wait(&bars->s_full[sb], (t >> 1) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 31);
          ok = false;
          break;
        }
        tc_fence_after();
        const int ms = t % kDqMetaStages;
        if (!warp_wait(&bars->meta_full[ms], (t / kDqMetaStages) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 32);
          ok = false;
          break;
        }
        const int2* km = meta + ms * (kKeys + 4);
        uint32_t sr[2][32], dr[2][32];
        tmem_ld32(tl + 128 * sb + 64 * wg, sr[0]);
        tmem_ld32(tl + 128 * sb + 64 * wg + 32, sr[1]);
        tmem_ld32(tl + 256 + 64 * wg, dr[0]);
        tmem_ld32(tl + 256 + 64 * wg + 32, dr[1]);
        tmem_wait_ld_dep(sr[0]);
        tmem_wait_ld_dep(sr[1]);
        tmem_wait_ld_dep(dr[0]);
        tmem_wait_ld_dep(dr[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dp_empty);  // the next dP may overwrite its columns
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c32 = 2 * wg + ch;
          const int2 sum = km[kKeys + c32];
          if (!(q >= sum.x && q < sum.y)) {  // some key of the chunk is not visible from this row
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int2 e = km[c32 * 32 + c];
              if (!(e.x <= q && q < e.y)) sr[ch][c] = 0xff800000u;
            }
          }
          // P = exp2(s scale_log2 - LSE2), dS = P (dP - Delta), packed in pairs
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float e0, e1;
            unpack2(fma2(pack2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), s2, n2), e0, e1);
            const uint64_t pp = pack2(ex2_approx(e0), ex2_approx(e1));
            const uint64_t dd = add2(pack2(__uint_as_float(dr[ch][c]), __uint_as_float(dr[ch][c + 1])), nd2);
            float d0, d1;
            unpack2(fma2(pp, dd, zero2), d0, d1);
            pk[c >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tl + 128 * sb + 64 * wg + 16 * ch, pk);  // over this warpgroup's own S columns
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->ds_full[sb]);
          mbar_arrive(&bars->meta_empty[ms]);
        }
      }
      if (!ok) break;
      // epilogue: this warpgroup's half of the dQ columns, scaled
      if (!warp_wait(&bars->o_full, n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_EPILOGUE, 31);
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int HC = D / 2;  // columns per warpgroup
      uint32_t acc[HC];
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(tl + 384 + HC * wg + 32 * cc, r);
        tmem_wait_ld_dep(r);
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[32 * cc + c] = r[c];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
      if (q <= x.q1) {
        float4* dst = reinterpret_cast<float4*>(p.dq + (((size_t)x.b * S + q) * p.Hq + x.h * G + g) * D + HC * wg);
#pragma unroll
        for (int u = 0; u < HC / 4; ++u)
          dst[u] = make_float4(__uint_as_float(acc[4 * u]) * p.scale, __uint_as_float(acc[4 * u + 1]) * p.scale,
                               __uint_as_float(acc[4 * u + 2]) * p.scale, __uint_as_float(acc[4 * u + 3]) * p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// bwd_dq_pair_kernel: query-major dQ on CTA pairs (D = 128)
// ---------------------------------------------------------------------------
// The dQ kernel above laid out for two SMs (tcgen05 cta_group::2), like the
// sparse forward: an item is one 256-row query tile (2P positions), CTA r
// holding rows 128 r .. 128 r + 127, and every M = 256 MMA, issued by the
// leader, spans both SMs -- half the MMA instructions per row, which is what
// bounds the single-CTA kernel (its one issuing thread).  K is the B operand of
// S = Q K^T (N = keys, split by keys: CTA r supplies keys 64 r .. 64 r + 63)
// and of dQ += dS K (N = dims, split by dims: CTA r supplies dims 64 r .. of
// all 128 keys), so each CTA keeps two views of every K tile at offsets that
// match across the pair: an S view [dh][64 keys] and a dQ view [128 keys] of
// its 64 dims (the 8 KB both contain are fetched twice); V, the B operand of
// dP = dO V^T (N = keys), only its S view.  Per tile each SM gathers 48 KB for
// its 128 rows (64 KB in the single-CTA kernel).  Loads of both CTAs complete
// on the leader's barriers, MMA commits arrive on both CTAs' barriers, and the
// elementwise warps of both CTAs arrive on the leader's barriers.
constexpr int kViewBytes = 64 * 128;  // 64 key rows x 128 bytes
constexpr int kPairKOps = 64;         // gather4 ops per K tile and CTA: S view 32, dQ view 32
constexpr int kPairVOps = 32;         // gather4 ops per V tile and CTA: S view
constexpr int kPairKPer = (kPairKOps + 2) / 3;  // the K loader, warps 12 and 14
constexpr int kPairVPer = (kPairVOps + 1) / 2;  // the V loader and warp 15

// dQ leaves by TMA: per elementwise warp two 1 KB slices of 32 rows x 8 fp32
constexpr int kDqEpiWarpBytes = 2048;

struct DqPairLayout {
  static constexpr int NSK = 3, NSV = 2;
  static constexpr int k_stage = 4 * kViewBytes;  // S view (2 x 8 KB), then dQ view (16 KB)
  static constexpr int v_stage = 2 * kViewBytes;  // S view
  static constexpr int q_off = 0;
  static constexpr int do_off = q_off + 2 * kBlockBytes;
  static constexpr int k_off = do_off + 2 * kBlockBytes;
  static constexpr int v_off = k_off + NSK * k_stage;
  static constexpr int meta_off = v_off + NSV * v_stage;
  static constexpr int meta_bytes = kDqMetaStages * (kKeys + 4) * 8;
  static constexpr int epi_off = (meta_off + meta_bytes + 1023) / 1024 * 1024;  // TMA sources: 128 B aligned
  static constexpr int bar_off = epi_off + 8 * kDqEpiWarpBytes;
  static constexpr int misc_off = bar_off + (int)sizeof(DqBars<NSK, NSV>);
  static constexpr int total = misc_off + 64 + 1024;
  static_assert(total <= 232448, "shared memory");
};

// Roles as in the single-CTA kernel (warp 0 key metadata, warp 1 TMEM and --
// leader only -- the MMA issuer, warps 2/3 Q and K / dO and V with warps 12-15
// helping with the gathers, warps 4-11 elementwise on this CTA's 128 rows).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kDqThreads, 1)
    bwd_dq_pair_kernel(const __grid_constant__ BwdParams p) {
  constexpr int D = 128;
  using L = DqPairLayout;
  constexpr int NSK = L::NSK, NSV = L::NSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  DqBars<NSK, NSV>* bars = reinterpret_cast<DqBars<NSK, NSV>*>(smem + L::bar_off);
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
    mbar_init(&bars->q_full, 2);  // the leader's Q and dO loader warps, for both CTAs' bytes
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->ds_full[i], 16);  // 8 elementwise warps in each CTA
    }
    mbar_init(&bars->dp_empty, 16);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 16);
    for (int i = 0; i < kDqMetaStages; ++i) {
      mbar_init(&bars->meta_full[i], 1);
      mbar_init(&bars->meta_empty[i], 8);  // this CTA's elementwise warps
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
  grid_dep_wait();
  grid_dep_launch();

  auto fail = [&](int site, int detail) {
    report_error(p.status, KVPOP_ERR_TIMEOUT, site, detail);
    *abort_flag = 1;
  };
  auto leader_bar = [&](uint64_t* bar) { return cluster_addr(smem_u32(bar), 0); };
  const uint32_t q_addr = sbase + L::q_off;
  const uint32_t do_addr = sbase + L::do_off;
  const uint32_t k_addr = sbase + L::k_off;
  const uint32_t v_addr = sbase + L::v_off;
  const int r64 = 64 * (int)rank;
  // gather4 op o of a gathered K (is_v false) or V tile: four key rows of 128
  // bytes.  K: o < 32 the S view (dims half o / 16, keys r64 + 4 (o % 16) ..),
  // o >= 32 the dQ view (this CTA's dims half, keys 4 (o - 32) ..).  V: the S view.
  auto op_target = [&](bool is_v, int o, int& key0, int& xcoord, int& dst) {
    if (is_v || o < 32) {
      const int dh = o >> 4, g4 = o & 15;
      key0 = r64 + 4 * g4;
      xcoord = dh * 64;
      dst = (is_v ? L::v_off : L::k_off) + dh * kViewBytes + g4 * 512;
    } else {
      const int g4 = o - 32;
      key0 = 4 * g4;
      xcoord = r64;
      dst = L::k_off + 2 * kViewBytes + g4 * 512;
    }
  };
  // rows of op o's four keys, read from the item's list before the stage is free
  auto gather_rows = [&](bool is_v, int o, const DqItem& x, int j, int row_base, int (&rows)[4]) {
    int key0, xc, dst;
    op_target(is_v, o, key0, xc, dst);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int pos = dq_gather_pos(x, j * kKeys + key0 + u, S);
      rows[u] = pos >= 0 ? row_base + pos * p.H : row_base;  // padding: any row, masked
    }
  };
  auto issue_gather = [&](bool is_v, int o, int st, const int (&rows)[4], uint32_t bar) {
    int key0, xc, dst;
    op_target(is_v, o, key0, xc, dst);
    tma_gather4_pair(smem + dst + st * (is_v ? L::v_stage : L::k_stage), is_v ? &p.tvr : &p.tkr, bar, xc, rows[0],
                     rows[1], rows[2], rows[3]);
  };

  if (warp >= 12) {
    setmaxnreg_dec<kDqRegsHelp>();
    // ---------------------------------------------------------- gather helpers
    // warps 12 and 14 (K) and 15 (V); warp 13 shares its SMSP with the MMA issuer
    // and stays idle, so that issuing gathers does not slow the issue of MMAs
    if (warp != 13) {
    const bool is_v = warp == 15;
    const int part = warp == 14 ? 2 : 1;  // part 0 is the loader warp itself
    const int per = is_v ? kPairVPer : kPairKPer;
    const int nops = is_v ? kPairVOps : kPairKOps;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    const int ns = is_v ? NSV : NSK;
    const int first = part * per;
    const int count = min(per, nops - first);
    bool ok = true;
    int t = 0;
    for (int it = it0; ok && it < p.nitems; it += dit) {
      const DqItem x = make_dq_item(p, it, true);
      const int row_base = x.b * S * p.H + x.h;
      for (int j = 0; j < x.NT; ++j, ++t) {
        const int st = t % ns;
        int rows[4];
        if (j < x.NTg && lane < count) gather_rows(is_v, first + lane, x, j, row_base, rows);
        // every tile, gathered or not: a parity wait is only exact while the
        // waiter is at most one phase ahead of the barrier
        if (!warp_wait(&empty[st], ((t / ns) & 1) ^ 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_PRODUCER, 43);
          ok = false;
          break;
        }
        if (j < x.NTg && lane < count) issue_gather(is_v, first + lane, st, rows, leader_bar(&full[st]));
        __syncwarp();
      }
    }
    }
  } else if (warp < 4) {
    setmaxnreg_dec<kDqRegsIo>();
    if (warp == 0) {
      // ---------------------------------------------------------- key metadata (this CTA's masks)
      bool ok = true;
      int t = 0;
      for (int it = it0; ok && it < p.nitems; it += dit) {
        const DqItem x = make_dq_item(p, it, true);
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
              if (pos <= x.q1) e[c] = make_int2(pos, __ldg(ev + pos));
            }
          }
        };
        int2 cur_e[4], nxt_e[4];
        load_tile(0, cur_e);
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int ms = t % kDqMetaStages;
          if (j + 1 < x.NT) load_tile(j + 1, nxt_e);
          if (!warp_wait(&bars->meta_empty[ms], ((t / kDqMetaStages) & 1) ^ 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 31);
            ok = false;
            break;
          }
          int2* m = meta + ms * (kKeys + 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = lane + 32 * c;
            int2 e = cur_e[c];
            if (e.x != 0x7fffffff && (e.x < 0 || e.x >= S)) {  // a corrupt list entry: never gathered
              report_error(p.status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 11);
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
      // TMEM of both CTAs: S of key tile t at 128 (t & 1), dP at 256, dQ at 384
      if (lane == 0 && leader && it0 < p.nitems) {
        constexpr uint32_t idesc_s = idesc_bf16(256, 128, 0);
        constexpr uint32_t idesc_dq = idesc_bf16(256, D, 1);
        // A B^T over D: A a 128-row block pair per CTA ([dh][128 rows]), B an S view
        // ([dh][64 keys]); descriptor low words stepped by constants
        auto issue_nt = [&](uint32_t a_lo, uint32_t b_lo, uint32_t d) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t w = (uint32_t)((ks & 3) * 32 >> 4);
            mma_ss_pair_lo(d, a_lo + (uint32_t)((ks >> 2) * kBlockBytes >> 4) + w,
                           b_lo + (uint32_t)((ks >> 2) * kViewBytes >> 4) + w, idesc_s, ks > 0 ? 1u : 0u);
          }
        };
        const uint32_t q_lo = desc_lo(q_addr, 16), do_lo = desc_lo(do_addr, 16);
        const uint32_t k_lo = desc_lo(k_addr, 16), v_lo = desc_lo(v_addr, 16);
        const uint32_t kq_lo = desc_lo(k_addr + 2 * kViewBytes, kBlockBytes);  // the dQ views, MN-major
        auto wait_bar = [&](uint64_t* bar, uint32_t ph, int detail) -> bool {
          if (!mbar_wait(bar, ph, abort_flag)) {
            fail(SITE_ATTN_MMA, detail);
            return false;
          }
          tc_fence_after();
          return true;
        };
        // S_t and dP_t of global tile t; item counter n
        auto issue_sdp = [&](int t, bool first_of_item, int n) -> bool {
          const int kst = t % NSK, vst = t % NSV;
          if (first_of_item && !wait_bar(&bars->q_full, n & 1, 31)) return false;
          if (!wait_bar(&bars->k_full[kst], (t / NSK) & 1, 32)) return false;
          issue_nt(q_lo, k_lo + (uint32_t)(kst * L::k_stage >> 4), tbase + 128u * (uint32_t)(t & 1));
          if (t > 0 && !wait_bar(&bars->dp_empty, (t - 1) & 1, 33)) return false;
          if (!wait_bar(&bars->v_full[vst], (t / NSV) & 1, 34)) return false;
          issue_nt(do_lo, v_lo + (uint32_t)(vst * L::v_stage >> 4), tbase + 256u);
          mma_commit_pair(&bars->s_full[t & 1]);
          mma_commit_pair(&bars->v_empty[vst]);
          return true;
        };
        DqItem x = make_dq_item(p, it0, true);
        int NTn = it0 + dit < p.nitems ? make_dq_item(p, it0 + dit, true).NT : 0;  // once per item
        bool ok = issue_sdp(0, true, 0);
        if (ok && x.NT == 1) mma_commit_pair(&bars->q_empty);
        int t = 0, n = 0;
        for (int it = it0; ok;) {
          for (int j = 0; ok && j < x.NT; ++j, ++t) {
            const int st = t % NSK;
            const bool last = j + 1 == x.NT;
            if (!last || NTn > 0) {
              const int NT1 = last ? NTn : x.NT;
              const int j1 = last ? 0 : j + 1;
              if (!(ok = issue_sdp(t + 1, j1 == 0, last ? n + 1 : n))) break;
              if (j1 == NT1 - 1) mma_commit_pair(&bars->q_empty);  // every S and dP of that item issued
            }
            if (!(ok = wait_bar(&bars->ds_full[t & 1], (t >> 1) & 1, 35))) break;
            if (j == 0 && !(ok = wait_bar(&bars->o_empty, (n & 1) ^ 1, 36))) break;
            const uint32_t b0 = kq_lo + (uint32_t)(st * L::k_stage >> 4);
            const uint32_t a0 = tbase + 128u * (uint32_t)(t & 1);
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int ks = 0; ks < kKeys / 16; ++ks) {
              // dS of keys 16 ks .. 16 ks + 15: warpgroup ks / 4 packed them over its own S columns
              mma_ts_pair_lo(tbase + 384, a0 + (uint32_t)(64 * (ks >> 2) + 8 * (ks & 3)),
                             b0 + (uint32_t)(ks * 2048 >> 4), idesc_dq, ks > 0 ? 1u : acc0);
            }
            mma_commit_pair(&bars->k_empty[st]);
            if (last) mma_commit_pair(&bars->o_full);
          }
          if (!ok) break;
          it += dit;
          ++n;
          if (it >= p.nitems) break;
          x = make_dq_item(p, it, true);
          NTn = it + dit < p.nitems ? make_dq_item(p, it + dit, true).NT : 0;
        }
        mma_commit_pair(&bars->drain);
      }
      // both CTAs: every pair MMA is done with this CTA's memory before teardown
      if (lane == 0 && it0 < p.nitems) mbar_wait(&bars->drain, 0, nullptr);
    } else {
      // ---------------------------------------------------------- loaders: warp 2 Q and K, warp 3 dO and V
      const bool is_v = warp == 3;
      const CUtensorMap* qmap = is_v ? &p.tdo : &p.tq;
      uint64_t* full = is_v ? bars->v_full : bars->k_full;
      uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
      const int qoff = is_v ? L::do_off : L::q_off;
      const int ns = is_v ? NSV : NSK;
      const int per = is_v ? kPairVPer : kPairKPer;
      // bytes per tile of both CTAs, counted on the leader's barrier
      const uint32_t tile_bytes = 2u * (uint32_t)(is_v ? L::v_stage : L::k_stage);
      if (lane == 0) tma_prefetch_desc(qmap);
      bool ok = true;
      int t = 0, n = 0;
      for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
        const DqItem x = make_dq_item(p, it, true);
        if (lane == 0) {
          ok = mbar_wait(&bars->q_empty, (n & 1) ^ 1, abort_flag);
          if (!ok) {
            fail(SITE_ATTN_PRODUCER, 37);
          } else {
            if (leader) mbar_arrive_expect_tx(&bars->q_full, 2 * 2 * kBlockBytes);
            const uint32_t qb = leader_bar(&bars->q_full);
            for (int dh = 0; dh < 2; ++dh)
              tma_load_4d_pair(smem + qoff + dh * kBlockBytes, qmap, qb, dh * 64, x.h * G, x.q0 + (int)rank * P, x.b);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int row_base = x.b * S * p.H + x.h;  // row of position t is row_base + t * H
        for (int j = 0; j < x.NT; ++j, ++t) {
          const int st = t % ns;
          const uint32_t ph = (t / ns) & 1;
          int rows[4];
          if (j < x.NTg && lane < per) gather_rows(is_v, lane, x, j, row_base, rows);
          if (!warp_wait(&empty[st], ph ^ 1, abort_flag)) {
            if (lane == 0) fail(SITE_ATTN_PRODUCER, 39);
            ok = false;
            break;
          }
          if (lane == 0 && leader) mbar_arrive_expect_tx(&full[st], tile_bytes);
          __syncwarp();
          const uint32_t fb = leader_bar(&full[st]);
          if (j < x.NTg) {
            // the first third of the tile's gather4 ops; warps 12-15 issue the rest
            if (lane < per) issue_gather(is_v, lane, st, rows, fb);
          } else if (lane == 0) {
            const int span_row = x.sp0 + (j - x.NTg) * kKeys;
            if (!is_v) {
              for (int dh = 0; dh < 2; ++dh)
                tma_load_4d_pair(smem + L::k_off + st * L::k_stage + dh * kViewBytes, &p.tk64, fb, dh * 64, x.h,
                                 span_row + r64, x.b);
              tma_load_4d_pair(smem + L::k_off + st * L::k_stage + 2 * kViewBytes, &p.tk, fb, r64, x.h, span_row,
                               x.b);
            } else {
              for (int dh = 0; dh < 2; ++dh)
                tma_load_4d_pair(smem + L::v_off + st * L::v_stage + dh * kViewBytes, &p.tv64, fb, dh * 64, x.h,
                                 span_row + r64, x.b);
            }
          }
          __syncwarp();
        }
      }
    }
  } else {
    setmaxnreg_inc<kDqRegsEw>();
    // ------------------------------------------------------------ elementwise
    const int wg = (warp - 4) >> 2;  // key half of each tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int p_row = row >> p.gshift;
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int t = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit, ++n) {
      const DqItem x = make_dq_item(p, it, true);
      const int qc = x.q0 + (int)rank * P;  // this CTA's first position
      const int q = qc + p_row;
      const size_t ro = ((size_t)(x.b * p.H + x.h) * p.Spad + qc) * G + row;
      const float nl2 = __ldg(p.nlse2 + ro);
      const float nd = __ldg(p.ndelta + ro);
      const uint64_t s2 = pack2(sl2, sl2), n2 = pack2(nl2, nl2), nd2 = pack2(nd, nd), zero2 = pack2(0.0f, 0.0f);
      for (int j = 0; j < x.NT; ++j, ++t) {
        const int sb = t & 1;
        if (!warp_wait(&bars->s_full[sb], (t >> 1) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 31);
          ok = false;
          break;
        }
        tc_fence_after();
        const int ms = t % kDqMetaStages;
        if (!warp_wait(&bars->meta_full[ms], (t / kDqMetaStages) & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 32);
          ok = false;
          break;
        }
        const int2* km = meta + ms * (kKeys + 4);
        uint32_t sr[2][32], dr[2][32];
        tmem_ld32(tl + 128 * sb + 64 * wg, sr[0]);
        tmem_ld32(tl + 128 * sb + 64 * wg + 32, sr[1]);
        tmem_ld32(tl + 256 + 64 * wg, dr[0]);
        tmem_ld32(tl + 256 + 64 * wg + 32, dr[1]);
        tmem_wait_ld_dep(sr[0]);
        tmem_wait_ld_dep(sr[1]);
        tmem_wait_ld_dep(dr[0]);
        tmem_wait_ld_dep(dr[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_bar(&bars->dp_empty));  // the next dP may overwrite its columns
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c32 = 2 * wg + ch;
          const int2 sum = km[kKeys + c32];
          if (!(q >= sum.x && q < sum.y)) {  // some key of the chunk is not visible from this row
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int2 e = km[c32 * 32 + c];
              if (!(e.x <= q && q < e.y)) sr[ch][c] = 0xff800000u;
            }
          }
          // P = exp2(s scale_log2 - LSE2), dS = P (dP - Delta), packed in pairs
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float e0, e1;
            unpack2(fma2(pack2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), s2, n2), e0, e1);
            const uint64_t pp = pack2(ex2_approx(e0), ex2_approx(e1));
            const uint64_t dd = add2(pack2(__uint_as_float(dr[ch][c]), __uint_as_float(dr[ch][c + 1])), nd2);
            float d0, d1;
            unpack2(fma2(pp, dd, zero2), d0, d1);
            pk[c >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tl + 128 * sb + 64 * wg + 16 * ch, pk);  // over this warpgroup's own S columns
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(leader_bar(&bars->ds_full[sb]));
          mbar_arrive(&bars->meta_empty[ms]);
        }
      }
      if (!ok) break;
      // epilogue: this warpgroup's half of the dQ columns, scaled
      if (!warp_wait(&bars->o_full, n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_EPILOGUE, 31);
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int HC = D / 2;  // columns per warpgroup
      uint32_t acc[HC];
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(tl + 384 + HC * wg + 32 * cc, r);
        tmem_wait_ld_dep(r);
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[32 * cc + c] = r[c];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_bar(&bars->o_empty));
      // the warp's 32 rows (32 / min(G, 32) positions x min(G, 32) heads, the order
      // of a dq box) leave by TMA, 8 columns at a time through two 1 KB slices, so
      // that the warp goes on while the stores drain; rows past S are clipped
      const int row0 = quarter * 32;
      const int ty = x.h * G + (row0 & (G - 1)), tz = qc + (row0 >> p.gshift);
      if (tz < S) {
        uint8_t* stw = smem + L::epi_off + (warp - 4) * kDqEpiWarpBytes;
#pragma unroll
        for (int sl = 0; sl < HC / 8; ++sl) {
          uint8_t* buf = stw + (sl & 1) * 1024;
          if (lane == 0) bulk_wait_read<1>();  // the slice stored two steps ago has been read
          __syncwarp();
          const int c = 8 * sl;
          *reinterpret_cast<float4*>(buf + lane * 32) =
              make_float4(__uint_as_float(acc[c]) * p.scale, __uint_as_float(acc[c + 1]) * p.scale,
                          __uint_as_float(acc[c + 2]) * p.scale, __uint_as_float(acc[c + 3]) * p.scale);
          *reinterpret_cast<float4*>(buf + lane * 32 + 16) =
              make_float4(__uint_as_float(acc[c + 4]) * p.scale, __uint_as_float(acc[c + 5]) * p.scale,
                          __uint_as_float(acc[c + 6]) * p.scale, __uint_as_float(acc[c + 7]) * p.scale);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&p.tdqs, buf, HC * wg + c, ty, tz, x.b);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every dq store complete before the CTA retires
  }

  // neither CTA releases its tensor or shared memory while the pair still works
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}


// ---------------------------------------------------------------------------
// bwd_dkdv: key-major dK, dV
// ---------------------------------------------------------------------------
// Epilogue staging of one elementwise warp: 32 keys x 16 fp32 columns, rows
// padded to 80 bytes (conflict-free row writes by the 32 key lanes).
constexpr int kEpiRow = 80;
constexpr int kEpiWarpBytes = 32 * kEpiRow;

template <int NQS>
struct KvBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[NQS], o_full[NQS], q_empty[NQS];  // stage: Q (+ -LSE2) landed, dO (+ -Delta) landed
  uint64_t s_full, s_free, d_full;  // S^T ready / held in registers by every warp; dP^T ready
  uint64_t p_full[2];                 // warpgroup h packed P^T and dS^T of its rows
  uint64_t acc_full, acc_empty;
  uint64_t drain;
};

template <int D>
struct KvLayout {
  static constexpr int DH = D / 64;
  static constexpr int NQS = D == 128 ? 2 : 4;  // Q/dO stages
  static constexpr int k_off = 0;
  static constexpr int v_off = k_off + DH * kBlockBytes;
  static constexpr int q_off = v_off + DH * kBlockBytes;           // stage i: Q at q_off + 2 i DH blocks
  static constexpr int stage_bytes = 2 * DH * kBlockBytes;         // Q then dO
  static constexpr int row_off = q_off + NQS * stage_bytes;        // stage i: 128 -LSE2 then 128 -Delta floats
  static constexpr int kmeta_off = row_off + NQS * 1024;
  static constexpr int epi_off = kmeta_off + kKeys * 8;          // per elementwise warp: kEpiWarpBytes
  static constexpr int bar_off = epi_off + 8 * kEpiWarpBytes;
  static constexpr int misc_off = bar_off + (int)sizeof(KvBars<NQS>);
  static constexpr int total = misc_off + 64 + 1024;
  static_assert(total <= 232448, "shared memory");
};

// Band item: keys [t0, t0 + 128) against rows t0 .. t0 + 126 + w.
// Long item: keys [128 c, 128 c + 128) of block blk's list against the rows of the block.
struct KvItem {
  int b, h, n;    // n: keys in the item (0: nothing to do)
  int t0;         // band: first key position
  const int2* keys;  // long: the item's list entries
  int qt0, NQ;    // first query tile and number of query tiles
};

template <bool LONG>
__device__ __forceinline__ KvItem make_kv_item(const BwdParams& p, int it) {
  KvItem x;
  const int nbh = p.H * p.nb;
  const int rank = it / nbh, rem = it - rank * nbh;
  x.h = rem % p.H;
  x.b = rem / p.H;
  x.keys = nullptr;
  x.t0 = 0;
  if (!LONG) {
    x.t0 = rank * kKeys;
    x.n = min(kKeys, p.S - x.t0);
    const int q_hi = min(p.S - 1, x.t0 + kKeys - 2 + p.w);
    x.qt0 = x.t0 / p.P;
    x.NQ = q_hi / p.P - x.qt0 + 1;
  } else {
    const int blk = p.nblk - 1 - rank / p.ctiles, c = rank % p.ctiles;
    const size_t bb = (size_t)(x.b * p.H + x.h) * p.nblk + blk;
    const int cnt = __ldg(p.nkeys + bb);
    x.n = min(kKeys, cnt - c * kKeys);
    x.keys = p.keys + bb * p.cap + c * kKeys;
    const int r0 = blk * kRows, r1 = min(r0 + kRows, p.S) - 1;
    x.qt0 = r0 / p.P;
    x.NQ = r1 / p.P - x.qt0 + 1;
  }
  if (x.n <= 0) x.n = 0;
  return x;
}

// Warp roles (384 threads):
//   warp 0      per query tile: Q and dO (TMA boxes) with the tile's LSE2 and
//               Delta rows (bulk copies) into a ring of NQS stages
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issuer
//   warp 2      the item's K tile (one TMA box, or gather4 from its list) and
//               the keys' (position, eviction row)
//   warp 3      the item's V tile
//   warps 4-11  elementwise: warpgroup h takes rows 64h .. 64h + 63 of each
//               query tile, one key per thread (TMEM lane); then the epilogue:
//               warpgroup 0 writes dv, warpgroup 1 dk
// TMEM columns: dV at 0, dK at D, S^T at 256 and dP^T at 384 (N = 128: the whole
// query tile; an N = 64 MMA costs an N = 128 one's cycles).  Warpgroup h owns rows
// 64 h .. 64 h + 63 (columns 64 h ..): it loads its S^T columns into registers and
// says so (the next S^T may then overwrite them), computes P, loads its dP^T columns,
// computes dS and packs P^T and dS^T over those 64 dP^T columns.  MMA order per query
// tile u: S^T of tile u + 1 (as soon as every warp holds S^T of tile u), dV, dK of
// rows 0-63, then of rows 64-127, as each warpgroup finishes, then dP^T of tile
// u + 1 -- so the S^T MMAs overlap the elementwise work instead of following it.
template <int D, bool LONG>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using L = KvLayout<D>;
  constexpr int DH = L::DH;
  constexpr int NQS = L::NQS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  KvBars<NQS>* bars = reinterpret_cast<KvBars<NQS>*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  int2* kmeta = reinterpret_cast<int2*>(smem + L::kmeta_off);
  const uint32_t sbase = smem_u32(smem);
  const int warp = warp_id(), lane = lane_id();
  const int S = p.S, G = p.G, P = p.P;
  const int it0 = blockIdx.x, dit = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 2);  // K (warp 2) and V (warp 3)
    mbar_init(&bars->kv_empty, 1);
    for (int i = 0; i < NQS; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 8);  // every elementwise warp
    mbar_init(&bars->d_full, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bars->p_full[i], 4);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
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
  grid_dep_wait();
  grid_dep_launch();

  auto fail = [&](int site, int detail) {
    report_error(p.status, KVPOP_ERR_TIMEOUT, site, detail);
    *abort_flag = 1;
  };
  const uint32_t k_addr = sbase + L::k_off;
  const uint32_t v_addr = sbase + L::v_off;
  auto q_stage = [&](int stg) { return sbase + L::q_off + stg * L::stage_bytes; };
  auto do_stage = [&](int stg) { return sbase + L::q_off + stg * L::stage_bytes + DH * kBlockBytes; };

  if (warp < 4) {
    setmaxnreg_dec<kRegsIo>();
    if (warp == 0) {
      // ---------------------------------------------------------- Q / dO / row constants
      if (lane == 0) {
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tdo);
        bool ok = true;
        int u = 0;
        for (int it = it0; ok && it < p.nitems; it += dit) {
          const KvItem x = make_kv_item<LONG>(p, it);
          if (x.n == 0) continue;
          const size_t rbase = (size_t)(x.b * p.H + x.h) * p.Spad * G;
          for (int i = 0; i < x.NQ; ++i, ++u) {
            const int stg = u % NQS;
            if (!mbar_wait(&bars->q_empty[stg], ((u / NQS) & 1) ^ 1, abort_flag)) {
              fail(SITE_ATTN_PRODUCER, 41);
              ok = false;
              break;
            }
            const int qt = x.qt0 + i;
            // Q (for the next S^T) lands on its own barrier, ahead of dO
            uint64_t* qb = &bars->q_full[stg];
            uint64_t* ob = &bars->o_full[stg];
            uint8_t* qs = smem + L::q_off + stg * L::stage_bytes;
            uint8_t* rs = smem + L::row_off + stg * 1024;
            mbar_arrive_expect_tx(qb, DH * kBlockBytes + 512);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(qs + dh * kBlockBytes, &p.tq, qb, dh * 64, x.h * G, qt * P, x.b);
            bulk_load(rs, p.nlse2 + rbase + (size_t)qt * 128, 512, qb);
            mbar_arrive_expect_tx(ob, DH * kBlockBytes + 512);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(qs + (DH + dh) * kBlockBytes, &p.tdo, ob, dh * 64, x.h * G, qt * P, x.b);
            bulk_load(rs + 512, p.ndelta + rbase + (size_t)qt * 128, 512, ob);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0);
        constexpr uint32_t idesc_acc = idesc_bf16(128, D, 1);
        auto wait_bar = [&](uint64_t* bar, uint32_t ph, int detail) -> bool {
          if (!mbar_wait(bar, ph, abort_flag)) {
            fail(SITE_ATTN_MMA, detail);
            return false;
          }
          tc_fence_after();
          return true;
        };
        // S^T = K Q^T into the S buffer once both warpgroups hold the previous S^T in
        // registers; dP^T = V dO^T into the dP buffer once the previous tile's dV and
        // dK products (whose A operands the warpgroups packed there) are issued.
        // Descriptor low words stepped by constants: the issuing thread shares its
        // SMSP with busy elementwise warps, so every MMA costs few instructions.
        auto issue_s = [&](int stg) {
          const uint32_t ka = desc_lo(k_addr, 16), qb = desc_lo(q_stage(stg), 16);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (uint32_t)(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
            mma_ss_lo(tbase + 256, ka + off, qb + off, idesc_s, ks > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full);
        };
        auto issue_dp = [&](int stg) {
          const uint32_t va = desc_lo(v_addr, 16), db = desc_lo(do_stage(stg), 16);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (uint32_t)(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
            mma_ss_lo(tbase + 384, va + off, db + off, idesc_s, ks > 0 ? 1u : 0u);
          }
          mma_commit(&bars->d_full);
        };
        // dV += P^T dO and dK += dS^T Q over rows 64 h .. 64 h + 63: warpgroup h packed
        // P^T over the first 32 and dS^T over the last 32 of its 64 dP^T columns
        auto issue_acc = [&](int stg, int h, bool first) {
          constexpr uint32_t lbo = DH > 1 ? kBlockBytes : 16;
          const uint32_t db = desc_lo(do_stage(stg) + h * kHalfBytes, lbo);
          const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_lo(tbase, tbase + 384 + 64 * h + ks * 8, db + (uint32_t)(ks * 2048 >> 4), idesc_acc,
                      ks > 0 ? 1u : acc0);
          const uint32_t qb = desc_lo(q_stage(stg) + h * kHalfBytes, lbo);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_lo(tbase + D, tbase + 384 + 64 * h + 32 + ks * 8, qb + (uint32_t)(ks * 2048 >> 4), idesc_acc,
                      ks > 0 ? 1u : acc0);
        };
        bool ok = true;
        int u = 0, n = 0;
        for (int it = it0; ok && it < p.nitems; it += dit) {
          const KvItem x = make_kv_item<LONG>(p, it);
          if (x.n == 0) continue;
          if (!(ok = wait_bar(&bars->kv_full, n & 1, 41))) break;
          if (!(ok = wait_bar(&bars->q_full[u % NQS], (u / NQS) & 1, 42))) break;
          // every warp holds the previous item's last S^T
          if (u > 0 && !(ok = wait_bar(&bars->s_free, (u - 1) & 1, 48))) break;
          issue_s(u % NQS);
          if (!(ok = wait_bar(&bars->o_full[u % NQS], (u / NQS) & 1, 49))) break;
          issue_dp(u % NQS);
          for (int i = 0; ok && i < x.NQ; ++i, ++u) {
            const int stg = u % NQS;
            const bool more = i + 1 < x.NQ;
            const int stg1 = (u + 1) % NQS;
            const uint32_t ph1 = ((u + 1) / NQS) & 1;
            // the next S^T while the warpgroups compute this tile's P and dS, if its
            // query tile has landed; otherwise after this tile's dV and dK products
            bool s_next = !more;
            if (more) {
              if (!(ok = wait_bar(&bars->s_free, u & 1, 47))) break;
              if (mbar_try_wait(&bars->q_full[stg1], ph1)) {
                tc_fence_after();
                issue_s(stg1);
                s_next = true;
              }
            }
            if (!(ok = wait_bar(&bars->p_full[0], u & 1, 43))) break;
            if (i == 0 && !(ok = wait_bar(&bars->acc_empty, (n & 1) ^ 1, 44))) break;
            issue_acc(stg, 0, i == 0);
            if (!s_next && mbar_try_wait(&bars->q_full[stg1], ph1)) {
              tc_fence_after();
              issue_s(stg1);
              s_next = true;
            }
            if (!(ok = wait_bar(&bars->p_full[1], u & 1, 46))) break;
            issue_acc(stg, 1, false);
            mma_commit(&bars->q_empty[stg]);
            if (more) {
              if (!s_next) {
                if (!(ok = wait_bar(&bars->q_full[stg1], ph1, 45))) break;
                issue_s(stg1);
              }
              // the next dP^T overwrites the columns these products read: the tensor
              // core runs them in issue order
              if (!(ok = wait_bar(&bars->o_full[stg1], ph1, 50))) break;
              issue_dp(stg1);
            }
            // K and V are read by S^T and dP^T only, the key metadata by the
            // elementwise warps before their first P: the next item may load once
            // the last tile's S^T and dP^T are issued and every warp is past tile 0
            if (i + 2 == x.NQ || x.NQ == 1) mma_commit(&bars->kv_empty);
          }
          if (!ok) break;
          mma_commit(&bars->acc_full);
          ++n;
        }
        mma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, nullptr);
      }
    } else {
      // ---------------------------------------------------------- K (warp 2) and V (warp 3) of each item
      const bool is_v = warp == 3;
      const CUtensorMap* rmap = is_v ? &p.tvr : &p.tkr;
      const CUtensorMap* tmap = is_v ? &p.tv : &p.tk;
      const int off = is_v ? L::v_off : L::k_off;
      bool ok = true;
      int n = 0;
      for (int it = it0; ok && it < p.nitems; it += dit) {
        const KvItem x = make_kv_item<LONG>(p, it);
        if (x.n == 0) continue;
        if (!warp_wait(&bars->kv_empty, (n & 1) ^ 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_PRODUCER, 42);
          ok = false;
          break;
        }
        if (!LONG) {
          if (!is_v) {
#pragma unroll
            for (int c = 0; c < 4; ++c) kmeta[lane + 32 * c] = make_int2(x.t0 + lane + 32 * c, S);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars->kv_full, DH * kBlockBytes);
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(smem + off + dh * kBlockBytes, tmap, &bars->kv_full, dh * 64, x.h, x.t0, x.b);
          }
        } else {
          const int row_base = x.b * S * p.H + x.h;
          int rows[4];
#pragma unroll
          for (int u2 = 0; u2 < 4; ++u2) {
            const int r = 4 * lane + u2;
            int2 e = r < x.n ? __ldg(x.keys + r) : make_int2(0x7fffffff, 0);
            if (e.x != 0x7fffffff && (e.x < 0 || e.x >= S)) {  // a corrupt entry: never gathered
              report_error(p.status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 12);
              e = make_int2(0x7fffffff, 0);
            }
            rows[u2] = e.x != 0x7fffffff ? row_base + e.x * p.H : row_base;  // padding: any row, masked
            if (!is_v) kmeta[r] = e;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(&bars->kv_full, DH * kBlockBytes);
          __syncwarp();
#pragma unroll
          for (int dh = 0; dh < DH; ++dh)
            tma_gather4(smem + off + dh * kBlockBytes + lane * 512, rmap, &bars->kv_full, dh * 64, rows[0], rows[1],
                        rows[2], rows[3]);
        }
        ++n;
      }
    }
  } else {
    setmaxnreg_inc<kRegsEw>();
    // ------------------------------------------------------------ elementwise
    const int hh = (warp - 4) >> 2;  // row half of each query tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // this thread's key (TMEM lane)
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    const uint64_t s2 = pack2(sl2, sl2), zero2 = pack2(0.0f, 0.0f);
    const int w = p.w, gs = p.gshift;
    bool ok = true;
    int u = 0, n = 0;
    for (int it = it0; ok && it < p.nitems; it += dit) {
      const KvItem x = make_kv_item<LONG>(p, it);
      if (x.n == 0) continue;
      if (!warp_wait(&bars->kv_full, n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_SOFTMAX, 41);
        ok = false;
        break;
      }
      const int2 me = kmeta[r];
      // band: rows [t, t + w) (and < S); long: rows [t + w, evict_at[t])
      const int lo = LONG ? (me.x == 0x7fffffff ? 0x7fffffff : me.x + w) : me.x;
      const int hi = LONG ? me.y : min(me.x + w, S);
      for (int i = 0; i < x.NQ; ++i, ++u) {
        const int stg = u % NQS;
        if (!warp_wait(&bars->s_full, u & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 42);
          ok = false;
          break;
        }
        tc_fence_after();
        // S^T into registers, then the S buffer goes back for the next tile's S^T
        uint32_t sr[2][32], dr[2][32];
        const uint32_t scol = 256 + 64 * hh, dcol = 384 + 64 * hh;  // this warpgroup's 64 rows
        tmem_ld32(tl + scol, sr[0]);
        tmem_ld32(tl + scol + 32, sr[1]);
        tmem_wait_ld_dep(sr[0]);
        tmem_wait_ld_dep(sr[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);
        // this half's rows: row 64 hh + c is at position pos_h + (c >> gshift);
        // the key sees the columns [clo, chi)
        const int pos_h = (x.qt0 + i) * P + ((64 * hh) >> gs);
        const int a = lo - pos_h, bnd = hi - pos_h;
        const int clo = a <= 0 ? 0 : min(64, min(a, 64) << gs);
        const int chi = bnd <= 0 ? 0 : min(64, min(bnd, 64) << gs);
        if (clo > 0 || chi < 64) {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (32 * ch + c < clo || 32 * ch + c >= chi) sr[ch][c] = 0xff800000u;
        }
        const float4* rl2 = reinterpret_cast<const float4*>(smem + L::row_off + stg * 1024) + 16 * hh;
        const float4* rdl = rl2 + 32;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 nl = rl2[(32 * ch + c) >> 2];  // -LSE2 of four rows (a broadcast read)
#pragma unroll
            for (int v2 = 0; v2 < 4; v2 += 2) {
              const uint64_t n2 = v2 == 0 ? pack2(nl.x, nl.y) : pack2(nl.z, nl.w);
              float e0, e1;
              unpack2(fma2(pack2(__uint_as_float(sr[ch][c + v2]), __uint_as_float(sr[ch][c + v2 + 1])), s2, n2), e0, e1);
              sr[ch][c + v2] = __float_as_uint(ex2_approx(e0));  // P in fp32
              sr[ch][c + v2 + 1] = __float_as_uint(ex2_approx(e1));
            }
          }
        }
        if (!warp_wait(&bars->d_full, u & 1, abort_flag)) {
          if (lane == 0) fail(SITE_ATTN_SOFTMAX, 43);
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld32(tl + dcol, dr[0]);
        tmem_ld32(tl + dcol + 32, dr[1]);
        tmem_wait_ld_dep(dr[0]);
        tmem_wait_ld_dep(dr[1]);
        // P^T over the first 32 of the warpgroup's dP^T columns, dS^T over the last 32
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 nd = rdl[(32 * ch + c) >> 2];  // -Delta of four rows
#pragma unroll
            for (int v2 = 0; v2 < 4; v2 += 2) {
              const uint64_t d2 = v2 == 0 ? pack2(nd.x, nd.y) : pack2(nd.z, nd.w);
              const uint64_t dd = add2(pack2(__uint_as_float(dr[ch][c + v2]), __uint_as_float(dr[ch][c + v2 + 1])), d2);
              const float p0 = __uint_as_float(sr[ch][c + v2]), p1 = __uint_as_float(sr[ch][c + v2 + 1]);
              float d0, d1;
              unpack2(fma2(pack2(p0, p1), dd, zero2), d0, d1);
              pk[(c + v2) >> 1] = pack_bf16x2(p0, p1);
              dk[(c + v2) >> 1] = pack_bf16x2(d0, d1);
            }
          }
          tmem_st16(tl + dcol + 16 * ch, pk);
          tmem_st16(tl + dcol + 32 + 16 * ch, dk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[hh]);
      }
      if (!ok) break;
      // epilogue: warpgroup 0 dV, warpgroup 1 dK (scaled)
      if (!warp_wait(&bars->acc_full, n & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_EPILOGUE, 41);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t acc[D];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tl + D * hh + 32 * cc, rr);
        tmem_wait_ld_dep(rr);
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[32 * cc + c] = rr[c];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
      // rows of the warp's 32 keys go out 16 columns at a time through shared
      // memory: each store (long: add) then covers 8 keys x 64 contiguous bytes
      // instead of 32 keys x 16 bytes
      {
        const float sc = hh == 1 ? p.scale : 1.0f;
        float* base = hh == 1 ? p.dk : p.dv;
        const bool valid = me.x >= 0 && me.x < S;  // padding and rejected entries hold 0x7fffffff
        const long long roff = valid ? (((long long)x.b * S + me.x) * p.H + x.h) * D : -1;
        const int kk = lane >> 2, c4 = lane & 3;
        long long offs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) offs[i] = __shfl_sync(0xffffffffu, roff, 8 * i + kk);
        uint8_t* stw = smem + L::epi_off + (warp - 4) * kEpiWarpBytes;
#pragma unroll
        for (int sl = 0; sl < D / 16; ++sl) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 16 * sl + 4 * j;
            *reinterpret_cast<float4*>(stw + lane * kEpiRow + 16 * j) =
                make_float4(__uint_as_float(acc[c]) * sc, __uint_as_float(acc[c + 1]) * sc,
                            __uint_as_float(acc[c + 2]) * sc, __uint_as_float(acc[c + 3]) * sc);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 val = *reinterpret_cast<const float4*>(stw + (8 * i + kk) * kEpiRow + 16 * c4);
            if (offs[i] >= 0) {
              float* dst = base + offs[i] + 16 * sl + 4 * c4;
              if (LONG) red_add_v4(dst, val);
              else *reinterpret_cast<float4*>(dst) = val;
            }
          }
          __syncwarp();
        }
      }
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename K>
kvpop_status prepare(K kern, int smem_bytes, const char* what, int regs_needed = kRegsNeeded) {
  kvpop_status st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes), what);
  if (st != KVPOP_OK) return st;
  cudaFuncAttributes fa;
  st = cuda_check(cudaFuncGetAttributes(&fa, kern), what);
  if (st != KVPOP_OK) return st;
  if (((fa.numRegs + 7) / 8) * 8 < regs_needed) {
    set_last_error("%s: kernel built with %d registers per thread, %d needed", what, fa.numRegs, regs_needed);
    return KVPOP_ERR_INTERNAL;
  }
  return KVPOP_OK;
}

template <int D>
kvpop_status launch_bwd(BwdParams prm, const void* O, const void* dO, const float* lse, float* nlse2, float* ndelta,
                        int2* keys, int32_t* nkeys, cudaStream_t cs) {
  const int b = prm.nb, S = prm.S, H = prm.H, G = prm.G;
  const int nbh = b * H;
  kvpop_status st;
  {
    const long long n = (long long)b * S * prm.Hq * (D / 8);
    const int blocks = (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, 8LL * num_sms()));
    st = cuda_check(launch_pdl(bwd_prep<D>, dim3(blocks), dim3(256), 0, cs,
                               static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), lse, b,
                               S, prm.Spad, H, G, nlse2, ndelta),
                    "kvpop_attn_bwd: prep");
    if (st != KVPOP_OK) return st;
  }
  st = cuda_check(launch_pdl(bwd_keys, dim3(prm.nblk * nbh), dim3(kRows), 0, cs, prm.evict_at, prm.lists, S, prm.s,
                             prm.w, prm.kk, prm.nL, prm.nblk, prm.cap, keys, nkeys),
                  "kvpop_attn_bwd: key lists");
  if (st != KVPOP_OK) return st;
  // dQ: CTA pairs for D = 128, single CTAs for D = 64
  if (D == 128) {
    auto kern = bwd_dq_pair_kernel;
    if ((st = prepare(kern, DqPairLayout::total, "kvpop_attn_bwd: dq", kDqRegsNeeded)) != KVPOP_OK) return st;
    BwdParams pq = prm;
    pq.nitems = prm.nqt2 * nbh;
    const int clusters = std::min(pq.nitems, num_sms() / 2);
    st = cuda_check(launch_pdl(kern, dim3(2 * clusters), dim3(kDqThreads), DqPairLayout::total, cs, pq),
                    "kvpop_attn_bwd: dq launch");
    if (st != KVPOP_OK) return st;
  } else {
    using L = DqLayout<D>;
    auto kern = bwd_dq_kernel<D>;
    if ((st = prepare(kern, L::total, "kvpop_attn_bwd: dq", kDqRegsNeeded)) != KVPOP_OK) return st;
    BwdParams pq = prm;
    pq.nitems = prm.nqt * nbh;
    st = cuda_check(launch_pdl(kern, dim3(std::min(pq.nitems, num_sms())), dim3(kDqThreads), L::total, cs, pq),
                    "kvpop_attn_bwd: dq launch");
    if (st != KVPOP_OK) return st;
  }
  // dK, dV: band items store, long items add
  using KL = KvLayout<D>;
  if (prm.w > 0) {
    auto kern = bwd_dkdv_kernel<D, false>;
    if ((st = prepare(kern, KL::total, "kvpop_attn_bwd: dkdv")) != KVPOP_OK) return st;
    BwdParams pb = prm;
    pb.nitems = ((S + kKeys - 1) / kKeys) * nbh;
    st = cuda_check(launch_pdl(kern, dim3(std::min(pb.nitems, num_sms())), dim3(kThreads), KL::total, cs, pb),
                    "kvpop_attn_bwd: band launch");
    if (st != KVPOP_OK) return st;
  } else {
    const size_t bytes = (size_t)b * S * H * D * sizeof(float);
    if ((st = cuda_check(cudaMemsetAsync(prm.dk, 0, bytes, cs), "kvpop_attn_bwd: zero dk")) != KVPOP_OK) return st;
    if ((st = cuda_check(cudaMemsetAsync(prm.dv, 0, bytes, cs), "kvpop_attn_bwd: zero dv")) != KVPOP_OK) return st;
  }
  {
    auto kern = bwd_dkdv_kernel<D, true>;
    if ((st = prepare(kern, KL::total, "kvpop_attn_bwd: dkdv")) != KVPOP_OK) return st;
    BwdParams pl = prm;
    pl.nitems = prm.nblk * prm.ctiles * nbh;
    st = cuda_check(launch_pdl(kern, dim3(std::min(pl.nitems, num_sms())), dim3(kThreads), KL::total, cs, pl),
                    "kvpop_attn_bwd: long launch");
  }
  return st;
}

struct BwdSizes {
  int G, P, Spad, nblk, cap, ctiles;
  size_t rows_bytes, keys_bytes, counts_bytes, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

kvpop_status bwd_sizes(int b, int S, int Hq, int H, kvpop_budget bud, BwdSizes* z, const char* who) {
  if (b <= 0 || S <= 0 || H <= 0 || Hq <= 0 || Hq % H != 0) {
    set_last_error("%s: bad shape b=%d S=%d Hq=%d H=%d", who, b, S, Hq, H);
    return KVPOP_ERR_INVALID_ARG;
  }
  if (bud.s < 0 || bud.w < 0 || bud.k < 0 || (long long)bud.s + bud.w + bud.k < 1) {
    set_last_error("%s: invalid budget", who);
    return KVPOP_ERR_INVALID_ARG;
  }
  z->G = Hq / H;
  if (128 % z->G != 0) {
    set_last_error("%s: G=%d must divide 128", who, z->G);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (b > 65535 || H > 65535 || S > (1 << 24)) {
    set_last_error("%s: b and H must be <= 65535, S <= 2^24", who);
    return KVPOP_ERR_UNSUPPORTED;
  }
  z->P = 128 / z->G;
  z->Spad = (S + 255) / 256 * 256;  // whole 256-row query tiles of the CTA-pair dQ kernel for every G
  z->nblk = (S + kRows - 1) / kRows;
  z->cap = bud.s + bud.k + kRows;
  z->ctiles = (z->cap + kKeys - 1) / kKeys;
  const long long items = (long long)z->nblk * z->ctiles * b * H;
  const long long qitems = (long long)(S + z->P - 1) / z->P * b * H;
  if (items > (1LL << 30) || qitems > (1LL << 30) || (long long)bud.s + bud.k > (1LL << 28)) {
    set_last_error("%s: problem too large for the work-item indexing", who);
    return KVPOP_ERR_UNSUPPORTED;
  }
  z->rows_bytes = align256((size_t)b * H * z->Spad * z->G * sizeof(float));
  z->keys_bytes = align256((size_t)b * H * z->nblk * z->cap * sizeof(int2));
  z->counts_bytes = align256((size_t)b * H * z->nblk * sizeof(int32_t));
  z->total = 2 * z->rows_bytes + z->keys_bytes + z->counts_bytes;
  return KVPOP_OK;
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_attn_bwd_workspace_size(int b, int S, int Hq, int H, kvpop_budget bud,
                                                      size_t* bytes) {
  if (!bytes) {
    set_last_error("kvpop_attn_bwd_workspace_size: bytes is NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  BwdSizes z;
  kvpop_status st = bwd_sizes(b, S, Hq, H, bud, &z, "kvpop_attn_bwd_workspace_size");
  if (st != KVPOP_OK) return st;
  *bytes = z.total;
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_attn_bwd(const void* q, const void* k, const void* v, const void* O, const void* dO,
                                       const float* lse, int b, int S, int Hq, int H, int D, float scale,
                                       const int32_t* evict_at, const int32_t* lists, kvpop_budget bud, float* dq,
                                       float* dk, float* dv, void* workspace, size_t workspace_bytes,
                                       kvpop_stream stream) {
  if (!q || !k || !v || !O || !dO || !lse || !evict_at || (!lists && bud.k > 0) || !dq || !dk || !dv) {
    set_last_error("kvpop_attn_bwd: q, k, v, O, dO, lse, evict_at, lists (k > 0), dq, dk, dv must be non-NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  BwdSizes z;
  kvpop_status st = bwd_sizes(b, S, Hq, H, bud, &z, "kvpop_attn_bwd");
  if (st != KVPOP_OK) return st;
  if (D != 64 && D != 128) {
    set_last_error("kvpop_attn_bwd: D=%d unsupported (64 or 128)", D);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (!workspace || workspace_bytes < z.total) {
    set_last_error("kvpop_attn_bwd: workspace of %zu bytes needed", z.total);
    return KVPOP_ERR_INVALID_ARG;
  }
  const uintptr_t am = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(O) |
                       reinterpret_cast<uintptr_t>(dO) | reinterpret_cast<uintptr_t>(dq) |
                       reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  if ((am & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
    set_last_error("kvpop_attn_bwd: tensors must be 16-byte aligned, the workspace 256-byte aligned");
    return KVPOP_ERR_UNSUPPORTED;
  }
  const int G = z.G, P = z.P;
  BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  {
    uint64_t dq4[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)S, (uint64_t)b};
    uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)S * Hq * D * 2};
    uint32_t bq[4] = {64, (uint32_t)G, (uint32_t)P, 1};
    uint64_t dk4[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)b};
    uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
    uint32_t bk[4] = {64, 1, 128, 1};
    uint32_t bk64[4] = {64, 1, 64, 1};
    if (!make_tmap_4d(&prm.tq, q, dq4, sq, bq) || !make_tmap_4d(&prm.tdo, dO, dq4, sq, bq) ||
        !make_tmap_4d(&prm.tk, k, dk4, sk, bk) || !make_tmap_4d(&prm.tv, v, dk4, sk, bk) ||
        !make_tmap_4d(&prm.tk64, k, dk4, sk, bk64) || !make_tmap_4d(&prm.tv64, v, dk4, sk, bk64) ||
        !make_tmap_rows(&prm.tkr, k, (uint64_t)D, (uint64_t)b * S * H, 64) ||
        !make_tmap_rows(&prm.tvr, v, (uint64_t)D, (uint64_t)b * S * H, 64))
      return KVPOP_ERR_CUDA;
    const uint32_t gb = (uint32_t)std::min(G, 32);
    uint64_t sq32[3] = {(uint64_t)D * 4, (uint64_t)Hq * D * 4, (uint64_t)S * Hq * D * 4};
    uint32_t bdq[4] = {8, gb, 32 / gb, 1};
    if (!make_tmap_4d_f32(&prm.tdqs, dq, dq4, sq32, bdq)) return KVPOP_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* nlse2 = reinterpret_cast<float*>(ws);
  float* ndelta = reinterpret_cast<float*>(ws + z.rows_bytes);
  int2* keys = reinterpret_cast<int2*>(ws + 2 * z.rows_bytes);
  int32_t* nkeys = reinterpret_cast<int32_t*>(ws + 2 * z.rows_bytes + z.keys_bytes);
  prm.evict_at = evict_at;
  prm.lists = reinterpret_cast<const int2*>(lists);
  prm.nlse2 = nlse2;
  prm.ndelta = ndelta;
  prm.keys = keys;
  prm.nkeys = nkeys;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.status = device_status_ptr();
  prm.S = S;
  prm.Spad = z.Spad;
  prm.Hq = Hq;
  prm.H = H;
  prm.G = G;
  prm.gshift = __builtin_ctz((unsigned)G);
  prm.P = P;
  prm.nb = b;
  prm.s = bud.s;
  prm.w = bud.w;
  prm.kk = bud.k;
  prm.nL = (S + KVPOP_LIST_QBLOCK - 1) / KVPOP_LIST_QBLOCK;
  prm.nqt = (S + P - 1) / P;
  prm.nqt2 = (S + 2 * P - 1) / (2 * P);
  prm.nblk = z.nblk;
  prm.cap = z.cap;
  prm.ctiles = z.ctiles;
  const float sc = scale > 0.0f ? scale : 1.0f / sqrtf((float)D);
  prm.scale = sc;
  prm.scale_log2 = sc * 1.4426950408889634f;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  return D == 128 ? launch_bwd<128>(prm, O, dO, lse, nlse2, ndelta, keys, nkeys, cs)
                  : launch_bwd<64>(prm, O, dO, lse, nlse2, ndelta, keys, nkeys, cs);
}
