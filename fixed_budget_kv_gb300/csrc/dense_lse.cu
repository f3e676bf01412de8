// Dense causal LSE of the teacher ("KVpop ... 精读笔记", section 2.2: A_{d,t} of
// the dense causal attention; section 2.3: its normaliser LSE_d), the
// QK^T-only pass behind kvpop_attn_fwd(O = NULL, no mask).
//
// A CTA owns four 128-row query tiles of one (batch, KV head): tile u covers
// 128/G consecutive positions (rows are (position, query head) pairs).  K
// tiles of 128 keys stream through a ring; for each, one M = 128, N = 128 MMA
// group per query tile writes S into that tile's 128 TMEM columns.  576
// threads: warp 0 TMA producer, warp 1 TMEM allocator and single-thread MMA
// issuer, warps 2-17 four softmax warpgroups (one per query tile, one thread
// per row = TMEM lane).  A tile's columns go back to the issuer as soon as its
// warps have read them, so the tensor core computes that tile's next S while
// the warps still sum exponentials.  Per row, l = sum 2^(s*scale*log2e - ref)
// against a reference that moves only when a chunk would overflow.
#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kNQ = 4;  // 128-row query tiles per CTA
constexpr int kThreads = (2 + 4 * kNQ) * 32;
constexpr int kKeys = 128;             // keys per K tile
constexpr int kBlockBytes = 128 * 128;  // 128 rows x 128 bytes

struct LseParams {
  CUtensorMap tq, tk;  // Q box 64 x G x P, K box 64 x 1 x 128
  float* lse;
  int* status;
  int S, Hq, H, G, P, npb, nbh;
  float scale_log2;
};

template <int NS>
struct LBars {
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS];
  uint64_t s_full[kNQ], s_empty[kNQ];
  uint64_t drain;
};

template <int D>
struct LLayout {
  static constexpr int DH = D / 64;
  static constexpr int NS = D == 128 ? 3 : 8;
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + kNQ * DH * kBlockBytes;
  static constexpr int bar_off = k_off + NS * DH * kBlockBytes;
  static constexpr int misc_off = bar_off + (int)sizeof(LBars<NS>);
  static constexpr int total = misc_off + 64 + 1024;
  static_assert(total <= 232448, "shared memory");
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dense_lse_kernel(const __grid_constant__ LseParams p) {
  using L = LLayout<D>;
  constexpr int DH = L::DH;
  constexpr int NS = L::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  LBars<NS>* bars = reinterpret_cast<LBars<NS>*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  const uint32_t sbase = smem_u32(smem);

  const int warp = warp_id(), lane = lane_id();
  // heaviest query blocks first across all (batch, head) pairs
  const int cid = (int)blockIdx.x;
  const int pblock = p.npb - 1 - cid / p.nbh;
  const int bh = cid % p.nbh;
  const int b = bh / p.H, h = bh % p.H;
  const int S = p.S, G = p.G, P = p.P;
  const int qb0 = pblock * kNQ * P;
  int nt[kNQ];  // K tiles each query tile needs (causal, up to the tile's last row)
#pragma unroll
  for (int u = 0; u < kNQ; ++u) {
    const int first = qb0 + u * P;
    const int last = min(first + P, S) - 1;
    nt[u] = last >= first ? last / kKeys + 1 : 0;
  }
  int NT = 0;
#pragma unroll
  for (int u = 0; u < kNQ; ++u) NT = max(NT, nt[u]);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_empty[i], 4);  // the tile's four softmax warps
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

  if (warp == 0) {
    if (lane == 0 && NT > 0) {
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tk);
      mbar_arrive_expect_tx(&bars->q_full, kNQ * DH * kBlockBytes);
      for (int u = 0; u < kNQ; ++u)
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(smem + L::q_off + (u * DH + dh) * kBlockBytes, &p.tq, &bars->q_full, dh * 64, h * G,
                      qb0 + u * P, b);
      for (int j = 0; j < NT; ++j) {
        const int st = j % NS;
        if (!mbar_wait(&bars->k_empty[st], ((j / NS) & 1) ^ 1, abort_flag)) {
          fail(SITE_ATTN_PRODUCER, 21);
          break;
        }
        mbar_arrive_expect_tx(&bars->k_full[st], DH * kBlockBytes);
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(smem + L::k_off + (st * DH + dh) * kBlockBytes, &p.tk, &bars->k_full[st], dh * 64, h,
                      j * kKeys, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && NT > 0) {
      {
        bool ok = mbar_wait(&bars->q_full, 0, abort_flag);
        if (!ok) fail(SITE_ATTN_MMA, 21);
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16(128, 128, 0);
        // descriptor low words stepped by constants: the issuing thread shares
        // its SMSP with four busy softmax warps, so every MMA costs few instructions
        const uint32_t q_lo = desc_lo(sbase + L::q_off, 16), k_lo = desc_lo(sbase + L::k_off, 16);
        for (int j = 0; ok && j < NT; ++j) {
          const int st = j % NS;
          if (!mbar_wait(&bars->k_full[st], (j / NS) & 1, abort_flag)) {
            fail(SITE_ATTN_MMA, 22);
            break;
          }
          tc_fence_after();
          for (int u = 0; u < kNQ; ++u) {
            if (j >= nt[u]) continue;
            if (!mbar_wait(&bars->s_empty[u], (j & 1) ^ 1, abort_flag)) {
              fail(SITE_ATTN_MMA, 23);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = q_lo + (uint32_t)(u * DH * kBlockBytes >> 4);
            const uint32_t b0 = k_lo + (uint32_t)(st * DH * kBlockBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (uint32_t)(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
              mma_ss_lo(tbase + 128 * u, a0 + off, b0 + off, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[u]);
          }
          mma_commit(&bars->k_empty[st]);
        }
        mma_commit(&bars->drain);
      }
      mbar_wait(&bars->drain, 0, nullptr);
    }
  } else {
    // softmax warpgroups: warps 2-5 -> tile 0, 6-9 -> tile 1, ...
    const int u = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int p_row = row / G, g = row - p_row * G;
    const int q_first = qb0 + u * P;
    const int q = q_first + p_row;
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16) + 128 * u;

    const float sl2 = p.scale_log2;
    const uint64_t s2 = pack2(sl2, sl2);
    float m_ref = neg_inf(), l = 0.0f;
    bool ok = true;
    const int ntq = nt[u];
    for (int j = 0; j < ntq; ++j) {
      if (!warp_wait(&bars->s_full[u], j & 1, abort_flag)) {
        if (lane == 0) fail(SITE_ATTN_SOFTMAX, 21);
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = (j * kKeys + kKeys - 1) > q_first;
      uint32_t ra[32], rb[32];
      tmem_ld32(tl, ra);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t(&cur)[32] = (ch & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (ch & 1) ? ra : rb;
        tmem_wait_ld_dep(cur);
        if (ch < 3) {
          tmem_ld32(tl + (ch + 1) * 32, nxt);
        } else {  // every column of this tile is in registers: hand TMEM back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->s_empty[u]);
        }
        if (diag) {
          const int t0 = j * kKeys + ch * 32;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (t0 + c > q) cur[c] = 0xff800000u;
        }
        if (m_ref == neg_inf()) {
          const float cm = max32(cur);
          if (cm == neg_inf()) continue;
          m_ref = cm;
        }
        float sum = exp2_sum32(cur, s2, pack2(-m_ref * sl2, -m_ref * sl2));
        if (!(sum <= 0x1p64f)) {  // a score far above the reference: move it
          const float cm = max32(cur);
          l *= ex2_approx((m_ref - cm) * sl2);
          m_ref = cm;
          sum = exp2_sum32(cur, s2, pack2(-m_ref * sl2, -m_ref * sl2));
        }
        l += sum;
      }
    }
    if (ok && q < S)
      p.lse[((size_t)b * p.Hq + h * G + g) * S + q] =
          l > 0.0f ? (m_ref * sl2 + __log2f(l)) * 0.69314718055994531f : neg_inf();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D>
kvpop_status launch_d(const LseParams& prm, cudaStream_t cs) {
  using L = LLayout<D>;
  auto kern = dense_lse_kernel<D>;
  kvpop_status st = cuda_check(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total),
      "dense LSE: smem attribute");
  if (st != KVPOP_OK) return st;
  return cuda_check(launch_pdl(kern, dim3(prm.npb * prm.nbh), dim3(kThreads), L::total, cs, prm),
                    "dense LSE: launch");
}

}  // namespace

// Called by kvpop_attn_fwd after argument validation (dense mode, O == NULL).
kvpop_status launch_dense_lse(const void* q, const void* k, int b, int S, int Hq, int H, int D,
                              float scale_log2, float* lse, cudaStream_t cs) {
  LseParams prm;
  memset(&prm, 0, sizeof(prm));
  const int G = Hq / H, P = 128 / G;
  uint64_t dq[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)S, (uint64_t)b};
  uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)S * Hq * D * 2};
  uint32_t bq[4] = {64, (uint32_t)G, (uint32_t)P, 1};
  uint64_t dk[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)b};
  uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
  uint32_t bk[4] = {64, 1, 128, 1};
  if (!make_tmap_4d(&prm.tq, q, dq, sq, bq) || !make_tmap_4d(&prm.tk, k, dk, sk, bk)) return KVPOP_ERR_CUDA;
  prm.lse = lse;
  prm.status = device_status_ptr();
  prm.S = S;
  prm.Hq = Hq;
  prm.H = H;
  prm.G = G;
  prm.P = P;
  prm.npb = (S + kNQ * P - 1) / (kNQ * P);
  prm.nbh = b * H;
  prm.scale_log2 = scale_log2;
  if ((long long)prm.npb * prm.nbh > 0x7fffffffLL) {
    set_last_error("dense LSE: grid too large");
    return KVPOP_ERR_UNSUPPORTED;
  }
  return D == 128 ? launch_d<128>(prm, cs) : launch_d<64>(prm, cs);
}

}  // namespace kvpop
