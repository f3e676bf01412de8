// kvpop_future_target: the transposed-attention pass of "KVpop ... 精读笔记",
// sections 2.2-2.3 (Eq. 8, Figure 2).  The future-attention mass of key t is a
// column sum of the dense attention map; with keys as rows and queries as
// columns it becomes a row sum that an attention-shaped kernel computes
// without materialising the map:
//   target[b,h,t] = log sum_{g<G} sum_{d>=t+w} exp(scale q_{d,hG+g}.k_t - LSE_{d,hG+g}).
// Every term is a probability (<= 1), so a plain fp32 sum needs no running max.
//
// One CTA owns four 128-key row tiles (512 keys) of one (batch, KV head) and a
// chunk of at most 64 query tiles (128/G positions x G heads = 128 columns
// each) among those the keys can see; each query tile fetched feeds four MMAs.
// 576 threads: warp 0 TMA producer (K once, Q tiles, and the LSE of each query
// tile, negated and in log2 units, by a 1-D bulk copy), warp 1 TMEM allocator
// and single-thread MMA issuer, warps 2-17 four warpgroups summing
// exponentials, one per row tile (one thread per key = TMEM lane).  A row
// tile's 128 TMEM columns are handed back as soon as they are read.  Chunks of
// the same keys add their partial sums into the output with one atomicAdd per
// key; a last pass takes the log.
#include <mutex>

#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kNR = 4;  // row tiles per CTA
constexpr int kThreads = (2 + 4 * kNR) * 32;
constexpr int kBlockBytes = 128 * 128;
constexpr int kLseStages = 4;
constexpr int kChunkTiles = 64;  // query tiles per CTA

struct TargetParams {
  CUtensorMap tq, tk;
  const float* lse2;  // [b, H, Spad, G] = -LSE * log2(e), -inf past S
  float* acc;         // [b, H, S] partial sums (the output buffer, zeroed first)
  int* status;
  int S, Spad, H, G, logG, P, nct, w, nchunk;
  float scale_log2;
};

template <int D>
struct TLayout {
  static constexpr int DH = D / 64;
  static constexpr int NS = D == 128 ? 2 : 4;
  static constexpr int k_off = 0;
  static constexpr int q_off = k_off + kNR * DH * kBlockBytes;
  static constexpr int lse_off = q_off + NS * DH * kBlockBytes;
  static constexpr int bar_off = lse_off + kLseStages * 512;
  static constexpr int nbar = 1 + 2 * NS + 2 * kNR + 2 * kLseStages + 1;
  static constexpr int misc_off = bar_off + nbar * 8;
  static constexpr int total = misc_off + 64 + 1024;
};

template <int NS>
struct TBars {
  uint64_t k_full;
  uint64_t q_full[NS], q_empty[NS];
  uint64_t s_full[kNR], s_empty[kNR];
  uint64_t l_full[kLseStages], l_empty[kLseStages];
  uint64_t drain;
};

__global__ void lse_prep(const float* __restrict__ lse, int b, int H, int G, int S, int Spad,
                         float* __restrict__ lse2) {
  grid_dep_wait();
  grid_dep_launch();
  const long long n = (long long)b * H * Spad * G;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(i % G);
    long long r = i / G;
    const int d = (int)(r % Spad);
    r /= Spad;
    const int h = (int)(r % H);
    const int bi = (int)(r / H);
    lse2[i] = d < S ? -lse[((size_t)bi * H * G + (size_t)h * G + g) * S + d] * 1.4426950408889634f
                    : __int_as_float(0xff800000);
  }
}

__global__ void target_finalize(float* __restrict__ t, long long n) {
  grid_dep_wait();
  grid_dep_launch();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float s = t[i];
    t[i] = s > 0.0f ? __log2f(s) * 0.69314718055994531f : __int_as_float(0xff800000);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) target_kernel(const __grid_constant__ TargetParams p) {
  using L = TLayout<D>;
  constexpr int DH = L::DH;
  constexpr int NS = L::NS;
  const int chunk = blockIdx.x, rb = blockIdx.y;
  const int b = blockIdx.z / p.H, h = blockIdx.z % p.H;
  const int S = p.S, P = p.P, G = p.G;
  const int t0 = rb * 128 * kNR;
  int c_start[kNR];
#pragma unroll
  for (int rt = 0; rt < kNR; ++rt) {
    const long long first = (long long)t0 + 128 * rt + p.w;  // first query position any key here sees
    c_start[rt] = first > S - 1 ? p.nct : (int)(first / P);
  }
  const int c_lo = c_start[0] + chunk * kChunkTiles;
  const int c_hi = min(p.nct, c_lo + kChunkTiles);
  if (c_lo >= c_hi) return;  // nothing left for this chunk (uniform over the CTA)
  const int NTc = c_hi - c_lo;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  TBars<NS>* bars = reinterpret_cast<TBars<NS>*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  const float* lse_s = reinterpret_cast<const float*>(smem + L::lse_off);
  const uint32_t sbase = smem_u32(smem);
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(&bars->k_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < kNR; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_empty[i], 4);
    }
    for (int i = 0; i < kLseStages; ++i) {
      mbar_init(&bars->l_full[i], 1);
      mbar_init(&bars->l_empty[i], 4 * kNR);
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
    if (lane == 0) {
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tk);
      mbar_arrive_expect_tx(&bars->k_full, kNR * DH * kBlockBytes);
      for (int rt = 0; rt < kNR; ++rt)
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(smem + L::k_off + (rt * DH + dh) * kBlockBytes, &p.tk, &bars->k_full, dh * 64, h,
                      t0 + 128 * rt, b);
      const float* lsrc = p.lse2 + ((size_t)b * p.H + h) * (size_t)p.Spad * G;
      for (int jc = 0; jc < NTc; ++jc) {
        const int c = c_lo + jc;
        const int st = jc % NS;
        if (!mbar_wait(&bars->q_empty[st], ((jc / NS) & 1) ^ 1, abort_flag)) {
          fail(SITE_TARGET_PRODUCER, 1);
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full[st], DH * kBlockBytes);
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(smem + L::q_off + (st * DH + dh) * kBlockBytes, &p.tq, &bars->q_full[st], dh * 64,
                      h * G, c * P, b);
        const int ls = jc % kLseStages;
        if (!mbar_wait(&bars->l_empty[ls], ((jc / kLseStages) & 1) ^ 1, abort_flag)) {
          fail(SITE_TARGET_PRODUCER, 2);
          break;
        }
        mbar_arrive_expect_tx(&bars->l_full[ls], 512);
        bulk_load(smem + L::lse_off + ls * 512, lsrc + (size_t)c * P * G, 512, &bars->l_full[ls]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(&bars->k_full, 0, abort_flag);
      if (!ok) fail(SITE_TARGET_MMA, 1);
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, 128, 0);
      const uint32_t k_lo = desc_lo(sbase + L::k_off, 16), q_lo = desc_lo(sbase + L::q_off, 16);
      int n_rt[kNR] = {0, 0, 0, 0};
      for (int jc = 0; ok && jc < NTc; ++jc) {
        const int c = c_lo + jc;
        const int st = jc % NS;
        if (!mbar_wait(&bars->q_full[st], (jc / NS) & 1, abort_flag)) {
          fail(SITE_TARGET_MMA, 2);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int rt = 0; rt < kNR; ++rt) {
          if (c < c_start[rt]) continue;
          const int n = n_rt[rt]++;
          if (!mbar_wait(&bars->s_empty[rt], (n & 1) ^ 1, abort_flag)) {
            fail(SITE_TARGET_MMA, 3);
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptor low words stepped by constants: the issuing thread shares
          // its SMSP with four busy warps, so every MMA costs few instructions
          const uint32_t a0 = k_lo + (uint32_t)(rt * DH * kBlockBytes >> 4);
          const uint32_t b0 = q_lo + (uint32_t)(st * DH * kBlockBytes >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (uint32_t)(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
            mma_ss_lo(tbase + 128 * rt, a0 + off, b0 + off, idesc, ks > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[rt]);
        }
        mma_commit(&bars->q_empty[st]);
      }
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr);
    }
  } else {
    // warpgroups: warps 2-5 -> row tile 0, 6-9 -> 1, 10-13 -> 2, 14-17 -> 3
    const int rt = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int t = t0 + 128 * rt + quarter * 32 + lane;  // this thread's key
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16) + 128 * rt;
    const float sl2 = p.scale_log2;
    const int row_first = t0 + 128 * rt;
    const int crt = c_start[rt];
    uint64_t acc0 = 0, acc1 = 0;  // packed fp32 pairs
    const uint64_t s2 = pack2(sl2, sl2);
    bool ok = true;
    int n = 0;
    for (int jc = 0; jc < NTc; ++jc) {
      const int c = c_lo + jc;
      const int ls = jc % kLseStages;
      if (!warp_wait(&bars->l_full[ls], (jc / kLseStages) & 1, abort_flag)) {
        if (lane == 0) fail(SITE_TARGET_SOFTMAX, 1);
        ok = false;
        break;
      }
      if (c >= crt) {
        if (!warp_wait(&bars->s_full[rt], n & 1, abort_flag)) {
          if (lane == 0) fail(SITE_TARGET_SOFTMAX, 2);
          ok = false;
          break;
        }
        ++n;
        tc_fence_after();
        const float* l2 = lse_s + ls * 128;
        const bool masked = (long long)c * P < (long long)row_first + 127 + p.w;
        uint32_t ra[32], rb[32];
        tmem_ld32(tl, ra);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t(&cur)[32] = (ch & 1) ? rb : ra;
          uint32_t(&nxt)[32] = (ch & 1) ? ra : rb;
          tmem_wait_ld_dep(cur);
          if (ch < 3) {
            tmem_ld32(tl + (ch + 1) * 32, nxt);
          } else {  // the whole S' row tile is in registers: hand TMEM back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_empty[rt]);
          }
          if (masked) {  // only the query tiles that straddle d = t + w
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
              const int d = c * P + ((ch * 32 + cc) >> p.logG);
              if (d < t + p.w) cur[cc] = 0xff800000u;
            }
          }
#pragma unroll
          for (int cc = 0; cc < 32; cc += 4) {
            const float4 lv = *reinterpret_cast<const float4*>(l2 + ch * 32 + cc);
            const uint64_t x0 = fma2(pack2(__uint_as_float(cur[cc]), __uint_as_float(cur[cc + 1])), s2,
                                     pack2(lv.x, lv.y));
            const uint64_t x1 = fma2(pack2(__uint_as_float(cur[cc + 2]), __uint_as_float(cur[cc + 3])), s2,
                                     pack2(lv.z, lv.w));
            float e0, e1, e2, e3;
            unpack2(x0, e0, e1);
            unpack2(x1, e2, e3);
            acc0 = add2(acc0, pack2(ex2_approx(e0), ex2_approx(e1)));
            acc1 = add2(acc1, pack2(ex2_approx(e2), ex2_approx(e3)));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->l_empty[ls]);
    }
    if (ok && t < S) {
      float y0, y1;
      unpack2(add2(acc0, acc1), y0, y1);
      const float sum = y0 + y1;
      if (sum > 0.0f) atomicAdd(p.acc + ((size_t)b * p.H + h) * S + t, sum);
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

template <int D>
kvpop_status launch_target(const TargetParams& prm, int b, int H, cudaStream_t cs) {
  using L = TLayout<D>;
  auto kern = target_kernel<D>;
  kvpop_status st = cuda_check(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total),
      "kvpop_future_target: smem attribute");
  if (st != KVPOP_OK) return st;
  const int nrb = (prm.S + 128 * kNR - 1) / (128 * kNR);
  dim3 grid(prm.nchunk, nrb, b * H);
  return cuda_check(launch_pdl(kern, grid, dim3(kThreads), L::total, cs, prm), "kvpop_future_target: launch");
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_future_target_workspace_size(int b, int S, int Hq, int H,
                                                           size_t* bytes) {
  if (!bytes || b <= 0 || S <= 0 || H <= 0 || Hq <= 0 || Hq % H != 0) {
    set_last_error("kvpop_future_target_workspace_size: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  const int G = Hq / H;
  if (128 % G != 0) {
    set_last_error("kvpop_future_target_workspace_size: G=%d must divide 128", G);
    return KVPOP_ERR_UNSUPPORTED;
  }
  const int P = 128 / G;
  const size_t spad = (size_t)((S + P - 1) / P) * P;
  *bytes = (size_t)b * H * spad * G * sizeof(float);
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_future_target(const void* q, const void* k, const float* lse, int b,
                                            int S, int Hq, int H, int D, float scale, int w,
                                            float* target, void* workspace, size_t ws_bytes,
                                            kvpop_stream stream) {
  if (!q || !k || !lse || !target || !workspace) {
    set_last_error("kvpop_future_target: q, k, lse, target and workspace must be non-NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (w < 0) {
    set_last_error("kvpop_future_target: w must be >= 0");
    return KVPOP_ERR_INVALID_ARG;
  }
  size_t need = 0;
  kvpop_status st = kvpop_future_target_workspace_size(b, S, Hq, H, &need);
  if (st != KVPOP_OK) return st;
  if (ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15)) {
    set_last_error("kvpop_future_target: workspace needs %zu bytes, 16-byte aligned", need);
    return KVPOP_ERR_INVALID_ARG;
  }
  if (D != 64 && D != 128) {
    set_last_error("kvpop_future_target: D=%d unsupported (64 or 128)", D);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k)) & 15) != 0) {
    set_last_error("kvpop_future_target: q and k must be 16-byte aligned");
    return KVPOP_ERR_UNSUPPORTED;
  }
  if ((long long)b * H > 65535) {
    set_last_error("kvpop_future_target: b*H must be <= 65535");
    return KVPOP_ERR_UNSUPPORTED;
  }
  const int G = Hq / H;
  const int P = 128 / G;
  TargetParams prm;
  memset(&prm, 0, sizeof(prm));
  {
    uint64_t dq[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)S, (uint64_t)b};
    uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)S * Hq * D * 2};
    uint32_t bq[4] = {64, (uint32_t)G, (uint32_t)P, 1};
    uint64_t dk[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)b};
    uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
    uint32_t bk[4] = {64, 1, 128, 1};
    if (!make_tmap_4d(&prm.tq, q, dq, sq, bq) || !make_tmap_4d(&prm.tk, k, dk, sk, bk))
      return KVPOP_ERR_CUDA;
  }
  prm.S = S;
  prm.nct = (S + P - 1) / P;
  prm.Spad = prm.nct * P;
  prm.H = H;
  prm.G = G;
  int lg = 0;
  while ((1 << lg) < G) ++lg;
  prm.logG = lg;
  prm.P = P;
  prm.w = w;
  prm.nchunk = (prm.nct + kChunkTiles - 1) / kChunkTiles;
  const float sc = scale > 0.0f ? scale : 1.0f / sqrtf((float)D);
  prm.scale_log2 = sc * 1.4426950408889634f;
  prm.lse2 = static_cast<const float*>(workspace);
  prm.acc = target;
  prm.status = device_status_ptr();
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const long long nout = (long long)b * H * S;
  st = cuda_check(cudaMemsetAsync(target, 0, (size_t)nout * sizeof(float), cs), "kvpop_future_target: zero");
  if (st != KVPOP_OK) return st;
  const long long n = (long long)b * H * prm.Spad * G;
  const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
  st = cuda_check(launch_pdl(lse_prep, dim3(blocks), dim3(256), 0, cs, lse, b, H, G, S, prm.Spad,
                             static_cast<float*>(workspace)),
                  "kvpop_future_target: lse prep");
  if (st != KVPOP_OK) return st;
  st = D == 128 ? launch_target<128>(prm, b, H, cs) : launch_target<64>(prm, b, H, cs);
  if (st != KVPOP_OK) return st;
  return cuda_check(launch_pdl(target_finalize, dim3((int)std::min<long long>((nout + 255) / 256, 4096)), dim3(256),
                               0, cs, target, nout),
                    "kvpop_future_target: finalize");
}

// ---------------------------------------------------------------------------
// Allocation-free variant of kvpop_future_target.
//
// Some callers cannot call cudaMalloc: a serving engine whose allocator has
// reserved all device memory up front for its KV pool, or a caller on a path
// where cudaMalloc's implicit device synchronisation is not allowed.  This
// entry point keeps the pass's scratch (the LSE rescaled to log2 units in
// query-tile order) in a file-scope device array instead of caller workspace.
// The array is part of the module image: every GPU that loads the library
// holds these 16 MiB until the process exits.
// ---------------------------------------------------------------------------
namespace kvpop {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB = 4,194,304 floats
static __device__ __align__(256) unsigned char g_target_scratch[kNoAllocScratchBytes];

// Device address of g_target_scratch, looked up once per device with that
// device current (the host-side symbol is only a stand-in, never a device address).
void* target_scratch_ptr(kvpop_status* st) {
  static void* cache[64] = {nullptr};
  static std::mutex mu;
  const int d = current_device();
  if (d < 0 || d >= 64) {
    set_last_error("kvpop_future_target_noalloc: device index %d out of range", d);
    *st = KVPOP_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[d] == nullptr) {
    void* p = nullptr;
    *st = cuda_check(cudaGetSymbolAddress(&p, g_target_scratch),
                     "kvpop_future_target_noalloc: cudaGetSymbolAddress");
    if (*st != KVPOP_OK) return nullptr;
    cache[d] = p;
  }
  *st = KVPOP_OK;
  return cache[d];
}

}  // namespace
}  // namespace kvpop

extern "C" kvpop_status kvpop_future_target_noalloc(const void* q, const void* k, const float* lse,
                                                    int b, int S, int Hq, int H, int D, float scale,
                                                    int w, float* target, kvpop_stream stream) {
  size_t need = 0;
  kvpop_status st = kvpop_future_target_workspace_size(b, S, Hq, H, &need);
  if (st != KVPOP_OK) return st;
  if (need > kvpop::kNoAllocScratchBytes) {
    kvpop::set_last_error(
        "kvpop_future_target_noalloc: needs %zu bytes of scratch (b*H*ceil(S/P)*P*G floats), "
        "above the built-in %zu; use kvpop_future_target with caller workspace",
        need, kvpop::kNoAllocScratchBytes);
    return KVPOP_ERR_UNSUPPORTED;
  }
  void* scratch = kvpop::target_scratch_ptr(&st);
  if (st != KVPOP_OK) return st;
  // Every element of the scratch that the pass reads is written by it first
  // (the LSE re-layout covers all b*H*Spad*G entries), so nothing is cleared.
  return kvpop_future_target(q, k, lse, b, S, Hq, H, D, scale, w, target, scratch,
                             kvpop::kNoAllocScratchBytes, stream);
}
