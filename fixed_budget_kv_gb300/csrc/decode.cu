// Fixed-budget decode cache ("KVpop ... 精读笔记", sections 2.4 and 3.3;
// "KVpop — 基于预测性在线剪枝的键值缓存压缩", section 2.4).
//
// Each (sequence, KV head) holds B = s + w + k slots: [0, s) sinks, [s, s+w) a
// ring for the protected window (position p >= s in slot s + (p - s) mod w),
// [s+w, B) the long-range set.  A decode step at position q:
//   1. update (one CTA per sequence x head): the token u = q - w leaving the
//      window takes a free long-range slot, or replaces the worst held token
//      (lowest priority, later position on ties) when its priority is strictly
//      greater, or is dropped; then token q is written into the ring;
//   2. split attention (flash-decoding): each CTA reads a contiguous range of
//      slots once -- K for the G query heads' scores, then V -- with 16-byte
//      coalesced loads; HBM-bound at 4 flop/byte;
//   3. combine the splits' (max, sum, partial O) into O and the LSE.
#include "common.cuh"

struct kvpop_cache {
  int n, H, G, D, s, w, k, B;
  int q_next;
  int nsplit, split_len;
  int device;
  __nv_bfloat16* kc;  // [n, H, B, D]
  __nv_bfloat16* vc;
  int32_t* slot_pos;  // [n, H, B]
  float* slot_prio;   // [n, H, B]
  int32_t* topk_cnt;  // [n, H]
  float* part_ml;     // [n, Hq, nsplit, 2]  (max in log2 units, sum)
  float* part_o;      // [n, Hq, nsplit, D]
};

namespace kvpop {
namespace {

constexpr int kSplit = 256;
constexpr int kUpdThreads = 256;
constexpr int kAttnThreads = 128;

__device__ __forceinline__ float prio_val(float p) { return p != p ? __int_as_float(0xff800000) : p; }

// worse(a, b): a is a worse long-range token than b (lower priority, or equal and later)
__device__ __forceinline__ bool worse(float va, int pa, float vb, int pb) {
  return va < vb || (va == vb && pa > pb);
}

__device__ __forceinline__ void copy_row(__nv_bfloat16* dst, const __nv_bfloat16* src, int D, int tid,
                                         int nthreads) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = tid; i < D / 8; i += nthreads) d[i] = s[i];
}

__global__ void __launch_bounds__(kUpdThreads)
    decode_update(kvpop_cache c, int q, const __nv_bfloat16* __restrict__ k_new,
                  const __nv_bfloat16* __restrict__ v_new, const float* __restrict__ prio_new,
                  int32_t* __restrict__ evicted_pos) {
  __shared__ float red_v[kUpdThreads / 32];
  __shared__ int red_p[kUpdThreads / 32];
  __shared__ int red_s[kUpdThreads / 32];
  __shared__ int s_dst, s_evicted, s_cnt;
  const int nh = blockIdx.x;  // sequence * H + head
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = c.D, B = c.B, s = c.s, w = c.w, k = c.k;
  const size_t slot0 = (size_t)nh * B;
  __nv_bfloat16* kc = c.kc + slot0 * D;
  __nv_bfloat16* vc = c.vc + slot0 * D;
  int32_t* spos = c.slot_pos + slot0;
  float* sprio = c.slot_prio + slot0;
  const __nv_bfloat16* kin = k_new + (size_t)nh * D;
  const __nv_bfloat16* vin = v_new + (size_t)nh * D;
  const float pin = prio_new[nh];

  if (q < s) {
    // sink
    copy_row(kc + (size_t)q * D, kin, D, tid, kUpdThreads);
    copy_row(vc + (size_t)q * D, vin, D, tid, kUpdThreads);
    if (tid == 0) {
      spos[q] = q;
      sprio[q] = pin;
      if (evicted_pos) evicted_pos[nh] = -1;
    }
    return;
  }
  // the competing token: u = q - w from the ring, or q itself when w == 0
  const int u = q - w;
  const int ring = w > 0 ? s + (q - s) % w : -1;
  if (tid == 0) {
    s_dst = -1;
    s_evicted = -1;
    s_cnt = c.topk_cnt[nh];
  }
  __syncthreads();
  if (u >= s) {
    const float pu = w > 0 ? sprio[ring] : pin;
    const int cnt = s_cnt;  // block-uniform
    if (k == 0) {
      if (tid == 0) s_evicted = u;
    } else if (cnt < k) {
      if (tid == 0) {
        s_dst = s + w + cnt;
        c.topk_cnt[nh] = cnt + 1;
      }
    } else {
      // worst held long-range token
      float bv = __int_as_float(0x7f800000);
      int bp = -1, bs = -1;
      for (int i = tid; i < k; i += kUpdThreads) {
        const int sl = s + w + i;
        const float v = prio_val(sprio[sl]);
        const int ps = spos[sl];
        if (bs < 0 || worse(v, ps, bv, bp)) {
          bv = v;
          bp = ps;
          bs = sl;
        }
      }
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (os >= 0 && (bs < 0 || worse(ov, op, bv, bp))) {
          bv = ov;
          bp = op;
          bs = os;
        }
      }
      if (lane == 0) {
        red_v[warp] = bv;
        red_p[warp] = bp;
        red_s[warp] = bs;
      }
      __syncthreads();
      if (tid == 0) {
        for (int i = 1; i < kUpdThreads / 32; ++i)
          if (red_s[i] >= 0 && (bs < 0 || worse(red_v[i], red_p[i], bv, bp))) {
            bv = red_v[i];
            bp = red_p[i];
            bs = red_s[i];
          }
        if (prio_val(pu) > bv) {  // strictly better than the worst held token
          s_dst = bs;
          s_evicted = bp;
        } else {
          s_evicted = u;
        }
      }
    }
    __syncthreads();
    const int dst = s_dst;
    if (dst >= 0) {
      if (w > 0) {
        copy_row(kc + (size_t)dst * D, kc + (size_t)ring * D, D, tid, kUpdThreads);
        copy_row(vc + (size_t)dst * D, vc + (size_t)ring * D, D, tid, kUpdThreads);
      } else {
        copy_row(kc + (size_t)dst * D, kin, D, tid, kUpdThreads);
        copy_row(vc + (size_t)dst * D, vin, D, tid, kUpdThreads);
      }
      if (tid == 0) {
        spos[dst] = u;
        sprio[dst] = pu;
      }
    }
  }
  __syncthreads();
  if (w > 0) {
    copy_row(kc + (size_t)ring * D, kin, D, tid, kUpdThreads);
    copy_row(vc + (size_t)ring * D, vin, D, tid, kUpdThreads);
    if (tid == 0) {
      spos[ring] = q;
      sprio[ring] = pin;
    }
  }
  if (tid == 0 && evicted_pos) evicted_pos[nh] = s_evicted;
}

// One CTA per (split, KV head, sequence).  D / 8 lanes cover one slot row with
// 16-byte loads; G query heads share every row.
template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads)
    decode_attn(kvpop_cache c, const __nv_bfloat16* __restrict__ q_new, float scale_log2) {
  constexpr int LPR = D / 8;                 // lanes per row
  constexpr int RPW = 32 / LPR;              // rows per warp step
  constexpr int NW = kAttnThreads / 32;
  __shared__ float sc[G][kSplit];
  __shared__ float red[G][NW];
  __shared__ float m_s[G], l_s[G];
  __shared__ float opart[kAttnThreads / LPR][G][D];
  const int sp = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = c.H, B = c.B;
  const int nh = n * H + h;
  const int slot_lo = sp * c.split_len;
  const int slot_hi = min(B, slot_lo + c.split_len);
  const int nslots = slot_hi - slot_lo;
  const __nv_bfloat16* kc = c.kc + ((size_t)nh * B) * D;
  const __nv_bfloat16* vc = c.vc + ((size_t)nh * B) * D;
  const int32_t* spos = c.slot_pos + (size_t)nh * B;
  const int sub = lane / LPR, li = lane % LPR;

  // query chunk of this lane for each head
  float qf[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 raw = *reinterpret_cast<const uint4*>(q_new + ((size_t)n * H * G + h * G + g) * D + li * 8);
    const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(pr[e]);
      qf[g][2 * e] = f.x * scale_log2;
      qf[g][2 * e + 1] = f.y * scale_log2;
    }
  }
  // phase 1: scores (log2 units)
  for (int r0 = warp * RPW; r0 < nslots; r0 += NW * RPW) {
    const int r = r0 + sub;
    const bool valid = r < nslots && spos[slot_lo + r] >= 0;
    float part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = 0.f;
    if (valid) {
      const uint4 raw = *reinterpret_cast<const uint4*>(kc + (size_t)(slot_lo + r) * D + li * 8);
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(pr[e]);
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = fmaf(f.x, qf[g][2 * e], fmaf(f.y, qf[g][2 * e + 1], part[g]));
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) part[g] += __shfl_xor_sync(0xffffffffu, part[g], o);
    }
    if (li == 0 && r < nslots) {
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g][r] = valid ? part[g] : __int_as_float(0xff800000);
    }
  }
  __syncthreads();
  // phase 2: per-head max and sum
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float m = __int_as_float(0xff800000);
    for (int r = tid; r < nslots; r += kAttnThreads) m = fmaxf(m, sc[g][r]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[g][warp] = m;
  }
  __syncthreads();
  if (tid < G) {
    float m = red[tid][0];
    for (int i = 1; i < NW; ++i) m = fmaxf(m, red[tid][i]);
    m_s[tid] = m;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = m_s[g];
    float l = 0.f;
    if (m != __int_as_float(0xff800000)) {
      for (int r = tid; r < nslots; r += kAttnThreads) {
        const float e = ex2_approx(sc[g][r] - m);
        sc[g][r] = e;
        l += e;
      }
    } else {
      for (int r = tid; r < nslots; r += kAttnThreads) sc[g][r] = 0.f;
    }
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) red[g][warp] = l;
  }
  __syncthreads();
  if (tid < G) {
    float l = 0.f;
    for (int i = 0; i < NW; ++i) l += red[tid][i];
    l_s[tid] = l;
  }
  // phase 3: partial O = sum_r p_r v_r
  float acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  const int grp = tid / LPR;                 // row group of this thread
  constexpr int NG = kAttnThreads / LPR;
  for (int r = grp; r < nslots; r += NG) {
    float pr_[G];
    bool any = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      pr_[g] = sc[g][r];
      any |= pr_[g] != 0.f;
    }
    if (!any) continue;
    const uint4 raw = *reinterpret_cast<const uint4*>(vc + (size_t)(slot_lo + r) * D + li * 8);
    const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(pv[e]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        acc[g][2 * e] = fmaf(pr_[g], f.x, acc[g][2 * e]);
        acc[g][2 * e + 1] = fmaf(pr_[g], f.y, acc[g][2 * e + 1]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) opart[grp][g][li * 8 + e] = acc[g][e];
  __syncthreads();
  const int Hq = H * G;
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int g = i / D, d = i % D;
    float o = 0.f;
#pragma unroll
    for (int r = 0; r < NG; ++r) o += opart[r][g][d];
    c.part_o[(((size_t)n * Hq + h * G + g) * c.nsplit + sp) * D + d] = o;
  }
  if (tid < G) {
    float* ml = c.part_ml + (((size_t)n * Hq + h * G + tid) * c.nsplit + sp) * 2;
    ml[0] = m_s[tid];
    ml[1] = l_s[tid];
  }
}

__global__ void decode_combine(kvpop_cache c, __nv_bfloat16* __restrict__ O, float* __restrict__ lse) {
  const int row = blockIdx.x;  // n * Hq + j
  const int D = c.D, ns = c.nsplit;
  const float* ml = c.part_ml + (size_t)row * ns * 2;
  float M = __int_as_float(0xff800000);
  for (int i = 0; i < ns; ++i) M = fmaxf(M, ml[2 * i]);
  float Lsum = 0.f;
  for (int i = 0; i < ns; ++i)
    if (ml[2 * i] != __int_as_float(0xff800000)) Lsum += ml[2 * i + 1] * ex2_approx(ml[2 * i] - M);
  const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float o = 0.f;
    for (int i = 0; i < ns; ++i)
      if (ml[2 * i] != __int_as_float(0xff800000))
        o += c.part_o[((size_t)row * ns + i) * D + d] * ex2_approx(ml[2 * i] - M);
    O[(size_t)row * D + d] = __float2bfloat16_rn(o * inv);
  }
  if (threadIdx.x == 0)
    lse[row] = Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : __int_as_float(0xff800000);
}

// Prefill: the retained set of row P-1 from evict_at over the prefix.
__global__ void __launch_bounds__(256)
    cache_prefill_kernel(kvpop_cache c, const __nv_bfloat16* __restrict__ k,
                         const __nv_bfloat16* __restrict__ v, const float* __restrict__ prio, int P,
                         const int32_t* __restrict__ evict_at) {
  __shared__ int wtot[8];
  __shared__ int running;
  const int nh = blockIdx.x, n = nh / c.H, h = nh % c.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = c.D, B = c.B, s = c.s, w = c.w, H = c.H;
  __nv_bfloat16* kc = c.kc + (size_t)nh * B * D;
  __nv_bfloat16* vc = c.vc + (size_t)nh * B * D;
  int32_t* spos = c.slot_pos + (size_t)nh * B;
  float* sprio = c.slot_prio + (size_t)nh * B;
  const float* pr = prio + (size_t)nh * P;
  const int32_t* ev = evict_at + (size_t)nh * P;
  const int last = P - 1;
  auto put = [&](int slot, int t) {
    const __nv_bfloat16* ks = k + (((size_t)n * P + t) * H + h) * D;
    const __nv_bfloat16* vs = v + (((size_t)n * P + t) * H + h) * D;
    for (int i = lane; i < D / 8; i += 32) {
      reinterpret_cast<uint4*>(kc + (size_t)slot * D)[i] = reinterpret_cast<const uint4*>(ks)[i];
      reinterpret_cast<uint4*>(vc + (size_t)slot * D)[i] = reinterpret_cast<const uint4*>(vs)[i];
    }
    if (lane == 0) {
      spos[slot] = t;
      sprio[slot] = pr[t];
    }
  };
  // sinks and window: one warp per token
  const int nsink = min(s, P);
  for (int t = warp; t < nsink; t += 8) put(t, t);
  if (w > 0)
    for (int t = max(s, P - w) + warp; t < P; t += 8) put(s + (t - s) % w, t);
  // long-range: tokens of E(P-1) still held at row P-1, in position order
  if (tid == 0) running = 0;
  __syncthreads();
  const int hi = last - w;  // E(P-1) = [s, P-1-w]
  for (int c0 = s; c0 <= hi; c0 += 256) {
    const int t = c0 + tid;
    const bool keep = t <= hi && ev[t] > last;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) wtot[warp] = __popc(bal);
    __syncthreads();
    int before = running;
    for (int i = 0; i < warp; ++i) before += wtot[i];
    before += __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int i = 0; i < 8; ++i) tot += wtot[i];
      running += tot;
    }
    // copy rows of the kept tokens (one thread per row, plain 16-byte copies)
    if (keep && before < c.k) {
      const int slot = s + w + before;
      const __nv_bfloat16* ks = k + (((size_t)n * P + t) * H + h) * D;
      const __nv_bfloat16* vs = v + (((size_t)n * P + t) * H + h) * D;
      for (int i = 0; i < D / 8; ++i) {
        reinterpret_cast<uint4*>(kc + (size_t)slot * D)[i] = reinterpret_cast<const uint4*>(ks)[i];
        reinterpret_cast<uint4*>(vc + (size_t)slot * D)[i] = reinterpret_cast<const uint4*>(vs)[i];
      }
      spos[slot] = t;
      sprio[slot] = pr[t];
    }
    __syncthreads();
  }
  if (tid == 0) c.topk_cnt[nh] = min(running, c.k);
}

template <int D>
kvpop_status launch_attn(const kvpop_cache& c, const void* q_new, float sl2, cudaStream_t cs) {
  dim3 grid(c.nsplit, c.H, c.n);
  switch (c.G) {
    case 1: decode_attn<D, 1><<<grid, kAttnThreads, 0, cs>>>(c, (const __nv_bfloat16*)q_new, sl2); break;
    case 2: decode_attn<D, 2><<<grid, kAttnThreads, 0, cs>>>(c, (const __nv_bfloat16*)q_new, sl2); break;
    case 4: decode_attn<D, 4><<<grid, kAttnThreads, 0, cs>>>(c, (const __nv_bfloat16*)q_new, sl2); break;
    case 8: decode_attn<D, 8><<<grid, kAttnThreads, 0, cs>>>(c, (const __nv_bfloat16*)q_new, sl2); break;
    default:
      set_last_error("kvpop_decode_step: G=%d unsupported (1, 2, 4 or 8)", c.G);
      return KVPOP_ERR_UNSUPPORTED;
  }
  return cuda_check(cudaGetLastError(), "kvpop_decode_step: attention launch");
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_cache_create(int n, int H, int G, int D, kvpop_budget bud,
                                           kvpop_cache** out) {
  if (!out || n <= 0 || H <= 0 || G <= 0) {
    set_last_error("kvpop_cache_create: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (bud.s < 0 || bud.w < 0 || bud.k < 0 || (long long)bud.s + bud.w + bud.k < 1 ||
      (long long)bud.s + bud.w + bud.k > (1 << 24)) {
    set_last_error("kvpop_cache_create: invalid budget");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (D != 64 && D != 128) {
    set_last_error("kvpop_cache_create: D=%d unsupported (64 or 128)", D);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (G != 1 && G != 2 && G != 4 && G != 8) {
    set_last_error("kvpop_cache_create: G=%d unsupported (1, 2, 4 or 8)", G);
    return KVPOP_ERR_UNSUPPORTED;
  }
  if ((long long)n * H > 65535 || H > 65535 || n > 65535) {
    set_last_error("kvpop_cache_create: n*H too large");
    return KVPOP_ERR_UNSUPPORTED;
  }
  kvpop_cache* c = new kvpop_cache();
  c->n = n;
  c->H = H;
  c->G = G;
  c->D = D;
  c->s = bud.s;
  c->w = bud.w;
  c->k = bud.k;
  c->B = bud.s + bud.w + bud.k;
  c->q_next = 0;
  c->split_len = kSplit;
  c->nsplit = (c->B + kSplit - 1) / kSplit;
  c->device = current_device();
  const size_t slots = (size_t)n * H * c->B;
  const size_t Hq = (size_t)H * G;
  kvpop_status st = KVPOP_OK;
  auto alloc = [&](void** p, size_t bytes, const char* what) {
    if (st == KVPOP_OK) st = cuda_check(cudaMalloc(p, bytes), what);
  };
  alloc((void**)&c->kc, slots * D * 2, "kvpop_cache_create: K");
  alloc((void**)&c->vc, slots * D * 2, "kvpop_cache_create: V");
  alloc((void**)&c->slot_pos, slots * 4, "kvpop_cache_create: slot_pos");
  alloc((void**)&c->slot_prio, slots * 4, "kvpop_cache_create: slot_prio");
  alloc((void**)&c->topk_cnt, (size_t)n * H * 4, "kvpop_cache_create: count");
  alloc((void**)&c->part_ml, (size_t)n * Hq * c->nsplit * 2 * 4, "kvpop_cache_create: partials");
  alloc((void**)&c->part_o, (size_t)n * Hq * c->nsplit * D * 4, "kvpop_cache_create: partials");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->slot_pos, 0xff, slots * 4), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->topk_cnt, 0, (size_t)n * H * 4), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->kc, 0, slots * D * 2), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->vc, 0, slots * D * 2), "kvpop_cache_create: init");
  if (st != KVPOP_OK) {
    kvpop_cache_destroy(c);
    return st;
  }
  *out = c;
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_cache_destroy(kvpop_cache* c) {
  if (!c) return KVPOP_OK;
  cudaFree(c->kc);
  cudaFree(c->vc);
  cudaFree(c->slot_pos);
  cudaFree(c->slot_prio);
  cudaFree(c->topk_cnt);
  cudaFree(c->part_ml);
  cudaFree(c->part_o);
  delete c;
  return KVPOP_OK;
}

extern "C" kvpop_status kvpop_cache_prefill(kvpop_cache* c, const void* k, const void* v,
                                            const float* prio, int P, const int32_t* evict_at,
                                            kvpop_stream stream) {
  if (!c || !k || !v || !prio || !evict_at || P <= 0) {
    set_last_error("kvpop_cache_prefill: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) != 0) {
    set_last_error("kvpop_cache_prefill: k and v must be 16-byte aligned");
    return KVPOP_ERR_UNSUPPORTED;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t slots = (size_t)c->n * c->H * c->B;
  kvpop_status st = cuda_check(cudaMemsetAsync(c->slot_pos, 0xff, slots * 4, cs), "prefill reset");
  if (st != KVPOP_OK) return st;
  cache_prefill_kernel<<<c->n * c->H, 256, 0, cs>>>(*c, (const __nv_bfloat16*)k,
                                                    (const __nv_bfloat16*)v, prio, P, evict_at);
  st = cuda_check(cudaGetLastError(), "kvpop_cache_prefill: launch");
  if (st == KVPOP_OK) c->q_next = P;
  return st;
}

extern "C" kvpop_status kvpop_decode_step(kvpop_cache* c, const void* q_new, const void* k_new,
                                          const void* v_new, const float* prio_new, void* O,
                                          float* lse, int32_t* evicted_pos, kvpop_stream stream) {
  if (!c || !q_new || !k_new || !v_new || !prio_new || !O || !lse) {
    set_last_error("kvpop_decode_step: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  const uintptr_t am = reinterpret_cast<uintptr_t>(q_new) | reinterpret_cast<uintptr_t>(k_new) |
                       reinterpret_cast<uintptr_t>(v_new);
  if (am & 15) {
    set_last_error("kvpop_decode_step: q_new, k_new, v_new must be 16-byte aligned");
    return KVPOP_ERR_UNSUPPORTED;
  }
  if (c->q_next == 0x7fffffff) {
    set_last_error("kvpop_decode_step: position overflow");
    return KVPOP_ERR_INVALID_ARG;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int q = c->q_next;
  decode_update<<<c->n * c->H, kUpdThreads, 0, cs>>>(*c, q, (const __nv_bfloat16*)k_new,
                                                     (const __nv_bfloat16*)v_new, prio_new,
                                                     evicted_pos);
  kvpop_status st = cuda_check(cudaGetLastError(), "kvpop_decode_step: update launch");
  if (st != KVPOP_OK) return st;
  const float sl2 = 1.4426950408889634f / sqrtf((float)c->D);
  st = c->D == 128 ? launch_attn<128>(*c, q_new, sl2, cs) : launch_attn<64>(*c, q_new, sl2, cs);
  if (st != KVPOP_OK) return st;
  decode_combine<<<c->n * c->H * c->G, 128, 0, cs>>>(*c, (__nv_bfloat16*)O, lse);
  st = cuda_check(cudaGetLastError(), "kvpop_decode_step: combine launch");
  if (st == KVPOP_OK) c->q_next = q + 1;
  return st;
}

extern "C" kvpop_status kvpop_cache_slots(const kvpop_cache* c, int32_t* slot_pos,
                                          kvpop_stream stream) {
  if (!c || !slot_pos) {
    set_last_error("kvpop_cache_slots: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  return cuda_check(cudaMemcpyAsync(slot_pos, c->slot_pos, (size_t)c->n * c->H * c->B * 4,
                                    cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)),
                    "kvpop_cache_slots: copy");
}

extern "C" kvpop_status kvpop_cache_position(const kvpop_cache* c, int32_t* q_next) {
  if (!c || !q_next) {
    set_last_error("kvpop_cache_position: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  *q_next = c->q_next;
  return KVPOP_OK;
}
