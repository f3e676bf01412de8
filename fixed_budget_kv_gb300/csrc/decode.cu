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
//      slots once -- K for the G query heads' scores, then V -- through a TMA
//      ring; the two small GEMMs run on warp-level tensor-core MMAs; HBM-bound
//      at 2G flop/byte;
//   3. the last split CTA of each (sequence, head) combines the splits' (max,
//      sum, partial O) into O and the LSE.
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
  int32_t* done_cnt;  // [n, H] split CTAs finished in this step (reset by the last one)
  int* status;        // device status words
  float* part_ml;     // [n, Hq, nsplit, 2]  (max in log2 units, sum)
  float* part_o;      // [n, Hq, nsplit, D]
  // K / V as 3-D bf16 tensors (D, B, n*H); box 64 columns x one 8 KB chunk of
  // slots, 128-byte swizzle; slots past B read as zeros
  CUtensorMap tk, tv;
};

namespace kvpop {
namespace {

constexpr int kSplit = 256;  // slots per attention CTA
constexpr int kUpdThreads = 256;
constexpr int kAttnThreads = 160;  // 4 compute warps + 1 producer warp

__device__ __forceinline__ int* device_status_from(const kvpop_cache& c) { return c.status; }

__device__ __forceinline__ float prio_val(float p) { return p != p ? __int_as_float(0xff800000) : p; }

// worse(a, b): a is a worse long-range token than b (lower priority, or equal and later)
__device__ __forceinline__ bool worse(float va, int pa, float vb, int pb) {
  return va < vb || (va == vb && pa > pb);
}

// One CTA per (sequence, head).  Every global value the step may need -- the
// long-range count, the long-range priorities and positions, the leaving
// token's priority and K/V row, the new K/V row -- is loaded up front in one
// batch, so the kernel costs one memory round trip, a block arg-min and the
// stores.
__global__ void __launch_bounds__(kUpdThreads)
    decode_update(kvpop_cache c, int q, const __nv_bfloat16* __restrict__ k_new,
                  const __nv_bfloat16* __restrict__ v_new, const float* __restrict__ prio_new,
                  int32_t* __restrict__ evicted_pos) {
  constexpr int kBatch = 8;  // long-range entries per thread per pass
  __shared__ float red_v[kUpdThreads / 32];
  __shared__ int red_p[kUpdThreads / 32];
  __shared__ int red_s[kUpdThreads / 32];
  __shared__ int s_dst, s_evicted;
  const int nh = blockIdx.x;  // sequence * H + head
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dep_launch();
  grid_dep_wait();  // nothing is read before the previous kernel has finished
  const int D = c.D, B = c.B, s = c.s, w = c.w, k = c.k;
  const int CH = D / 8;  // 16-byte pieces per row
  const size_t slot0 = (size_t)nh * B;
  uint4* kc = reinterpret_cast<uint4*>(c.kc + slot0 * D);
  uint4* vc = reinterpret_cast<uint4*>(c.vc + slot0 * D);
  int32_t* spos = c.slot_pos + slot0;
  float* sprio = c.slot_prio + slot0;
  const float pin = prio_new[nh];
  // the competing token: u = q - w from the ring, or q itself when w == 0
  const int u = q - w;
  const int ring = w > 0 && q >= s ? s + (q - s) % w : -1;
  const bool compete = q >= s && u >= s;
  // threads [0, CH) hold the new K piece, [CH, 2CH) the new V piece,
  // [2CH, 3CH) the ring's K piece, [3CH, 4CH) the ring's V piece
  const int role = tid < 4 * CH ? tid / CH : 4, piece = tid % CH;
  uint4 row = make_uint4(0, 0, 0, 0);
  if (role == 0) row = reinterpret_cast<const uint4*>(k_new + (size_t)nh * D)[piece];
  if (role == 1) row = reinterpret_cast<const uint4*>(v_new + (size_t)nh * D)[piece];
  if (role == 2 && compete && ring >= 0) row = kc[(size_t)ring * CH + piece];
  if (role == 3 && compete && ring >= 0) row = vc[(size_t)ring * CH + piece];
  if (q < s) {
    // sink
    if (role == 0) kc[(size_t)q * CH + piece] = row;
    if (role == 1) vc[(size_t)q * CH + piece] = row;
    if (tid == 0) {
      spos[q] = q;
      sprio[q] = pin;
      if (evicted_pos) evicted_pos[nh] = -1;
    }
    return;
  }
  int cnt = 0;
  float pu = pin;
  if (compete && k > 0) {
    cnt = c.topk_cnt[nh];
    if (ring >= 0) pu = sprio[ring];
    // worst held long-range token: lowest priority, later position on ties
    float bv = __int_as_float(0x7f800000);
    int bp = -1, bs = -1;
    for (int i0 = tid; i0 < k; i0 += kUpdThreads * kBatch) {
      float vv[kBatch];
      int pp[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {  // all loads of the batch in flight together
        const int i = i0 + j * kUpdThreads;
        vv[j] = i < k ? prio_val(sprio[s + w + i]) : 0.0f;
        pp[j] = i < k ? spos[s + w + i] : -1;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * kUpdThreads;
        if (i < k && (bs < 0 || worse(vv[j], pp[j], bv, bp))) {
          bv = vv[j];
          bp = pp[j];
          bs = s + w + i;
        }
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
      if (cnt < k) {  // a free long-range slot
        s_dst = s + w + cnt;
        s_evicted = -1;
        c.topk_cnt[nh] = cnt + 1;
      } else {
        for (int i = 1; i < kUpdThreads / 32; ++i)
          if (red_s[i] >= 0 && (bs < 0 || worse(red_v[i], red_p[i], bv, bp))) {
            bv = red_v[i];
            bp = red_p[i];
            bs = red_s[i];
          }
        const bool take = prio_val(pu) > bv;  // strictly better than the worst held token
        s_dst = take ? bs : -1;
        s_evicted = take ? bp : u;
      }
    }
    __syncthreads();
  } else if (tid == 0) {
    s_dst = -1;
    s_evicted = compete ? u : -1;  // k == 0: the leaving token is dropped
  }
  if (!(compete && k > 0)) __syncthreads();
  const int dst = s_dst;
  if (dst >= 0) {
    // the competitor's row: the ring's old contents, or the new token when w == 0
    if (w > 0) {
      if (role == 2) kc[(size_t)dst * CH + piece] = row;
      if (role == 3) vc[(size_t)dst * CH + piece] = row;
    } else {
      if (role == 0) kc[(size_t)dst * CH + piece] = row;
      if (role == 1) vc[(size_t)dst * CH + piece] = row;
    }
    if (tid == 0) {
      spos[dst] = u;
      sprio[dst] = pu;
    }
  }
  if (ring >= 0) {
    if (role == 0) kc[(size_t)ring * CH + piece] = row;
    if (role == 1) vc[(size_t)ring * CH + piece] = row;
    if (tid == 0) {
      spos[ring] = q;
      sprio[ring] = pin;
    }
  }
  if (tid == 0 && evicted_pos) evicted_pos[nh] = s_evicted;
}

// One CTA per (split of kSplit slots, KV head, sequence), 5 warps.  Warp 4
// streams the split's K rows and then its V rows through a kStages-deep ring
// of 8 KB chunks with 3-D TMA boxes in the 128-byte-swizzled layout, so every
// CTA keeps kStages chunks of HBM reads in flight.  The G query heads of a KV
// head against a chunk of keys, and the probabilities against a chunk of
// values, are small GEMMs (G x D x 32 keys): warps 0-3 run them with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate; the heads fill the first G of
// 16 rows) fed by conflict-free ldmatrix from the swizzled chunks, which
// keeps the instruction count far below the HBM time.  Softmax over the split
// in fp32.  Empty slots hold finite data (zeros or stale rows) and get weight
// 0.  The last CTA of a (sequence, head) to finish merges the splits' (max,
// sum, partial O).
constexpr int kChunkBytes = 8192;  // one ring chunk: 8 KB of slot rows
constexpr int kStages = 4;         // ring depth (5 CTAs per SM fit)
constexpr int kCompute = 128;      // compute threads (warps 0-3)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// C (16x8 fp32) += A (16x16 bf16, row-major) * B (16x8 bf16, col-major)
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads)
    decode_attn(const __grid_constant__ kvpop_cache c, const __nv_bfloat16* __restrict__ q_new, float scale_log2, __nv_bfloat16* __restrict__ O,
                float* __restrict__ lse) {
  constexpr int NW = kCompute / 32;
  constexpr int DH = D / 64;                     // 64-column halves
  constexpr int kChunk = kChunkBytes / (D * 2);  // slot rows per chunk (32 or 64)
  constexpr int HALF = kChunk * 128;             // bytes of one 64-column half of a chunk
  constexpr int NTW = kChunk / 8 / NW;           // key n-tiles per warp in the score GEMM
  constexpr int DW = D / NW;                     // output columns per warp in the P.V GEMM
  constexpr int NDW = DW / 8;                    // d n-tiles per warp
  constexpr int kPer = kSplit / kCompute;
  static_assert(G <= 8, "at most 8 query heads fill the 16 MMA rows");
  static_assert(NTW >= 1 && NDW % 2 == 0, "tile split");
  extern __shared__ __align__(1024) uint8_t dsm[];  // ring: kStages x 8 KB, 1024-byte aligned
  __shared__ __align__(16) float sct[kSplit * G];   // scores, then weights: [slot][head]
  __shared__ float red[G][NW];
  __shared__ float m_s[G], l_s[G], inv_s[G], lse_s[G];
  __shared__ int s_last;
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ volatile int abort_flag;
  uint8_t* ring = dsm + ((1024 - (smem_u32(dsm) & 1023)) & 1023);
  const uint32_t ring_addr = smem_u32(ring);
  const int sp = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = c.H, B = c.B, Hq = H * G;
  const int nh = n * H + h;
  const int slot_lo = sp * c.split_len;
  const int nslots = min(B, slot_lo + c.split_len) - slot_lo;
  const int nch = (nslots + kChunk - 1) / kChunk;  // chunks of K, then as many of V
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NW);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == NW && lane == 0) {
    tma_prefetch_desc(&c.tk);
    tma_prefetch_desc(&c.tv);
  }
  grid_dep_launch();
  grid_dep_wait();  // the update of this step has finished: slots, K and V are final
  __syncthreads();
  bool ok = true;
  if (warp == NW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      for (int i = 0; i < 2 * nch; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, &abort_flag)) {
          ok = false;
          abort_flag = 1;
          break;
        }
        const bool is_k = i < nch;
        const int ci = is_k ? i : i - nch;
        mbar_arrive_expect_tx(&full[st], kChunkBytes);
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(ring + st * kChunkBytes + dh * HALF, is_k ? &c.tk : &c.tv, &full[st], dh * 64,
                      slot_lo + ci * kChunk, nh, 0);
      }
    }
  } else {
    // ---------------------------------------------------------------- compute
    const int g = lane >> 2, t = lane & 3;  // MMA fragment coordinates
    const int32_t* spos = c.slot_pos + (size_t)nh * B + slot_lo;
    // Q as MMA A fragments: row g < G holds query head h*G+g, columns are d
    uint32_t aq[D / 16][2];
    {
      const __nv_bfloat16* qrow = q_new + ((size_t)n * Hq + h * G + (g < G ? g : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        aq[ks][0] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t) : 0u;
        aq[ks][1] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * t) : 0u;
      }
    }
    bool occ[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = tid + j * kCompute;
      occ[j] = r < nslots && spos[r] >= 0;
    }
    // phase 1: S = Q K^T per chunk; warp w takes key n-tiles w*NTW .. w*NTW+NTW-1
    for (int ci = 0; ci < nch; ++ci) {
      const int st = ci % kStages;
      if (ok && !mbar_wait(&full[st], (ci / kStages) & 1, &abort_flag)) {
        ok = false;
        abort_flag = 1;
      }
      const uint32_t cb = ring_addr + st * kChunkBytes;
      float sacc[NTW][4];
#pragma unroll
      for (int j = 0; j < NTW; ++j) {
        sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
        const int r = (warp * NTW + j) * 8 + (lane & 7);  // key row this lane addresses
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          const int cc16 = 2 * ks + (lane >> 3);  // 16-byte column chunk 0 .. D/8-1
          const uint32_t addr = cb + (cc16 >> 3) * HALF + r * 128 + (((cc16 & 7) ^ (r & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma16816(sacc[j], aq[ks][0], 0u, aq[ks][1], 0u, b0, b1);
          mma16816(sacc[j], aq[ks + 1][0], 0u, aq[ks + 1][1], 0u, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (g < G) {
#pragma unroll
        for (int j = 0; j < NTW; ++j) {
          const int key = ci * kChunk + (warp * NTW + j) * 8 + 2 * t;
          if (key < nslots) sct[key * G + g] = sacc[j][0] * scale_log2;
          if (key + 1 < nslots) sct[(key + 1) * G + g] = sacc[j][1] * scale_log2;
        }
      }
    }
    named_barrier_sync(1, kCompute);
    // phase 2: per-head max and sum over the split; scores become weights
    {
      float m[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) m[gg] = __int_as_float(0xff800000);
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (occ[j]) {
#pragma unroll
          for (int gg = 0; gg < G; ++gg) m[gg] = fmaxf(m[gg], sct[(tid + j * kCompute) * G + gg]);
        }
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        for (int o = 16; o > 0; o >>= 1) m[gg] = fmaxf(m[gg], __shfl_xor_sync(0xffffffffu, m[gg], o));
        if (lane == 0) red[gg][warp] = m[gg];
      }
    }
    named_barrier_sync(1, kCompute);
    if (tid < G) {
      float m = red[tid][0];
      for (int i = 1; i < NW; ++i) m = fmaxf(m, red[tid][i]);
      m_s[tid] = m;
    }
    named_barrier_sync(1, kCompute);
    {
      float l[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) l[gg] = 0.f;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int r = tid + j * kCompute;
        if (r >= nslots) break;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float mg = m_s[gg];
          const float e = (occ[j] && mg != __int_as_float(0xff800000)) ? ex2_approx(sct[r * G + gg] - mg) : 0.f;
          sct[r * G + gg] = e;
          l[gg] += e;
        }
      }
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        for (int o = 16; o > 0; o >>= 1) l[gg] += __shfl_xor_sync(0xffffffffu, l[gg], o);
        if (lane == 0) red[gg][warp] = l[gg];
      }
    }
    named_barrier_sync(1, kCompute);
    if (tid < G) {
      float l = 0.f;
      for (int i = 0; i < NW; ++i) l += red[tid][i];
      l_s[tid] = l;
    }
    // phase 3: O = P V per chunk; warp w owns output columns w*DW .. w*DW+DW-1
    float oacc[NDW][4];
#pragma unroll
    for (int j = 0; j < NDW; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    for (int ci = 0; ci < nch; ++ci) {
      const int i = nch + ci;
      const int st = i % kStages;
      if (ok && !mbar_wait(&full[st], (i / kStages) & 1, &abort_flag)) {
        ok = false;
        abort_flag = 1;
      }
      const uint32_t cb = ring_addr + st * kChunkBytes;
#pragma unroll
      for (int kk = 0; kk < kChunk; kk += 16) {
        // A: probabilities of heads g (rows) for keys kk .. kk+15 (columns), bf16
        uint32_t a0 = 0u, a2 = 0u;
        if (g < G) {
          const int k0 = ci * kChunk + kk + 2 * t;
          const float p0 = k0 < nslots ? sct[k0 * G + g] : 0.f;
          const float p1 = k0 + 1 < nslots ? sct[(k0 + 1) * G + g] : 0.f;
          const float p8 = k0 + 8 < nslots ? sct[(k0 + 8) * G + g] : 0.f;
          const float p9 = k0 + 9 < nslots ? sct[(k0 + 9) * G + g] : 0.f;
          a0 = pack_bf16x2(p0, p1);
          a2 = pack_bf16x2(p8, p9);
        }
        const int r = kk + (lane & 7) + ((lane >> 3) & 1) * 8;  // value row this lane addresses
#pragma unroll
        for (int j = 0; j < NDW; j += 2) {
          const int cc16 = (warp * DW + j * 8) / 8 + (lane >> 4);
          const uint32_t addr = cb + (cc16 >> 3) * HALF + r * 128 + (((cc16 & 7) ^ (r & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma16816(oacc[j], a0, 0u, a2, 0u, b0, b1);
          mma16816(oacc[j + 1], a0, 0u, a2, 0u, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // partial O: lane (g, t) holds O[g][d = warp*DW + j*8 + 2t, +1]
    if (g < G) {
      float* po = c.part_o + (((size_t)n * Hq + h * G + g) * c.nsplit + sp) * D + warp * DW + 2 * t;
#pragma unroll
      for (int j = 0; j < NDW; ++j) *reinterpret_cast<float2*>(po + j * 8) = make_float2(oacc[j][0], oacc[j][1]);
    }
    if (tid < G) {
      float* ml = c.part_ml + (((size_t)n * Hq + h * G + tid) * c.nsplit + sp) * 2;
      ml[0] = m_s[tid];
      ml[1] = l_s[tid];
    }
  }
  // the last CTA of this (sequence, head) to finish merges all splits
  __threadfence();
  __syncthreads();
  if (!ok) report_error(device_status_from(c), KVPOP_ERR_TIMEOUT, SITE_DECODE, 1);
  if (tid == 0) {
    const int prev = atomicAdd(c.done_cnt + nh, 1);
    s_last = prev == c.nsplit - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int ns = c.nsplit;
  float* wgt = sct;  // [G][ns] weight of each split
  const size_t row0 = (size_t)n * Hq + h * G;
  for (int i = tid; i < G * ns; i += kAttnThreads) wgt[i] = __ldcg(c.part_ml + (row0 * ns + i) * 2);
  __syncthreads();
  if (tid < G) {
    float M = __int_as_float(0xff800000);
    for (int i = 0; i < ns; ++i) M = fmaxf(M, wgt[tid * ns + i]);
    float Lsum = 0.f;
    for (int i = 0; i < ns; ++i) {
      const float mi = wgt[tid * ns + i];
      const float wi = mi != __int_as_float(0xff800000) ? ex2_approx(mi - M) : 0.f;
      Lsum += __ldcg(c.part_ml + ((row0 + tid) * ns + i) * 2 + 1) * wi;
      wgt[tid * ns + i] = wi;
    }
    inv_s[tid] = Lsum > 0.f ? 1.0f / Lsum : 0.f;
    lse_s[tid] = Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : __int_as_float(0xff800000);
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int gg = i / D, d = i % D;
    const float* po = c.part_o + ((row0 + gg) * ns) * D + d;
    float o = 0.f;
#pragma unroll 8
    for (int sidx = 0; sidx < ns; ++sidx) o += __ldcg(po + (size_t)sidx * D) * wgt[gg * ns + sidx];
    O[(row0 + gg) * D + d] = __float2bfloat16_rn(o * inv_s[gg]);
  }
  if (tid < G) lse[row0 + tid] = lse_s[tid];
  if (tid == 0) c.done_cnt[nh] = 0;  // ready for the next step
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

template <int D, int G>
kvpop_status launch_attn_g(const kvpop_cache& c, const void* q_new, float sl2, void* O, float* lse,
                           cudaStream_t cs) {
  auto kern = decode_attn<D, G>;
  const int smem = kStages * kChunkBytes + 1024;  // + alignment slack for the swizzled ring
  kvpop_status st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                               "kvpop_decode_step: smem attribute");
  if (st != KVPOP_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.nsplit, c.H, c.n);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, kern, c, (const __nv_bfloat16*)q_new, sl2, (__nv_bfloat16*)O, lse),
                    "kvpop_decode_step: attention launch");
}

template <int D>
kvpop_status launch_attn(const kvpop_cache& c, const void* q_new, float sl2, void* O, float* lse,
                         cudaStream_t cs) {
  switch (c.G) {
    case 1: return launch_attn_g<D, 1>(c, q_new, sl2, O, lse, cs);
    case 2: return launch_attn_g<D, 2>(c, q_new, sl2, O, lse, cs);
    case 4: return launch_attn_g<D, 4>(c, q_new, sl2, O, lse, cs);
    case 8: return launch_attn_g<D, 8>(c, q_new, sl2, O, lse, cs);
    default:
      set_last_error("kvpop_decode_step: G=%d unsupported (1, 2, 4 or 8)", c.G);
      return KVPOP_ERR_UNSUPPORTED;
  }
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
      (long long)bud.s + bud.w + bud.k > (long long)kSplit * kSplit) {  // the merge holds kSplit splits
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
  c->status = device_status_ptr();
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
  alloc((void**)&c->done_cnt, (size_t)n * H * 4, "kvpop_cache_create: split counters");
  alloc((void**)&c->part_ml, (size_t)n * Hq * c->nsplit * 2 * 4, "kvpop_cache_create: partials");
  alloc((void**)&c->part_o, (size_t)n * Hq * c->nsplit * D * 4, "kvpop_cache_create: partials");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->slot_pos, 0xff, slots * 4), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->topk_cnt, 0, (size_t)n * H * 4), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->done_cnt, 0, (size_t)n * H * 4), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->kc, 0, slots * D * 2), "kvpop_cache_create: init");
  if (st == KVPOP_OK) st = cuda_check(cudaMemset(c->vc, 0, slots * D * 2), "kvpop_cache_create: init");
  if (st == KVPOP_OK) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)c->B, (uint64_t)n * H, 1};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)c->B * D * 2, (uint64_t)n * H * c->B * D * 2};
    const uint32_t box[4] = {64, (uint32_t)(kChunkBytes / (D * 2)), 1, 1};
    if (!make_tmap_4d(&c->tk, c->kc, dims, strides, box) || !make_tmap_4d(&c->tv, c->vc, dims, strides, box))
      st = KVPOP_ERR_CUDA;
  }
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
  cudaFree(c->done_cnt);
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
  // both kernels use programmatic dependent launch: each starts while the
  // previous kernel of the stream drains and waits for it before any read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c->n * c->H);
  cfg.blockDim = dim3(kUpdThreads);
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  kvpop_status st = cuda_check(cudaLaunchKernelEx(&cfg, decode_update, *c, q, (const __nv_bfloat16*)k_new,
                                                  (const __nv_bfloat16*)v_new, prio_new, evicted_pos),
                               "kvpop_decode_step: update launch");
  if (st != KVPOP_OK) return st;
  const float sl2 = 1.4426950408889634f / sqrtf((float)c->D);
  st = c->D == 128 ? launch_attn<128>(*c, q_new, sl2, O, lse, cs) : launch_attn<64>(*c, q_new, sl2, O, lse, cs);
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
