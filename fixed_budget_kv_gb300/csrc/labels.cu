// Training-side passes built on the future-attention target ("KVpop ... 精读笔记",
// section 2.2):
//   kvpop_target_normalize -- r_t = log(eps + (1/G) sum_g m_t^g), m_t^g the
//                             future mass averaged over its N_t = S - t - w queries;
//   kvpop_teacher_labels   -- per row q, the teacher's top-k of E(q) = {s..q-w}
//                             under the decayed score r_t + floor((q-t)/n) log gamma,
//                             the cutoff t_bnd the leaving token t_new = q - w has
//                             to beat, and y = +1 (kept) / -1 (dropped);
//   kvpop_boundary_loss    -- the pairwise logistic loss on (t_new, t_bnd) with the
//                             same decay on the predicted scores, and its gradient.
//
// Labels: one CTA per (64-row chunk, batch x head) walks its rows; per row the
// k-th best "other" token is found among the candidates by their 64-bit keys
// (decayed score in order-preserving form, then the inverted index so that the
// lower index wins ties).  The CTA carries a band of scores around the cutoff
// from row to row and re-scores only the candidates whose score changed; full
// rows count against the previous cutoff and, failing that, take a radix select
// (8 bits per pass, a shared-memory histogram fed by warp-aggregated
// increments, stopping as soon as one candidate is left) -- see the kernel.  The
// decayed score is computed in fp32 with one rounding after the product and one
// after the sum (no contraction), -0 read as +0 and NaN as -inf, so the integer
// outputs are exactly those of that definition.
#include <algorithm>

#include "common.cuh"

namespace kvpop {
namespace {

constexpr int kLabelThreads = 512;
constexpr int kLabelRowsPerCta = 64;
constexpr int kCacheFloats = 32768;  // targets kept in shared memory when S fits (128 KB)
constexpr int kWindow = 512;         // keys kept around the pivot on a full row
constexpr int kBand = 2048;          // candidates kept in the score band

__device__ __forceinline__ float decayed_score(float r, int q, int t, int n, float lg) {
  const float m = (float)((q - t) / n);
  const float dec = __fmul_rn(m, lg);
  float sc = __fadd_rn(r, dec);
  if (sc != sc) sc = __int_as_float(0xff800000);
  return sc == 0.0f ? 0.0f : sc;  // -0 == +0
}

// larger key = better token: (score desc, index asc)
__device__ __forceinline__ unsigned long long label_key(float sc, int t) {
  uint32_t u = __float_as_uint(sc);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (0xffffffffu - (uint32_t)t);
}

// floor(d / n) for 0 <= d < 2^24 through the fp32 reciprocal, corrected by one step
__device__ __forceinline__ int div_floor(int d, int n, float inv_n) {
  int m = __float2int_rz(__fmul_rn((float)d, inv_n));
  if (m * n > d) --m;
  else if ((m + 1) * n <= d) ++m;
  return m;
}

__device__ __forceinline__ float decayed_score_m(float r, int m, float lg) {
  float sc = __fadd_rn(r, __fmul_rn((float)m, lg));
  if (sc != sc) sc = __int_as_float(0xff800000);
  return sc == 0.0f ? 0.0f : sc;  // -0 == +0
}

// Band: from row to row only two things change -- the candidate that joins
// (the previous row's leaving token) and the candidates whose decay step
// floor((q - t) / n) grows at this row (t = q mod n, one in n); every other
// score is bit for bit what it was.  So the CTA keeps a band of scores
// [lo, hi] around the cutoff: the number of candidates above hi, and the list
// of those inside (index and target, in shared memory).  A row updates the
// count and the list from the joining and the decaying candidates only
// (scores only fall, so a listed candidate never rises above hi; one that
// falls below lo stays listed and is skipped), then selects the cutoff among
// the listed candidates -- the previous cutoff tried first, a radix select
// over the list otherwise.  When the cutoff leaves the band, or the list
// overflows, the row takes the full path below and the band is rebuilt
// around the new cutoff in one more pass.
//
// Full path: one pass over all candidates against the previous row's cutoff as
// pivot counts the keys above it and gathers, in shared memory, the keys whose
// score lies within +-delta of the pivot's.  When the cutoff moved by d places,
// the new one is the d-th nearest key above (or below) the pivot; if the window
// holds at least d of them it is found there.  delta adapts so the window holds
// a few dozen to a few hundred keys; a row whose window was too narrow, or
// overflowed, falls back to a radix select.
template <bool kFastDiv>
__global__ void __launch_bounds__(kLabelThreads)
    teacher_labels_kernel(const float* __restrict__ r_tgt, int H, int S, int s, int w, int k, int n, float inv_n,
                          const float* __restrict__ log_gamma, int32_t* __restrict__ t_bnd,
                          int32_t* __restrict__ y, int cache, int* status) {
  extern __shared__ float rs[];  // the row of targets, when it fits
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need, s_left, s_found, s_wcount;
  __shared__ int red[kLabelThreads / 32];
  __shared__ unsigned long long wbuf[kWindow];
  __shared__ int band_t[kBand];
  __shared__ float band_r[kBand];
  __shared__ int s_bn;
  const int bh = blockIdx.y;
  const int h = bh % H;
  const float* r = r_tgt + (size_t)bh * S;
  const float lg = log_gamma[h];
  const int q0 = blockIdx.x * kLabelRowsPerCta;
  const int q1 = min(S, q0 + kLabelRowsPerCta);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tmax = max(0, q1 - 1 - w);  // candidates of this CTA's rows are t < tmax
  if (cache)
    for (int t = tid; t < tmax; t += kLabelThreads) rs[t] = r[t];
  __syncthreads();
  auto score_of = [&](int q, int t) -> float {
    const float rt = cache ? rs[t] : __ldg(r + t);
    return kFastDiv ? decayed_score_m(rt, div_floor(q - t, n, inv_n), lg) : decayed_score(rt, q, t, n, lg);
  };
  auto block_sum = [&](int v) -> int {
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int i = 0; i < kLabelThreads / 32; ++i) tot += red[i];
    __syncthreads();
    return tot;
  };
  float delta = 1.0f / 64.0f;  // half-width of the window, in score units
  int prev = -1;               // the previous row's cutoff
  // band state (uniform over the CTA)
  bool band_ok = false;
  float b_lo = 0.0f, b_hi = 0.0f, bdelta = 1.0f / 32.0f;
  int ahi = 0;       // candidates scored above b_hi
  int band_age = 0;  // rows served by the current band
  auto cat = [&](float sc) -> int { return sc > b_hi ? 2 : (sc >= b_lo ? 1 : 0); };  // NaN -> 0
  auto append = [&](int t, float rt) {
    const int slot = atomicAdd(&s_bn, 1);
    if (slot < kBand) {
      band_t[slot] = t;
      band_r[slot] = rt;
    }
  };
  auto band_score = [&](int q, int i) -> float {
    const int t = band_t[i];
    return decayed_score_m(band_r[i], kFastDiv ? div_floor(q - t, n, inv_n) : (q - t) / n, lg);
  };
  // the row's cutoff from the band, or -1 when it left the band (band_ok falls)
  auto band_row = [&](int q, int tn) -> int {
    // candidates whose decay step grows at this row: t = q (mod n), already candidates at q - 1
    int dA = 0;
    for (int t = s + (q - s) % n + n * tid; t < tn - 1; t += n * kLabelThreads) {
      const float rt = cache ? rs[t] : __ldg(r + t);
      const int mq = kFastDiv ? div_floor(q - t, n, inv_n) : (q - t) / n;
      const int oc = cat(decayed_score_m(rt, mq - 1, lg)), nc = cat(decayed_score_m(rt, mq, lg));
      if (oc == 2 && nc != 2) {
        --dA;
        if (nc == 1) append(t, rt);
      }
    }
    if (tid == 0) {  // the candidate that joins: the previous row's leaving token
      const int t = tn - 1;
      const float rt = cache ? rs[t] : __ldg(r + t);
      const int c = cat(decayed_score_m(rt, kFastDiv ? div_floor(q - t, n, inv_n) : (q - t) / n, lg));
      if (c == 2) ++dA;
      if (c == 1) append(t, rt);
    }
    ahi += block_sum(dA);  // its barriers also publish the list
    const int bn = s_bn;
    const int need = k - ahi;  // the cutoff is the need-th best listed candidate
    if (bn > kBand || need < 1) return -1;
    // listed candidates still in the band, and those above the previous cutoff
    const float sp = prev >= 0 ? score_of(q, prev) : 0.0f;
    const bool piv = prev >= 0 && sp >= b_lo;  // (then it is listed: it was the cutoff)
    const unsigned long long pk = piv ? label_key(sp, prev) : 0ull;
    int alive = 0, above = 0;
    for (int i = tid; i < bn; i += kLabelThreads) {
      const float sc = band_score(q, i);
      if (sc >= b_lo) {
        ++alive;
        above += piv && label_key(sc, band_t[i]) > pk;
      }
    }
    alive = block_sum(alive);
    above = block_sum(above);
    if (alive < need) return -1;
    if (piv && above == need - 1) return prev;
    // radix select of the need-th largest key among the listed candidates in the band
    unsigned long long prefix = 0, mask = 0;
    int nd = need;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kLabelThreads) hist[i] = 0;
      __syncthreads();
      for (int i0 = 0; i0 < bn; i0 += kLabelThreads) {  // warp-uniform loop
        const int i = i0 + tid;
        bool match = false;
        unsigned long long key = 0;
        if (i < bn) {
          const float sc = band_score(q, i);
          key = label_key(sc, band_t[i]);
          match = sc >= b_lo && (key & mask) == prefix;
        }
        const uint32_t active = __ballot_sync(0xffffffffu, match);
        if (match) {
          const uint32_t bin = (uint32_t)(key >> shift) & 255u;
          const uint32_t peers = __match_any_sync(active, bin);
          if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
        }
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t cnt[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = hist[255 - 8 * lane - j];
          tot += cnt[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - tot;
        if (excl < (uint32_t)nd && (uint32_t)nd <= incl) {
          uint32_t run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + cnt[j] >= (uint32_t)nd) {
              s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - j) << shift);
              s_need = nd - (int)run;
              s_left = (int)cnt[j];
              break;
            }
            run += cnt[j];
          }
        }
      }
      __syncthreads();
      prefix = s_prefix;
      mask |= 255ull << shift;
      nd = s_need;
      const int left = s_left;
      __syncthreads();
      if (left == 1 || shift == 0) break;
    }
    // the one listed candidate that carries the prefix (keys are distinct)
    if (tid == 0) s_found = -1;
    __syncthreads();
    for (int i = tid; i < bn; i += kLabelThreads) {
      const float sc = band_score(q, i);
      if (sc >= b_lo && (label_key(sc, band_t[i]) & mask) == prefix) atomicMax(&s_found, band_t[i]);
    }
    __syncthreads();
    const int res = s_found;
    __syncthreads();
    return res;
  };
  // a band of scores around the cutoff `cut` of row q, from one pass over T(q)
  auto build_band = [&](int q, int tn, int cut) {
    const float sc0 = score_of(q, cut);
    band_ok = false;
    // scores never rise only while the decay factor is at most 1 (log gamma <= 0)
    if (!(lg <= 0.0f) || !(sc0 > __int_as_float(0xff800000) && sc0 < __int_as_float(0x7f800000))) return;
    b_lo = sc0 - bdelta;
    b_hi = sc0 + bdelta;
    if (tid == 0) s_bn = 0;
    __syncthreads();
    int a = 0;
    for (int t = s + tid; t < tn; t += kLabelThreads) {
      const float rt = cache ? rs[t] : __ldg(r + t);
      const int c = cat(decayed_score_m(rt, kFastDiv ? div_floor(q - t, n, inv_n) : (q - t) / n, lg));
      a += c == 2;
      if (c == 1) append(t, rt);
    }
    ahi = block_sum(a);
    const int bn = s_bn;
    if (bn > kBand) {
      bdelta *= 0.5f;
      return;
    }
    if (bn > kBand / 2) bdelta *= 0.75f;
    band_ok = true;
    band_age = 0;
  };
  for (int q = q0; q < q1; ++q) {
    const int tn = q - w;
    const size_t out = (size_t)bh * S + q;
    if (tn < s || k == 0 || tn - s < k) {  // uniform over the CTA
      band_ok = false;
      if (tid == 0) {
        t_bnd[out] = -1;
        y[out] = tn < s ? 0 : (k == 0 ? -1 : 1);
      }
      continue;
    }
    int found = -1;
    if (band_ok) {
      found = band_row(q, tn);
      if (found >= 0) {
        ++band_age;
      } else {
        band_ok = false;
        if (band_age < 16) bdelta *= 2.0f;  // the cutoff left the band quickly: widen it
      }
    }
    const bool rebuild = found < 0;
    const float sp = (found < 0 && prev >= 0) ? score_of(q, prev) : 0.0f;
    // (a pivot scored -inf ties with NaN candidates, which the plain comparisons
    // below do not see: such rows take the radix select)
    if (found < 0 && prev >= 0 && sp != __int_as_float(0xff800000)) {
      const unsigned long long pk = label_key(sp, prev);
      const float lo = sp - delta, hi = sp + delta;
      if (tid == 0) {
        s_wcount = 0;
        s_found = -1;
      }
      __syncthreads();
      int c = 0;
      // this thread's candidates t = s + tid + 512 i: q - t falls by 512 per step,
      // so floor((q - t) / n) follows by a subtraction and one carry
      int t = s + tid;
      int m = 0, rem = 0;
      if (t < tn) {
        m = kFastDiv ? div_floor(q - t, n, inv_n) : (q - t) / n;
        rem = q - t - m * n;
      }
      const int step_m = kLabelThreads / n, step_r = kLabelThreads % n;
      // the decayed score exactly as defined (one rounding after the product and
      // one after the sum); plain comparisons already treat -0 as +0 and put NaN
      // below a finite pivot, as the key order does
      auto visit = [&](int tt, float rt, int mm) {
        const float sc = __fadd_rn(rt, __fmul_rn((float)mm, lg));
        c += (sc > sp) || (sc == sp && tt < prev);
        if (sc >= lo && sc <= hi && tt != prev) {
          const int slot = atomicAdd(&s_wcount, 1);
          if (slot < kWindow) wbuf[slot] = label_key(sc == 0.0f ? 0.0f : sc, tt);
        }
      };
      auto advance = [&]() {
        rem -= step_r;
        m -= step_m;
        if (rem < 0) {
          rem += n;
          --m;
        }
      };
      // four candidates per round, their loads issued together
      for (; t + 3 * kLabelThreads < tn; t += 4 * kLabelThreads) {
        float rv[4];
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) rv[u4] = cache ? rs[t + u4 * kLabelThreads] : __ldg(r + t + u4 * kLabelThreads);
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          visit(t + u4 * kLabelThreads, rv[u4], m);
          advance();
        }
      }
      for (; t < tn; t += kLabelThreads) {
        visit(t, cache ? rs[t] : __ldg(r + t), m);
        advance();
      }
      c = block_sum(c);  // its barriers also publish the window
      const int wc = s_wcount;
      const int dm = c - (k - 1);  // places the cutoff moved: > 0 up, < 0 down
      if (dm == 0) {
        found = prev;
      } else if (wc <= kWindow) {
        const bool up = dm > 0;
        const int want = up ? dm - 1 : -dm - 1;  // keys strictly between the pivot and the new cutoff
        for (int i = tid; i < wc; i += kLabelThreads) {
          const unsigned long long e = wbuf[i];
          if (up ? e > pk : e < pk) {
            int rank = 0;
            for (int j = 0; j < wc && rank <= want; ++j) {
              const unsigned long long f = wbuf[j];
              rank += up ? (f > pk && f < e) : (f < pk && f > e);
            }
            if (rank == want) s_found = (int)(0xffffffffu - (uint32_t)e);
          }
        }
        __syncthreads();
        found = s_found;
      }
      // keep the window at a few dozen keys (uniform decisions)
      if (wc > kWindow) delta *= 0.25f;
      else if (found < 0) delta *= 4.0f;
      else if (wc > kWindow / 4) delta *= 0.75f;
      else if (wc < kWindow / 32) delta *= 1.5f;
      __syncthreads();
    }
    // otherwise a radix select of the k-th largest key among t in [s, tn)
    unsigned long long prefix = 0, mask = 0;
    int need = k;
    for (int shift = 56; found < 0 && shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kLabelThreads) hist[i] = 0;
      __syncthreads();
      for (int t0 = s; t0 < tn; t0 += kLabelThreads) {  // warp-uniform loop
        const int t = t0 + tid;
        const bool valid = t < tn;
        unsigned long long key = 0;
        if (valid) key = label_key(score_of(q, t), t);
        const bool match = valid && (key & mask) == prefix;
        const uint32_t active = __ballot_sync(0xffffffffu, match);
        if (match) {
          const uint32_t bin = (uint32_t)(key >> shift) & 255u;
          const uint32_t peers = __match_any_sync(active, bin);
          if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
        }
      }
      __syncthreads();
      if (warp == 0) {
        // bins from the top: lane l owns bins 255 - 8l .. 248 - 8l
        uint32_t cnt[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cnt[i] = hist[255 - 8 * lane - i];
          tot += cnt[i];
        }
        uint32_t incl = tot;  // inclusive scan over lanes (higher bins first)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - tot;
        if (excl < (uint32_t)need && (uint32_t)need <= incl) {
          uint32_t run = excl;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run + cnt[i] >= (uint32_t)need) {
              s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - i) << shift);
              s_need = need - (int)run;
              s_left = (int)cnt[i];
              break;
            }
            run += cnt[i];
          }
        }
      }
      __syncthreads();
      prefix = s_prefix;
      mask |= 255ull << shift;
      need = s_need;
      const int left = s_left;
      __syncthreads();
      if (left == 1 || shift == 0) {
        // one candidate carries the prefix: find it
        if (tid == 0) s_found = -1;
        __syncthreads();
        for (int t = s + tid; t < tn; t += kLabelThreads) {
          const unsigned long long key = label_key(score_of(q, t), t);
          if ((key & mask) == prefix) atomicMax(&s_found, t);
        }
        __syncthreads();
        found = s_found;
        __syncthreads();
        break;
      }
    }
    if (rebuild && found >= 0) build_band(q, tn, found);
    prev = found;
    if (tid == 0) {
      int yy = -1;
      if (found >= 0) {
        const float sb = score_of(q, found);
        const float sn = decayed_score(__ldg(r + tn), q, tn, n, lg);
        yy = sn > sb ? 1 : -1;  // t_new has the larger index: it loses ties
      } else {
        report_error(status, KVPOP_ERR_INTERNAL, SITE_INTERNAL_CHECK, 20);
      }
      t_bnd[out] = found;
      y[out] = yy;
    }
  }
}

__global__ void target_normalize_kernel(const float* __restrict__ target, long long total, int S, int G, int w,
                                        float eps, float* __restrict__ r) {
  const float leps = eps > 0.0f ? logf(eps) : __int_as_float(0xff800000);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i % S);
    const int nt = S - t - w;
    // x = log((1/G) sum_g m_t^g) = target - log(G * N_t)
    const float x = nt > 0 ? target[i] - logf((float)G * (float)nt) : __int_as_float(0xff800000);
    float out;
    if (!(eps > 0.0f)) {
      out = x;
    } else {  // log(eps + e^x), stably
      const float hi = fmaxf(leps, x), lo = fminf(leps, x);
      out = lo == __int_as_float(0xff800000) ? hi : hi + log1pf(expf(lo - hi));
    }
    r[i] = out;
  }
}

__device__ __forceinline__ float softplus_f(float z) { return z > 0.0f ? z + log1pf(expf(-z)) : log1pf(expf(z)); }
__device__ __forceinline__ float sigmoid_f(float z) {
  return z >= 0.0f ? 1.0f / (1.0f + expf(-z)) : expf(z) / (1.0f + expf(z));
}

// Sum of the weighted pair losses and the unscaled gradient; acc[0] += loss sum,
// acc[1] += number of pairs.
__global__ void __launch_bounds__(256)
    boundary_loss_kernel(const float* __restrict__ r_hat, const int32_t* __restrict__ t_bnd,
                         const int32_t* __restrict__ y, const float* __restrict__ omega, int H, int S, int w,
                         int n, const float* __restrict__ log_gamma, float inv_tau, long long total,
                         float* __restrict__ acc, float* __restrict__ grad) {
  __shared__ float red_l[8], red_c[8];
  float lsum = 0.0f, cnt = 0.0f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int yy = y[i], tb = t_bnd[i];
    if (yy == 0 || tb < 0) continue;
    const long long bh = i / S;
    const int q = (int)(i - bh * S);
    const int tn = q - w;
    if (tn < 0 || tb >= S) continue;  // labels from kvpop_teacher_labels never do this
    const float lg = log_gamma[bh % H];
    const float* rr = r_hat + bh * S;
    const float dn = __fadd_rn(rr[tn], __fmul_rn((float)((q - tn) / n), lg));
    const float db = __fadd_rn(rr[tb], __fmul_rn((float)((q - tb) / n), lg));
    const float z = -(float)yy * (dn - db) * inv_tau;
    const float om = omega ? omega[i] : 1.0f;
    lsum += om * softplus_f(z);
    cnt += 1.0f;
    const float g = om * sigmoid_f(z) * (-(float)yy * inv_tau);
    atomicAdd(grad + bh * S + tn, g);
    atomicAdd(grad + bh * S + tb, -g);
  }
  for (int o = 16; o > 0; o >>= 1) {
    lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_l[warp] = lsum;
    red_c[warp] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f, c = 0.0f;
    for (int i = 0; i < 8; ++i) {
      a += red_l[i];
      c += red_c[i];
    }
    if (c > 0.0f) {
      atomicAdd(acc, a);
      atomicAdd(acc + 1, c);
    }
  }
}

// loss = sum / pairs, grad /= pairs (the mean over pairs)
__global__ void boundary_loss_finalize(float* __restrict__ acc, float* __restrict__ grad, long long total) {
  const float c = acc[1];
  const float inv = c > 0.0f ? 1.0f / c : 0.0f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x)
    grad[i] *= inv;
}

__global__ void boundary_loss_mean(float* __restrict__ acc) {
  if (threadIdx.x == 0) acc[0] = acc[1] > 0.0f ? acc[0] / acc[1] : 0.0f;
}

int grid_for(long long total, int threads) {
  const long long want = (total + threads - 1) / threads;
  return (int)std::min<long long>(std::max<long long>(want, 1), (long long)num_sms() * 8);
}

}  // namespace
}  // namespace kvpop

using namespace kvpop;

extern "C" kvpop_status kvpop_target_normalize(const float* target, int b, int H, int S, int G, int w, float eps,
                                               float* r_tgt, kvpop_stream stream) {
  if (!target || !r_tgt || b <= 0 || H <= 0 || S <= 0 || G <= 0 || w < 0 || !(eps >= 0.0f)) {
    set_last_error("kvpop_target_normalize: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  const long long total = (long long)b * H * S;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  target_normalize_kernel<<<grid_for(total, 256), 256, 0, cs>>>(target, total, S, G, w, eps, r_tgt);
  return cuda_check(cudaGetLastError(), "kvpop_target_normalize: launch");
}

extern "C" kvpop_status kvpop_teacher_labels(const float* r_tgt, int b, int H, int S, kvpop_budget bud, int n,
                                             const float* log_gamma, int32_t* t_bnd, int32_t* y,
                                             kvpop_stream stream) {
  if (!r_tgt || !log_gamma || !t_bnd || !y || b <= 0 || H <= 0 || S <= 0 || n <= 0) {
    set_last_error("kvpop_teacher_labels: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  if (bud.s < 0 || bud.w < 0 || bud.k < 0) {
    set_last_error("kvpop_teacher_labels: invalid budget");
    return KVPOP_ERR_INVALID_ARG;
  }
  if ((long long)b * H > 65535 || S > (1 << 30)) {
    set_last_error("kvpop_teacher_labels: b*H must be <= 65535");
    return KVPOP_ERR_UNSUPPORTED;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  dim3 grid((S + kLabelRowsPerCta - 1) / kLabelRowsPerCta, b * H);
  const float inv_n = 1.0f / (float)n;
  const int cache = S <= kCacheFloats ? 1 : 0;
  const int smem = cache ? S * 4 : 0;
  auto kern = S < (1 << 24) ? teacher_labels_kernel<true> : teacher_labels_kernel<false>;
  kvpop_status st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCacheFloats * 4),
                               "kvpop_teacher_labels: smem attribute");
  if (st != KVPOP_OK) return st;
  kern<<<grid, kLabelThreads, smem, cs>>>(r_tgt, H, S, bud.s, bud.w, bud.k, n, inv_n, log_gamma, t_bnd, y, cache,
                                          device_status_ptr());
  return cuda_check(cudaGetLastError(), "kvpop_teacher_labels: launch");
}

extern "C" kvpop_status kvpop_boundary_loss(const float* r_hat, const int32_t* t_bnd, const int32_t* y,
                                            const float* omega, int b, int H, int S, int w, int n,
                                            const float* log_gamma, float tau, float* loss, float* grad,
                                            kvpop_stream stream) {
  if (!r_hat || !t_bnd || !y || !log_gamma || !loss || !grad || b <= 0 || H <= 0 || S <= 0 || w < 0 || n <= 0 ||
      !(tau > 0.0f)) {
    set_last_error("kvpop_boundary_loss: bad arguments");
    return KVPOP_ERR_INVALID_ARG;
  }
  const long long total = (long long)b * H * S;
  if (total > (1LL << 24)) {  // the pair count is kept exactly in fp32
    set_last_error("kvpop_boundary_loss: b*H*S must be <= 2^24");
    return KVPOP_ERR_UNSUPPORTED;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  kvpop_status st = cuda_check(cudaMemsetAsync(loss, 0, 2 * sizeof(float), cs), "kvpop_boundary_loss: clear");
  if (st == KVPOP_OK) st = cuda_check(cudaMemsetAsync(grad, 0, total * sizeof(float), cs), "kvpop_boundary_loss: clear");
  if (st != KVPOP_OK) return st;
  boundary_loss_kernel<<<grid_for(total, 256), 256, 0, cs>>>(r_hat, t_bnd, y, omega, H, S, w, n, log_gamma,
                                                              1.0f / tau, total, loss, grad);
  st = cuda_check(cudaGetLastError(), "kvpop_boundary_loss: launch");
  if (st != KVPOP_OK) return st;
  boundary_loss_finalize<<<grid_for(total, 256), 256, 0, cs>>>(loss, grad, total);
  st = cuda_check(cudaGetLastError(), "kvpop_boundary_loss: launch");
  if (st != KVPOP_OK) return st;
  boundary_loss_mean<<<1, 32, 0, cs>>>(loss);
  return cuda_check(cudaGetLastError(), "kvpop_boundary_loss: launch");
}
