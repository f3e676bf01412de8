/*
 * kvpop.h -- C ABI of libkvpop, the GB300 (sm_103a) hot path of KVpop
 * fixed-budget KV-cache eviction.
 *
 * Sources (page title and section / equation):
 *   [notes]   "KVpop -- Key-Value Cache Compression with Predictive Online
 *             Pruning 精读笔记" (liuzhao09.github.io)
 *   [summary] "KVpop — 基于预测性在线剪枝的键值（KV）缓存压缩" (gist.science)
 *
 * Notation: b batch, H KV heads, G query heads per KV head, Hq = H*G, D head
 * dim, S sequence length.  Query head j reads KV head j / G.  The per-head
 * budget is B = s + w + k: s sink tokens, a protected window of the w most
 * recent tokens and k long-range slots chosen by a static per-token priority
 * ([notes] section 2.1, Eq. B; [summary] section 2.1).
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers owned by the caller, except the
 *     opaque kvpop_cache, which the library owns.  Only kvpop_cache_create
 *     allocates device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise, except kvpop_device_status.
 *   - Arguments are validated on the host; a bad argument returns
 *     KVPOP_ERR_INVALID_ARG / KVPOP_ERR_UNSUPPORTED before anything is
 *     launched, and kvpop_last_error() gives a one-line reason (thread-local).
 *   - Kernels never trap.  A wait that exceeds its time limit makes the kernel
 *     record KVPOP_ERR_TIMEOUT in the per-device status words and return;
 *     read them with kvpop_device_status.
 *   - Layouts: q, O [b, S, Hq, D] bf16; k, v [b, S, H, D] bf16 (BSHD,
 *     contiguous, 16-byte aligned); LSE [b, Hq, S] fp32 natural log;
 *     priorities [b, H, S] fp32; rank, tau, evict_at [b, H, S] int32;
 *     target [b, H, S] fp32 natural log.
 *   - Supported head dims: D = 64 or 128.  Hq % H == 0 and 128 % G == 0.
 */
#ifndef KVPOP_H
#define KVPOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvpop_stream; /* a cudaStream_t */

typedef enum {
  KVPOP_OK = 0,
  KVPOP_ERR_INVALID_ARG = 1,
  KVPOP_ERR_UNSUPPORTED = 2,
  KVPOP_ERR_CUDA = 3,
  KVPOP_ERR_TIMEOUT = 4,
  KVPOP_ERR_INTERNAL = 5
} kvpop_status;

/* B = s + w + k; all >= 0 and B >= 1. */
typedef struct {
  int32_t s; /* sink tokens, always kept */
  int32_t w; /* protected window of the most recent tokens */
  int32_t k; /* long-range slots chosen by priority */
} kvpop_budget;

/* tau value meaning "every eligible token is kept" (|E(q)| <= k). */
#define KVPOP_TAU_ALL 2147483647
/* Query positions covered by one long-range list (see kvpop_mask). */
#define KVPOP_LIST_QBLOCK 64

const char* kvpop_status_string(kvpop_status status);
/* Detail of the last failing call on this thread ("" if none). */
const char* kvpop_last_error(void);
int kvpop_version(void);

/*
 * Synchronises the current device, copies its four status words to `out`
 * ([0] first error code, [1] kernel site, [2] detail, [3] error count) and,
 * if `reset` is non-zero, clears them.  Returns out[0] as a status.
 */
kvpop_status kvpop_device_status(int32_t out[4], int reset);

/* ------------------------------------------------------------------------
 * kvpop_mask -- fixed-budget retained set from static priorities.
 *
 * [notes] section 2.2 (eligible set E(q) = {t : s <= t <= q - w}) and
 * section 2.3 (M_{q,t} = [t<s] v [q-t<w] v ([t in E(q)] ^ [rank(t) <= tau_q]),
 * tau_q the rank of the k-th best eligible token); [summary] section 2.4
 * (running threshold over static priorities, no dense S x S mask).
 *
 * Per (batch, KV head), with the order (priority desc, index asc), NaN
 * counting as -inf and -0.0 == +0.0:
 *   rank[t]     position of token t in that order, 0 = best;
 *   tau[q]      rank of the k-th best token of E(q); KVPOP_TAU_ALL when
 *               |E(q)| <= k; -1 when k == 0;
 *   evict_at[t] first row q >= t + w at which t is no longer retained
 *               (S if never; S for sinks).  Row q retains t exactly when
 *               t <= q < evict_at[t], so the retained set of row q is
 *               {t <= q : q < evict_at[t]} and holds min(q+1, B) keys.
 *   lists       (nullable) [b, H, ceil(S/64), k] pairs of int32
 *               (position, evict_at): list i holds the long-range keys
 *               retained at row 64*i, i.e. {t in E(64 i) : 64 i < evict_at[t]};
 *               first those still retained at row 64 i + 63, then those
 *               dropped inside rows 64 i .. 64 i + 63, each group in
 *               increasing position.  Its length is
 *               min(k, max(0, 64 i - w - s + 1)); the rest of the row is
 *               unspecified.  kvpop_attn_fwd reads it.
 * prio [b, H, S] fp32.  workspace: device scratch of at least
 * kvpop_mask_workspace_size() bytes, 256-byte aligned.
 * Supported S: 1 .. 131072.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_mask_workspace_size(int b, int H, int S, kvpop_budget budget, size_t* bytes);
kvpop_status kvpop_mask_lists_size(int b, int H, int S, kvpop_budget budget, size_t* bytes);
kvpop_status kvpop_mask(const float* prio, int b, int H, int S, kvpop_budget budget,
                        int32_t* rank, int32_t* tau, int32_t* evict_at, int32_t* lists,
                        void* workspace, size_t workspace_bytes, kvpop_stream stream);

/* ------------------------------------------------------------------------
 * kvpop_attn_fwd -- causal GQA softmax attention, sparse or dense.
 *
 * [notes] section 2.1 (sparse softmax attention over the retained set) and
 * section 2.3 (the attention call returns the log-sum-exp normaliser LSE);
 * [summary] section 2.2.
 *
 * Sparse mode (evict_at and lists from kvpop_mask with the same budget): row
 * q of query head j attends over {t <= q : q < evict_at[t]} of KV head j / G.
 * Dense mode (evict_at == lists == NULL): all t <= q (the dense teacher).
 *   O   [b, S, Hq, D] bf16, nullable: NULL computes the LSE only.
 *   lse [b, Hq, S] fp32, natural log of sum_t exp(scale * q.k_t).
 * scale <= 0 selects 1/sqrt(D).  bf16 inputs, fp32 accumulation.
 * Errors: INVALID_ARG, UNSUPPORTED (D, G, alignment), CUDA.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_attn_fwd(const void* q, const void* k, const void* v, int b, int S, int Hq,
                            int H, int D, float scale, const int32_t* evict_at,
                            const int32_t* lists, kvpop_budget budget, void* O, float* lse,
                            kvpop_stream stream);

/* ------------------------------------------------------------------------
 * kvpop_attn_bwd -- gradient of the sparse attention (the training path).
 *
 * [notes] section 2.1 (Figure 1 and the training flow: the student runs the
 * sparse attention over the retained set and the backbone is trained through
 * it).  For the sparse rows of kvpop_attn_fwd -- same q, k, v, evict_at, lists,
 * budget and scale -- and an upstream gradient dO = dL/dO, with
 * P_{q,t} = exp(scale * q.k_t - lse_q) over {t <= q : q < evict_at[t]}:
 *   dv_t     = sum_q P_{q,t} dO_q
 *   dS_{q,t} = P_{q,t} (dO_q . v_t - dO_q . O_q)
 *   dq_q     = scale * sum_t dS_{q,t} k_t
 *   dk_t     = scale * sum_q dS_{q,t} q_q
 * where the sums over q run over the G query heads of the KV head too.
 *   O, lse     the forward's outputs for these inputs: [b, S, Hq, D] bf16 and
 *              [b, Hq, S] fp32 (dO . O stands in for sum_t P dP)
 *   dO         [b, S, Hq, D] bf16
 *   dq         [b, S, Hq, D] fp32; dk, dv [b, S, H, D] fp32; all overwritten
 * workspace: kvpop_attn_bwd_workspace_size() bytes, 256-byte aligned (row
 * constants and per-block key lists; contents undefined between calls).
 * D 64 or 128, G dividing 128, tensors 16-byte aligned, b and H <= 65535,
 * S <= 2^24.  bf16 operands (P and dS rounded to bf16 before their products),
 * fp32 accumulation; dk and dv take fp32 atomic additions, so their last bits
 * vary from run to run.  Errors: INVALID_ARG (NULL pointer, bad shape or budget,
 * workspace too small), UNSUPPORTED (D, G, alignment, sizes), CUDA.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_attn_bwd_workspace_size(int b, int S, int Hq, int H, kvpop_budget budget, size_t* bytes);
kvpop_status kvpop_attn_bwd(const void* q, const void* k, const void* v, const void* O, const void* dO,
                            const float* lse, int b, int S, int Hq, int H, int D, float scale,
                            const int32_t* evict_at, const int32_t* lists, kvpop_budget budget, float* dq,
                            float* dk, float* dv, void* workspace, size_t workspace_bytes,
                            kvpop_stream stream);

/* ------------------------------------------------------------------------
 * kvpop_future_target -- transposed-attention pass for the future mass.
 *
 * [notes] section 2.2 (m_t = (1/N_t) sum_{d=t+w}^{S-1} A_{d,t}) and section
 * 2.3 (Eq. 8 and Figure 2: keys as rows, queries as columns, the stored LSE
 * reused, mask d >= t + w).  Output, per (batch, KV head h, token t):
 *   target[b,h,t] = log sum_{g<G} sum_{d=t+w}^{S-1}
 *                   exp(scale * q_{d,hG+g} . k_t - lse[b, hG+g, d])
 * (natural log, no 1/N_t, 1/G or epsilon; -inf when t + w > S - 1).
 * lse is the dense causal LSE from kvpop_attn_fwd (dense mode).  workspace:
 * device scratch of kvpop_future_target_workspace_size() bytes (16-byte
 * aligned) that receives the LSE rescaled to log2 units in query-tile order.
 * scale <= 0 selects 1/sqrt(D).  Terms below about 1e-38 underflow to zero.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_future_target_workspace_size(int b, int S, int Hq, int H, size_t* bytes);
kvpop_status kvpop_future_target(const void* q, const void* k, const float* lse, int b, int S,
                                 int Hq, int H, int D, float scale, int w, float* target,
                                 void* workspace, size_t workspace_bytes, kvpop_stream stream);

/* ------------------------------------------------------------------------
 * kvpop_future_target_noalloc -- kvpop_future_target without caller scratch.
 *
 * The paper has no counterpart: this exists for callers that cannot call
 * cudaMalloc -- e.g. an engine whose allocator has reserved all device memory
 * for its own pools, or a path where cudaMalloc's implicit device
 * synchronisation is not allowed.  Same arguments and result as
 * kvpop_future_target minus the workspace; it allocates nothing.
 *   - Scratch is a 16 MiB file-scope device array (every GPU that loads the
 *     library holds it until exit).  Calls needing more than that
 *     (b*H*ceil(S/P)*P*G floats, P = 128/G, above 4,194,304) return
 *     KVPOP_ERR_UNSUPPORTED with a message; nothing is launched.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams, no ordering between them) race.  Every scratch element a call
 *     reads is written by that call first, so no clearing is needed.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_future_target_noalloc(const void* q, const void* k, const float* lse, int b,
                                         int S, int Hq, int H, int D, float scale, int w,
                                         float* target, kvpop_stream stream);

/* ------------------------------------------------------------------------
 * Training-side passes on the future-attention target ([notes] section 2.2).
 *
 * kvpop_target_normalize: r_tgt[b,h,t] = log(eps + (1/G) sum_g m_t^g) with
 *   m_t^g = (1/N_t) sum_{d=t+w}^{S-1} A_{d,t}^g and N_t = S - t - w, from the
 *   unnormalised target of kvpop_future_target (natural log) -- i.e.
 *   log(eps + exp(target) / (G N_t)); a key with no future query (N_t <= 0)
 *   has mass 0, so log(eps) (-inf when eps == 0).  target, r_tgt: [b, H, S]
 *   fp32 device; r_tgt may equal target.  eps >= 0.  Errors: INVALID_ARG, CUDA.
 *
 * kvpop_teacher_labels: per row q, the token t_new = q - w leaves the window;
 *   the teacher ranks E(q) = {s..q-w} by the decayed score
 *     r_t(q) = r_tgt[t] + floor((q - t) / n) * log_gamma[h]
 *   (fp32: rounded after the product and after the sum; NaN counts as -inf,
 *   -0 as +0; ties go to the lower index) and keeps its top k.
 *     t_bnd[b,h,q] = the k-th best token of E(q) other than t_new -- the
 *                    cutoff t_new has to beat (when t_new is dropped it is the
 *                    lowest-scoring member of the teacher top-k); -1 when
 *                    fewer than k other tokens are eligible or k == 0;
 *     y[b,h,q]     = +1 if t_new is in the teacher top-k, -1 if not, 0 when the
 *                    row has no leaving token (q - w < s).
 *   r_tgt [b, H, S] fp32, log_gamma [H] fp32 (log of the per-head decay factor,
 *   <= 0), t_bnd and y [b, H, S] int32, all device.  n >= 1.  Cost: one
 *   radix select over E(q) per row, O(S^2) per (batch, head).
 *   Errors: INVALID_ARG, UNSUPPORTED (b*H > 65535), CUDA.
 *
 * kvpop_boundary_loss: the pairwise logistic loss over the rows with y != 0
 *   and t_bnd >= 0:
 *     loss[0] = mean of omega[q] * softplus(-y[q] (rh_new(q) - rh_bnd(q)) / tau),
 *     rh_t(q) = r_hat[t] + floor((q - t) / n) * log_gamma[h]  (the same decay on
 *     the predicted scores), t_new = q - w;
 *     loss[1] = the number of such pairs (0 pairs: loss[0] = 0, grad = 0);
 *     grad = d loss[0] / d r_hat, [b, H, S] fp32, overwritten.
 *   r_hat [b, H, S] fp32; omega [b, H, S] fp32 or NULL (all 1); t_bnd, y as
 *   from kvpop_teacher_labels; loss: 2 floats.  tau > 0.  b*H*S <= 2^24.  Sums
 *   use fp32 atomics, so the last bits vary between runs.
 *   Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 * ---------------------------------------------------------------------- */
kvpop_status kvpop_target_normalize(const float* target, int b, int H, int S, int G, int w, float eps,
                                    float* r_tgt, kvpop_stream stream);
kvpop_status kvpop_teacher_labels(const float* r_tgt, int b, int H, int S, kvpop_budget budget, int n,
                                  const float* log_gamma, int32_t* t_bnd, int32_t* y,
                                  kvpop_stream stream);
kvpop_status kvpop_boundary_loss(const float* r_hat, const int32_t* t_bnd, const int32_t* y,
                                 const float* omega, int b, int H, int S, int w, int n,
                                 const float* log_gamma, float tau, float* loss, float* grad,
                                 kvpop_stream stream);

/* ------------------------------------------------------------------------
 * Fixed-budget decode cache ([notes] section 2.4 and section 3.3: B slots
 * per KV head, the token u = q - w leaving the window is kept or evicted by
 * comparing its priority with the worst held long-range token; [summary]
 * section 2.4).
 *
 * Slots of each (sequence, KV head): [0, s) sinks, [s, s+w) window ring
 * (position p >= s sits in slot s + (p - s) mod w), [s+w, B) long-range.
 * All n sequences advance together: the cache holds one next position q.
 * ---------------------------------------------------------------------- */
typedef struct kvpop_cache kvpop_cache;

/* Allocates the device state (K/V [n,H,B,D] bf16, slot positions and
 * priorities, split-softmax partials); the caller owns the handle and frees it
 * with kvpop_cache_destroy.  q starts at 0.  Limits: D in {64, 128}, G in
 * {1, 2, 4, 8}, 1 <= B <= 65536, n*H <= 65535; otherwise
 * KVPOP_ERR_INVALID_ARG (bad budget) or KVPOP_ERR_UNSUPPORTED. */
kvpop_status kvpop_cache_create(int n, int H, int G, int D, kvpop_budget budget,
                                kvpop_cache** out);
kvpop_status kvpop_cache_destroy(kvpop_cache* cache);

/* Loads a prefix of P tokens: k, v [n, P, H, D] bf16, prio [n, H, P] fp32 and
 * evict_at [n, H, P] from kvpop_mask over the prefix (same budget).  The cache
 * then holds the retained set of row P-1 and its next position is P. */
kvpop_status kvpop_cache_prefill(kvpop_cache* cache, const void* k, const void* v,
                                 const float* prio, int P, const int32_t* evict_at,
                                 kvpop_stream stream);

/* One decode step at the cache's position q (then q += 1).  Two kernels on
 * `stream` (the update, then the split attention with the split merge fused
 * into its last CTA), both with programmatic dependent launch: neither reads
 * any buffer before the previous kernel of the stream has completed.
 * q_new, k_new, v_new must be 16-byte aligned (else KVPOP_ERR_UNSUPPORTED).
 *   1. the token u = q - w leaves the window; if u >= s it takes a free
 *      long-range slot, or replaces the worst held token m (lowest priority,
 *      later index on ties) when its priority is strictly greater, else it is
 *      dropped;
 *   2. the new token (k_new, v_new [n, H, D], prio_new [n, H]) enters;
 *   3. the G query heads q_new [n, Hq, D] attend over the min(q+1, B) held
 *      slots: O [n, Hq, D] bf16, lse [n, Hq] fp32.
 * evicted_pos [n, H] (nullable): the position that left the retained set at
 * this step, or -1. */
kvpop_status kvpop_decode_step(kvpop_cache* cache, const void* q_new, const void* k_new,
                               const void* v_new, const float* prio_new, void* O, float* lse,
                               int32_t* evicted_pos, kvpop_stream stream);

/* slot_pos [n, H, B] int32 device buffer: position held by each slot, -1 if empty. */
kvpop_status kvpop_cache_slots(const kvpop_cache* cache, int32_t* slot_pos, kvpop_stream stream);
/* Host value of the next decode position. */
kvpop_status kvpop_cache_position(const kvpop_cache* cache, int32_t* q_next);

#ifdef __cplusplus
}
#endif

#endif /* KVPOP_H */
