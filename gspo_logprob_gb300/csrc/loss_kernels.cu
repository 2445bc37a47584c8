// O(N) kernels: split merge -> LSE / logp, the GRPO token objective and its
// reductions, the GSPO segment seam, group-normalised advantages, and the
// bounded-wait self-test.  All floating-point sums run in a fixed order
// (strided partial sums in token order, then a xor butterfly and a fixed
// order across warps), so results are deterministic without floating-point
// atomics; integer counts are exact in any order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace gh {

namespace {

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- merge
// LSE_i = M + log(sum_k s_k e^{m_k - M}) over the splits k (one per 256-column tile).
// Fold of the split partials of rows blockIdx.x * 32 + lane (256 threads: warp
// g = 0..7 is a split group, lane a row).  M = max over splits of part_m (exact
// in any order); S = sum over splits of part_s * exp(part_m - M), where group g
// sums the splits k = g, g + 8, g + 16, ... in increasing order and the eight
// group sums are then added in group order.  The order depends on the split
// count only (a function of V), never on N or on how the rows were batched.
// Returns the LSE in warp 0's lanes (meaningless in the others).
__device__ __forceinline__ float fold_splits(int N, int splits, const float* __restrict__ part_m,
                                             const float* __restrict__ part_s, float (*red)[33]) {
  // Loads are issued FOLD_BATCH splits at a time (all in flight together) and
  // then used in increasing split order, so the sums keep the order above.
  constexpr int FOLD_BATCH = 16;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 32 + lane;
  const bool ok = i < N;
  float mx = -INFINITY;
  if (ok) {
    for (int k0 = g; k0 < splits; k0 += 8 * FOLD_BATCH) {
      float v[FOLD_BATCH];
#pragma unroll
      for (int b = 0; b < FOLD_BATCH; ++b) {
        const int k = k0 + 8 * b;
        v[b] = k < splits ? __ldg(part_m + static_cast<size_t>(k) * N + i) : -INFINITY;
      }
#pragma unroll
      for (int b = 0; b < FOLD_BATCH; ++b) mx = fmaxf(mx, v[b]);
    }
  }
  red[g][lane] = mx;
  __syncthreads();
  float M = red[0][lane];
#pragma unroll
  for (int h = 1; h < 8; ++h) M = fmaxf(M, red[h][lane]);
  __syncthreads();
  float s = 0.f;
  if (ok && M != -INFINITY) {
    for (int k0 = g; k0 < splits; k0 += 8 * FOLD_BATCH) {
      float vm[FOLD_BATCH], vs[FOLD_BATCH];
#pragma unroll
      for (int b = 0; b < FOLD_BATCH; ++b) {
        const int k = k0 + 8 * b;
        vm[b] = k < splits ? __ldg(part_m + static_cast<size_t>(k) * N + i) : -INFINITY;
        vs[b] = k < splits ? __ldg(part_s + static_cast<size_t>(k) * N + i) : 0.f;
      }
#pragma unroll
      for (int b = 0; b < FOLD_BATCH; ++b)
        if (vm[b] != -INFINITY) s += vs[b] * expf(vm[b] - M);
    }
  }
  red[g][lane] = s;
  __syncthreads();
  float S = red[0][lane];
#pragma unroll
  for (int h = 1; h < 8; ++h) S += red[h][lane];
  return M + logf(S);
}

__global__ void __launch_bounds__(256) merge_kernel(int N, int V, int splits, const float* __restrict__ part_m,
                                                    const float* __restrict__ part_s, const float* __restrict__ zy,
                                                    const int* __restrict__ targets,
                                                    const uint8_t* __restrict__ mask, float* logp, float* lse,
                                                    int* status, int* zero_ctl) {
  // the control words of the multi-CTA GRPO loss launched next on the stream
  if (zero_ctl && blockIdx.x == 0 && threadIdx.x < GRPO_CTL_WORDS) zero_ctl[threadIdx.x] = 0;
  __shared__ float red[8][33];
  const float L = fold_splits(N, splits, part_m, part_s, red);
  const int i = blockIdx.x * 32 + (threadIdx.x & 31);
  if (threadIdx.x >= 32 || i >= N) return;
  lse[i] = L;
  const int y = targets[i];
  const bool act = mask[i] != 0;
  float lp;
  if (y >= 0 && y < V) {
    lp = zy[i] - L;
  } else if (act) {
    lp = __int_as_float(0x7fc00000);
    atomicOr(status, GH_DEV_TARGET_OOR);
  } else {
    lp = 0.f;
  }
  logp[i] = lp;
  if (!isfinite(L) || (act && y >= 0 && y < V && !isfinite(lp))) atomicOr(status, GH_DEV_NONFINITE);
}

// merge of vocabulary-parallel partials: the splits of all shards in global
// order (the same fold as merge_kernel), the target logit from the shard that
// owns the target column
__global__ void __launch_bounds__(256) merge_shards_kernel(int N, int V_total, int splits,
                                                           const float* __restrict__ part_m,
                                                           const float* __restrict__ part_s,
                                                           const float* __restrict__ zy, const ShardBounds sb,
                                                           const int* __restrict__ targets,
                                                           const uint8_t* __restrict__ mask, float* logp, float* lse,
                                                           int* status) {
  __shared__ float red[8][33];
  const float L = fold_splits(N, splits, part_m, part_s, red);
  const int i = blockIdx.x * 32 + (threadIdx.x & 31);
  if (threadIdx.x >= 32 || i >= N) return;
  lse[i] = L;
  const int y = targets[i];
  const bool act = mask[i] != 0;
  float lp;
  if (y >= 0 && y < V_total) {
    int owner = 0;
    while (owner + 1 < sb.num_shards && y >= sb.start[owner + 1]) ++owner;
    lp = zy[static_cast<size_t>(owner) * N + i] - L;
  } else if (act) {
    lp = __int_as_float(0x7fc00000);
    atomicOr(status, GH_DEV_TARGET_OOR);
  } else {
    lp = 0.f;
  }
  logp[i] = lp;
  if (!isfinite(L) || (act && y >= 0 && y < V_total && !isfinite(lp))) atomicOr(status, GH_DEV_NONFINITE);
}

// ---------------------------------------------------------------- per-sequence CTAs
// The GRPO loss and the GSPO seam give each sequence (segment) to one CTA of
// LB threads.  Thread t takes the sequence's tokens b + t, b + t + LB, ... in
// order, and the block adds the threads' sums in a fixed order (a xor
// butterfly in each warp, then the warp sums in warp order).  The CTA finds
// the sequence's token range [b, e) itself, by a block-wide search of the
// nondecreasing ids, so a sequence's sums depend neither on where it sits in
// the batch nor on how many CTAs run.  Per-sequence results go to a small
// global scratch and the last CTA to finish (elected by an atomic counter
// after a fence; nothing waits) adds them in sequence order.  Without scratch
// one CTA runs the same code over every sequence with the results in shared
// memory, and gives the same bits.
constexpr int LB = 512;
constexpr int LW = LB / 32;
// calls of at most this many tokens get coef from the folding CTA rather than
// from a separate token-parallel kernel
constexpr int LAST_CTA_COEF_MAX = 4096;

struct Red {
  float f0, f1, f2;
  int i0, i1;
};

__device__ __forceinline__ Red red_zero() { return Red{0.f, 0.f, 0.f, 0, 0}; }

__device__ __forceinline__ Red red_warp(Red v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.f0 += __shfl_xor_sync(0xffffffffu, v.f0, o);
    v.f1 += __shfl_xor_sync(0xffffffffu, v.f1, o);
    v.f2 += __shfl_xor_sync(0xffffffffu, v.f2, o);
    v.i0 += __shfl_xor_sync(0xffffffffu, v.i0, o);
    v.i1 += __shfl_xor_sync(0xffffffffu, v.i1, o);
  }
  return v;
}

// Block-wide sum in a fixed order; every thread gets the same bits (the xor
// butterfly is symmetric, and fp32 addition commutes).  sh: LW entries.
__device__ __forceinline__ Red red_block(Red v, Red* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = red_warp(v);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  Red r = lane < LW ? sh[lane] : red_zero();
  r = red_warp(r);
  __syncthreads();
  return r;
}

// First index in [lo, hi) whose key fails `pred`, for keys on which pred holds
// on a prefix (on other keys: some index in [lo, hi]).  Block-wide: LB-way
// sampling narrows the range until one probe per thread decides it.
template <class Pred>
__device__ int block_partition_point(const int* __restrict__ key, int lo, int hi, Pred pred) {
  while (hi - lo > LB) {
    const int step = (hi - lo + LB - 1) / LB;
    const int T = (hi - lo + step - 1) / step;
    const int t = threadIdx.x;
    const bool pr = t < T && pred(key[lo + t * step]);
    const int c = __syncthreads_count(pr);
    const int nlo = c > 0 ? lo + (c - 1) * step + 1 : lo;
    const int nhi = c < T ? lo + c * step : hi;
    lo = nlo;
    hi = nhi;
  }
  const int i = lo + static_cast<int>(threadIdx.x);
  const bool pr = i < hi && pred(key[i]);
  return lo + __syncthreads_count(pr);
}

// Loads of values other CTAs wrote (the last-CTA fold): L2, not a stale L1.
template <bool GLOBAL, class T>
__device__ __forceinline__ T ld_other(const T* p) {
  if constexpr (GLOBAL) return __ldcg(p);
  return *p;
}

// Tokens [a, z) of this CTA's even share of N (the layout checks).
__device__ __forceinline__ void cta_token_slice(int N, long long& a, long long& z) {
  a = static_cast<long long>(blockIdx.x) * N / gridDim.x;
  z = static_cast<long long>(blockIdx.x + 1) * N / gridDim.x;
}

// ---------------------------------------------------------------- GRPO
struct GrpoP {
  int N;
  const float* logp;
  const float* old_logp;
  const float* ref_logp;
  const float* adv;
  const int* seq_id;
  const uint8_t* mask;
  int num_seqs;
  int reduction;
  float eps_low, eps_high, beta, delta;
  int seq_level;
  double norm;
  float* coef;
  float* loss3;
  float* seq_policy;
  float* seq_kl;
  int* seq_count;
  int* num_clipped;
  int* status;
  int direct;    // coef weights known before the reduction (norm > 0 or fixed): written per sequence
  float scale0;  // 1 / norm when direct
};

// Scratch of the multi-CTA GRPO loss: per sequence P, K (sums of the policy
// and KL terms), R (sequence ratio), n (active tokens); ctl: [0] CTAs done,
// [1] bad layout, [2] clipped tokens, [3] scale bits, [4] no-active flag.
struct GrpoScr {
  float* P;
  float* K;
  float* R;
  int* n;
  int* ctl;
};

struct TokTerms {
  float r, pg, kl, d;
  bool act;
};

// Token objective for ratio r: u = min(r, delta) A (cap off when delta <= 0),
// v = clip(r, lo, hi) A, pg = -min(u, v); d pg / d log r = -A r act where act
// follows the active branch (ties count as the unclipped term): the unclipped
// term moves with r unless the cap binds, the clipped one only inside the band.
__device__ __forceinline__ TokTerms grpo_terms(float r, float lp, float rf, float A, float lo, float hi,
                                               float delta) {
  TokTerms t;
  t.r = r;
  const float c = fminf(fmaxf(r, lo), hi);
  const float rr = delta > 0.f ? fminf(r, delta) : r;
  const float u = rr * A, v = c * A;
  t.pg = -fminf(u, v);
  t.d = rf - lp;
  t.kl = expm1f(t.d) - t.d;  // exp(d) - d - 1
  t.act = (u <= v) ? (delta <= 0.f || r <= delta) : (r >= lo && r <= hi);
  return t;
}

// coef_i = w (-A r act + beta (1 - exp(d))) for an active token i of a
// sequence with advantage A, sequence ratio rs (sequence level) and weight w
__device__ __forceinline__ float grpo_coef_of(const GrpoP& p, int i, float A, float rs, float w, float lo,
                                              float hi) {
  const float lp = p.logp[i];
  const float r = p.seq_level ? rs : expf(lp - p.old_logp[i]);
  const TokTerms tt = grpo_terms(r, lp, p.ref_logp ? p.ref_logp[i] : lp, A, lo, hi, p.delta);
  return w * (-A * tt.r * (tt.act ? 1.f : 0.f) - p.beta * expm1f(tt.d));
}

// sequence ratio exp(mean active log-ratio) of tokens [b, e); block-wide
__device__ __forceinline__ float grpo_seq_ratio(const GrpoP& p, int b, int e, Red* sh) {
  Red v = red_zero();
  for (int i = b + static_cast<int>(threadIdx.x); i < e; i += LB) {
    if (!p.mask[i]) continue;
    v.f0 += p.logp[i] - p.old_logp[i];
    v.i0 += 1;
  }
  v = red_block(v, sh);
  return expf(v.i0 > 0 ? v.f0 / static_cast<float>(v.i0) : 0.f);
}

__device__ __forceinline__ float grpo_weight(const GrpoP& p, float scale, int n) {
  return p.reduction == GH_SEQ_MEAN ? (n > 0 ? scale / static_cast<float>(n) : 0.f) : scale;
}

// Normaliser and (loss, policy, kl) from per-sequence totals, summed over
// sequences in index order (lane-strided, then a xor butterfly).  Run by one
// warp; shared by the single-call loss and by grpo_loss_from_sequence_totals so
// that a batch split across data-parallel ranks reduces to the same bits.
// Returns the per-token weight scale (1/T, 1/L or 1/C) and sets *flag_out
// when the normaliser is zero.
template <bool GLOBAL>
__device__ __forceinline__ float grpo_reduce_warp(const float* sP, const float* sK, const int* sN, int num_seqs,
                                                  int reduction, double norm, float beta, int lane, float* loss3,
                                                  int* status, int* flag_out) {
  long long tot = 0;
  int live = 0;
  for (int s = lane; s < num_seqs; s += 32) {
    const int n = ld_other<GLOBAL>(sN + s);
    tot += n;
    live += n > 0 ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    live += __shfl_xor_sync(0xffffffffu, live, o);
  }
  float scale = 0.f;
  int flag = 0;
  if (reduction == GH_TOKEN_MEAN) {
    const double den = norm > 0.0 ? norm : static_cast<double>(tot);
    if (den > 0.0)
      scale = static_cast<float>(1.0 / den);
    else
      flag = 1;
  } else if (reduction == GH_SEQ_MEAN) {
    const double den = norm > 0.0 ? norm : static_cast<double>(live);
    if (den > 0.0)
      scale = static_cast<float>(1.0 / den);
    else
      flag = 1;
  } else {
    scale = static_cast<float>(1.0 / norm);
  }
  float pol = 0.f, kl = 0.f;
  if (!flag) {
    for (int s = lane; s < num_seqs; s += 32) {
      const int n = ld_other<GLOBAL>(sN + s);
      float w = scale;
      if (reduction == GH_SEQ_MEAN) w = n > 0 ? scale / static_cast<float>(n) : 0.f;
      pol += ld_other<GLOBAL>(sP + s) * w;
      kl += ld_other<GLOBAL>(sK + s) * w;
    }
    pol = wsum(pol);
    kl = wsum(kl);
  }
  if (lane == 0) {
    if (flag && status) atomicOr(status, GH_DEV_NO_ACTIVE);
    if (loss3) {
      loss3[0] = pol + beta * kl;
      loss3[1] = pol;
      loss3[2] = kl;
    }
  }
  *flag_out = flag;
  return scale;
}

// The GRPO loss.  SINGLE: one CTA, per-sequence results in dynamic shared
// memory (3 * num_seqs words).  Otherwise a grid of CTAs with GrpoScr, the last
// CTA folding; when the weights are not known upfront, grpo_coef_kernel
// writes coef afterwards.
template <bool SINGLE>
__global__ void __launch_bounds__(LB) grpo_loss_kernel(GrpoP p, GrpoScr g) {
  extern __shared__ float sh_dyn[];
  __shared__ Red red_sh[LW];
  __shared__ int s_bad, s_last, s_clip;
  __shared__ float s_scale;
  __shared__ int s_flag;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  float* P = SINGLE ? sh_dyn : g.P;
  float* K = SINGLE ? sh_dyn + p.num_seqs : g.K;
  int* nn = SINGLE ? reinterpret_cast<int*>(sh_dyn + 2 * p.num_seqs) : g.n;
  if (t == 0) {
    s_bad = 0;
    s_clip = 0;
  }
  __syncthreads();
  const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;

  // layout check of this CTA's share of the tokens: ids in range, nondecreasing
  {
    long long a, z;
    cta_token_slice(p.N, a, z);
    bool bad = false;
    for (long long i = a + t; i < z; i += LB) {
      const int s = p.seq_id[i];
      if (s < 0 || s >= p.num_seqs) bad = true;
      if (i > 0 && p.seq_id[i - 1] > s) bad = true;
    }
    if (__syncthreads_or(bad) && t == 0) {
      if (SINGLE)
        s_bad = 1;
      else
        atomicOr(g.ctl + 1, 1);
    }
  }
  __syncthreads();

  bool nonfinite = false;
  if (!(SINGLE && s_bad)) {
    for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x) {
      const int b = block_partition_point(p.seq_id, 0, p.N, [s](int v) { return v < s; });
      const int e = block_partition_point(p.seq_id, b, p.N, [s](int v) { return v <= s; });
      const float A = p.adv[s];
      const float rs = p.seq_level ? grpo_seq_ratio(p, b, e, red_sh) : 1.f;
      Red v = red_zero();
      for (int i = b + t; i < e; i += LB) {
        if (!p.mask[i]) continue;
        const float lp = p.logp[i];
        const float r = p.seq_level ? rs : expf(lp - p.old_logp[i]);
        const TokTerms tt = grpo_terms(r, lp, p.ref_logp ? p.ref_logp[i] : lp, A, lo, hi, p.delta);
        v.f0 += tt.pg;
        v.f1 += tt.kl;
        v.i0 += 1;
        v.i1 += tt.act ? 0 : 1;
        if (!isfinite(tt.pg) || !isfinite(tt.kl)) nonfinite = true;
      }
      v = red_block(v, red_sh);
      if (t == 0) {
        P[s] = v.f0;
        K[s] = v.f1;
        nn[s] = v.i0;
        if (!SINGLE) g.R[s] = rs;
        if (p.seq_policy) p.seq_policy[s] = v.f0;
        if (p.seq_kl) p.seq_kl[s] = v.f1;
        if (p.seq_count) p.seq_count[s] = v.i0;
        if (SINGLE)
          s_clip += v.i1;
        else if (v.i1)
          atomicAdd(g.ctl + 2, v.i1);
      }
      if (p.coef && p.direct) {
        const float w = grpo_weight(p, p.scale0, v.i0);
        for (int i = b + t; i < e; i += LB) p.coef[i] = p.mask[i] ? grpo_coef_of(p, i, A, rs, w, lo, hi) : 0.f;
      }
    }
  }
  if (nonfinite) atomicOr(p.status, GH_DEV_NONFINITE);

  if (!SINGLE) {
    // the last CTA to finish folds (every other CTA's writes precede its count)
    __threadfence();
    __syncthreads();
    if (t == 0) s_last = atomicAdd(g.ctl, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  __syncthreads();
  const int bad = SINGLE ? s_bad : ld_other<true>(g.ctl + 1);
  if (bad) {
    if (t == 0) {
      atomicOr(p.status, GH_DEV_BAD_SEQ);
      if (p.loss3) p.loss3[0] = p.loss3[1] = p.loss3[2] = __int_as_float(0x7fc00000);
      if (p.num_clipped) *p.num_clipped = 0;
      if (!SINGLE) g.ctl[4] = 1;
    }
    if (p.coef)
      for (int i = t; i < p.N; i += LB) p.coef[i] = 0.f;
    return;
  }
  if (warp == 0) {
    int flag;
    const float scale = grpo_reduce_warp<!SINGLE>(P, K, nn, p.num_seqs, p.reduction, p.norm, p.beta, lane, p.loss3,
                                                  p.status, &flag);
    if (lane == 0) {
      s_scale = scale;
      s_flag = flag;
      if (!SINGLE) {
        g.ctl[3] = __float_as_int(scale);
        g.ctl[4] = flag;
      }
      if (p.num_clipped) *p.num_clipped = SINGLE ? s_clip : ld_other<true>(g.ctl + 2);
    }
  }
  __syncthreads();
  if (!SINGLE && p.coef && !p.direct && p.N <= LAST_CTA_COEF_MAX) {
    // a small call: the folding CTA writes coef itself (one launch fewer)
    const int flag = s_flag;
    for (int i = t; i < p.N; i += LB) {
      float c = 0.f;
      if (p.mask[i] && !flag) {
        const int s = p.seq_id[i];
        c = grpo_coef_of(p, i, p.adv[s], ld_other<true>(g.R + s), grpo_weight(p, s_scale, ld_other<true>(g.n + s)),
                         lo, hi);
      }
      p.coef[i] = c;
    }
    return;
  }
  if (SINGLE && p.coef && !p.direct) {
    // coef_i = w_i (-A r act + beta (1 - exp(d))); at the sequence level r and
    // act are the sequence's (every token of a sequence has the same weight,
    // so the gradient of the shared ratio lands on each token with that weight)
    if (s_flag) {
      for (int i = t; i < p.N; i += LB) p.coef[i] = 0.f;
      return;
    }
    for (int s = 0; s < p.num_seqs; ++s) {
      const int b = block_partition_point(p.seq_id, 0, p.N, [s](int v) { return v < s; });
      const int e = block_partition_point(p.seq_id, b, p.N, [s](int v) { return v <= s; });
      const float A = p.adv[s];
      const float rs = p.seq_level ? grpo_seq_ratio(p, b, e, red_sh) : 1.f;
      const float w = grpo_weight(p, s_scale, nn[s]);
      for (int i = b + t; i < e; i += LB) p.coef[i] = p.mask[i] ? grpo_coef_of(p, i, A, rs, w, lo, hi) : 0.f;
    }
  }
}

// coef of every token once the fold has set the scale (multi-CTA loss with
// the normaliser taken from this call); same arithmetic as grpo_coef_of
// inside the loss kernel
__global__ void __launch_bounds__(256) grpo_coef_kernel(GrpoP p, GrpoScr g) {
  if (g.ctl[1]) return;  // bad layout: the fold already zeroed coef
  const float scale = __int_as_float(g.ctl[3]);
  const int flag = g.ctl[4];
  const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.N; i += gridDim.x * blockDim.x) {
    float c = 0.f;
    if (p.mask[i] && !flag) {
      const int s = p.seq_id[i];
      c = grpo_coef_of(p, i, p.adv[s], g.R[s], grpo_weight(p, scale, g.n[s]), lo, hi);
    }
    p.coef[i] = c;
  }
}

// loss from gathered per-sequence totals (one warp; dynamic shared memory 3 * num_seqs)
__global__ void grpo_totals_kernel(int num_seqs, const float* seq_policy, const float* seq_kl, const int* seq_count,
                                   int reduction, double norm, float beta, float* loss3, int* status) {
  extern __shared__ float sh[];
  float* sP = sh;
  float* sK = sh + num_seqs;
  int* sN = reinterpret_cast<int*>(sh + 2 * num_seqs);
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
    sP[s] = seq_policy[s];
    sK[s] = seq_kl[s];
    sN[s] = seq_count[s];
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int flag;
    grpo_reduce_warp<false>(sP, sK, sN, num_seqs, reduction, norm, beta, threadIdx.x, loss3, status, &flag);
  }
}

// ---------------------------------------------------------------- GSPO
enum { GSPO_FULL = 0, GSPO_PARTIALS = 1, GSPO_FINISH = 2 };

struct GspoP {
  int N;
  const float* logp;
  const float* old_logp;
  const float* ref_logp;  // nullable (beta == 0)
  const uint8_t* mask;
  const int* seg_id;
  int num_segments;
  const float* seg_adv;
  float eps_low, eps_high, beta;
  double divisor;
  int token_weighted;
  float* loss;
  float* seg_ratio;
  float* coef;
  float* mean_logp;
  int* num_clipped;
  int* status;
  int mode;             // GSPO_FULL: one call over the batch; GSPO_PARTIALS / GSPO_FINISH: sequence-parallel steps
  float* fsum;          // PARTIALS out: [2S + 1]
  int* cnt;             // PARTIALS out: [S + 1]
  int R;                // FINISH: pieces
  const float* fsum_all;  // FINISH: [R, 2S + 1]
  const int* cnt_all;     // FINISH: [R, S + 1]
};

// Scratch of the multi-CTA seam: per segment sL (loss term) and lps (sum of
// m logp over this call's tokens); ctl: [0] CTAs done, [1] bad layout,
// [2] clipped segments, [3] active tokens.
struct GspoScr {
  float* sL;
  float* lps;
  int* ctl;
};

struct SegTerms {
  float rho, ell, g, kb;
  bool act;
};

// rho_s = exp(S_s / n_s), l_s = -min(rho A, clip(rho) A), K_s = mean k3 KL:
// the segment's loss term (omega_s / divisor)(l_s + beta K_s), its policy
// gradient per active token g and KL gradient scale kb (zero for n_s = 0,
// where rho is reported as 1)
__device__ __forceinline__ SegTerms gspo_seg_terms(const GspoP& p, float S, float K, int n, float A) {
  SegTerms r{1.f, 0.f, 0.f, 0.f, true};
  if (n <= 0) return r;
  const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;
  const float inv_div = static_cast<float>(1.0 / p.divisor);
  const float nf = static_cast<float>(n);
  r.rho = expf(S / nf);
  const float c = fminf(fmaxf(r.rho, lo), hi);
  const float u = r.rho * A, v = c * A;
  const float pol = -fminf(u, v);
  r.act = (u <= v) ? true : (r.rho >= lo && r.rho <= hi);
  const float omega = p.token_weighted ? nf : 1.f;
  r.ell = omega * inv_div * (pol + p.beta * (K / nf));
  r.g = r.act ? (omega * inv_div) * (-A * r.rho) / nf : 0.f;
  r.kb = (omega * inv_div) * p.beta / nf;
  return r;
}

// The GSPO seam (one call, or one step of the sequence-parallel pair).
// SINGLE: one CTA, sL / lps in dynamic shared memory (2 * S words).
template <bool SINGLE>
__global__ void __launch_bounds__(LB) gspo_seam_kernel(GspoP p, GspoScr g) {
  extern __shared__ float sh_dyn[];
  __shared__ Red red_sh[LW];
  __shared__ int s_bad, s_last, s_clip, s_cnt;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int S = p.num_segments;
  float* sL = SINGLE ? sh_dyn : g.sL;
  float* lps = SINGLE ? sh_dyn + S : g.lps;
  if (t == 0) {
    s_bad = 0;
    s_clip = 0;
    s_cnt = 0;
  }
  __syncthreads();

  // layout check of this CTA's share: ids in [-1, S); ids >= 0 nondecreasing;
  // -1 only as a tail, with mask 0
  {
    long long a, z;
    cta_token_slice(p.N, a, z);
    bool bad = false;
    for (long long i = a + t; i < z; i += LB) {
      const int sg = p.seg_id[i];
      if (sg < -1 || sg >= S) bad = true;
      if (sg < 0 && p.mask[i]) bad = true;
      if (i > 0) {
        const int q = p.seg_id[i - 1];
        if (q < 0 && sg >= 0) bad = true;
        if (q >= 0 && sg >= 0 && q > sg) bad = true;
      }
    }
    if (__syncthreads_or(bad) && t == 0) {
      if (SINGLE)
        s_bad = 1;
      else
        atomicOr(g.ctl + 1, 1);
    }
  }
  __syncthreads();
  const bool writes_coef = p.mode != GSPO_PARTIALS && p.coef;
  bool nonfinite = false;
  if (!(SINGLE && s_bad)) {
    const int nvalid = block_partition_point(p.seg_id, 0, p.N, [](int v) { return v >= 0; });
    if (writes_coef)  // the -1 tail: this CTA's share
      for (int i = nvalid + blockIdx.x * LB + t; i < p.N; i += gridDim.x * LB) p.coef[i] = 0.f;
    for (int sg = blockIdx.x; sg < S; sg += gridDim.x) {
      const int b = block_partition_point(p.seg_id, 0, nvalid, [sg](int v) { return v < sg; });
      const int e = block_partition_point(p.seg_id, b, nvalid, [sg](int v) { return v <= sg; });
      Red v = red_zero();
      for (int i = b + t; i < e; i += LB) {
        if (!p.mask[i]) continue;
        const float lp = p.logp[i];
        if (p.mode != GSPO_FINISH) {
          v.f0 += lp - p.old_logp[i];
          if (p.ref_logp) {
            const float d = p.ref_logp[i] - lp;
            v.f1 += expm1f(d) - d;
          }
        }
        v.f2 += lp;
        v.i0 += 1;
      }
      v = red_block(v, red_sh);
      if (p.mode == GSPO_PARTIALS) {
        if (t == 0) {
          p.fsum[sg] = v.f0;
          p.fsum[S + sg] = v.f1;
          p.cnt[sg] = v.i0;
          lps[sg] = v.f2;
          if (SINGLE)
            s_cnt += v.i0;
          else if (v.i0)
            atomicAdd(g.ctl + 3, v.i0);
          if (!isfinite(v.f0) || !isfinite(v.f1)) nonfinite = true;
        }
        continue;
      }
      // the segment's sums over every piece, in piece order (one piece: 0 + x)
      float Ssum = 0.f, Ksum = 0.f;
      int n = 0;
      if (p.mode == GSPO_FULL) {
        Ssum += v.f0;
        Ksum += v.f1;
        n += v.i0;
      } else {
        for (int r = 0; r < p.R; ++r) {
          Ssum += p.fsum_all[static_cast<size_t>(r) * (2 * S + 1) + sg];
          Ksum += p.fsum_all[static_cast<size_t>(r) * (2 * S + 1) + S + sg];
          n += p.cnt_all[static_cast<size_t>(r) * (S + 1) + sg];
        }
      }
      const SegTerms st = gspo_seg_terms(p, Ssum, Ksum, n, n > 0 ? p.seg_adv[sg] : 0.f);
      if (t == 0) {
        sL[sg] = st.ell;
        lps[sg] = v.f2;
        if (p.seg_ratio) p.seg_ratio[sg] = st.rho;
        const int clipped = (n > 0 && !st.act) ? 1 : 0;
        if (SINGLE) {
          s_clip += clipped;
          s_cnt += v.i0;
        } else {
          if (clipped) atomicAdd(g.ctl + 2, 1);
          if (v.i0) atomicAdd(g.ctl + 3, v.i0);
        }
        if (!isfinite(v.f0) || !isfinite(v.f1) || (n > 0 && (!isfinite(st.rho) || !isfinite(st.ell))))
          nonfinite = true;
      }
      if (writes_coef)
        for (int i = b + t; i < e; i += LB) {
          float c = 0.f;
          if (p.mask[i]) {
            c = st.g;
            if (p.ref_logp) c -= st.kb * expm1f(p.ref_logp[i] - p.logp[i]);
          }
          p.coef[i] = c;
        }
    }
  }
  if (nonfinite) atomicOr(p.status, GH_DEV_NONFINITE);

  if (!SINGLE) {
    __threadfence();
    __syncthreads();
    if (t == 0) s_last = atomicAdd(g.ctl, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  __syncthreads();
  const int bad = SINGLE ? s_bad : ld_other<true>(g.ctl + 1);
  if (bad) {
    if (t == 0) {
      atomicOr(p.status, GH_DEV_BAD_SEQ);
      if (p.mode != GSPO_PARTIALS && p.loss) p.loss[0] = __int_as_float(0x7fc00000);
      if (p.num_clipped) *p.num_clipped = 0;
    }
    if (writes_coef)
      for (int i = t; i < p.N; i += LB) p.coef[i] = 0.f;
    return;
  }
  if (warp != 0) return;
  // segment-ordered sums of the per-segment results (lane-strided, then a xor butterfly)
  float L = 0.f, a = 0.f;
  for (int sg = lane; sg < S; sg += 32) {
    if (p.mode != GSPO_PARTIALS) L += ld_other<!SINGLE>(sL + sg);
    if (p.mode != GSPO_FINISH) a += ld_other<!SINGLE>(lps + sg);
  }
  L = wsum(L);
  a = wsum(a);
  if (lane != 0) return;
  const int total = SINGLE ? s_cnt : ld_other<true>(g.ctl + 3);
  if (p.mode == GSPO_PARTIALS) {
    p.fsum[2 * S] = a;
    p.cnt[S] = total;
    return;
  }
  p.loss[0] = L;
  if (p.num_clipped) *p.num_clipped = SINGLE ? s_clip : ld_other<true>(g.ctl + 2);
  if (p.mean_logp) {
    // the new_logprobs metric over every piece, in piece order (one piece: 0 + x)
    float sa = 0.f;
    int sn = 0;
    if (p.mode == GSPO_FULL) {
      sa += a;
      sn += total;
    } else {
      for (int r = 0; r < p.R; ++r) {
        sa += p.fsum_all[static_cast<size_t>(r) * (2 * S + 1) + 2 * S];
        sn += p.cnt_all[static_cast<size_t>(r) * (S + 1) + S];
      }
    }
    p.mean_logp[0] = sn > 0 ? sa / static_cast<float>(sn) : 0.f;
  }
}

// ---------------------------------------------------------------- advantages
__global__ void advantage_kernel(const float* rewards, int num_seqs, int group_size, float eps, float* adv) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  const int groups = num_seqs / group_size;
  if (g >= groups) return;
  const float* r = rewards + static_cast<size_t>(g) * group_size;
  double mean = 0.0;
  for (int k = 0; k < group_size; ++k) mean += r[k];
  mean /= group_size;
  double var = 0.0;
  for (int k = 0; k < group_size; ++k) var += (r[k] - mean) * (r[k] - mean);
  const double sd = group_size > 1 ? sqrt(var / (group_size - 1)) : 0.0;
  for (int k = 0; k < group_size; ++k)
    adv[static_cast<size_t>(g) * group_size + k] = static_cast<float>((r[k] - mean) / (sd + eps));
}

// ---------------------------------------------------------------- dH shard merge
__global__ void dh_merge_kernel(int num_shards, size_t n, bool to_bf16, const float* __restrict__ partials,
                                void* out) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float v = 0.f;
    for (int r = 0; r < num_shards; ++r) v += partials[static_cast<size_t>(r) * n + i];
    if (to_bf16)
      static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    else
      static_cast<float*>(out)[i] = v;
  }
}

// ---------------------------------------------------------------- timeout probe
__global__ void timeout_probe_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: the bounded wait must give up and report it
    mbar_wait_bounded(&bar, 0, &abort_flag, status, GH_DEV_TIMEOUT, timeout_ns);
  }
  __syncthreads();
}

}  // namespace

// The counters inside the GRPO loss's scratch: after the four per-sequence
// arrays of grpo_loss_scratch_seqs(N) entries, each 256-byte aligned.
int* grpo_scratch_ctl(void* scratch, int64_t N) {
  const size_t a = align_up(static_cast<size_t>(grpo_loss_scratch_seqs(N)) * 4, 256);
  return reinterpret_cast<int*>(static_cast<char*>(scratch) + 4 * a);
}

cudaError_t launch_merge(int N, int V, int splits, const float* part_m, const float* part_s, const float* zy,
                         const int32_t* targets, const uint8_t* mask, float* logp, float* lse, int* status,
                         void* grpo_scratch, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  int* ctl = grpo_scratch ? grpo_scratch_ctl(grpo_scratch, N) : nullptr;
  merge_kernel<<<static_cast<unsigned>(ceil_div(N, 32)), 256, 0, st>>>(N, V, splits, part_m, part_s, zy, targets,
                                                                        mask, logp, lse, status, ctl);
  return cudaGetLastError();
}

cudaError_t launch_merge_shards(int N, int V_total, int splits, const float* part_m, const float* part_s,
                                const float* zy, const ShardBounds& sb, const int32_t* targets, const uint8_t* mask,
                                float* logp, float* lse, int* status, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  merge_shards_kernel<<<static_cast<unsigned>(ceil_div(N, 32)), 256, 0, st>>>(N, V_total, splits, part_m, part_s, zy,
                                                                               sb, targets, mask, logp, lse, status);
  return cudaGetLastError();
}

size_t grpo_loss_scratch_bytes(int64_t N) {
  if (N <= 0) return 0;  // nothing to spread over CTAs
  const int64_t cap = grpo_loss_scratch_seqs(N);
  return align_up(static_cast<size_t>(cap) * 4, 256) * 4 + 256;
}

int64_t grpo_loss_scratch_seqs(int64_t N) {
  const int64_t c = N / 8 > 64 ? N / 8 : 64;
  return c < MAX_SEQS ? c : MAX_SEQS;
}

// CTAs of the multi-CTA loss kernels: one per sequence, at most four per SM
static unsigned loss_grid(int num_seqs) {
  const int cap = 4 * num_sms();
  return static_cast<unsigned>(num_seqs < cap ? num_seqs : cap);
}

static bool loss_one_cta_knob() {
  static const int v = [] {
    const char* e = getenv("GH_LOSS_ONE_CTA");
    return e && atoi(e) == 1 ? 1 : 0;
  }();
  return v == 1;
}

cudaError_t launch_grpo(int N, const float* logp, const uint8_t* mask, const gh_grpo* g, float* coef, float* loss3,
                        int* status, void* scratch, bool ctl_zeroed, cudaStream_t st) {
  GrpoP p;
  p.N = N;
  p.logp = logp;
  p.old_logp = g->old_logp;
  p.ref_logp = g->ref_logp;
  p.adv = g->adv;
  p.seq_id = g->seq_id;
  p.mask = mask;
  p.num_seqs = g->num_seqs;
  p.reduction = g->reduction;
  p.eps_low = g->eps_low;
  p.eps_high = g->eps_high;
  p.beta = g->beta;
  p.delta = g->delta;
  p.seq_level = g->ratio_level;
  p.norm = g->norm;
  p.coef = coef;
  p.loss3 = loss3;
  p.seq_policy = g->seq_policy;
  p.seq_kl = g->seq_kl;
  p.seq_count = g->seq_count;
  p.num_clipped = g->num_clipped;
  p.status = status;
  p.direct = (g->reduction == GH_FIXED || g->norm > 0.0) ? 1 : 0;
  p.scale0 = p.direct ? static_cast<float>(1.0 / g->norm) : 0.f;
  const int S = g->num_seqs;
  GrpoScr gs{};
  if (scratch && S <= grpo_loss_scratch_seqs(N) && !loss_one_cta_knob()) {
    const size_t a = align_up(static_cast<size_t>(grpo_loss_scratch_seqs(N)) * 4, 256);
    char* b = static_cast<char*>(scratch);
    gs.P = reinterpret_cast<float*>(b);
    gs.K = reinterpret_cast<float*>(b + a);
    gs.R = reinterpret_cast<float*>(b + 2 * a);
    gs.n = reinterpret_cast<int*>(b + 3 * a);
    gs.ctl = grpo_scratch_ctl(scratch, N);
    cudaError_t e = cudaSuccess;
    if (!ctl_zeroed) e = cudaMemsetAsync(gs.ctl, 0, GRPO_CTL_WORDS * sizeof(int), st);
    if (e != cudaSuccess) return e;
    grpo_loss_kernel<false><<<loss_grid(S), LB, 0, st>>>(p, gs);
    e = cudaGetLastError();
    if (e != cudaSuccess || !coef || p.direct || N <= LAST_CTA_COEF_MAX) return e;
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(ceil_div(N, 256), 4 * num_sms()));
    grpo_coef_kernel<<<blocks, 256, 0, st>>>(p, gs);
    count_extra_launch();
    return cudaGetLastError();
  }
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(grpo_loss_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  grpo_loss_kernel<true><<<1, LB, static_cast<size_t>(3) * S * sizeof(float), st>>>(p, gs);
  return cudaGetLastError();
}

cudaError_t launch_grpo_totals(int num_seqs, const float* seq_policy, const float* seq_kl, const int32_t* seq_count,
                               int reduction, double norm, float beta, float* loss3, int* status, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(grpo_totals_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  grpo_totals_kernel<<<1, 256, static_cast<size_t>(3) * num_seqs * sizeof(float), st>>>(
      num_seqs, seq_policy, seq_kl, seq_count, reduction, norm, beta, loss3, status);
  return cudaGetLastError();
}

size_t gspo_scratch_bytes(int num_segments) {
  return align_up(static_cast<size_t>(num_segments) * 4, 256) * 2 + 256;
}

static GspoP gspo_params(const GspoArgs& g) {
  GspoP p{};
  p.N = g.N;
  p.logp = g.logp;
  p.old_logp = g.old_logp;
  p.ref_logp = g.ref_logp;
  p.mask = g.mask;
  p.seg_id = g.seg_id;
  p.num_segments = g.num_segments;
  p.seg_adv = g.seg_adv;
  p.eps_low = g.eps_low;
  p.eps_high = g.eps_high;
  p.beta = g.beta;
  p.divisor = g.divisor;
  p.token_weighted = g.token_weighted;
  p.loss = g.loss;
  p.seg_ratio = g.seg_ratio;
  p.coef = g.coef;
  p.mean_logp = g.mean_logp;
  p.num_clipped = g.num_clipped;
  p.status = g.status;
  return p;
}

// One launch of the seam in either shape: a grid of CTAs over the caller's
// scratch, or one CTA with shared memory when there is none.
static cudaError_t launch_seam(GspoP p, void* scratch, cudaStream_t st) {
  const int S = p.num_segments;
  GspoScr gs{};
  if (scratch && !loss_one_cta_knob()) {
    const size_t a = align_up(static_cast<size_t>(S) * 4, 256);
    char* b = static_cast<char*>(scratch);
    gs.sL = reinterpret_cast<float*>(b);
    gs.lps = reinterpret_cast<float*>(b + a);
    gs.ctl = reinterpret_cast<int*>(b + 2 * a);
    cudaError_t e = cudaMemsetAsync(gs.ctl, 0, 8 * sizeof(int), st);
    if (e != cudaSuccess) return e;
    gspo_seam_kernel<false><<<loss_grid(S), LB, 0, st>>>(p, gs);
    return cudaGetLastError();
  }
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gspo_seam_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         2 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  gspo_seam_kernel<true><<<1, LB, static_cast<size_t>(2) * S * sizeof(float), st>>>(p, gs);
  return cudaGetLastError();
}

cudaError_t launch_gspo(const GspoArgs& g, void* scratch, cudaStream_t st) {
  GspoP p = gspo_params(g);
  p.mode = GSPO_FULL;
  return launch_seam(p, scratch, st);
}

cudaError_t launch_gspo_partials(const GspoArgs& g, float* fsum, int32_t* cnt, void* scratch, cudaStream_t st) {
  GspoP p = gspo_params(g);
  p.mode = GSPO_PARTIALS;
  p.fsum = fsum;
  p.cnt = cnt;
  return launch_seam(p, scratch, st);
}

cudaError_t launch_gspo_finish(const GspoArgs& g, int R, const float* fsum_all, const int32_t* cnt_all, void* scratch,
                               cudaStream_t st) {
  GspoP p = gspo_params(g);
  p.mode = GSPO_FINISH;
  p.R = R;
  p.fsum_all = fsum_all;
  p.cnt_all = cnt_all;
  return launch_seam(p, scratch, st);
}

cudaError_t launch_advantage(const float* rewards, int num_seqs, int group_size, float eps, float* adv,
                             cudaStream_t st) {
  const int groups = num_seqs / group_size;
  if (groups <= 0) return cudaSuccess;
  advantage_kernel<<<static_cast<unsigned>(ceil_div(groups, 128)), 128, 0, st>>>(rewards, num_seqs, group_size, eps,
                                                                                 adv);
  return cudaGetLastError();
}

cudaError_t launch_dh_merge(int num_shards, size_t n, bool to_bf16, const float* partials, void* out,
                            cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 152 * 16));
  dh_merge_kernel<<<blocks, 256, 0, st>>>(num_shards, n, to_bf16, partials, out);
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* status, uint64_t tmo, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(status, tmo);
  return cudaGetLastError();
}

}  // namespace gh
