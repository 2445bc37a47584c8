// O(N) kernels: split merge -> LSE / logp, the GRPO token objective and its
// reductions, the GSPO segment seam, group-normalised advantages, and the
// bounded-wait self-test.  All sums run in a fixed order (lane-strided partial
// sums in token order, then a xor butterfly or a fixed shared-memory tree), so
// results are deterministic without floating-point atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace gh {

namespace {

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int wsum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// first index in [lo, hi) with key[idx] >= v (key nondecreasing on [lo, hi))
__device__ __forceinline__ int lower_bound_i(const int* key, int lo, int hi, int v) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (key[mid] < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
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
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 32 + lane;
  const bool ok = i < N;
  float mx = -INFINITY;
  if (ok)
    for (int k = g; k < splits; k += 8) mx = fmaxf(mx, part_m[static_cast<size_t>(k) * N + i]);
  red[g][lane] = mx;
  __syncthreads();
  float M = red[0][lane];
#pragma unroll
  for (int h = 1; h < 8; ++h) M = fmaxf(M, red[h][lane]);
  __syncthreads();
  float s = 0.f;
  if (ok && M != -INFINITY) {
    for (int k = g; k < splits; k += 8) {
      const float mk = part_m[static_cast<size_t>(k) * N + i];
      if (mk != -INFINITY) s += part_s[static_cast<size_t>(k) * N + i] * expf(mk - M);
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
                                                    int* status) {
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
  int* status;
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

// Sequence s's tokens [b, e): mean active log-ratio (lane-strided partial sums
// in token order, then a xor butterfly) and active count.  The same code runs
// wherever the sequence sits in the batch, so the bits do not depend on it.
__device__ __forceinline__ void seq_log_ratio(const GrpoP& p, int b, int e, int lane, float& lr, int& n) {
  float acc = 0.f;
  int cnt = 0;
  for (int i = b + lane; i < e; i += 32) {
    if (!p.mask[i]) continue;
    acc += p.logp[i] - p.old_logp[i];
    cnt += 1;
  }
  acc = wsum(acc);
  cnt = wsum_i(cnt);
  n = cnt;
  lr = cnt > 0 ? acc / static_cast<float>(cnt) : 0.f;
}

// Normaliser and (loss, policy, kl) from per-sequence totals, summed over
// sequences in index order (lane-strided, then a xor butterfly).  Run by one
// warp; shared by the single-call loss and by grpo_loss_from_sequence_totals so
// that a batch split across data-parallel ranks reduces to the same bits.
// Returns the per-token weight scale (1/T, 1/L or 1/C) and sets *flag when
// the normaliser is zero.
__device__ __forceinline__ float grpo_reduce_warp(const float* sP, const float* sK, const int* sN, int num_seqs,
                                                  int reduction, double norm, float beta, int lane, float* loss3,
                                                  int* status, int* flag_out) {
  long long tot = 0;
  int live = 0;
  for (int s = lane; s < num_seqs; s += 32) {
    tot += sN[s];
    live += sN[s] > 0 ? 1 : 0;
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
      float w = scale;
      if (reduction == GH_SEQ_MEAN) w = sN[s] > 0 ? scale / static_cast<float>(sN[s]) : 0.f;
      pol += sP[s] * w;
      kl += sK[s] * w;
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

// one CTA of 1024 threads; dynamic shared memory: 3 * num_seqs words
__global__ void __launch_bounds__(1024) grpo_kernel(GrpoP p) {
  extern __shared__ float sh[];
  float* sP = sh;
  float* sK = sh + p.num_seqs;
  int* sN = reinterpret_cast<int*>(sh + 2 * p.num_seqs);
  __shared__ float s_scale;
  __shared__ int s_flag;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, nw = blockDim.x >> 5;
  const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;

  // phase 0: layout check -- ids in range and nondecreasing
  bool bad = false;
  for (int i = t; i < p.N; i += blockDim.x) {
    const int s = p.seq_id[i];
    if (s < 0 || s >= p.num_seqs) bad = true;
    if (i > 0 && p.seq_id[i - 1] > s) bad = true;
  }
  if (__syncthreads_or(bad)) {
    if (t == 0) {
      atomicOr(p.status, GH_DEV_BAD_SEQ);
      if (p.loss3) p.loss3[0] = p.loss3[1] = p.loss3[2] = __int_as_float(0x7fc00000);
    }
    if (p.coef)
      for (int i = t; i < p.N; i += blockDim.x) p.coef[i] = 0.f;
    return;
  }

  // phase 1: per-sequence totals of m*pg, m*kl and active counts (warp per sequence)
  bool nonfinite = false;
  for (int s = warp; s < p.num_seqs; s += nw) {
    const int b = lower_bound_i(p.seq_id, 0, p.N, s);
    const int e = lower_bound_i(p.seq_id, b, p.N, s + 1);
    const float A = p.adv[s];
    float rs = 1.f;
    if (p.seq_level) {
      float lr;
      int n;
      seq_log_ratio(p, b, e, lane, lr, n);
      rs = expf(lr);
    }
    float ap = 0.f, ak = 0.f;
    int an = 0;
    for (int i = b + lane; i < e; i += 32) {
      if (!p.mask[i]) continue;
      const float lp = p.logp[i];
      const float r = p.seq_level ? rs : expf(lp - p.old_logp[i]);
      const TokTerms tt = grpo_terms(r, lp, p.ref_logp ? p.ref_logp[i] : lp, A, lo, hi, p.delta);
      ap += tt.pg;
      ak += tt.kl;
      an += 1;
      if (!isfinite(tt.pg) || !isfinite(tt.kl)) nonfinite = true;
    }
    ap = wsum(ap);
    ak = wsum(ak);
    an = wsum_i(an);
    if (lane == 0) {
      sP[s] = ap;
      sK[s] = ak;
      sN[s] = an;
      if (p.seq_policy) p.seq_policy[s] = ap;
      if (p.seq_kl) p.seq_kl[s] = ak;
      if (p.seq_count) p.seq_count[s] = an;
    }
  }
  if (nonfinite) atomicOr(p.status, GH_DEV_NONFINITE);
  __syncthreads();

  // phase 2 (warp 0): normaliser, then (loss, policy, kl)
  if (warp == 0) {
    int flag;
    const float scale = grpo_reduce_warp(sP, sK, sN, p.num_seqs, p.reduction, p.norm, p.beta, lane, p.loss3,
                                         p.status, &flag);
    if (lane == 0) {
      s_scale = scale;
      s_flag = flag;
    }
  }
  __syncthreads();

  // phase 3 (warp per sequence): coef_i = w_i (-A r act + beta (1 - exp(d)));
  // at the sequence level r and act are the sequence's (every token of a
  // sequence has the same weight, so the gradient of the shared ratio lands
  // on each token with that weight)
  if (p.coef) {
    const float scale = s_scale;
    const int flag = s_flag;
    for (int i = t; i < p.N; i += blockDim.x)
      if (!p.mask[i] || flag) p.coef[i] = 0.f;
    if (!flag) {
      for (int s = warp; s < p.num_seqs; s += nw) {
        const int b = lower_bound_i(p.seq_id, 0, p.N, s);
        const int e = lower_bound_i(p.seq_id, b, p.N, s + 1);
        const float A = p.adv[s];
        float rs = 1.f;
        if (p.seq_level) {
          float lr;
          int n;
          seq_log_ratio(p, b, e, lane, lr, n);
          rs = expf(lr);
        }
        const float w = p.reduction == GH_SEQ_MEAN ? (sN[s] > 0 ? scale / static_cast<float>(sN[s]) : 0.f) : scale;
        for (int i = b + lane; i < e; i += 32) {
          if (!p.mask[i]) continue;
          const float lp = p.logp[i];
          const float r = p.seq_level ? rs : expf(lp - p.old_logp[i]);
          const TokTerms tt = grpo_terms(r, lp, p.ref_logp ? p.ref_logp[i] : lp, A, lo, hi, p.delta);
          p.coef[i] = w * (-A * tt.r * (tt.act ? 1.f : 0.f) - p.beta * expm1f(tt.d));
        }
      }
    }
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
    grpo_reduce_warp(sP, sK, sN, num_seqs, reduction, norm, beta, threadIdx.x, loss3, status, &flag);
  }
}

// ---------------------------------------------------------------- GSPO
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
  int* status;
};

// Layout check (ids in [-1, S); ids >= 0 nondecreasing; -1 only as a tail,
// with mask 0) and the start of the -1 tail.  Block-wide; false on a bad
// layout, after flagging it and zeroing coef.
__device__ bool gspo_layout(const GspoP& p, int* s_nvalid) {
  const int t = threadIdx.x;
  bool bad = false;
  for (int i = t; i < p.N; i += blockDim.x) {
    const int sg = p.seg_id[i];
    if (sg < -1 || sg >= p.num_segments) bad = true;
    if (sg < 0 && p.mask[i]) bad = true;
    if (i > 0) {
      const int q = p.seg_id[i - 1];
      if (q < 0 && sg >= 0) bad = true;
      if (q >= 0 && sg >= 0 && q > sg) bad = true;
    }
  }
  if (__syncthreads_or(bad)) {
    if (t == 0) {
      atomicOr(p.status, GH_DEV_BAD_SEQ);
      if (p.loss) p.loss[0] = __int_as_float(0x7fc00000);
    }
    if (p.coef)
      for (int i = t; i < p.N; i += blockDim.x) p.coef[i] = 0.f;
    return false;
  }
  if (t == 0) {
    int lo_i = 0, hi_i = p.N;
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i) >> 1;
      if (p.seg_id[mid] >= 0)
        lo_i = mid + 1;
      else
        hi_i = mid;
    }
    *s_nvalid = lo_i;
  }
  __syncthreads();
  return true;
}

// Per-segment partial sums of this call's tokens (warp per segment, lane-
// strided in token order, then a xor butterfly): fS[s] = sum m (logp - old),
// fK[s] = sum m kl, cnt[s] = active tokens; and *lps / *lpn = sum m logp and
// sum m over all tokens (fixed shared-memory tree).
__device__ void gspo_partials(const GspoP& p, int nvalid, float* fS, float* fK, int* cnt, float* lps, int* lpn,
                              float* red_a, int* red_b) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, nw = blockDim.x >> 5;
  bool nonfinite = false;
  for (int sg = warp; sg < p.num_segments; sg += nw) {
    const int b = lower_bound_i(p.seg_id, 0, nvalid, sg);
    const int e = lower_bound_i(p.seg_id, b, nvalid, sg + 1);
    float acc = 0.f, kacc = 0.f;
    int c = 0;
    for (int i = b + lane; i < e; i += 32) {
      if (!p.mask[i]) continue;
      const float lp = p.logp[i];
      acc += lp - p.old_logp[i];
      if (p.ref_logp) {
        const float d = p.ref_logp[i] - lp;
        kacc += expm1f(d) - d;
      }
      c += 1;
    }
    acc = wsum(acc);
    kacc = wsum(kacc);
    c = wsum_i(c);
    if (!isfinite(acc) || !isfinite(kacc)) nonfinite = true;
    if (lane == 0) {
      fS[sg] = acc;
      fK[sg] = kacc;
      cnt[sg] = c;
    }
  }
  if (nonfinite) atomicOr(p.status, GH_DEV_NONFINITE);
  float a = 0.f;
  int n = 0;
  for (int i = t; i < p.N; i += blockDim.x)
    if (p.mask[i]) {
      a += p.logp[i];
      n += 1;
    }
  a = wsum(a);
  n = wsum_i(n);
  if (lane == 0) {
    red_a[warp] = a;
    red_b[warp] = n;
  }
  __syncthreads();
  if (warp == 0) {
    float x = lane < nw ? red_a[lane] : 0.f;
    int y = lane < nw ? red_b[lane] : 0;
    x = wsum(x);
    y = wsum_i(y);
    if (lane == 0) {
      *lps = x;
      *lpn = y;
    }
  }
  __syncthreads();
}

// Loss from the partials of R contiguous pieces of the batch (R = 1 for one
// call; sequence-parallel ranks otherwise), summed over pieces in order:
// rho_s = exp(S_s / n_s), l_s = -min(rho A, clip(rho) A), K_s = mean k3 KL,
// loss = sum_s (omega_s / divisor)(l_s + beta K_s).  Leaves per segment
// sL = loss term, sG = policy gradient per active token, sB = KL gradient
// scale per active token (these may alias fS, fK, cnt when R = 1: each
// segment is read and then written by the same thread).  Writes loss,
// seg_ratio and mean_logp.
__device__ void gspo_finish(const GspoP& p, int R, int fstride, int cstride, const float* fS, const float* fK,
                            const int* cnt, const float* lps, const int* lpn, float* sL, float* sG, float* sB) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;
  const float inv_div = static_cast<float>(1.0 / p.divisor);
  bool nonfinite = false;
  for (int sg = t; sg < p.num_segments; sg += blockDim.x) {
    float S = 0.f, K = 0.f;
    int n = 0;
    for (int r = 0; r < R; ++r) {
      S += fS[r * fstride + sg];
      K += fK[r * fstride + sg];
      n += cnt[r * cstride + sg];
    }
    float rho = 1.f, ell = 0.f, g = 0.f, kb = 0.f;
    if (n > 0) {
      const float A = p.seg_adv[sg];
      const float nf = static_cast<float>(n);
      rho = expf(S / nf);
      const float c = fminf(fmaxf(rho, lo), hi);
      const float u = rho * A, v = c * A;
      const float pol = -fminf(u, v);
      const bool act = (u <= v) ? true : (rho >= lo && rho <= hi);
      const float omega = p.token_weighted ? nf : 1.f;
      ell = omega * inv_div * (pol + p.beta * (K / nf));
      g = act ? (omega * inv_div) * (-A * rho) / nf : 0.f;
      kb = (omega * inv_div) * p.beta / nf;
      if (!isfinite(rho) || !isfinite(ell)) nonfinite = true;
    }
    sL[sg] = ell;
    sG[sg] = g;
    sB[sg] = kb;
    if (p.seg_ratio) p.seg_ratio[sg] = rho;
  }
  if (nonfinite) atomicOr(p.status, GH_DEV_NONFINITE);
  __syncthreads();
  if (warp == 0) {
    float L = 0.f;
    for (int sg = lane; sg < p.num_segments; sg += 32) L += sL[sg];
    L = wsum(L);
    if (lane == 0) {
      p.loss[0] = L;
      if (p.mean_logp) {
        float a = 0.f;
        int n = 0;
        for (int r = 0; r < R; ++r) {
          a += lps[r * fstride];
          n += lpn[r * cstride];
        }
        p.mean_logp[0] = n > 0 ? a / static_cast<float>(n) : 0.f;
      }
    }
  }
}

// coef_i = m_i (sG[s] + sB[s] (1 - exp(ref_i - logp_i))) for this call's tokens
__device__ void gspo_coef(const GspoP& p, const float* sG, const float* sB) {
  for (int i = threadIdx.x; i < p.N; i += blockDim.x) {
    const int sg = p.seg_id[i];
    float c = 0.f;
    if (sg >= 0 && p.mask[i]) {
      c = sG[sg];
      if (p.ref_logp) c -= sB[sg] * expm1f(p.ref_logp[i] - p.logp[i]);
    }
    p.coef[i] = c;
  }
}

// one call over the whole batch: one CTA of 1024 threads; dynamic shared
// memory 3 * num_segments words (partials, reused for the per-segment results)
__global__ void __launch_bounds__(1024) gspo_kernel(GspoP p) {
  extern __shared__ float sh[];
  float* fS = sh;
  float* fK = sh + p.num_segments;
  int* cnt = reinterpret_cast<int*>(sh + 2 * p.num_segments);
  __shared__ float red_a[32];
  __shared__ int red_b[32];
  __shared__ int s_nvalid;
  __shared__ float s_lps;
  __shared__ int s_lpn;
  if (!gspo_layout(p, &s_nvalid)) return;
  gspo_partials(p, s_nvalid, fS, fK, cnt, &s_lps, &s_lpn, red_a, red_b);
  gspo_finish(p, 1, 0, 0, fS, fK, cnt, &s_lps, &s_lpn, fS, fK, reinterpret_cast<float*>(cnt));
  __syncthreads();
  gspo_coef(p, fS + p.num_segments, reinterpret_cast<float*>(cnt));
}

// sequence-parallel step 1: this rank's partials to global memory
// fsum [2S + 1] = (S_s..., K_s..., sum m logp), cnt [S + 1] = (n_s..., sum m)
__global__ void __launch_bounds__(1024) gspo_partials_kernel(GspoP p, float* fsum, int* cnt) {
  __shared__ float red_a[32];
  __shared__ int red_b[32];
  __shared__ int s_nvalid;
  if (!gspo_layout(p, &s_nvalid)) return;
  const int S = p.num_segments;
  gspo_partials(p, s_nvalid, fsum, fsum + S, cnt, fsum + 2 * S, cnt + S, red_a, red_b);
}

// sequence-parallel step 2: loss from R ranks' gathered partials, coef for
// this rank's tokens; dynamic shared memory 3 * num_segments words
__global__ void __launch_bounds__(1024) gspo_finish_kernel(GspoP p, int R, const float* fsum_all,
                                                           const int* cnt_all) {
  extern __shared__ float sh[];
  float* sL = sh;
  float* sG = sh + p.num_segments;
  float* sB = sh + 2 * p.num_segments;
  __shared__ int s_nvalid;
  if (!gspo_layout(p, &s_nvalid)) return;
  const int S = p.num_segments;
  gspo_finish(p, R, 2 * S + 1, S + 1, fsum_all, fsum_all + S, cnt_all, fsum_all + 2 * S, cnt_all + S, sL, sG, sB);
  __syncthreads();
  gspo_coef(p, sG, sB);
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

cudaError_t launch_merge(int N, int V, int splits, const float* part_m, const float* part_s, const float* zy,
                         const int32_t* targets, const uint8_t* mask, float* logp, float* lse, int* status,
                         cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  merge_kernel<<<static_cast<unsigned>(ceil_div(N, 32)), 256, 0, st>>>(N, V, splits, part_m, part_s, zy, targets,
                                                                        mask, logp, lse, status);
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

cudaError_t launch_grpo(int N, const float* logp, const uint8_t* mask, const gh_grpo* g, float* coef, float* loss3,
                        int* status, cudaStream_t st) {
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
  p.status = status;
  const size_t sm = static_cast<size_t>(3) * g->num_seqs * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(grpo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  grpo_kernel<<<1, 1024, sm, st>>>(p);
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

static GspoP gspo_params(const GspoArgs& g) {
  GspoP p;
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
  p.status = g.status;
  return p;
}

cudaError_t launch_gspo(const GspoArgs& g, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gspo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  gspo_kernel<<<1, 1024, static_cast<size_t>(3) * g.num_segments * sizeof(float), st>>>(gspo_params(g));
  return cudaGetLastError();
}

cudaError_t launch_gspo_partials(const GspoArgs& g, float* fsum, int32_t* cnt, cudaStream_t st) {
  gspo_partials_kernel<<<1, 1024, 0, st>>>(gspo_params(g), fsum, cnt);
  return cudaGetLastError();
}

cudaError_t launch_gspo_finish(const GspoArgs& g, int R, const float* fsum_all, const int32_t* cnt_all,
                               cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gspo_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * MAX_SEQS * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  gspo_finish_kernel<<<1, 1024, static_cast<size_t>(3) * g.num_segments * sizeof(float), st>>>(gspo_params(g), R,
                                                                                               fsum_all, cnt_all);
  return cudaGetLastError();
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
