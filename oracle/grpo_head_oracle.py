"""Plain fp64 definitions of everything the fused GRPO/GSPO head computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by tests/,
``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs, never by the
product path.

Sources (pages):
  [Liger]  Liger-Kernel PR #1160 "[GRPO] add chunked grpo streaming over vocab"
  [RLK]    RL-Kernel PR #291 "[WS2][PR5][Logp] Add deterministic DP-aware GRPO
           loss on the TP-aware logprob path"
  [FLLM]   Fast-LLM PR #554 "Fuse the GSPO segment seam into compiled blocks (#507)"

The pages print no formula for the ratio, clip, KL or advantage; the
standard GRPO/PPO/GSPO definitions below are the plainest reading of the
names the pages use (ratio, clipping, reference KL, group-relative advantage,
per-segment ratio), and each reading is listed in the design doc.

Pins (tests/test_oracle_*.py):
  head_logits / selected_logprob : W=0 closed form (log V), one-hot gather
      closed form, softmax rows sum to 1, scipy logsumexp, shift invariance
  streamed_lse : equals the plain LSE for chunk sizes 1, 7, 64, 256, V;
      all-padding chunk is the identity
  group_advantages : numpy mean/std(ddof=1) of each group, zero-spread groups
  grpo_loss : ratio==1 & beta=0 closed form, clip-free band, k3 >= 0 and 0 at
      equality, reductions coincide on equal lengths, worked example fixture,
      finite differences of the loss w.r.t. logp (token and sequence ratios,
      with and without the two-sided cap), the cap's worked example, a cap
      above every ratio changes nothing, one-token sequences and constant
      per-sequence log-ratios reduce the sequence level to the token level
  gspo_loss : length-1 segments reduce to token PPO-clip (with the KL term:
      to the token-level GRPO loss with the same fixed normaliser), one
      segment closed form, np.bincount counts, finite differences w.r.t. logp
      with and without the KL term
  dlogits / head_backward : finite differences of the loss w.r.t. H and W,
      row sums of dlogits and column sums of dW vanish
No function is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np


class OracleError(ValueError):
    """Raised where the method defines an error (zero active tokens, ...)."""


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------
def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored inputs: float32 arrays, or bf16 held as
    uint16 bit patterns (the upper half of a float32)."""
    if dtype == "bf16":
        b = np.ascontiguousarray(x, dtype=np.uint16)
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "fp64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# selected-token log-prob  ([Liger] "Summary"; [RLK] PR description,
# "LogprobOutputSpec": fp32 selected logprob and fp32 vocab LSE)
# --------------------------------------------------------------------------
def head_logits(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = H W^T over the real vocabulary only ([Liger] "Summary": the loss
    takes hidden states and the head weight, fused-linear)."""
    return H @ W.T


def selected_logprob(H: np.ndarray, W: np.ndarray, targets: np.ndarray,
                     mask: Optional[np.ndarray] = None, chunk_rows: int = 1024):
    """logp_i = z_{i,y_i} - LSE_i and LSE_i = log sum_j exp(z_ij), j < V.

    Plain definition: each row chunk materialises its full [rows, V] logits
    and takes a max-shifted log-sum-exp.  Padded vocabulary columns do not
    exist here ([RLK] PR description: padded columns are masked before the
    local partials, so they must not change the result).

    Targets outside [0, V): an active token gets NaN (and counts in the
    returned ``bad_targets``); an inactive one gets logp 0.  The mask is
    authoritative ([RLK] "MaskMode": inactive targets need not hold
    ignore_index).

    Returns (logp[N], lse[N], bad_targets)."""
    N = H.shape[0]
    V = W.shape[0]
    if mask is None:
        mask = np.ones(N, dtype=np.uint8)
    logp = np.empty(N, dtype=np.float64)
    lse = np.empty(N, dtype=np.float64)
    bad = 0
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        Z = head_logits(H[r0:r1], W)
        zmax = Z.max(axis=1)
        lse[r0:r1] = zmax + np.log(np.exp(Z - zmax[:, None]).sum(axis=1))
        for i in range(r0, r1):
            y = int(targets[i])
            if 0 <= y < V:
                logp[i] = Z[i - r0, y] - lse[i]
            elif mask[i]:
                logp[i] = math.nan
                bad += 1
            else:
                logp[i] = 0.0
    return logp, lse, bad


def streamed_lse(Z: np.ndarray, chunk: int, padded_width: Optional[int] = None) -> np.ndarray:
    """LSE by streaming the vocabulary in chunks, as the pages describe.

    [RLK] PR description ("ReductionSpec", identity partial): each chunk of a
    row gives a local partial (max m_t, sumexp s_t = sum exp(z - m_t)) with
    padded columns at -inf; partials merge in fixed chunk order by
    (m, s) (+) (m', s') = (M, s e^{m-M} + s' e^{m'-M}), M = max(m, m'); a
    chunk whose columns are all padding contributes the identity (-inf, 0)
    and exp(-inf - (-inf)) is never evaluated.  ``padded_width`` > V appends
    -inf columns to exercise the identity."""
    n, V = Z.shape
    width = V if padded_width is None else padded_width
    Zp = np.full((n, width), -np.inf)
    Zp[:, :V] = Z
    out = np.empty(n)
    for i in range(n):
        m, s = -math.inf, 0.0                       # identity partial
        for c0 in range(0, width, chunk):
            blk = Zp[i, c0:c0 + chunk]
            mt = float(blk.max())
            if mt == -math.inf:
                continue                            # (-inf, 0): nothing to merge
            st = float(np.exp(blk - mt).sum())
            M = max(m, mt)
            s = (s * math.exp(m - M) if m != -math.inf else 0.0) + st * math.exp(mt - M)
            m = M
        out[i] = m + math.log(s) if s > 0 else -math.inf
    return out


# --------------------------------------------------------------------------
# group-normalised advantage ([RLK] "Reference Op": group-relative advantage
# computed from gathered rewards; review note: the two-pass variance form
# subtracts the mean before squaring)
# --------------------------------------------------------------------------
def group_advantages(rewards: np.ndarray, group_size: int, eps: float = 1e-4) -> np.ndarray:
    """A = (r - mean_g) / (std_g + eps) over consecutive groups of
    ``group_size`` sequences; std is the unbiased (n-1) two-pass standard
    deviation; a group of one has std 0."""
    r = np.asarray(rewards, dtype=np.float64)
    n = r.shape[0]
    if group_size <= 0 or n % group_size != 0:
        raise OracleError("number of sequences must be a multiple of the group size")
    A = np.empty(n)
    for g0 in range(0, n, group_size):
        grp = r[g0:g0 + group_size]
        mean = 0.0
        for v in grp:
            mean += v
        mean /= group_size
        var = 0.0
        for v in grp:
            var += (v - mean) ** 2
        std = math.sqrt(var / (group_size - 1)) if group_size > 1 else 0.0
        for k in range(group_size):
            A[g0 + k] = (grp[k] - mean) / (std + eps)
    return A


# --------------------------------------------------------------------------
# GRPO token objective and reduction
# --------------------------------------------------------------------------
REDUCTIONS = ("token_mean", "seq_mean", "fixed")


def _token_terms(logp, old, ref, A_tok, eps_low, eps_high, delta=0.0, log_ratio=None):
    """Per-token PPO-clip surrogate and k3 KL ([RLK] "Overview": ratio,
    clipping and reference KL act per token).

    r = exp(logp - old) (or exp(log_ratio) when given: the sequence-level
    ratio); c = clip(r, 1-eps_low, 1+eps_high); with the two-sided clip
    ([Liger] test parameter delta) the unclipped ratio is capped at delta:
    u = min(r, delta) A, else u = r A; v = c A; pg = -min(u, v);
    d = ref - logp; kl = exp(d) - d - 1.  d pg / d log r = -A r act with
    act = 1 when the unclipped term is the minimum (ties count as unclipped)
    and the cap does not bind (r <= delta), or when the clipped term is the
    minimum and r lies inside the clip band; act = 0 otherwise."""
    r = np.exp(logp - old) if log_ratio is None else np.exp(log_ratio)
    c = np.clip(r, 1.0 - eps_low, 1.0 + eps_high)
    rr = np.minimum(r, delta) if delta > 0 else r
    u = rr * A_tok
    v = c * A_tok
    pg = -np.minimum(u, v)
    d = ref - logp
    kl = np.exp(d) - d - 1.0
    # the gradient follows the active branch: the unclipped (capped) term
    # moves with r unless the cap binds; the clipped term moves with r only
    # inside the clip band (where clip(r) = r)
    in_band = (r >= 1.0 - eps_low) & (r <= 1.0 + eps_high)
    below_cap = (r <= delta) if delta > 0 else np.ones_like(r, dtype=bool)
    act = np.where(u <= v, below_cap, in_band)
    return r, pg, kl, act.astype(np.float64), d


def grpo_loss(logp, old, ref, mask, seq_id, adv, num_seqs: int, eps_low: float,
              eps_high: float, beta: float, reduction: str = "token_mean",
              norm: float = 0.0, delta: float = 0.0, ratio_level: str = "token"):
    """Masked GRPO loss, its (policy, kl) parts and d loss / d logp.

    Reductions ([RLK] "Key Changes: Loss Contract", token_normalizer):
      token_mean  w_i = m_i / T     T = active tokens (global_active_tokens)
      seq_mean    w_i = m_i / (n_s L)   n_s active tokens of sequence s,
                  L = sequences with n_s > 0 (per_sequence_then_mean)
      fixed       w_i = m_i / C     (fixed_constant, Dr.GRPO)
    ``norm`` > 0 replaces T (token_mean), L (seq_mean) or gives C (fixed; it
    must then be > 0).  Totals are formed per sequence first and then summed
    over sequences in index order ([RLK] "Key Changes: Reference Op":
    slots -> per-sequence totals -> scalar).  policy = sum w pg,
    kl = sum w kl, loss = policy + beta kl  ([RLK] "Reference Op":
    (loss, policy_loss, kl)).  With no active tokens token_mean and
    seq_mean raise (review note on the zero-active-token guard), fixed gives 0.

    ``delta`` > 0 caps the unclipped ratio ([Liger] "Testing Done": the
    two-sided clip parameter, 2.0 in the failing cases).  ``ratio_level`` =
    "sequence" uses one ratio per sequence, exp of the mean active log-ratio
    of the sequence ([Liger] "Testing Done": the "sequence" importance
    sampling level), for every token of the sequence; the KL stays per token.

    coef_j = d loss / d logp_j; token level: w_j (-A_s r_j act_j + beta (1 - e^{d_j}));
    sequence level: w_j beta (1 - e^{d_j}) + (m_j / n_s) sum_{i in s} w_i (-A_s r_s act_s)."""
    if reduction not in REDUCTIONS:
        raise OracleError(reduction)
    if ratio_level not in ("token", "sequence"):
        raise OracleError(ratio_level)
    logp = np.asarray(logp, dtype=np.float64)
    N = logp.shape[0]
    m = np.asarray(mask, dtype=np.float64)
    seq = np.asarray(seq_id, dtype=np.int64)
    A = np.asarray(adv, dtype=np.float64)
    A_tok = A[seq]
    # inactive tokens may carry NaN log-probs (bad target); they are excluded.
    lp = np.where(m > 0, logp, 0.0)
    od = np.where(m > 0, np.asarray(old, dtype=np.float64), 0.0)
    rf = np.where(m > 0, np.asarray(ref, dtype=np.float64), 0.0) if ref is not None else lp

    # explicit loop: per-sequence active counts (and mean log-ratios)
    n = np.zeros(num_seqs, dtype=np.int64)
    lr_sum = np.zeros(num_seqs)
    for i in range(N):
        if m[i] > 0:
            n[seq[i]] += 1
            lr_sum[seq[i]] += lp[i] - od[i]
    log_ratio = None
    if ratio_level == "sequence":
        seq_lr = np.where(n > 0, lr_sum / np.maximum(n, 1), 0.0)
        log_ratio = np.where(m > 0, seq_lr[seq], 0.0)
    r, pg, kl, act, d = _token_terms(lp, od, rf, A_tok, eps_low, eps_high, delta, log_ratio)

    # explicit loop: per-sequence totals in token order
    P = np.zeros(num_seqs)
    K = np.zeros(num_seqs)
    for i in range(N):
        if m[i] > 0:
            P[seq[i]] += pg[i]
            K[seq[i]] += kl[i]

    total = int(n.sum())
    live = int((n > 0).sum())
    if reduction == "token_mean":
        denom = norm if norm > 0 else float(total)
        if denom <= 0:
            raise OracleError("no active tokens")
        seq_scale = np.full(num_seqs, 1.0 / denom)
    elif reduction == "seq_mean":
        Lden = norm if norm > 0 else float(live)
        if Lden <= 0:
            raise OracleError("no active tokens")
        seq_scale = np.where(n > 0, 1.0 / (np.maximum(n, 1) * Lden), 0.0)
    else:
        if not norm > 0:
            raise OracleError("fixed reduction needs a positive constant")
        seq_scale = np.full(num_seqs, 1.0 / norm)

    policy = 0.0
    klsum = 0.0
    for s in range(num_seqs):
        policy += P[s] * seq_scale[s]
        klsum += K[s] * seq_scale[s]
    loss = policy + beta * klsum
    w = m * seq_scale[seq]
    if ratio_level == "token":
        coef = w * (-A_tok * r * act + beta * (1.0 - np.exp(d)))
    else:
        wsum = np.zeros(num_seqs)
        g = np.zeros(num_seqs)
        for i in range(N):
            if m[i] > 0:
                wsum[seq[i]] += w[i]
                g[seq[i]] = -A_tok[i] * r[i] * act[i]      # shared by the sequence
        coef = w * beta * (1.0 - np.exp(d)) + (m / np.maximum(n[seq], 1)) * wsum[seq] * g[seq]
    coef = np.where(m > 0, coef, 0.0)
    abs_terms = float(np.sum(np.abs(w * (pg + beta * kl))))
    return dict(loss=loss, policy=policy, kl=klsum, coef=coef, per_seq_policy=P,
                per_seq_kl=K, counts=n, weights=w, ratio=r, act=act, abs_terms=abs_terms)


# --------------------------------------------------------------------------
# GSPO sequence-level variant ([FLLM] "What": per-token weights ->
# index_add_ into num_segments bins -> per-segment loss, new_logprobs metric
# and the unscaled per-token backward coefficient; "/ divisor" and
# grad_output applied outside)
# --------------------------------------------------------------------------
def gspo_loss(logp, old, mask, seg_id, num_segments: int, seg_adv, eps_low: float,
              eps_high: float, divisor: float, token_weighted: bool = False, ref=None, beta: float = 0.0):
    """S_s = sum_{i in s} m_i (logp_i - old_i) and n_s = sum m_i (explicit
    loop: the index_add_ of the seam); rho_s = exp(S_s / n_s);
    l_s = -min(rho_s A_s, clip(rho_s, 1-eps_low, 1+eps_high) A_s);
    with a reference policy, K_s = (1/n_s) sum_{i in s} m_i kl_i (k3, the
    segment mean, matching the sequence-level ratio);
    loss = sum_s omega_s (l_s + beta K_s) / divisor with omega_s = 1 (or n_s
    when token_weighted); coef_i = d loss / d logp_i =
    (omega_s / divisor) (-A_s rho_s act_s + beta (1 - e^{d_i})) m_i / n_s;
    segments with n_s = 0 contribute 0 and report rho = 1; tokens with
    seg_id = -1 belong to no segment; new_logprobs = mean active logp."""
    logp = np.asarray(logp, dtype=np.float64)
    old = np.asarray(old, dtype=np.float64)
    N = logp.shape[0]
    if not divisor > 0:
        raise OracleError("divisor must be positive")
    use_kl = ref is not None and beta != 0.0
    rf = np.asarray(ref, dtype=np.float64) if use_kl else None
    S = np.zeros(num_segments)
    K = np.zeros(num_segments)
    n = np.zeros(num_segments, dtype=np.int64)
    lp_sum = 0.0
    act_tokens = 0
    for i in range(N):                                   # index_add_
        s = int(seg_id[i])
        if mask[i] and s >= 0:
            S[s] += logp[i] - old[i]
            n[s] += 1
            if use_kl:
                d = rf[i] - logp[i]
                K[s] += math.exp(d) - d - 1.0
        if mask[i]:
            lp_sum += logp[i]
            act_tokens += 1
    A = np.asarray(seg_adv, dtype=np.float64)
    rho = np.ones(num_segments)
    ell = np.zeros(num_segments)
    g = np.zeros(num_segments)                           # policy part of d loss / d logp, per active token
    seg_act = np.zeros(num_segments, dtype=bool)         # the policy term moves with rho (not cut by the clip)
    kb = np.zeros(num_segments)                          # KL part scale, per active token
    loss = 0.0
    abs_terms = 0.0
    for s in range(num_segments):
        if n[s] == 0:
            continue
        rho[s] = math.exp(S[s] / n[s])
        c = min(max(rho[s], 1.0 - eps_low), 1.0 + eps_high)
        u, v = rho[s] * A[s], c * A[s]
        ell[s] = -min(u, v)
        act = True if u <= v else (1.0 - eps_low <= rho[s] <= 1.0 + eps_high)
        seg_act[s] = act
        omega = float(n[s]) if token_weighted else 1.0
        term = ell[s] + (beta * K[s] / n[s] if use_kl else 0.0)
        loss += omega * term / divisor
        abs_terms += abs(omega * term / divisor)
        g[s] = (omega / divisor) * (-A[s] * rho[s] * (1.0 if act else 0.0)) / n[s]
        kb[s] = (omega / divisor) * beta / n[s]
    coef = np.zeros(N)
    for i in range(N):
        s = int(seg_id[i])
        if mask[i] and s >= 0:
            coef[i] = g[s]
            if use_kl:
                coef[i] += kb[s] * (1.0 - math.exp(rf[i] - logp[i]))
    mean_logp = lp_sum / act_tokens if act_tokens > 0 else 0.0
    return dict(loss=loss, seg_ratio=rho, seg_loss=ell, coef=coef, counts=n, seg_act=seg_act,
                seg_sum=S, seg_kl=K, mean_logp=mean_logp, abs_terms=abs_terms)


# --------------------------------------------------------------------------
# backward ([RLK] review of the logprob op: p is derived from the logits and
# lse; here the logits are recomputed instead of saved)
# --------------------------------------------------------------------------
def dlogits(H, W, targets, lse, coef, g0: float = 1.0):
    """G_ij = g0 coef_i (1[j = y_i] - exp(z_ij - LSE_i)) over the real
    vocabulary (d loss / d z, since d logp_i / d z_ij = 1[j=y_i] - p_ij)."""
    Z = head_logits(H, W)
    P = np.exp(Z - np.asarray(lse)[:, None])
    onehot = np.zeros_like(P)
    V = W.shape[0]
    for i, y in enumerate(targets):
        if 0 <= int(y) < V:
            onehot[i, int(y)] = 1.0
    return g0 * np.asarray(coef)[:, None] * (onehot - P)


def head_backward(H, W, targets, lse, coef, g0: float = 1.0, chunk_rows: int = 1024):
    """dH = G W and dW = G^T H with G from ``dlogits``, row chunk by chunk
    (dW summed over chunks)."""
    N, D = H.shape
    V = W.shape[0]
    dH = np.zeros((N, D))
    dW = np.zeros((V, D))
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        G = dlogits(H[r0:r1], W, targets[r0:r1], lse[r0:r1], coef[r0:r1], g0)
        dH[r0:r1] = G @ W
        dW += G.T @ H[r0:r1]
    return dH, dW


# --------------------------------------------------------------------------
# convenience: one whole forward + backward from synth inputs
# --------------------------------------------------------------------------
def forward_backward(H, W, targets, mask, seq_id, adv, num_seqs, old, ref, eps_low,
                     eps_high, beta, reduction="token_mean", norm=0.0, g0=1.0,
                     with_grads=True):
    logp, lse, bad = selected_logprob(H, W, targets, mask)
    res = grpo_loss(logp, old, ref, mask, seq_id, adv, num_seqs, eps_low, eps_high, beta,
                    reduction, norm)
    res.update(logp=logp, lse=lse, bad_targets=bad)
    if with_grads:
        dH, dW = head_backward(H, W, targets, lse, res["coef"], g0)
        res.update(dH=dH, dW=dW)
    return res
