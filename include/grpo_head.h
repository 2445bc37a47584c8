/*
 * grpo_head.h -- C ABI of the fused LM-head GRPO / GSPO loss for GB300 (sm_103a).
 *
 * The library computes, from hidden states H[N,D] and the LM-head weight
 * W[V,D], each token's selected-token log-probability
 *     logp_i = z_{i,y_i} - LSE_i,   z = H W^T,   LSE_i = log sum_{j<V} exp(z_ij)
 * by streaming the vocabulary in 256-column tiles (never materialising the
 * [N,V] logits), the GRPO clipped-ratio + k3-KL loss and its GSPO
 * sequence-level variant on top, and the backward dH = G W, dW = G^T H with
 * G = dloss/dz recomputed tile by tile.
 *
 * Sources: Liger-Kernel PR #1160 "[GRPO] add chunked grpo streaming over vocab"
 * (Summary: selected-token log-probs by streaming over vocab, fused-linear
 * API); RL-Kernel PR #291 "[WS2][PR5][Logp] Add deterministic DP-aware GRPO
 * loss on the TP-aware logprob path" (PR description: fp32 (max, sumexp)
 * merge in fixed tile order, padded columns at -inf, (-inf, 0) identity
 * partial, fp32 logp and LSE outputs, explicit active mask; Key Changes: token
 * normalisers, per-sequence totals then scalar, (loss, policy_loss, kl));
 * Fast-LLM PR #554 "Fuse the GSPO segment seam into compiled blocks (#507)"
 * (What: per-token weights -> index_add_ into segments -> per-segment loss,
 * new_logprobs metric and per-token backward coefficient; divisor and
 * grad_output applied outside).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates or frees device memory and keeps no device data between
 *    calls, apart from the fixed scratch array of grpo_head_forward_noalloc
 *    (scratch space is otherwise the caller's `ws` buffer, sized by the
 *    *_workspace_size calls).  Host state it does keep for the life of the
 *    process: per-device launch set-up (kernel attributes, the number of CTA
 *    pairs that fit, device properties, the no-allocation array's address),
 *    tuning knobs read once from the environment, the calling thread's last
 *    error message, and the process-wide instrumentation counters below.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).  Nothing synchronises.  The work
 *    is kernels and asynchronous memsets only, so these calls can be captured
 *    into a CUDA graph (a captured call keeps the `ws` address it was given);
 *    grpo_head_forward_noalloc is described on its own below.
 *  - The return value reports argument and launch errors (gh_status); a
 *    message for the last error of the calling thread is in gh_last_error().
 *  - Data-dependent problems are OR-ed into the caller's device word
 *    `int32_t *status` (GH_DEV_* bits) without a host synchronisation; the
 *    caller reads it when it chooses.  `status` must be zeroed by the caller.
 *  - Row-major layouts; 16-byte aligned base pointers; bf16 rows need
 *    D % 8 == 0 (16-byte TMA row pitch); fp32 rows take any D (vector loads
 *    when D % 4 == 0, scalar loads otherwise).
 *  - Results are deterministic (no floating-point atomics) and logp/LSE are
 *    bitwise independent of row_tile and of the other rows in the batch.
 */
#ifndef GRPO_HEAD_H_
#define GRPO_HEAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host-side status */
typedef enum {
  GH_OK = 0,
  GH_ERR_INVALID_ARG = 1, /* a pointer, size, alignment or enum is invalid */
  GH_ERR_UNSUPPORTED = 2, /* valid but not built (e.g. no sm_103a device)  */
  GH_ERR_WORKSPACE = 3,   /* ws is NULL or smaller than *_workspace_size   */
  GH_ERR_CUDA = 4         /* a CUDA runtime/driver call failed             */
} gh_status;

/* device-side status bits OR-ed into *status */
enum {
  GH_DEV_TARGET_OOR = 1,  /* an active token's target is outside [0,V); its logp is NaN */
  GH_DEV_NONFINITE = 2,   /* a non-finite LSE/logp/loss term was produced              */
  GH_DEV_TIMEOUT = 4,     /* a bounded pipeline wait gave up; outputs are incomplete   */
  GH_DEV_NO_ACTIVE = 8,   /* token/sequence mean with no active token: loss 0, coef 0  */
  GH_DEV_BAD_SEQ = 16     /* seq_id/seg_id out of range or not laid out as documented  */
};

typedef enum { GH_BF16 = 0, GH_FP32 = 1 } gh_dtype;

/* token normalisers (RL-Kernel PR #291, Key Changes: Loss Contract) */
typedef enum {
  GH_TOKEN_MEAN = 0, /* w_i = m_i / T, T = active tokens (or `norm` if > 0)            */
  GH_SEQ_MEAN = 1,   /* w_i = m_i / (n_s L), L = live sequences (or `norm` if > 0)     */
  GH_FIXED = 2       /* w_i = m_i / C, C = `norm` (> 0), Dr.GRPO constant              */
} gh_reduction;

/* The LM-head problem shared by forward and backward. */
typedef struct {
  int64_t N;              /* tokens (rows of H)                                          */
  int64_t D;              /* hidden size                                                 */
  int64_t V;              /* real vocabulary size; padding to 256 columns is internal     */
  int32_t dtype;          /* gh_dtype of H, W and dH: bf16 (fp32 accumulate, tensor
                             cores) or fp32 (exact fp32 FMA, no TF32)                    */
  int32_t row_tile;       /* 0 = default | 64 | 128 | 256: rows per work unit (bf16: 64
                             and 128 run single-CTA tiles, 256 and the default CTA-pair
                             tiles; fp32: rows per CTA, default 64); the results do not
                             depend on it (bitwise)                                      */
  const void* H;          /* [N, D] row-major                                            */
  const void* W;          /* [V, D] row-major                                            */
  const int32_t* targets; /* [N] selected token ids y_i                                  */
  const uint8_t* mask;    /* [N] 1 = active token; authoritative (inactive targets may
                             hold any value; inactive rows still get an LSE)             */
} gh_head;

/* GRPO loss parameters (RL-Kernel PR #291, Overview / Key Changes). */
typedef struct {
  const float* old_logp;  /* [N] behaviour-policy log-probs                               */
  const float* ref_logp;  /* [N] reference-policy log-probs; NULL allowed iff beta == 0   */
  const float* adv;       /* [num_seqs] per-sequence advantage A_s                        */
  const int32_t* seq_id;  /* [N] sequence of each token, nondecreasing, in [0, num_seqs)  */
  int32_t num_seqs;
  int32_t reduction;      /* gh_reduction                                                 */
  float eps_low;          /* ratio clipped to [1 - eps_low, 1 + eps_high]                 */
  float eps_high;
  float beta;             /* weight of the k3 KL term exp(d) - d - 1, d = ref - logp      */
  float delta;            /* > 0: two-sided clip, the unclipped ratio is capped at delta
                             (Liger-Kernel PR #1160, Testing Done: the delta parameter);
                             0: off                                                      */
  double norm;            /* > 0: explicit normaliser (T, L or C above, e.g. the active
                             token count of the whole step across micro-batches or
                             data-parallel ranks); 0: from this call (token/seq mean)   */
  int32_t ratio_level;    /* 0: token ratios exp(logp - old); 1: one ratio per sequence,
                             exp of the mean active log-ratio of the sequence (the
                             "sequence" importance-sampling level of the same tests)    */
  int32_t reserved;       /* must be 0                                                    */
  float* seq_policy;      /* optional out [num_seqs]: sum over the sequence's active
                             tokens of the policy term (before the normaliser)           */
  float* seq_kl;          /* optional out [num_seqs]: same for the KL term               */
  int32_t* seq_count;     /* optional out [num_seqs]: active tokens of each sequence     */
  int32_t* num_clipped;   /* optional out [1]: active tokens whose policy gradient the
                             clip (or the delta cap) cuts off, act = 0 below: the
                             clipped-token count behind the usual clip fraction       */
} gh_grpo;

/*
 * Bytes of scratch `ws` grpo_head_forward needs for this problem: the split
 * partials and target logits of the log-prob, per-sequence slots of the GRPO
 * loss for up to max(64, N / 8) sequences (capped at 16384), and 256 bytes of
 * counters (the loss's control words and the forward's tile counter, all set
 * by the call itself).  With more sequences than slots the loss runs on one
 * CTA instead of one CTA per sequence, with the same results, bit for bit.
 */
size_t grpo_head_forward_workspace_size(const gh_head* head);
/*
 * Bytes of scratch `ws` grpo_head_backward needs for this problem: one
 * dlogits block (bf16: at most 16384 vocabulary columns, plus an fp32 dH
 * accumulator when the vocabulary spans several blocks; fp32: at most 1024
 * columns, plus partials of the GEMMs' K slices that run in parallel) for a
 * chunk of rows.  The rows per chunk keep this at most three quarters of
 * N * V * 2 bytes (the size of the bf16 [N, V] logits), except on problems too
 * small for it: a chunk holds at least min(N, 128) rows (bf16; 64 for fp32) of
 * at least one 256-column tile.
 */
size_t grpo_head_backward_workspace_size(const gh_head* head);
/*
 * Bytes of scratch grpo_head_backward_shard needs for the vocabulary shard
 * `head` of a V_total-column vocabulary (0 for invalid arguments).
 */
size_t grpo_head_backward_shard_workspace_size(const gh_head* head, int64_t V_total);

/*
 * Forward: selected-token log-prob and LSE for every row, and, when `grpo` is
 * not NULL, the GRPO loss and d loss / d logp.
 *   logp  [N] fp32 out: z_{i,y_i} - LSE_i (NaN for an active token with an
 *         out-of-range target, 0 for an inactive one).
 *   lse   [N] fp32 out: LSE_i over the real vocabulary.
 *   coef  [N] fp32 out (may be NULL; needs grpo): coef_i = d loss / d logp_i =
 *         w_i (-A_s r_i act_i + beta (1 - exp(ref_i - logp_i))), with r the
 *         token (or sequence) ratio and act = 1 where the PPO term moving with
 *         r is the minimum: the unclipped term below the delta cap, or the
 *         clipped term inside the clip band.
 *   loss3 [3] fp32 out (may be NULL; needs grpo): (loss, policy_loss, kl) with
 *         loss = policy_loss + beta kl, summed per sequence first and then over
 *         sequences in index order.
 * Errors: GH_ERR_INVALID_ARG for bad sizes/pointers/alignment/enums,
 * GH_ERR_WORKSPACE for a short ws, GH_ERR_CUDA for a failed launch.
 */
gh_status grpo_head_forward(const gh_head* head, const gh_grpo* grpo, float* logp, float* lse,
                            float* coef, float* loss3, int32_t* status, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * Vocabulary-parallel (tensor-parallel) log-prob, RL-Kernel PR #291, PR
 * description: each rank holds a vocabulary shard of W; padded columns are
 * masked before the local (max, sumexp) partials; partials are moved by
 * all-gather and merged in fixed global shard order; cross-degree bitwise
 * equality needs a tile decomposition that does not depend on the number of
 * shards.  Here the decomposition is the global grid of 256-column splits:
 * shard bounds are multiples of 256 (gh_vocab_shard_bounds gives an even
 * split), every shard's splits are global splits, and the merged result is
 * bitwise the one grpo_head_forward gives on the whole vocabulary.
 *
 * gh_vocab_shard_bounds: columns [*start, *start + *len) of shard `rank` of
 * `num_shards` over V_total (whole splits, the remainder spread over the first
 * shards; num_shards <= ceil(V_total / 256)).  Host only.
 */
gh_status gh_vocab_shard_bounds(int64_t V_total, int32_t num_shards, int32_t rank, int64_t* start, int64_t* len);

/*
 * Number of vocabulary splits of a V-column vocabulary (or shard): the row
 * count of the split partial arrays part_m / part_s that
 * grpo_head_logprob_shard writes and grpo_logprob_merge reads.  Returns 0 for
 * V < 1.  Host only.
 */
int64_t gh_vocab_splits(int64_t V);

/*
 * One rank's shard: head->W is the shard [head->V, D] holding global columns
 * [vocab_start, vocab_start + head->V) of V_total; targets are global ids.
 * Writes the shard's split partials part_m, part_s [S_shard, N] fp32
 * (S_shard = ceil(head->V / 256)) and zy [N] = z_{i, y_i} for the rows whose
 * target lies in the shard (other rows untouched).  vocab_start must be a
 * multiple of 256 and every shard but the last whole splits.
 */
gh_status grpo_head_logprob_shard(const gh_head* head, int64_t vocab_start, int64_t V_total, float* part_m,
                                  float* part_s, float* zy, int32_t* status, void* stream);

/*
 * Merge of the gathered shard outputs: part_m, part_s [S_total, N] are the
 * shards' partials concatenated in shard order (= global split order), zy
 * [num_shards, N] their zy rows, shard_starts (HOST array, num_shards + 1
 * entries) the bounds.  Writes logp and lse [N] exactly as grpo_head_forward.
 */
gh_status grpo_logprob_merge(int64_t N, int64_t V_total, int32_t num_shards, const int64_t* shard_starts,
                             const float* part_m, const float* part_s, const float* zy, const int32_t* targets,
                             const uint8_t* mask, float* logp, float* lse, int32_t* status, void* stream);

/*
 * Backward of one vocabulary shard (the tensor-parallel counterpart of
 * grpo_head_backward): head->W is the shard holding global columns
 * [vocab_start, vocab_start + head->V); lse and coef are the full-vocabulary
 * per-row values (from grpo_logprob_merge and the loss), identical on every
 * rank.  Writes dW [head->V, D] fp32 for the shard's rows (added to dW when
 * accumulate_dW) and dH_partial [N, D] fp32 = G_shard W_shard; the shards'
 * partials summed in shard order (grpo_dh_merge) give dH.  The shard's dW rows
 * are bitwise the rows grpo_head_backward gives on the whole vocabulary (both
 * add dW over the same row chunks, which depend on V_total, not on the
 * shard).  Workspace: at least grpo_head_backward_shard_workspace_size(head,
 * V_total) bytes.
 */
gh_status grpo_head_backward_shard(const gh_head* head, int64_t vocab_start, int64_t V_total, const float* lse,
                                   const float* coef, const float* grad_out, float* dH_partial, float* dW,
                                   int32_t accumulate_dW, int32_t* status, void* ws, size_t ws_bytes, void* stream);

/*
 * dH [N, D] (in dtype) = sum over shards, in shard order, of the gathered fp32
 * partials dH_partials [num_shards, N, D] (a deterministic reduction in place
 * of a float all-reduce).
 */
gh_status grpo_dh_merge(int32_t num_shards, int64_t N, int64_t D, int32_t dtype, const float* dH_partials, void* dH,
                        int32_t* status, void* stream);

/*
 * (loss, policy_loss, kl) from per-sequence totals gathered across
 * data-parallel ranks (RL-Kernel PR #291, Key Changes: Reference Op: each rank
 * owns whole sequences; per-sequence totals are all-gathered as a
 * [num_sequences] vector and summed in sequence order, never all-reduced).
 * seq_policy, seq_kl [num_seqs] fp32 and seq_count [num_seqs] int32 are the
 * concatenation, in global sequence order, of the gh_grpo.seq_* outputs of
 * every rank's grpo_head_forward; the sum runs in the same order and code as
 * a single-call forward over the whole batch, so the result is bitwise the
 * same as that call's loss3.  `norm` as in gh_grpo.  loss3 [3] out.
 */
gh_status grpo_loss_from_sequence_totals(int32_t num_seqs, const float* seq_policy, const float* seq_kl,
                                         const int32_t* seq_count, int32_t reduction, double norm, float beta,
                                         float* loss3, int32_t* status, void* stream);

/*
 * GSPO sequence-level loss over packed documents (Fast-LLM PR #554, What):
 *   S_s = sum_{i in s} m_i (logp_i - old_i), n_s = sum_{i in s} m_i,
 *   rho_s = exp(S_s / n_s), l_s = -min(rho_s A_s, clip(rho_s) A_s),
 *   K_s = (1/n_s) sum_{i in s} m_i (exp(d_i) - d_i - 1), d = ref - logp,
 *   loss = sum_s omega_s (l_s + beta K_s) / divisor, omega_s = 1 (or n_s if
 *   token_weighted),
 *   coef_i = (omega_s / divisor)(-A_s rho_s act_s + beta (1 - exp(d_i))) m_i / n_s.
 * seg_id [N]: document of each token; ids >= 0 are nondecreasing and -1 marks
 * an unused tail (whose mask must be 0).  Segments with n_s = 0 contribute 0
 * and report seg_ratio 1.  ref_logp may be NULL when beta == 0.  Outputs:
 * loss [1], seg_ratio [num_segments], coef [N], mean_logp [1] (the
 * new_logprobs metric: mean active logp), num_clipped [1] (live segments
 * whose policy gradient the clip cuts off, act_s = 0); seg_ratio, mean_logp
 * and num_clipped may be NULL.
 * ws: gspo_segment_workspace_size(num_segments) bytes of scratch, or NULL.
 * With it each segment gets its own CTA; without it one CTA does every
 * segment.  Both give the same results, bit for bit.
 */
size_t gspo_segment_workspace_size(int32_t num_segments);
gh_status gspo_segment_loss(int64_t N, const float* logp, const float* old_logp, const float* ref_logp,
                            const uint8_t* mask, const int32_t* seg_id, int32_t num_segments, const float* seg_adv,
                            float eps_low, float eps_high, float beta, double divisor, int32_t token_weighted,
                            float* loss, float* seg_ratio, float* coef, float* mean_logp, int32_t* num_clipped,
                            int32_t* status, void* ws, size_t ws_bytes, void* stream);

/*
 * GSPO under sequence parallelism (Fast-LLM PR #554, What / Correctness: the
 * segment sums are reduced across the sequence-data-parallel ranks between
 * the pre- and post-aggregation blocks; a document may span ranks).  Each
 * rank holds a contiguous piece of the packed token sequence (same seg_id
 * layout rule within its piece) and calls gspo_segment_partials, which writes
 *   fsum [2 * num_segments + 1] = (S_s partial..., KL partial..., sum m logp),
 *   cnt  [num_segments + 1]     = (n_s partial..., sum m);
 * ref_logp NULL skips the KL partials.  The ranks gather fsum and cnt in rank
 * order ([num_ranks, 2S + 1] and [num_ranks, S + 1]) and each calls
 * gspo_segment_loss_from_partials for its own tokens: the partials are summed
 * over ranks in rank order (no float all-reduce, so the result does not depend
 * on the collective's topology), then loss, seg_ratio, mean_logp, num_clipped
 * and this rank's coef follow as in gspo_segment_loss.  With one rank the
 * result is bitwise gspo_segment_loss's.  ws as in gspo_segment_loss.
 */
gh_status gspo_segment_partials(int64_t N, const float* logp, const float* old_logp, const float* ref_logp,
                                const uint8_t* mask, const int32_t* seg_id, int32_t num_segments, float* fsum,
                                int32_t* cnt, int32_t* status, void* ws, size_t ws_bytes, void* stream);
gh_status gspo_segment_loss_from_partials(int64_t N, const float* logp, const float* ref_logp, const uint8_t* mask,
                                          const int32_t* seg_id, int32_t num_segments, int32_t num_ranks,
                                          const float* fsum_all, const int32_t* cnt_all, const float* seg_adv,
                                          float eps_low, float eps_high, float beta, double divisor,
                                          int32_t token_weighted, float* loss, float* seg_ratio, float* coef,
                                          float* mean_logp, int32_t* num_clipped, int32_t* status, void* ws,
                                          size_t ws_bytes, void* stream);

/*
 * Backward of the head given each row's LSE and coef (from grpo_head_forward
 * or gspo_segment_loss): per vocabulary block the logits are recomputed,
 *   G_ij = g coef_i (1[j = y_i] - exp(z_ij - LSE_i))   (g = *grad_out, or 1 if NULL)
 * and dH = G W (fp32 accumulation over blocks in increasing vocabulary order,
 * written in `dtype`), dW = G^T H (fp32; added to dW when accumulate_dW != 0,
 * e.g. across micro-batches).  dH [N, D] in dtype; dW [V, D] fp32.  When the
 * vocabulary is narrow next to the block and accumulator rows, the rows are
 * processed in chunks (see grpo_head_backward_workspace_size), each adding its
 * dW contribution in chunk order; the chunks depend on N, D, dtype and V only.
 * A row's dH does not depend on the chunks or on the other rows of the batch.
 */
gh_status grpo_head_backward(const gh_head* head, const float* lse, const float* coef,
                             const float* grad_out, void* dH, float* dW, int32_t accumulate_dW,
                             int32_t* status, void* ws, size_t ws_bytes, void* stream);

/*
 * Group-normalised advantages (RL-Kernel PR #291, Reference Op: group-relative
 * advantage from gathered rewards; review note: two-pass variance):
 * A = (r - mean_g) / (std_g + eps) over consecutive groups of group_size
 * sequences, std unbiased (n - 1), 0 for a group of one.  rewards, adv:
 * [num_seqs] fp32; num_seqs must be a multiple of group_size.
 */
gh_status grpo_group_advantage(const float* rewards, int32_t num_seqs, int32_t group_size, float eps,
                               float* adv, int32_t* status, void* stream);

/*
 * Forward without a caller workspace.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- their
 * device memory is wholly owned by another allocator (a framework's caching
 * allocator that has reserved the pool, or a memory plan fixed before the
 * step), or they must not call cudaMalloc mid-step because it can synchronise
 * the device -- and so cannot hand grpo_head_forward its `ws` buffer.
 *
 * Same arguments, outputs and results as grpo_head_forward (bitwise), minus
 * `ws`/`ws_bytes`: the scratch lives in a fixed, file-scope device array of
 * GH_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  Nothing is allocated or freed by the call.  A problem whose
 * forward scratch (grpo_head_forward_workspace_size) exceeds that size is
 * rejected with GH_ERR_INVALID_ARG and a message in gh_last_error() before
 * any GPU work.  The array's device address is looked up on the first call
 * made on each device (with that device current), so make that first call
 * before any stream capture; it is looked up again when a call comes from a
 * different CUDA context than the one it was found in (after
 * cudaDeviceReset, for example).  All calls share the one array and it keeps the
 * last call's contents (nothing in it needs to start at zero): calls whose GPU
 * work overlaps in time, e.g. on two streams, race on it and must be
 * serialised by the caller.
 */
#define GH_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
gh_status grpo_head_forward_noalloc(const gh_head* head, const gh_grpo* grpo, float* logp, float* lse,
                                    float* coef, float* loss3, int32_t* status, void* stream);

/* Human-readable name of a gh_status. */
const char* gh_status_string(gh_status s);
/* Message of the last error returned on the calling thread ("" if none). */
const char* gh_last_error(void);
/* ABI version (major * 100 + minor). */
int32_t gh_abi_version(void);

/*
 * Instrumentation (used by the benchmark; off by default).  When enabled, each
 * kernel the library launches is bracketed by CUDA events on its stream and
 * counted per kernel kind; gh_profile_read returns, for kind k, the launch
 * count and the summed event time (ms) since the last reset (it synchronises
 * the recorded events).  gh_launch_count counts all launches since load.
 * The instrumentation state is process-wide and unsynchronised: enable it only
 * while a single host thread calls the library, and not during a CUDA-graph
 * capture.
 * Kinds: 0 fwd logits+LSE, 1 merge, 2 GRPO loss, 3 GSPO loss, 4 dlogits,
 * 5 dH GEMM, 6 dW GEMM, 7 advantage, 8 fp32 forward, 9 fp32 dlogits,
 * 10 fp32 GEMM, 11 timeout probe, 12 GRPO loss from sequence totals, 13 shard merge,
 * 14 GSPO partials, 15 GSPO loss from partials, 16 dH shard merge, 17 dH and dW
 * GEMMs of a vocabulary block in one launch.
 */
#define GH_NUM_KERNEL_KINDS 18
void gh_profile_enable(int32_t on);
void gh_profile_reset(void);
gh_status gh_profile_read(int32_t kind, int64_t* launches, double* total_ms);
int64_t gh_launch_count(void);
const char* gh_kernel_kind_name(int32_t kind);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing will complete, with a limit of timeout_ns; the wait gives
 * up, sets GH_DEV_TIMEOUT in *status and the kernel returns normally.
 */
gh_status gh_timeout_probe(int32_t* status, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GRPO_HEAD_H_ */
