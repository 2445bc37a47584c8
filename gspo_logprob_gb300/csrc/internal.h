// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>

#include "grpo_head.h"

namespace gh {

// Column tiling of the vocabulary: 256-column tiles; each tile is one split,
// whose per-row (max, sum exp) partial the merge folds in a fixed order.  The
// split count depends on V only, which keeps logp/LSE bitwise independent of N,
// the row tile, the task schedule and the GPU's SM count.
constexpr int VTILE = 256;
constexpr int TILES_PER_SPLIT = 1;
constexpr int SPLIT_COLS = VTILE * TILES_PER_SPLIT;
static_assert(SPLIT_COLS == 256, "the fp32 logits kernels write one partial per 256-column tile");
// Backward vocabulary block (columns of dlogits held in the workspace at once):
// 16384 by default (fewer fp32 dH read-modify-write passes), or a multiple of
// 256 from GH_BWD_BLOCK_COLS (a tuning knob; dW and the dlogits are the same
// for any width, dH differs only in the fp32 rounding of its accumulation).
int bwd_block_cols();
// Maximum sequences / segments handled by the single-CTA loss kernels.
constexpr int MAX_SEQS = 16384;

enum KernelKind {
  K_FWD_TC = 0,
  K_MERGE = 1,
  K_GRPO = 2,
  K_GSPO = 3,
  K_DLOGITS_TC = 4,
  K_DH_TC = 5,
  K_DW_TC = 6,
  K_ADV = 7,
  K_FWD_F32 = 8,
  K_DLOGITS_F32 = 9,
  K_GEMM_F32 = 10,
  K_PROBE = 11,
  K_GRPO_TOTALS = 12,
  K_MERGE_SHARDS = 13,
  K_GSPO_PARTIALS = 14,
  K_GSPO_FINISH = 15,
  K_DH_MERGE = 16,
  K_DHDW_TC = 17,
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// bf16 2-D tensor map (row-major [outer, inner], row stride in bytes), 128-byte
// swizzle, zero fill out of bounds.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

int num_sms();
uint64_t timeout_ns();
// Sets the calling thread's gh_last_error() message.
void set_error_message(const std::string& msg);

// --- tcgen05 launchers (tc_kernels.cu) ---------------------------------------
struct TcFwdArgs {
  int N, D, V, row_tile;
  const void* H;
  const void* W;
  const int32_t* targets;
  float* part_m;
  float* part_s;
  float* zy;
  int* status;
  int col_offset;  // vocabulary shards: global id of local column 0 (else 0)
  int* task_ctr;   // nullable: a device int for tiles handed out on demand (fwd_dynamic)
};
// Forward logits + LSE.  With a task counter and fwd_dynamic(), the pairs take
// tiles from *task_ctr (the call zeroes it first), so they stay within about a
// tile of each other and a W tile is still in L2 for the rest of its raster
// group; otherwise tiles are dealt round-robin.  The bits are the same.
cudaError_t launch_fwd_tc(const TcFwdArgs& a, cudaStream_t st);

struct TcDlogitsArgs {
  int N, D, V, vb0, width, ldg;
  const void* H;
  const void* W;
  const int32_t* targets;
  const float* lse;
  const float* coef;
  const float* grad_out;
  void* G;
  int* status;
  int col_offset;
  int* zero_word;  // nullable: set to 0 by the launch (the fused dH/dW tile counter that follows)
};
cudaError_t launch_dlogits_tc(const TcDlogitsArgs& a, cudaStream_t st);

struct TcDhArgs {  // dH (+)= G[:, :width] W[vb0:vb0+width, :]
  int N, D, V, vb0, width, ldg;
  const void* G;
  const void* W;
  int mode;  // EpiStore mode
  float* acc32;
  void* out16;
  int* status;
};
cudaError_t launch_dh_tc(const TcDhArgs& a, cudaStream_t st);

struct TcDwArgs {  // dW[vb0:vb0+width] (+)= G[:, :width]^T H
  int N, D, V, vb0, width, ldg;
  const void* G;
  const void* H;
  int accumulate;
  float* dW;
  int* status;
};
cudaError_t launch_dw_tc(const TcDwArgs& a, cudaStream_t st);
// dH and dW of one vocabulary block in one launch of CTA pairs with tiles
// handed out from *task_ctr, which must read 0 when the launch starts: the
// call zeroes it first unless ctr_zeroed says an earlier launch on the same
// stream (the dlogits launch given it as zero_word) already did.  Used when
// dhdw_fused() (the CTA-pair kernels are on and GH_BWD_FUSED is not 0).
bool dhdw_fused();
cudaError_t launch_dhdw_tc(const TcDhArgs& h, const TcDwArgs& w, int* task_ctr, bool ctr_zeroed, cudaStream_t st);

// --- fp32 SIMT launchers (simt_kernels.cu) ----------------------------------
struct F32FwdArgs {
  int N, D, V, row_tile;
  const float* H;
  const float* W;
  const int32_t* targets;
  float* part_m;
  float* part_s;
  float* zy;
  int col_offset;
};
cudaError_t launch_fwd_f32(const F32FwdArgs& a, cudaStream_t st);

struct F32DlogitsArgs {
  int N, D, V, vb0, width, ldg;
  const float* H;
  const float* W;
  const int32_t* targets;
  const float* lse;
  const float* coef;
  const float* grad_out;
  float* G;
  int col_offset;
};
cudaError_t launch_dlogits_f32(const F32DlogitsArgs& a, cudaStream_t st);

// C[row_off + m, n] (+)= sum_k A(m,k) B(k,n),  A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn]
//
// K is cut into slices of F32_SLICE (the last may be shorter).  Each output is
// C0 + p_0 + p_1 + ... added left to right, where p_s is the fmaf chain of
// slice s in increasing k and C0 is C (accumulate) or absent (C = p_0 + ...).
// The slices run either one after the other inside each CTA (par <= 1, no
// scratch) or `par` at a time in parallel CTAs that write their partials to
// `scratch` [par, M, Nn], each wave then added to C in slice order by a
// reduce kernel.  Both orders give the same bits, so `par` (chosen from the
// output grid and the scratch available) never changes the result: it may
// depend on M, and a data-parallel rank's dH rows or a vocabulary shard's dW
// rows come out bitwise equal to the whole problem's.
constexpr int F32_SLICE = 512;
struct F32GemmArgs {
  int M, Nn, K;
  const float* A;
  long long sam, sak;
  const float* B;
  long long sbk, sbn;
  float* C;
  long long ldc;
  int row_off;
  int accumulate;
  int par;         // slices run in parallel per wave (1 = all slices inside each CTA)
  float* scratch;  // [par, M, Nn] partials when par > 1
  int slice0;      // set by launch_gemm_f32: first slice of the current wave
};
cudaError_t launch_gemm_f32(const F32GemmArgs& a, cudaStream_t st);
// slices to run in parallel for an M x Nn output with a K range, given
// `scratch_bytes` of scratch (1 when the output grid alone fills the GPU)
int gemm_f32_par(long long M, long long Nn, long long K, size_t scratch_bytes);
// one more kernel launched inside a counted call (gh_launch_count)
void count_extra_launch();

// --- loss kernels (loss_kernels.cu) -----------------------------------------
// grpo_scratch (nullable): the scratch of the GRPO loss launched next on the
// same stream, whose control words the merge zeroes.
cudaError_t launch_merge(int N, int V, int splits, const float* part_m, const float* part_s, const float* zy,
                         const int32_t* targets, const uint8_t* mask, float* logp, float* lse, int* status,
                         void* grpo_scratch, cudaStream_t st);
// Shard bounds (global vocabulary ids, num_shards + 1 entries) for the merge of
// vocabulary-parallel partials; zy is [num_shards, N].
constexpr int MAX_SHARDS = 64;
struct ShardBounds {
  int num_shards;
  int start[MAX_SHARDS + 1];
};
cudaError_t launch_merge_shards(int N, int V_total, int splits, const float* part_m, const float* part_s,
                                const float* zy, const ShardBounds& sb, const int32_t* targets, const uint8_t* mask,
                                float* logp, float* lse, int* status, cudaStream_t st);
// GRPO loss.  `scratch` (nullable): grpo_loss_scratch_bytes(N) bytes from the
// forward workspace; with it, and at most grpo_loss_scratch_seqs(N) sequences,
// the loss runs one CTA per sequence, otherwise one CTA over all of them (the
// same bits either way).  ctl_zeroed: the merge before it on the stream was
// given the same scratch and zeroed its control words (else the call does).
cudaError_t launch_grpo(int N, const float* logp, const uint8_t* mask, const gh_grpo* g, float* coef,
                        float* loss3, int* status, void* scratch, bool ctl_zeroed, cudaStream_t st);
size_t grpo_loss_scratch_bytes(int64_t N);
int64_t grpo_loss_scratch_seqs(int64_t N);
// The 256-byte block of counters at the end of that scratch: words
// [0, GRPO_CTL_WORDS) are the loss's control words, word FWD_TILE_CTR_WORD the
// forward's tile counter.
constexpr int GRPO_CTL_WORDS = 8;
constexpr int FWD_TILE_CTR_WORD = 32;
int* grpo_scratch_ctl(void* scratch, int64_t N);
cudaError_t launch_grpo_totals(int num_seqs, const float* seq_policy, const float* seq_kl, const int32_t* seq_count,
                               int reduction, double norm, float beta, float* loss3, int* status, cudaStream_t st);
struct GspoArgs {
  int N;
  const float* logp;
  const float* old_logp;
  const float* ref_logp;
  const uint8_t* mask;
  const int32_t* seg_id;
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
};
// GSPO seam steps.  `scratch` (nullable): gspo_scratch_bytes(num_segments)
// bytes; with it one CTA per segment, otherwise one CTA (the same bits).
size_t gspo_scratch_bytes(int num_segments);
cudaError_t launch_gspo(const GspoArgs& g, void* scratch, cudaStream_t st);
cudaError_t launch_gspo_partials(const GspoArgs& g, float* fsum, int32_t* cnt, void* scratch, cudaStream_t st);
cudaError_t launch_gspo_finish(const GspoArgs& g, int R, const float* fsum_all, const int32_t* cnt_all, void* scratch,
                               cudaStream_t st);
cudaError_t launch_advantage(const float* rewards, int num_seqs, int group_size, float eps, float* adv,
                             cudaStream_t st);
// dH = sum over shards (in shard order) of the fp32 partials [num_shards, n]
cudaError_t launch_dh_merge(int num_shards, size_t n, bool to_bf16, const float* partials, void* out,
                            cudaStream_t st);
cudaError_t launch_timeout_probe(int* status, uint64_t timeout_ns, cudaStream_t st);

}  // namespace gh
