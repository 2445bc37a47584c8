// C ABI of the fused LM-head GRPO / GSPO loss: argument validation, workspace
// layout, launch sequencing and the optional per-kernel event instrumentation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "grpo_head.h"
#include "internal.h"

namespace gh {

static thread_local std::string g_last_error;

static gh_status fail(gh_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static gh_status fail(gh_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

void set_error_message(const std::string& msg) { g_last_error = msg; }

static gh_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- device facts
static std::mutex g_mu;

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

static bool device_is_sm103() {
  static int cache[64] = {0};  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 0 || dev >= 64) return false;
  if (cache[dev] == 0) {
    int ma = 0, mi = 0;
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    cache[dev] = (ma == 10 && mi == 3) ? 1 : 2;
  }
  return cache[dev] == 1;
}

int bwd_block_cols() {
  static int v = 0;
  if (v == 0) {
    const char* e = getenv("GH_BWD_BLOCK_COLS");
    const int x = e ? atoi(e) : 0;
    v = (x >= VTILE && x % VTILE == 0 && x <= (1 << 20)) ? x : 16384;
  }
  return v;
}

uint64_t timeout_ns() {
  static uint64_t t = 0;
  if (t == 0) {
    const char* e = getenv("GH_TIMEOUT_NS");
    unsigned long long v = e ? strtoull(e, nullptr, 10) : 0ull;
    t = v > 0 ? v : 2000000000ull;  // 2 s
  }
  return t;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- instrumentation
struct Prof {
  bool on = false;
  int64_t launches_total = 0;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  size_t pool_next = 0;
  int64_t count[GH_NUM_KERNEL_KINDS] = {0};
  double ms[GH_NUM_KERNEL_KINDS] = {0};
};
static Prof g_prof;

static cudaEvent_t pool_event() {
  if (g_prof.pool_next < g_prof.pool.size()) return g_prof.pool[g_prof.pool_next++];
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  g_prof.pool.push_back(e);
  g_prof.pool_next = g_prof.pool.size();
  return e;
}

void count_extra_launch() { ++g_prof.launches_total; }

template <class F>
static cudaError_t run(int kind, cudaStream_t st, F&& f) {
  ++g_prof.launches_total;
  if (!g_prof.on) return f();
  cudaEvent_t a = pool_event(), b = pool_event();
  if (a) cudaEventRecord(a, st);
  cudaError_t e = f();
  if (b) cudaEventRecord(b, st);
  if (a && b) g_prof.recs.push_back({kind, a, b});
  return e;
}

static void prof_collect() {
  for (auto& r : g_prof.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      g_prof.count[r.kind] += 1;
      g_prof.ms[r.kind] += ms;
    }
  }
  g_prof.recs.clear();
  g_prof.pool_next = 0;
}

// ---------------------------------------------------------------- validation helpers
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static gh_status check_head(const gh_head* h) {
  if (!h) return fail(GH_ERR_INVALID_ARG, "head is NULL");
  if (h->N < 0 || h->N > (int64_t(1) << 30)) return fail(GH_ERR_INVALID_ARG, "N=%lld out of range", (long long)h->N);
  if (h->D < 1 || h->D > (int64_t(1) << 20)) return fail(GH_ERR_INVALID_ARG, "D=%lld out of range", (long long)h->D);
  if (h->V < 1 || h->V > (int64_t(1) << 28)) return fail(GH_ERR_INVALID_ARG, "V=%lld out of range", (long long)h->V);
  if (h->dtype != GH_BF16 && h->dtype != GH_FP32) return fail(GH_ERR_INVALID_ARG, "dtype=%d unknown", h->dtype);
  if (h->row_tile != 0 && h->row_tile != 64 && h->row_tile != 128 && h->row_tile != 256)
    return fail(GH_ERR_INVALID_ARG, "row_tile=%d (expected 0, 64, 128 or 256)", h->row_tile);
  if (!h->W) return fail(GH_ERR_INVALID_ARG, "W is NULL");
  if (h->N > 0 && (!h->H || !h->targets || !h->mask)) return fail(GH_ERR_INVALID_ARG, "H/targets/mask is NULL");
  if (h->dtype == GH_BF16) {
    if (h->D % 8 != 0) return fail(GH_ERR_INVALID_ARG, "bf16 needs D %% 8 == 0 (D=%lld)", (long long)h->D);
    if (!aligned16(h->W) || (h->N > 0 && !aligned16(h->H)))
      return fail(GH_ERR_INVALID_ARG, "bf16 H and W must be 16-byte aligned");
  } else {
    if (!aligned16(h->W) || (h->N > 0 && !aligned16(h->H)))
      return fail(GH_ERR_INVALID_ARG, "fp32 H and W must be 16-byte aligned");
  }
  return GH_OK;
}

static int64_t num_splits(int64_t V) { return ceil_div(ceil_div(V, VTILE), TILES_PER_SPLIT); }

struct FwdWs {
  float* part_m;
  float* part_s;
  float* zy;
  void* loss;  // per-sequence slots of the GRPO loss
  size_t bytes;
};
static FwdWs fwd_layout(const gh_head* h, void* base) {
  const int64_t S = num_splits(h->V), N = h->N;
  const size_t a = align_up(static_cast<size_t>(S * N) * 4, 256);
  const size_t z = align_up(static_cast<size_t>(N) * 4, 256);
  char* b = static_cast<char*>(base);
  FwdWs w;
  w.part_m = reinterpret_cast<float*>(b);
  w.part_s = reinterpret_cast<float*>(b + a);
  w.zy = reinterpret_cast<float*>(b + 2 * a);
  w.loss = b + 2 * a + z;
  w.bytes = 2 * a + z + grpo_loss_scratch_bytes(N);
  return w;
}

// Backward plan.  The vocabulary is walked in blocks of vb columns (the bf16
// dlogits block G [rows, vb] lives in the workspace) and the rows in chunks of
// nc tokens, each chunk finishing its dH over all blocks before the next one
// starts and adding its dW contribution to dW.  nc keeps the workspace within
// three quarters of N * V * 2 bytes (the bf16 [N, V] logits the method never
// forms): one chunk of all N rows unless the vocabulary is narrow next to the
// block and accumulator rows.  nc depends on N, D, dtype and the WHOLE
// vocabulary only (V_total, also for a vocabulary shard), so that every
// vocabulary shard adds dW over the same row chunks as the single-shard call
// and its dW rows come out bitwise equal.  dH rows never depend on nc.
constexpr double BWD_MEM_FRACTION = 0.75;

// Vocabulary block width: bf16 16384 columns (GH_BWD_BLOCK_COLS), fp32 at most
// 1024 (the fp32 dlogits block is twice as wide in bytes, and narrow blocks
// keep whole-batch row chunks on small problems); never wider than the padded
// vocabulary.
static int64_t vocab_block(int64_t V, int dtype) {
  const int64_t Vp = ceil_div(V, VTILE) * VTILE;
  int64_t cols = bwd_block_cols();
  if (dtype != GH_BF16 && cols > 1024) cols = 1024;
  return Vp < cols ? Vp : cols;
}

static double bwd_budget(int64_t N, int64_t V) {
  return BWD_MEM_FRACTION * 2.0 * static_cast<double>(N) * static_cast<double>(V);
}

static int64_t bwd_rows_per_chunk(int64_t N, int64_t D, int64_t V_total, int dtype) {
  const bool bf16 = dtype == GH_BF16;
  const int64_t vb = vocab_block(V_total, dtype);
  const int64_t nblk = ceil_div(ceil_div(V_total, VTILE) * VTILE, vb);
  const double per_row = static_cast<double>(vb) * (bf16 ? 2 : 4) + ((bf16 && nblk > 1) ? 4.0 * D : 0.0);
  const double budget = bwd_budget(N, V_total);
  const int64_t gran = bf16 ? 128 : 64;  // one row tile of the single-CTA tensor-core / fp32 kernels
  if (N <= gran || static_cast<double>(N) * per_row <= budget) return N;
  // the most rows that fit, in whole row tiles (at least one), then spread
  // evenly over the chunks that takes
  int64_t nc_max = static_cast<int64_t>(budget / per_row) / gran * gran;
  if (nc_max < gran) nc_max = gran;
  const int64_t nch = ceil_div(N, nc_max);
  int64_t nc = ceil_div(ceil_div(N, nch), gran) * gran;
  if (nc > nc_max) nc = nc_max;
  return nc < N ? nc : N;
}

struct BwdWs {
  void* G;
  float* acc32;
  int* task_ctr;  // tile counter of the fused dH/dW launch
  float* slices;  // fp32 path: partials of the K slices that run in parallel
  size_t slice_bytes;
  int64_t vb;     // block width (columns)
  int64_t nblk;   // blocks
  int64_t nc;     // rows per chunk
  int64_t nch;    // chunks
  size_t bytes;
};
// dh_partial: a vocabulary shard's backward, whose fp32 dH partial is the
// caller's output (no accumulator needed)
static BwdWs bwd_layout(const gh_head* h, void* base, int64_t V_total, bool dh_partial) {
  const int64_t Vp = ceil_div(h->V, VTILE) * VTILE;
  BwdWs w;
  w.vb = vocab_block(h->V, h->dtype);
  w.nblk = ceil_div(Vp, w.vb);
  w.nc = bwd_rows_per_chunk(h->N, h->D, V_total, h->dtype);
  w.nch = w.nc > 0 ? ceil_div(h->N, w.nc) : 0;
  const bool bf16 = h->dtype == GH_BF16;
  const size_t g = align_up(static_cast<size_t>(w.nc) * w.vb * (bf16 ? 2 : 4), 256);
  const size_t acc = (bf16 && w.nblk > 1 && !dh_partial) ? align_up(static_cast<size_t>(w.nc) * h->D * 4, 256) : 0;
  // fp32: scratch for the K slices of the dH / dW GEMMs that run in parallel,
  // as much as their output grids can use within what the budget leaves (at
  // most 64 MB; none means every GEMM runs its slices inside each CTA)
  size_t sk = 0;
  if (!bf16) {
    const double left = bwd_budget(h->N, h->V) - static_cast<double>(g + acc + 256);
    size_t room = left > 0 ? static_cast<size_t>(left) / 256 * 256 : 0;
    if (room > (size_t(64) << 20)) room = size_t(64) << 20;
    const int p_dh = gemm_f32_par(w.nc, h->D, w.vb, room);
    const int p_dw = gemm_f32_par(w.vb, h->D, w.nc, room);
    const size_t s_dh = p_dh > 1 ? static_cast<size_t>(p_dh) * w.nc * h->D * 4 : 0;
    const size_t s_dw = p_dw > 1 ? static_cast<size_t>(p_dw) * w.vb * h->D * 4 : 0;
    sk = align_up(s_dh > s_dw ? s_dh : s_dw, 256);
  }
  char* b = static_cast<char*>(base);
  w.G = b;
  w.acc32 = acc ? reinterpret_cast<float*>(b + g) : nullptr;
  w.task_ctr = reinterpret_cast<int*>(b + g + acc);
  w.slices = sk ? reinterpret_cast<float*>(b + g + acc + 256) : nullptr;
  w.slice_bytes = sk;
  w.bytes = g + acc + 256 + sk;
  return w;
}

}  // namespace gh

using namespace gh;

extern "C" {

int32_t gh_abi_version(void) { return 106; }

const char* gh_status_string(gh_status s) {
  switch (s) {
    case GH_OK: return "GH_OK";
    case GH_ERR_INVALID_ARG: return "GH_ERR_INVALID_ARG";
    case GH_ERR_UNSUPPORTED: return "GH_ERR_UNSUPPORTED";
    case GH_ERR_WORKSPACE: return "GH_ERR_WORKSPACE";
    case GH_ERR_CUDA: return "GH_ERR_CUDA";
  }
  return "GH_ERR_UNKNOWN";
}

const char* gh_last_error(void) { return g_last_error.c_str(); }

size_t grpo_head_forward_workspace_size(const gh_head* head) {
  if (check_head(head) != GH_OK) return 0;
  return fwd_layout(head, nullptr).bytes;
}

size_t grpo_head_backward_workspace_size(const gh_head* head) {
  if (check_head(head) != GH_OK) return 0;
  return bwd_layout(head, nullptr, head->V, false).bytes;
}

size_t grpo_head_backward_shard_workspace_size(const gh_head* head, int64_t V_total) {
  if (check_head(head) != GH_OK) return 0;
  if (V_total < head->V || V_total > (int64_t(1) << 28)) return 0;
  return bwd_layout(head, nullptr, V_total, true).bytes;
}

gh_status grpo_head_forward(const gh_head* head, const gh_grpo* grpo, float* logp, float* lse, float* coef,
                            float* loss3, int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  gh_status s = check_head(head);
  if (s != GH_OK) return s;
  if (!status) return fail(GH_ERR_INVALID_ARG, "status is NULL");
  if (head->N > 0 && (!logp || !lse)) return fail(GH_ERR_INVALID_ARG, "logp/lse is NULL");
  if ((coef || loss3) && !grpo) return fail(GH_ERR_INVALID_ARG, "coef/loss3 requested without GRPO parameters");
  if (grpo) {
    if (head->N > 0 && (!grpo->old_logp || !grpo->adv || !grpo->seq_id))
      return fail(GH_ERR_INVALID_ARG, "old_logp/adv/seq_id is NULL");
    if (!grpo->ref_logp && grpo->beta != 0.f) return fail(GH_ERR_INVALID_ARG, "ref_logp is NULL with beta != 0");
    if (grpo->num_seqs < 1 || grpo->num_seqs > MAX_SEQS)
      return fail(GH_ERR_INVALID_ARG, "num_seqs=%d out of [1, %d]", grpo->num_seqs, MAX_SEQS);
    if (grpo->reduction < GH_TOKEN_MEAN || grpo->reduction > GH_FIXED)
      return fail(GH_ERR_INVALID_ARG, "reduction=%d unknown", grpo->reduction);
    if (grpo->reduction == GH_FIXED && !(grpo->norm > 0.0))
      return fail(GH_ERR_INVALID_ARG, "fixed reduction needs norm > 0");
    if (!(grpo->eps_low >= 0.f) || !(grpo->eps_high >= 0.f) || !std::isfinite(grpo->beta) || grpo->norm < 0.0)
      return fail(GH_ERR_INVALID_ARG, "eps_low/eps_high/beta/norm invalid");
    if (!(grpo->delta >= 0.f) || !std::isfinite(grpo->delta))
      return fail(GH_ERR_INVALID_ARG, "delta must be finite and >= 0 (0 = no cap)");
    if (grpo->ratio_level != 0 && grpo->ratio_level != 1)
      return fail(GH_ERR_INVALID_ARG, "ratio_level=%d (expected 0 token or 1 sequence)", grpo->ratio_level);
    if (grpo->reserved != 0) return fail(GH_ERR_INVALID_ARG, "gh_grpo.reserved must be 0");
  }
  const size_t need = fwd_layout(head, nullptr).bytes;
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GH_ERR_WORKSPACE, "forward workspace needs %zu bytes, got %zu", need, ws ? ws_bytes : size_t(0));
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = static_cast<int>(head->N), D = static_cast<int>(head->D), V = static_cast<int>(head->V);
  if (N > 0) {
    FwdWs w = fwd_layout(head, ws);
    cudaError_t e;
    if (head->dtype == GH_BF16) {
      // tile counter of the on-demand forward: a word of the loss scratch's counter block
      int* ctr = grpo_scratch_ctl(w.loss, N) + FWD_TILE_CTR_WORD;
      TcFwdArgs a{N, D, V, head->row_tile, head->H, head->W, head->targets, w.part_m, w.part_s, w.zy, status, 0, ctr};
      e = run(K_FWD_TC, st, [&] { return launch_fwd_tc(a, st); });
    } else {
      F32FwdArgs a{N, D, V, head->row_tile, static_cast<const float*>(head->H), static_cast<const float*>(head->W),
                   head->targets, w.part_m, w.part_s, w.zy};
      e = run(K_FWD_F32, st, [&] { return launch_fwd_f32(a, st); });
    }
    if (e != cudaSuccess) return cuda_fail(e, "forward logits/LSE launch");
    e = run(K_MERGE, st, [&] {
      return launch_merge(N, V, static_cast<int>(num_splits(V)), w.part_m, w.part_s, w.zy, head->targets, head->mask,
                          logp, lse, status, grpo ? w.loss : nullptr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  if (grpo) {
    // with N > 0 the merge above was given this scratch and zeroed its control words
    void* scratch = (ws && N > 0) ? fwd_layout(head, ws).loss : nullptr;
    cudaError_t e = run(K_GRPO, st, [&] {
      return launch_grpo(N, logp, head->mask, grpo, coef, loss3, status, scratch, scratch != nullptr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "GRPO loss launch");
  }
  return GH_OK;
}

int64_t gh_vocab_splits(int64_t V) { return V < 1 ? 0 : num_splits(V); }

gh_status gh_vocab_shard_bounds(int64_t V_total, int32_t num_shards, int32_t rank, int64_t* start, int64_t* len) {
  g_last_error.clear();
  if (!start || !len) return fail(GH_ERR_INVALID_ARG, "start/len is NULL");
  if (V_total < 1) return fail(GH_ERR_INVALID_ARG, "V_total must be >= 1");
  const int64_t S = ceil_div(V_total, SPLIT_COLS);
  if (num_shards < 1 || num_shards > MAX_SHARDS || num_shards > S)
    return fail(GH_ERR_INVALID_ARG, "num_shards=%d must be in [1, min(%d, %lld splits)]", num_shards, MAX_SHARDS,
                (long long)S);
  if (rank < 0 || rank >= num_shards) return fail(GH_ERR_INVALID_ARG, "rank out of range");
  const int64_t base = S / num_shards, extra = S % num_shards;
  const int64_t s0 = rank * base + (rank < extra ? rank : extra);
  const int64_t ns = base + (rank < extra ? 1 : 0);
  const int64_t c0 = s0 * SPLIT_COLS;
  const int64_t c1 = (s0 + ns) * SPLIT_COLS < V_total ? (s0 + ns) * SPLIT_COLS : V_total;
  *start = c0;
  *len = c1 - c0;
  return GH_OK;
}

gh_status grpo_head_logprob_shard(const gh_head* head, int64_t vocab_start, int64_t V_total, float* part_m,
                                  float* part_s, float* zy, int32_t* status, void* stream) {
  g_last_error.clear();
  gh_status s = check_head(head);
  if (s != GH_OK) return s;
  if (!status) return fail(GH_ERR_INVALID_ARG, "status is NULL");
  if (head->N > 0 && (!part_m || !part_s || !zy)) return fail(GH_ERR_INVALID_ARG, "part_m/part_s/zy is NULL");
  if (vocab_start < 0 || vocab_start % SPLIT_COLS != 0)
    return fail(GH_ERR_INVALID_ARG, "vocab_start=%lld must be a multiple of %d", (long long)vocab_start, SPLIT_COLS);
  if (V_total > (int64_t(1) << 28) || vocab_start + head->V > V_total)
    return fail(GH_ERR_INVALID_ARG, "shard [%lld, %lld) exceeds V_total=%lld", (long long)vocab_start,
                (long long)(vocab_start + head->V), (long long)V_total);
  if (vocab_start + head->V < V_total && head->V % SPLIT_COLS != 0)
    return fail(GH_ERR_INVALID_ARG, "a shard other than the last must hold whole %d-column splits", SPLIT_COLS);
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = static_cast<int>(head->N), D = static_cast<int>(head->D), V = static_cast<int>(head->V);
  if (N == 0) return GH_OK;
  cudaError_t e;
  if (head->dtype == GH_BF16) {
    TcFwdArgs a{N, D, V, head->row_tile, head->H, head->W, head->targets, part_m, part_s, zy, status,
                static_cast<int>(vocab_start)};
    e = run(K_FWD_TC, st, [&] { return launch_fwd_tc(a, st); });
  } else {
    F32FwdArgs a{N, D, V, head->row_tile, static_cast<const float*>(head->H), static_cast<const float*>(head->W),
                 head->targets, part_m, part_s, zy, static_cast<int>(vocab_start)};
    e = run(K_FWD_F32, st, [&] { return launch_fwd_f32(a, st); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "shard forward launch");
  return GH_OK;
}

gh_status grpo_logprob_merge(int64_t N, int64_t V_total, int32_t num_shards, const int64_t* shard_starts,
                             const float* part_m, const float* part_s, const float* zy, const int32_t* targets,
                             const uint8_t* mask, float* logp, float* lse, int32_t* status, void* stream) {
  g_last_error.clear();
  if (N < 0 || N > (int64_t(1) << 30)) return fail(GH_ERR_INVALID_ARG, "N out of range");
  if (V_total < 1 || V_total > (int64_t(1) << 28)) return fail(GH_ERR_INVALID_ARG, "V_total out of range");
  if (!status || !shard_starts) return fail(GH_ERR_INVALID_ARG, "status/shard_starts is NULL");
  if (N > 0 && (!part_m || !part_s || !zy || !targets || !mask || !logp || !lse))
    return fail(GH_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (num_shards < 1 || num_shards > MAX_SHARDS)
    return fail(GH_ERR_INVALID_ARG, "num_shards=%d out of [1, %d]", num_shards, MAX_SHARDS);
  ShardBounds sb;
  sb.num_shards = num_shards;
  if (shard_starts[0] != 0 || shard_starts[num_shards] != V_total)
    return fail(GH_ERR_INVALID_ARG, "shard bounds must start at 0 and end at V_total");
  for (int r = 0; r < num_shards; ++r) {
    if (shard_starts[r + 1] <= shard_starts[r] || shard_starts[r] % SPLIT_COLS != 0)
      return fail(GH_ERR_INVALID_ARG, "shard %d bounds [%lld, %lld) are not increasing multiples of %d", r,
                  (long long)shard_starts[r], (long long)shard_starts[r + 1], SPLIT_COLS);
    sb.start[r] = static_cast<int>(shard_starts[r]);
  }
  sb.start[num_shards] = static_cast<int>(V_total);
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = run(K_MERGE_SHARDS, st, [&] {
    return launch_merge_shards(static_cast<int>(N), static_cast<int>(V_total), static_cast<int>(num_splits(V_total)),
                               part_m, part_s, zy, sb, targets, mask, logp, lse, status, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "shard merge launch");
  return GH_OK;
}

gh_status grpo_loss_from_sequence_totals(int32_t num_seqs, const float* seq_policy, const float* seq_kl,
                                         const int32_t* seq_count, int32_t reduction, double norm, float beta,
                                         float* loss3, int32_t* status, void* stream) {
  g_last_error.clear();
  if (!seq_policy || !seq_kl || !seq_count || !loss3 || !status)
    return fail(GH_ERR_INVALID_ARG, "seq_policy/seq_kl/seq_count/loss3/status is NULL");
  if (num_seqs < 1 || num_seqs > MAX_SEQS)
    return fail(GH_ERR_INVALID_ARG, "num_seqs=%d out of [1, %d]", num_seqs, MAX_SEQS);
  if (reduction < GH_TOKEN_MEAN || reduction > GH_FIXED) return fail(GH_ERR_INVALID_ARG, "reduction=%d unknown", reduction);
  if (reduction == GH_FIXED && !(norm > 0.0)) return fail(GH_ERR_INVALID_ARG, "fixed reduction needs norm > 0");
  if (norm < 0.0 || !std::isfinite(beta)) return fail(GH_ERR_INVALID_ARG, "norm/beta invalid");
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = run(K_GRPO_TOTALS, st, [&] {
    return launch_grpo_totals(num_seqs, seq_policy, seq_kl, seq_count, reduction, norm, beta, loss3, status, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "sequence-totals launch");
  return GH_OK;
}

static gh_status check_gspo_common(int64_t N, const float* logp, const uint8_t* mask, const int32_t* seg_id,
                                   int32_t num_segments, int32_t* status) {
  if (N < 0 || N > (int64_t(1) << 30)) return fail(GH_ERR_INVALID_ARG, "N out of range");
  if (!status) return fail(GH_ERR_INVALID_ARG, "status is NULL");
  if (N > 0 && (!logp || !mask || !seg_id)) return fail(GH_ERR_INVALID_ARG, "logp/mask/seg_id is NULL");
  if (num_segments < 1 || num_segments > MAX_SEQS)
    return fail(GH_ERR_INVALID_ARG, "num_segments=%d out of [1, %d]", num_segments, MAX_SEQS);
  return GH_OK;
}

static gh_status check_gspo_loss_args(const float* ref_logp, float beta, const float* seg_adv, float eps_low,
                                      float eps_high, double divisor, float* loss, float* coef, int64_t N) {
  if (!loss || !seg_adv) return fail(GH_ERR_INVALID_ARG, "loss/seg_adv is NULL");
  if (N > 0 && !coef) return fail(GH_ERR_INVALID_ARG, "coef is NULL");
  if (!(divisor > 0.0) || !std::isfinite(divisor)) return fail(GH_ERR_INVALID_ARG, "divisor must be > 0");
  if (!(eps_low >= 0.f) || !(eps_high >= 0.f)) return fail(GH_ERR_INVALID_ARG, "eps must be >= 0");
  if (!std::isfinite(beta) || (beta != 0.f && !ref_logp))
    return fail(GH_ERR_INVALID_ARG, "beta must be finite, and ref_logp given when beta != 0");
  return GH_OK;
}

size_t gspo_segment_workspace_size(int32_t num_segments) {
  if (num_segments < 1 || num_segments > MAX_SEQS) return 0;
  return gspo_scratch_bytes(num_segments);
}

// ws of a seam call: NULL (one CTA) or at least gspo_segment_workspace_size bytes
static gh_status check_gspo_ws(int32_t num_segments, void* ws, size_t ws_bytes) {
  if (ws && ws_bytes < gspo_scratch_bytes(num_segments))
    return fail(GH_ERR_WORKSPACE, "GSPO workspace needs %zu bytes, got %zu", gspo_scratch_bytes(num_segments),
                ws_bytes);
  if (ws && !aligned16(ws)) return fail(GH_ERR_INVALID_ARG, "GSPO workspace must be 16-byte aligned");
  return GH_OK;
}

gh_status gspo_segment_loss(int64_t N, const float* logp, const float* old_logp, const float* ref_logp,
                            const uint8_t* mask, const int32_t* seg_id, int32_t num_segments, const float* seg_adv,
                            float eps_low, float eps_high, float beta, double divisor, int32_t token_weighted,
                            float* loss, float* seg_ratio, float* coef, float* mean_logp, int32_t* num_clipped,
                            int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  gh_status s = check_gspo_common(N, logp, mask, seg_id, num_segments, status);
  if (s != GH_OK) return s;
  if (N > 0 && !old_logp) return fail(GH_ERR_INVALID_ARG, "old_logp is NULL");
  s = check_gspo_loss_args(ref_logp, beta, seg_adv, eps_low, eps_high, divisor, loss, coef, N);
  if (s != GH_OK) return s;
  s = check_gspo_ws(num_segments, ws, ws_bytes);
  if (s != GH_OK) return s;
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GspoArgs g{static_cast<int>(N), logp, old_logp, beta != 0.f ? ref_logp : nullptr, mask, seg_id, num_segments,
             seg_adv, eps_low, eps_high, beta, divisor, token_weighted, loss, seg_ratio, coef, mean_logp,
             num_clipped, status};
  cudaError_t e = run(K_GSPO, st, [&] { return launch_gspo(g, ws, st); });
  if (e != cudaSuccess) return cuda_fail(e, "GSPO launch");
  return GH_OK;
}

gh_status gspo_segment_partials(int64_t N, const float* logp, const float* old_logp, const float* ref_logp,
                                const uint8_t* mask, const int32_t* seg_id, int32_t num_segments, float* fsum,
                                int32_t* cnt, int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  gh_status s = check_gspo_common(N, logp, mask, seg_id, num_segments, status);
  if (s != GH_OK) return s;
  if (N > 0 && !old_logp) return fail(GH_ERR_INVALID_ARG, "old_logp is NULL");
  if (!fsum || !cnt) return fail(GH_ERR_INVALID_ARG, "fsum/cnt is NULL");
  s = check_gspo_ws(num_segments, ws, ws_bytes);
  if (s != GH_OK) return s;
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GspoArgs g{static_cast<int>(N), logp, old_logp, ref_logp, mask, seg_id, num_segments, nullptr, 0.f, 0.f, 0.f,
             1.0, 0, nullptr, nullptr, nullptr, nullptr, nullptr, status};
  cudaError_t e = run(K_GSPO_PARTIALS, st, [&] { return launch_gspo_partials(g, fsum, cnt, ws, st); });
  if (e != cudaSuccess) return cuda_fail(e, "GSPO partials launch");
  return GH_OK;
}

gh_status gspo_segment_loss_from_partials(int64_t N, const float* logp, const float* ref_logp, const uint8_t* mask,
                                          const int32_t* seg_id, int32_t num_segments, int32_t num_ranks,
                                          const float* fsum_all, const int32_t* cnt_all, const float* seg_adv,
                                          float eps_low, float eps_high, float beta, double divisor,
                                          int32_t token_weighted, float* loss, float* seg_ratio, float* coef,
                                          float* mean_logp, int32_t* num_clipped, int32_t* status, void* ws,
                                          size_t ws_bytes, void* stream) {
  g_last_error.clear();
  gh_status s = check_gspo_common(N, logp, mask, seg_id, num_segments, status);
  if (s != GH_OK) return s;
  s = check_gspo_loss_args(ref_logp, beta, seg_adv, eps_low, eps_high, divisor, loss, coef, N);
  if (s != GH_OK) return s;
  if (num_ranks < 1 || num_ranks > 4096) return fail(GH_ERR_INVALID_ARG, "num_ranks out of [1, 4096]");
  if (!fsum_all || !cnt_all) return fail(GH_ERR_INVALID_ARG, "fsum_all/cnt_all is NULL");
  s = check_gspo_ws(num_segments, ws, ws_bytes);
  if (s != GH_OK) return s;
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GspoArgs g{static_cast<int>(N), logp, nullptr, beta != 0.f ? ref_logp : nullptr, mask, seg_id, num_segments,
             seg_adv, eps_low, eps_high, beta, divisor, token_weighted, loss, seg_ratio, coef, mean_logp,
             num_clipped, status};
  cudaError_t e =
      run(K_GSPO_FINISH, st, [&] { return launch_gspo_finish(g, num_ranks, fsum_all, cnt_all, ws, st); });
  if (e != cudaSuccess) return cuda_fail(e, "GSPO finish launch");
  return GH_OK;
}

// Backward body shared by the whole-vocabulary and the vocabulary-shard
// entry points.  col_offset: global id of local column 0 (targets are global).
// V_total: the whole vocabulary (it fixes the row chunks).  dh_partial: dH is
// an fp32 [N, D] partial over this vocabulary (no cast).
static gh_status backward_impl(const gh_head* head, const float* lse, const float* coef, const float* grad_out,
                               void* dH, float* dW, int32_t accumulate_dW, int32_t* status, void* ws,
                               size_t ws_bytes, void* stream, int col_offset, int64_t V_total, bool dh_partial) {
  if (!status || !dW) return fail(GH_ERR_INVALID_ARG, "status/dW is NULL");
  if (head->N > 0 && (!lse || !coef || !dH)) return fail(GH_ERR_INVALID_ARG, "lse/coef/dH is NULL");
  if (!aligned16(dW) || (head->N > 0 && !aligned16(dH))) return fail(GH_ERR_INVALID_ARG, "dH/dW must be 16-byte aligned");
  const size_t need = bwd_layout(head, nullptr, V_total, dh_partial).bytes;
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GH_ERR_WORKSPACE, "backward workspace needs %zu bytes, got %zu", need, ws ? ws_bytes : size_t(0));
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = static_cast<int>(head->N), D = static_cast<int>(head->D), V = static_cast<int>(head->V);
  if (N == 0) {
    if (!accumulate_dW) {
      cudaError_t e = cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * D * sizeof(float), st);
      if (e != cudaSuccess) return cuda_fail(e, "dW clear");
    }
    return GH_OK;
  }
  BwdWs w = bwd_layout(head, ws, V_total, dh_partial);
  const int64_t Vp = ceil_div(V, VTILE) * VTILE;
  const bool bf16 = head->dtype == GH_BF16;
  const size_t in_elt = bf16 ? 2 : 4;
  const size_t dh_elt = (bf16 && !dh_partial) ? 2 : 4;
  for (int64_t c = 0; c < w.nch; ++c) {
    // rows [r0, r0 + n): this chunk's dH is finished over every block before
    // the next chunk starts; its dW contribution is added to dW
    const int64_t r0 = c * w.nc;
    const int n = static_cast<int>((N - r0) < w.nc ? (N - r0) : w.nc);
    const void* Hc = static_cast<const char*>(head->H) + static_cast<size_t>(r0) * D * in_elt;
    const int32_t* yc = head->targets + r0;
    const float* lse_c = lse + r0;
    const float* coef_c = coef + r0;
    void* dHc = static_cast<char*>(dH) + static_cast<size_t>(r0) * D * dh_elt;
    const int acc_dW = (c > 0 || accumulate_dW) ? 1 : 0;
    for (int64_t b = 0; b < w.nblk; ++b) {
      const int vb0 = static_cast<int>(b * w.vb);
      const int width = static_cast<int>((Vp - vb0) < w.vb ? (Vp - vb0) : w.vb);
      const int ldg = static_cast<int>(w.vb);
      cudaError_t e;
      if (bf16) {
        // the dlogits launch zeroes the fused launch's tile counter on entry
        TcDlogitsArgs da{n,   D,      V,          vb0, width, ldg, Hc, head->W, yc, lse_c, coef_c, grad_out, w.G,
                         status, col_offset, dhdw_fused() ? w.task_ctr : nullptr};
        e = run(K_DLOGITS_TC, st, [&] { return launch_dlogits_tc(da, st); });
        if (e != cudaSuccess) return cuda_fail(e, "dlogits launch");
        int mode;
        float* acc32 = w.acc32;
        if (dh_partial) {
          mode = b == 0 ? 0 : 1;  // fp32 partial accumulated in place
          acc32 = static_cast<float*>(dHc);
        } else if (w.nblk == 1) {
          mode = 3;
        } else if (b == 0) {
          mode = 0;
        } else if (b == w.nblk - 1) {
          mode = 2;
        } else {
          mode = 1;
        }
        TcDhArgs ha{n, D, V, vb0, width, ldg, w.G, head->W, mode, acc32, dHc, status};
        TcDwArgs wa{n, D, V, vb0, width, ldg, w.G, Hc, acc_dW, dW, status};
        if (dhdw_fused()) {
          e = run(K_DHDW_TC, st, [&] { return launch_dhdw_tc(ha, wa, w.task_ctr, true, st); });
          if (e != cudaSuccess) return cuda_fail(e, "dH/dW launch");
        } else {
          e = run(K_DH_TC, st, [&] { return launch_dh_tc(ha, st); });
          if (e != cudaSuccess) return cuda_fail(e, "dH launch");
          e = run(K_DW_TC, st, [&] { return launch_dw_tc(wa, st); });
          if (e != cudaSuccess) return cuda_fail(e, "dW launch");
        }
      } else {
        const float* H = static_cast<const float*>(Hc);
        const float* W = static_cast<const float*>(head->W);
        float* G = static_cast<float*>(w.G);
        F32DlogitsArgs da{n, D, V, vb0, width, ldg, H, W, yc, lse_c, coef_c, grad_out, G, col_offset};
        e = run(K_DLOGITS_F32, st, [&] { return launch_dlogits_f32(da, st); });
        if (e != cudaSuccess) return cuda_fail(e, "dlogits launch");
        const int real = static_cast<int>((V - vb0) < width ? (V - vb0) : width);
        // dH[rows, D] (+)= G[:, :real] W[vb0:vb0+real, :]
        F32GemmArgs ha{n, D, real, G, ldg, 1, W + static_cast<size_t>(vb0) * D, D, 1, static_cast<float*>(dHc), D,
                       0, b > 0 ? 1 : 0, gemm_f32_par(n, D, real, w.slice_bytes), w.slices, 0};
        e = run(K_GEMM_F32, st, [&] { return launch_gemm_f32(ha, st); });
        if (e != cudaSuccess) return cuda_fail(e, "dH launch");
        // dW[vb0 + v, :] (+)= sum over the chunk's rows i of G[i, v] H[i, :]
        F32GemmArgs wa{real, D, n, G, 1, ldg, H, D, 1, dW, D, vb0, acc_dW, gemm_f32_par(real, D, n, w.slice_bytes),
                       w.slices, 0};
        e = run(K_GEMM_F32, st, [&] { return launch_gemm_f32(wa, st); });
        if (e != cudaSuccess) return cuda_fail(e, "dW launch");
      }
    }
  }
  return GH_OK;
}

gh_status grpo_head_backward(const gh_head* head, const float* lse, const float* coef, const float* grad_out,
                             void* dH, float* dW, int32_t accumulate_dW, int32_t* status, void* ws, size_t ws_bytes,
                             void* stream) {
  g_last_error.clear();
  gh_status s = check_head(head);
  if (s != GH_OK) return s;
  return backward_impl(head, lse, coef, grad_out, dH, dW, accumulate_dW, status, ws, ws_bytes, stream, 0, head->V,
                       false);
}

gh_status grpo_head_backward_shard(const gh_head* head, int64_t vocab_start, int64_t V_total, const float* lse,
                                   const float* coef, const float* grad_out, float* dH_partial, float* dW,
                                   int32_t accumulate_dW, int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  gh_status s = check_head(head);
  if (s != GH_OK) return s;
  if (vocab_start < 0 || vocab_start % SPLIT_COLS != 0)
    return fail(GH_ERR_INVALID_ARG, "vocab_start=%lld must be a multiple of %d", (long long)vocab_start, SPLIT_COLS);
  if (V_total > (int64_t(1) << 28) || vocab_start + head->V > V_total)
    return fail(GH_ERR_INVALID_ARG, "shard exceeds V_total");
  return backward_impl(head, lse, coef, grad_out, dH_partial, dW, accumulate_dW, status, ws, ws_bytes, stream,
                       static_cast<int>(vocab_start), V_total, true);
}

gh_status grpo_dh_merge(int32_t num_shards, int64_t N, int64_t D, int32_t dtype, const float* dH_partials, void* dH,
                        int32_t* status, void* stream) {
  g_last_error.clear();
  if (!status || (N > 0 && (!dH_partials || !dH))) return fail(GH_ERR_INVALID_ARG, "a pointer is NULL");
  if (num_shards < 1 || num_shards > MAX_SHARDS) return fail(GH_ERR_INVALID_ARG, "num_shards out of range");
  if (N < 0 || D < 1 || N * D > (int64_t(1) << 40)) return fail(GH_ERR_INVALID_ARG, "N/D out of range");
  if (dtype != GH_BF16 && dtype != GH_FP32) return fail(GH_ERR_INVALID_ARG, "dtype unknown");
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = run(K_DH_MERGE, st, [&] {
    return launch_dh_merge(num_shards, static_cast<size_t>(N) * static_cast<size_t>(D), dtype == GH_BF16,
                           dH_partials, dH, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dH merge launch");
  return GH_OK;
}

gh_status grpo_group_advantage(const float* rewards, int32_t num_seqs, int32_t group_size, float eps, float* adv,
                               int32_t* status, void* stream) {
  g_last_error.clear();
  if (!rewards || !adv || !status) return fail(GH_ERR_INVALID_ARG, "rewards/adv/status is NULL");
  if (group_size < 1 || num_seqs < 1 || num_seqs % group_size != 0)
    return fail(GH_ERR_INVALID_ARG, "num_seqs=%d must be a positive multiple of group_size=%d", num_seqs, group_size);
  if (!(eps >= 0.f)) return fail(GH_ERR_INVALID_ARG, "eps must be >= 0");
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      run(K_ADV, st, [&] { return launch_advantage(rewards, num_seqs, group_size, eps, adv, st); });
  if (e != cudaSuccess) return cuda_fail(e, "advantage launch");
  return GH_OK;
}

void gh_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof.on = on != 0;
}

void gh_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  prof_collect();
  for (int k = 0; k < GH_NUM_KERNEL_KINDS; ++k) {
    g_prof.count[k] = 0;
    g_prof.ms[k] = 0.0;
  }
}

gh_status gh_profile_read(int32_t kind, int64_t* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (kind < 0 || kind >= GH_NUM_KERNEL_KINDS || !launches || !total_ms)
    return fail(GH_ERR_INVALID_ARG, "bad profile query");
  prof_collect();
  *launches = g_prof.count[kind];
  *total_ms = g_prof.ms[kind];
  return GH_OK;
}

int64_t gh_launch_count(void) { return g_prof.launches_total; }

const char* gh_kernel_kind_name(int32_t kind) {
  static const char* names[GH_NUM_KERNEL_KINDS] = {
      "fwd_logits_lse_tc", "merge_lse", "grpo_loss", "gspo_segment", "dlogits_tc", "dh_gemm_tc",
      "dw_gemm_tc", "group_advantage", "fwd_logits_lse_f32", "dlogits_f32", "gemm_f32", "timeout_probe",
      "grpo_sequence_totals", "merge_lse_shards", "gspo_partials", "gspo_finish", "dh_merge",
      "dhdw_gemm_tc"};
  if (kind < 0 || kind >= GH_NUM_KERNEL_KINDS) return "";
  return names[kind];
}

gh_status gh_timeout_probe(int32_t* status, uint64_t timeout_ns_, void* stream) {
  g_last_error.clear();
  if (!status) return fail(GH_ERR_INVALID_ARG, "status is NULL");
  if (timeout_ns_ == 0 || timeout_ns_ > 10000000000ull) return fail(GH_ERR_INVALID_ARG, "timeout out of (0, 10 s]");
  if (!device_is_sm103()) return fail(GH_ERR_UNSUPPORTED, "current device is not an sm_103 (GB300) GPU");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = run(K_PROBE, st, [&] { return launch_timeout_probe(status, timeout_ns_, st); });
  if (e != cudaSuccess) return cuda_fail(e, "probe launch");
  return GH_OK;
}

}  // extern "C"
