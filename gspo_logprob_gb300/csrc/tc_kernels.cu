// tcgen05 kernels of the bf16 path: logits + online LSE (forward), dlogits
// recompute (backward) and the dH / dW GEMMs, as instances of the CTA-pair
// kernel (tc_gemm_pair_kernel), its on-demand form with one or two jobs
// (tc_dual_pair_kernel) and the single-CTA kernel (tc_gemm_kernel).
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "tc_gemm.cuh"
#include "tc_gemm_pair.cuh"
#include "tc_gemm_dual.cuh"

namespace gh {

namespace {

// Tuning knobs (read once from the environment): which kernel runs each
// product, its CTA row-tile height (1 or 2 blocks of 128 rows), the raster
// group size, the epilogue warps and the tile hand-out.  Every setting
// computes the same result; they only change tile shape, order and which
// warps or CTAs do the work.
int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e ? atoi(e) : dflt;
}
// per kernel kind: 1 = 128 x 256 tiles (double-buffered accumulator), 2 = 256 x 256.
// Defaults from a sweep on the 8B-vocabulary workload: dlogits and dW run 256-row
// tiles (their epilogues are short next to K); dH keeps 128-row tiles because
// its fp32 read-modify-write epilogue needs the second accumulator to hide.
int kind_mt(const char* name, int dflt) {
  const int v = env_int(name, dflt);
  return v == 1 || v == 2 ? v : dflt;
}
int dlogits_mt() {
  static const int v = kind_mt("GH_DLOGITS_MT", 2);
  return v;
}
int dh_mt() {
  static const int v = kind_mt("GH_DH_MT", 1);
  return v;
}
int dw_mt() {
  static const int v = kind_mt("GH_DW_MT", 2);
  return v;
}
// epilogue warps per TMEM row for the 256-row tiles (1 or 2)
int dlogits_cg() {
  static const int v = kind_mt("GH_DLOGITS_CG", 1);
  return v;
}
int dh_cg() {
  static const int v = kind_mt("GH_DH_CG", 1);
  return v;
}
int dw_cg() {
  static const int v = kind_mt("GH_DW_CG", 1);
  return v;
}
int kind_group_m(const char* name, int dflt) {
  const int v = env_int(name, dflt);
  return v > 0 ? v : dflt;
}
// forward raster group (row tiles per group; 0 = all row tiles of a tile
// column before the next).  16: H's rows for a group stay in L2 while W tiles
// stream past; on the 8B-vocabulary step it cut DRAM reads and ran 0.9% faster
// under the power cap than a group of all 32 row tiles
int fwd_group_m() {
  static const int v = env_int("GH_FWD_GROUP_M", 16);
  return v > 0 ? v : 0;
}
// forward epilogue groups of the CTA-pair kernel: 2 (two tiles' epilogues at
// once) when a tile's MMAs are short next to its epilogue -- K of at most 16
// blocks (D <= 1024) -- else 1; GH_FWD_EPI_GROUPS = 1 or 2 forces it.  The
// results are the same bits either way.
int fwd_epi_groups(int num_kb) {
  static const int v = env_int("GH_FWD_EPI_GROUPS", 0);
  if (v == 1 || v == 2) return v;
  return num_kb <= 16 ? 2 : 1;
}
// forward tiles handed out on demand (1) or dealt round-robin (0).  Default:
// on demand for K of more than 32 blocks (D > 2048), where a launch is long
// enough for round-robin pairs to drift apart and re-read W from DRAM (at
// D = 4096 on demand read a third of the bytes); at D = 2048 the hand-out's
// per-tile cost was 1-2% and round-robin stayed faster.
int fwd_dynamic(int num_kb) {
  static const int v = env_int("GH_FWD_DYNAMIC", -1);
  if (v == 0 || v == 1) return v;
  return num_kb > 32 && fwd_epi_groups(num_kb) == 1 ? 1 : 0;
}
int dlogits_group_m() {
  static const int v = kind_group_m("GH_DLOGITS_GROUP_M", 16);
  return v;
}
// dH / dW: groups of 8 row tiles (a 76-tile wave then touches the fewest
// distinct operand bytes; measured +0.7% over 16 on the fused launch)
int dh_group_m() {
  static const int v = kind_group_m("GH_DH_GROUP_M", 8);
  return v;
}
int dw_group_m() {
  static const int v = kind_group_m("GH_DW_GROUP_M", 8);
  return v;
}

// Launch set-up of one kernel instance, done once per device under a lock:
// the dynamic shared-memory limit is a per-device function attribute, and the
// number of CTA pairs that fit is queried after it is set.
struct KernSetup {
  std::mutex mu;
  bool done[64] = {};
  int pairs[64] = {};
};

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev < 0 || dev >= 64 ? 0 : dev;
}

// sets the shared-memory attribute; with `cluster_pairs` also returns how many
// 2-CTA clusters of `threads` threads fit on the device (at most max_pairs())
int max_pairs();
cudaError_t kern_setup(KernSetup& s, const void* kern, int smem, int threads, bool cluster_pairs, int* pairs) {
  const int dev = current_device();
  std::lock_guard<std::mutex> g(s.mu);
  if (!s.done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    if (cluster_pairs) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(2 * max_pairs());
      q.blockDim = dim3(threads);
      q.dynamicSmemBytes = smem;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) n = max_pairs();
      (void)cudaGetLastError();
      if (n > max_pairs()) n = max_pairs();
    }
    s.pairs[dev] = n;
    s.done[dev] = true;
  }
  if (pairs) *pairs = s.pairs[dev];
  return cudaSuccess;
}

template <int MT, int CG, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const TcSched& sc, int b_off_n, int b_off_k,
                      const typename Epi::Params& ep, int* status, cudaStream_t st) {
  using C = TcCfg<MT, CG>;
  auto kern = tc_gemm_kernel<MT, CG, A_MN, B_MN, Epi>;
  static KernSetup setup;  // per instantiation
  cudaError_t e = kern_setup(setup, reinterpret_cast<const void*>(kern), C::SMEM_BYTES, C::THREADS, false, nullptr);
  if (e != cudaSuccess) return e;
  if (sc.num_tasks <= 0) return cudaSuccess;
  const int grid = static_cast<int>(sc.num_tasks < num_sms() ? sc.num_tasks : num_sms());
  kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(ta, tb, sc, b_off_n, b_off_k, ep, status, timeout_ns());
  return cudaGetLastError();
}

// CTA-pair kernels (cta_group::2, 256 x 256 tiles over two SMs) per kind: 1 on
// (default; measured faster for every kind on the 8B-vocabulary workload), 0 the
// single-CTA kernels selected by the tile-height knobs below
int pair_knob(const char* name, int dflt) {
  const int v = env_int(name, dflt);
  return v == 0 || v == 1 ? v : dflt;
}
int fwd_pair() {
  static const int v = pair_knob("GH_FWD_PAIR", 1);
  return v;
}
int dlogits_pair() {
  static const int v = pair_knob("GH_DLOGITS_PAIR", 1);
  return v;
}
int dh_pair() {
  static const int v = pair_knob("GH_DH_PAIR", 1);
  return v;
}
int dw_pair() {
  static const int v = pair_knob("GH_DW_PAIR", 1);
  return v;
}

// dH and dW of a block in one launch with dynamically handed-out tiles (1,
// default) or as two launches (0); only with both pair knobs on
int bwd_fused_knob() {
  static const int v = pair_knob("GH_BWD_FUSED", 1);
  return v;
}

int max_pairs() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) cache[dev] = num_sms() / 2 > 0 ? num_sms() / 2 : 1;
  return cache[dev];
}

template <bool A_MN, bool B_MN, class Epi, int EG = 1>
cudaError_t launch_tc_pair(const CUtensorMap& ta, const CUtensorMap& tb, const TcSched& sc, int b_off_n, int b_off_k,
                           const typename Epi::Params& ep, int* status, cudaStream_t st) {
  using C = TcPairCfg;
  constexpr int THREADS = tc_pair_threads(EG);
  if (EG > 1 && sc.n_per_task != 1) return cudaErrorInvalidValue;  // groups take whole tasks of one tile
  auto kern = tc_gemm_pair_kernel<A_MN, B_MN, Epi, EG>;
  static KernSetup setup;  // per instantiation
  int pairs_fit = 0;
  cudaError_t e0 = kern_setup(setup, reinterpret_cast<const void*>(kern), C::SMEM_BYTES, THREADS, true, &pairs_fit);
  if (e0 != cudaSuccess) return e0;
  if (sc.num_tasks <= 0) return cudaSuccess;
  const int pairs = sc.num_tasks < pairs_fit ? sc.num_tasks : pairs_fit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, sc, b_off_n, b_off_k, ep, status, timeout_ns());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

TcSched make_sched(int num_m_blocks, int num_n_blocks, int n_per_task, int num_kb, int m_step, int group_m) {
  TcSched sc;
  sc.num_m_blocks = num_m_blocks;
  sc.num_n_blocks = num_n_blocks;
  sc.n_per_task = n_per_task;
  sc.num_kb = num_kb;
  sc.m_step = m_step;
  sc.group_m = group_m < 1 ? 1 : (group_m > num_m_blocks ? num_m_blocks : group_m);
  sc.num_ng = static_cast<int>(ceil_div(num_n_blocks, n_per_task));
  sc.num_tasks = num_m_blocks * sc.num_ng;
  return sc;
}

// One launch of tc_dual_pair_kernel: the tiles of j0, then of j1, handed out
// from *task_ctr, which must read 0 at the start (the call zeroes it unless
// ctr_zeroed says an earlier launch on the stream did).
template <class Epi>
cudaError_t launch_dual(const CUtensorMap& ta0, const CUtensorMap& tb0, const CUtensorMap& ta1, const CUtensorMap& tb1,
                        const PairJob& j0, const PairJob& j1, const typename Epi::Params& e0,
                        const typename Epi::Params& e1, int* task_ctr, bool ctr_zeroed, int* status,
                        cudaStream_t st) {
  const int tasks = j0.sc.num_tasks + j1.sc.num_tasks;
  if (tasks <= 0) return cudaSuccess;
  auto kern = tc_dual_pair_kernel<Epi>;
  static KernSetup setup;  // per instantiation
  int pairs_fit = 0;
  cudaError_t e = kern_setup(setup, reinterpret_cast<const void*>(kern), DUAL_SMEM_BYTES, TcPairCfg::THREADS, true,
                             &pairs_fit);
  if (e != cudaSuccess) return e;
  if (!ctr_zeroed) {
    e = cudaMemsetAsync(task_ctr, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  const int pairs = tasks < pairs_fit ? tasks : pairs_fit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(TcPairCfg::THREADS);
  cfg.dynamicSmemBytes = DUAL_SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta0, tb0, ta1, tb1, j0, j1, e0, e1, task_ctr, status, timeout_ns());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const TcFwdArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = H [N, D] K-major, B = W [V, D] K-major
  if (!make_tmap_bf16(&ta, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN)) return cudaErrorInvalidValue;
  const int num_vt = static_cast<int>(ceil_div(a.V, VTILE));
  const int nkb = static_cast<int>(ceil_div(a.D, TC_BK));
  EpiFwdLse::Params ep;
  ep.N = a.N;
  ep.V = a.V;
  ep.part_m = a.part_m;
  ep.part_s = a.part_s;
  ep.zy = a.zy;
  ep.targets = a.targets;
  ep.col_offset = a.col_offset;
  // row tiles in raster groups (fwd_group_m) before the next tile column: a
  // tile column's W tiles are shared in L2 by the CTAs working on it
  if (a.row_tile == 64 || a.row_tile == 128) {
    const int m_step = a.row_tile;
    const int num_m = static_cast<int>(ceil_div(a.N, m_step));
    TcSched sc = make_sched(num_m, num_vt, TILES_PER_SPLIT, nkb, m_step, fwd_group_m() ? fwd_group_m() : num_m);
    return launch_tc<1, 1, false, false, EpiFwdLse>(ta, tb, sc, 0, 0, ep, a.status, st);
  }
  const int num_m = static_cast<int>(ceil_div(a.N, 2 * TC_BM));
  TcSched sc = make_sched(num_m, num_vt, TILES_PER_SPLIT, nkb, 2 * TC_BM, fwd_group_m() ? fwd_group_m() : num_m);
  if (fwd_pair()) {
    CUtensorMap tb2;  // each CTA of the pair stages 128 of the 256 columns
    if (!make_tmap_bf16(&tb2, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN / 2))
      return cudaErrorInvalidValue;
    if (a.task_ctr && fwd_dynamic(nkb)) {
      static_assert(TILES_PER_SPLIT == 1, "a task is one split: the epilogue ends it with the tile's column");
      PairJob j, none;
      j.sc = sc;
      j.b_off_n = j.b_off_k = 0;
      j.a_mn = j.b_mn = 0;
      none = j;
      none.sc.num_tasks = 0;
      return launch_dual<EpiFwdLse>(ta, tb2, ta, tb2, j, none, ep, ep, a.task_ctr, false, a.status, st);
    }
    if (fwd_epi_groups(nkb) == 2) return launch_tc_pair<false, false, EpiFwdLse, 2>(ta, tb2, sc, 0, 0, ep, a.status, st);
    return launch_tc_pair<false, false, EpiFwdLse>(ta, tb2, sc, 0, 0, ep, a.status, st);
  }
  return launch_tc<2, 1, false, false, EpiFwdLse>(ta, tb, sc, 0, 0, ep, a.status, st);
}

cudaError_t launch_dlogits_tc(const TcDlogitsArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN)) return cudaErrorInvalidValue;
  EpiDlogits::Params ep;
  ep.N = a.N;
  ep.V = a.V;
  ep.vb0 = a.vb0;
  ep.ldg = a.ldg;
  ep.lse = a.lse;
  ep.coef = a.coef;
  ep.grad_out = a.grad_out;
  ep.targets = a.targets;
  ep.col_offset = a.col_offset;
  ep.G = static_cast<__nv_bfloat16*>(a.G);
  ep.zero_word = a.zero_word;
  const int nkb = static_cast<int>(ceil_div(a.D, TC_BK));
  const int nn = static_cast<int>(ceil_div(a.width, TC_BN));
  if (dlogits_mt() == 1) {
    TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, TC_BM)), nn, 1, nkb, TC_BM, dlogits_group_m());
    return launch_tc<1, 1, false, false, EpiDlogits>(ta, tb, sc, a.vb0, 0, ep, a.status, st);
  }
  TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, 2 * TC_BM)), nn, 1, nkb, 2 * TC_BM, dlogits_group_m());
  if (dlogits_pair()) {
    CUtensorMap tb2;
    if (!make_tmap_bf16(&tb2, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN / 2))
      return cudaErrorInvalidValue;
    return launch_tc_pair<false, false, EpiDlogits>(ta, tb2, sc, a.vb0, 0, ep, a.status, st);
  }
  if (dlogits_cg() == 2) return launch_tc<2, 2, false, false, EpiDlogits>(ta, tb, sc, a.vb0, 0, ep, a.status, st);
  return launch_tc<2, 1, false, false, EpiDlogits>(ta, tb, sc, a.vb0, 0, ep, a.status, st);
}

cudaError_t launch_dh_tc(const TcDhArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = G [N, ldg] K-major (K = vocabulary column); B = W [V, D] MN-major (N = D, K = vocabulary row)
  if (!make_tmap_bf16(&ta, a.G, a.ldg, a.N, static_cast<uint64_t>(a.ldg) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  EpiStore::Params ep;
  ep.M_valid = a.N;
  ep.N_valid = a.D;
  ep.row_off = 0;
  ep.ld = a.D;
  ep.mode = a.mode;
  ep.out32 = a.acc32;
  ep.out16 = static_cast<__nv_bfloat16*>(a.out16);
  const int nkb = static_cast<int>(ceil_div(a.width, TC_BK));
  const int nn = static_cast<int>(ceil_div(a.D, TC_BN));
  if (dh_pair()) {
    TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, 2 * TC_BM)), nn, 1, nkb, 2 * TC_BM, dh_group_m());
    return launch_tc_pair<false, true, EpiStore>(ta, tb, sc, 0, a.vb0, ep, a.status, st);
  }
  if (dh_mt() == 1) {
    TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, TC_BM)), nn, 1, nkb, TC_BM, dh_group_m());
    return launch_tc<1, 1, false, true, EpiStore>(ta, tb, sc, 0, a.vb0, ep, a.status, st);
  }
  TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, 2 * TC_BM)), nn, 1, nkb, 2 * TC_BM, dh_group_m());
  if (dh_cg() == 2) return launch_tc<2, 2, false, true, EpiStore>(ta, tb, sc, 0, a.vb0, ep, a.status, st);
  return launch_tc<2, 1, false, true, EpiStore>(ta, tb, sc, 0, a.vb0, ep, a.status, st);
}

cudaError_t launch_dw_tc(const TcDwArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = G^T: G [N, ldg] read MN-major (M = vocabulary column, K = token row);
  // B = H [N, D] MN-major (N = D, K = token row)
  if (!make_tmap_bf16(&ta, a.G, a.ldg, a.N, static_cast<uint64_t>(a.ldg) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  const int rows = a.V - a.vb0 < a.width ? a.V - a.vb0 : a.width;
  EpiStore::Params ep;
  ep.M_valid = rows;
  ep.N_valid = a.D;
  ep.row_off = a.vb0;
  ep.ld = a.D;
  ep.mode = a.accumulate ? 1 : 0;
  ep.out32 = a.dW;
  ep.out16 = nullptr;
  const int nkb = static_cast<int>(ceil_div(a.N, TC_BK));
  const int nn = static_cast<int>(ceil_div(a.D, TC_BN));
  if (dw_pair()) {
    TcSched sc = make_sched(static_cast<int>(ceil_div(rows, 2 * TC_BM)), nn, 1, nkb, 2 * TC_BM, dw_group_m());
    return launch_tc_pair<true, true, EpiStore>(ta, tb, sc, 0, 0, ep, a.status, st);
  }
  if (dw_mt() == 1) {
    TcSched sc = make_sched(static_cast<int>(ceil_div(rows, TC_BM)), nn, 1, nkb, TC_BM, dw_group_m());
    return launch_tc<1, 1, true, true, EpiStore>(ta, tb, sc, 0, 0, ep, a.status, st);
  }
  TcSched sc = make_sched(static_cast<int>(ceil_div(rows, 2 * TC_BM)), nn, 1, nkb, 2 * TC_BM, dw_group_m());
  if (dw_cg() == 2) return launch_tc<2, 2, true, true, EpiStore>(ta, tb, sc, 0, 0, ep, a.status, st);
  return launch_tc<2, 1, true, true, EpiStore>(ta, tb, sc, 0, 0, ep, a.status, st);
}

bool dhdw_fused() { return bwd_fused_knob() == 1 && dh_pair() == 1 && dw_pair() == 1; }

cudaError_t launch_dhdw_tc(const TcDhArgs& h, const TcDwArgs& w, int* task_ctr, bool ctr_zeroed, cudaStream_t st) {
  // dH: A = G [N, ldg] K-major, B = W [V, D] MN-major (rows vb0.. of the block)
  CUtensorMap ta_h, tb_h, ta_w, tb_w;
  if (!make_tmap_bf16(&ta_h, h.G, h.ldg, h.N, static_cast<uint64_t>(h.ldg) * 2, TC_BK, TC_BM))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb_h, h.W, h.D, h.V, static_cast<uint64_t>(h.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  // dW: A = G^T (G read MN-major), B = H [N, D] MN-major
  if (!make_tmap_bf16(&ta_w, w.G, w.ldg, w.N, static_cast<uint64_t>(w.ldg) * 2, 64, TC_BK))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb_w, w.H, w.D, w.N, static_cast<uint64_t>(w.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  EpiStore::Params eh;
  eh.M_valid = h.N;
  eh.N_valid = h.D;
  eh.row_off = 0;
  eh.ld = h.D;
  eh.mode = h.mode;
  eh.out32 = h.acc32;
  eh.out16 = static_cast<__nv_bfloat16*>(h.out16);
  const int rows = w.V - w.vb0 < w.width ? w.V - w.vb0 : w.width;
  EpiStore::Params ew;
  ew.M_valid = rows;
  ew.N_valid = w.D;
  ew.row_off = w.vb0;
  ew.ld = w.D;
  ew.mode = w.accumulate ? 1 : 0;
  ew.out32 = w.dW;
  ew.out16 = nullptr;
  PairJob jh, jw;
  jh.sc = make_sched(static_cast<int>(ceil_div(h.N, 2 * TC_BM)), static_cast<int>(ceil_div(h.D, TC_BN)), 1,
                     static_cast<int>(ceil_div(h.width, TC_BK)), 2 * TC_BM, dh_group_m());
  jh.b_off_n = 0;
  jh.b_off_k = h.vb0;
  jh.a_mn = 0;
  jh.b_mn = 1;
  jw.sc = make_sched(static_cast<int>(ceil_div(rows, 2 * TC_BM)), static_cast<int>(ceil_div(w.D, TC_BN)), 1,
                     static_cast<int>(ceil_div(w.N, TC_BK)), 2 * TC_BM, dw_group_m());
  jw.b_off_n = 0;
  jw.b_off_k = 0;
  jw.a_mn = 1;
  jw.b_mn = 1;
  // the product with the deeper K (longer tiles) first: the short tiles of
  // the other fill the end of the list
  if (jw.sc.num_kb > jh.sc.num_kb)
    return launch_dual<EpiStore>(ta_w, tb_w, ta_h, tb_h, jw, jh, ew, eh, task_ctr, ctr_zeroed, h.status, st);
  return launch_dual<EpiStore>(ta_h, tb_h, ta_w, tb_w, jh, jw, eh, ew, task_ctr, ctr_zeroed, h.status, st);
}

}  // namespace gh
