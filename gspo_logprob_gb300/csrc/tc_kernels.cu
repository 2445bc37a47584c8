// tcgen05 kernels of the bf16 path: logits + online LSE (forward), dlogits
// recompute (backward) and the dH / dW GEMMs, all instances of tc_gemm_kernel.
#include "internal.h"
#include "tc_gemm.cuh"

namespace gh {

namespace {

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const TcSched& sc, int b_off_n, int b_off_k,
                      const typename Epi::Params& ep, int* status, cudaStream_t st) {
  auto kern = tc_gemm_kernel<A_MN, B_MN, Epi>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (sc.num_tasks <= 0) return cudaSuccess;
  const int grid = static_cast<int>(sc.num_tasks < num_sms() ? sc.num_tasks : num_sms());
  kern<<<grid, TC_THREADS, TC_SMEM_BYTES, st>>>(ta, tb, sc, b_off_n, b_off_k, ep, status, timeout_ns());
  return cudaGetLastError();
}

TcSched make_sched(int num_m_blocks, int num_n_blocks, int m_per_task, int n_per_task, int num_kb, int m_step) {
  TcSched sc;
  sc.num_m_blocks = num_m_blocks;
  sc.num_n_blocks = num_n_blocks;
  sc.m_per_task = m_per_task;
  sc.n_per_task = n_per_task;
  sc.num_kb = num_kb;
  sc.m_step = m_step;
  sc.num_mg = static_cast<int>(ceil_div(num_m_blocks, m_per_task));
  sc.num_tasks = sc.num_mg * static_cast<int>(ceil_div(num_n_blocks, n_per_task));
  return sc;
}

}  // namespace

cudaError_t launch_fwd_tc(const TcFwdArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = H [N, D] K-major, B = W [V, D] K-major
  if (!make_tmap_bf16(&ta, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN)) return cudaErrorInvalidValue;
  const int m_step = a.row_tile == 64 ? 64 : 128;
  const int m_per_task = a.row_tile == 256 ? 2 : 1;
  const int num_m = static_cast<int>(ceil_div(a.N, m_step));
  const int num_vt = static_cast<int>(ceil_div(a.V, VTILE));
  TcSched sc = make_sched(num_m, num_vt, m_per_task, TILES_PER_SPLIT, static_cast<int>(ceil_div(a.D, TC_BK)), m_step);
  EpiFwdLse::Params ep;
  ep.N = a.N;
  ep.V = a.V;
  ep.part_m = a.part_m;
  ep.part_s = a.part_s;
  ep.zy = a.zy;
  ep.targets = a.targets;
  return launch_tc<false, false, EpiFwdLse>(ta, tb, sc, 0, 0, ep, a.status, st);
}

cudaError_t launch_dlogits_tc(const TcDlogitsArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, TC_BK, TC_BN)) return cudaErrorInvalidValue;
  TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, TC_BM)), static_cast<int>(ceil_div(a.width, TC_BN)), 1, 1,
                          static_cast<int>(ceil_div(a.D, TC_BK)), TC_BM);
  EpiDlogits::Params ep;
  ep.N = a.N;
  ep.V = a.V;
  ep.vb0 = a.vb0;
  ep.ldg = a.ldg;
  ep.lse = a.lse;
  ep.coef = a.coef;
  ep.grad_out = a.grad_out;
  ep.targets = a.targets;
  ep.G = static_cast<__nv_bfloat16*>(a.G);
  return launch_tc<false, false, EpiDlogits>(ta, tb, sc, a.vb0, 0, ep, a.status, st);
}

cudaError_t launch_dh_tc(const TcDhArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = G [N, ldg] K-major (K = vocabulary column); B = W [V, D] MN-major (N = D, K = vocabulary row)
  if (!make_tmap_bf16(&ta, a.G, a.ldg, a.N, static_cast<uint64_t>(a.ldg) * 2, TC_BK, TC_BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, a.D, a.V, static_cast<uint64_t>(a.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  TcSched sc = make_sched(static_cast<int>(ceil_div(a.N, TC_BM)), static_cast<int>(ceil_div(a.D, TC_BN)), 1, 1,
                          static_cast<int>(ceil_div(a.width, TC_BK)), TC_BM);
  EpiStore::Params ep;
  ep.M_valid = a.N;
  ep.N_valid = a.D;
  ep.row_off = 0;
  ep.ld = a.D;
  ep.mode = a.mode;
  ep.out32 = a.acc32;
  ep.out16 = static_cast<__nv_bfloat16*>(a.out16);
  return launch_tc<false, true, EpiStore>(ta, tb, sc, 0, a.vb0, ep, a.status, st);
}

cudaError_t launch_dw_tc(const TcDwArgs& a, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = G^T: G [N, ldg] read MN-major (M = vocabulary column, K = token row);
  // B = H [N, D] MN-major (N = D, K = token row)
  if (!make_tmap_bf16(&ta, a.G, a.ldg, a.N, static_cast<uint64_t>(a.ldg) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.H, a.D, a.N, static_cast<uint64_t>(a.D) * 2, 64, TC_BK)) return cudaErrorInvalidValue;
  const int rows = a.V - a.vb0 < a.width ? a.V - a.vb0 : a.width;
  TcSched sc = make_sched(static_cast<int>(ceil_div(rows, TC_BM)), static_cast<int>(ceil_div(a.D, TC_BN)), 1, 1,
                          static_cast<int>(ceil_div(a.N, TC_BK)), TC_BM);
  EpiStore::Params ep;
  ep.M_valid = rows;
  ep.N_valid = a.D;
  ep.row_off = a.vb0;
  ep.ld = a.D;
  ep.mode = a.accumulate ? 1 : 0;
  ep.out32 = a.dW;
  ep.out16 = nullptr;
  return launch_tc<true, true, EpiStore>(ta, tb, sc, 0, 0, ep, a.status, st);
}

}  // namespace gh
