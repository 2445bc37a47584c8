// Two GEMMs in one launch on CTA pairs (the dH and dW products of a backward
// vocabulary block), with 256 x 256 tiles handed out dynamically.  The
// long-K forward runs here too, as one job with an empty second one.
//
// The pair kernel of tc_gemm_pair.cuh deals tiles round-robin, so a launch of
// 512 dH tiles over 76 pairs runs 6.74 waves and idles a quarter of the GPU
// in its last one; dW does the same.  Here both products share one launch and
// one task list (the job with the deeper K first, then the other), and each
// pair takes its next tile from a global counter, so the pairs finish within
// about one tile of each other.  A tile is still computed whole by one pair,
// in the same K order, so the results do not depend on which pair takes which
// tile.
//
// Task hand-off inside a pair: the even CTA's producer thread draws the task
// index (atomicAdd on *task_ctr, zeroed before the launch) while
// the last 16 K blocks of its current tile are still to be loaded, and
// publishes it in a ring of DUAL_RING slots in both CTAs' shared memory (a
// remote st.shared::cluster plus a release arrive on the peer's slot barrier).
// The slot's consumers -- the even CTA's MMA thread and epilogue warps, the odd
// CTA's producer and epilogue warps -- read it after an acquire wait and free
// it with an arrive on the even CTA's slot-empty barrier.  An index past the
// end of the list tells every role of the pair to stop.
//
// Roles, pipeline, TMEM use and the bounded waits are those of
// tc_gemm_pair_kernel; the tensor maps, K depth and epilogue parameters are
// chosen per task from its job, and each tile's load and MMA loops are
// instantiated for the job's operand majors (with the majors as run-time
// values the same loops ran about 12% slower).
#pragma once
#include "tc_gemm_pair.cuh"

namespace gh {

struct PairJob {
  TcSched sc;  // tiles of this product (n_per_task = 1, m_step = 256)
  int b_off_n, b_off_k;
  int a_mn, b_mn;  // operand majors (1 = MN-major)
};

constexpr int DUAL_RING = 8;
constexpr int DUAL_SMEM_BYTES = TcPairCfg::STAGES * TcPairCfg::STAGE_BYTES + 1024 + 512;

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded with cluster-scope acquire (the barrier is arrived on, and
// the data it guards written, by the other CTA of the pair)
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                          int* status, uint64_t timeout_ns) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if ((++it & 63u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        if (status) atomicOr(status, GH_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// a job's fields in registers: selecting a reference to one of two kernel
// parameters would make every later use a load through a generic address
__device__ __forceinline__ PairJob job_copy(bool second, const PairJob& j0, const PairJob& j1) {
  PairJob J;
  J.sc.num_m_blocks = second ? j1.sc.num_m_blocks : j0.sc.num_m_blocks;
  J.sc.num_n_blocks = second ? j1.sc.num_n_blocks : j0.sc.num_n_blocks;
  J.sc.n_per_task = second ? j1.sc.n_per_task : j0.sc.n_per_task;
  J.sc.num_kb = second ? j1.sc.num_kb : j0.sc.num_kb;
  J.sc.m_step = second ? j1.sc.m_step : j0.sc.m_step;
  J.sc.group_m = second ? j1.sc.group_m : j0.sc.group_m;
  J.sc.num_ng = second ? j1.sc.num_ng : j0.sc.num_ng;
  J.sc.num_tasks = second ? j1.sc.num_tasks : j0.sc.num_tasks;
  J.b_off_n = second ? j1.b_off_n : j0.b_off_n;
  J.b_off_k = second ? j1.b_off_k : j0.b_off_k;
  J.a_mn = second ? j1.a_mn : j0.a_mn;
  J.b_mn = second ? j1.b_mn : j0.b_mn;
  return J;
}

// One tile's loads (producer thread) and MMAs (even CTA's issuer) with the
// operand majors as compile-time constants, as in tc_gemm_pair_kernel.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ bool dual_load_tile(uint8_t* smem, uint64_t* full, uint64_t* empty, int& stage,
                                               uint32_t& phase, uint32_t rank, const CUtensorMap* mA,
                                               const CUtensorMap* mB, int m0, int n0, int b_off_k, int num_kb,
                                               int draw_kb, int* task_ctr, int& next, bool& have_next,
                                               volatile int* abort_flag, int* status, uint64_t timeout_ns) {
  using C = TcPairCfg;
  for (int kb = 0; kb < num_kb; ++kb) {
    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) return false;
    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
    const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
    uint8_t* sA = smem + stage * C::STAGE_BYTES;
    uint8_t* sB = sA + C::A_BYTES;
    const int k0 = kb * TC_BK;
    if (!A_MN) {
      tma_load_2d_pair(sA, mA, bar, k0, m0);
    } else {
      tma_load_2d_pair(sA, mA, bar, m0, k0);
      tma_load_2d_pair(sA + 8192, mA, bar, m0 + 64, k0);
    }
    if (!B_MN) {
      tma_load_2d_pair(sB, mB, bar, k0 + b_off_k, n0);
    } else {
      tma_load_2d_pair(sB, mB, bar, n0, k0 + b_off_k);
      tma_load_2d_pair(sB + 8192, mB, bar, n0 + 64, k0 + b_off_k);
    }
    if (kb == draw_kb) {
      next = atomicAdd(task_ctr, 1);
      have_next = true;
    }
    if (++stage == C::STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ bool dual_mma_tile(uint8_t* smem, uint64_t* full, uint64_t* empty, int& stage,
                                              uint32_t& phase, uint32_t d_tmem, int num_kb, volatile int* abort_flag,
                                              int* status, uint64_t timeout_ns) {
  using C = TcPairCfg;
  constexpr uint32_t IDESC = idesc_bf16_f32(2 * TC_BM, TC_BN, A_MN, B_MN);
  for (int kb = 0; kb < num_kb; ++kb) {
    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) return false;
    tc_fence_after();
    const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
    const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
    for (int kk = 0; kk < TC_BK / 16; ++kk) {
      const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024) : sdesc_sw128(a_base + kk * 32, 16, 1024);
      const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024) : sdesc_sw128(b_base + kk * 32, 16, 1024);
      umma_pair_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
    }
    umma_pair_commit_mc(&empty[stage], 0x3);
    if (++stage == C::STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

template <class Epi>
__global__ void __launch_bounds__(TcPairCfg::THREADS, 1)
    tc_dual_pair_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                        const PairJob j0, const PairJob j1, const typename Epi::Params ep0,
                        const typename Epi::Params ep1, int* task_ctr, int* status,
                        const uint64_t timeout_ns) {
  using C = TcPairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* rfull = drain + 1;           // [DUAL_RING] task slot written (both CTAs)
  uint64_t* rempty = rfull + DUAL_RING;  // [DUAL_RING] task slot read by all consumers (even CTA's are used)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rempty + DUAL_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ring = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [DUAL_RING]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int T0 = j0.sc.num_tasks;
  const int T = T0 + j1.sc.num_tasks;
  // consumers of a slot: even CTA's MMA thread + epilogue warps, odd CTA's producer + epilogue warps
  constexpr uint32_t SLOT_CONSUMERS = 2 * (1 + C::EPI_WARPS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int r = 0; r < DUAL_RING; ++r) {
      mbar_init(&rfull[r], 1);
      mbar_init(&rempty[r], SLOT_CONSUMERS);
      ring[r] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TC_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ task source + TMA producer (both CTAs)
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      int next = 0;
      bool have_next = false;
      while (ok) {
        const int slot = it % DUAL_RING;
        const uint32_t rph = static_cast<uint32_t>(it / DUAL_RING) & 1u;
        int t;
        if (rank == 0) {
          if (!mbar_wait_cluster_bounded(&rempty[slot], rph ^ 1u, abort_flag, status, timeout_ns)) break;
          if (!have_next) next = atomicAdd(task_ctr, 1);
          have_next = false;
          t = (next >= 0 && next < T) ? next : T;  // past the end (or a counter never zeroed): stop
          ring[slot] = t;
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&ring[slot])), 1), static_cast<uint32_t>(t));
          mbar_arrive(&rfull[slot]);
          mbar_arrive_cluster(mapa_shared(smem_u32(&rfull[slot]), 1));
        } else {
          if (!mbar_wait_cluster_bounded(&rfull[slot], rph, abort_flag, status, timeout_ns)) break;
          t = ring[slot];
          mbar_arrive_cluster(mapa_shared(smem_u32(&rempty[slot]), 0));
        }
        ++it;
        if (t >= T) break;
        const bool second = t >= T0;
        const PairJob J = job_copy(second, j0, j1);
        const CUtensorMap* mA = second ? &tmA1 : &tmA0;
        const CUtensorMap* mB = second ? &tmB1 : &tmB0;
        int m_blk, n_blk;
        tc_task_of(J.sc, second ? t - T0 : t, m_blk, n_blk);
        const int m0 = m_blk * J.sc.m_step + static_cast<int>(rank) * TC_BM;
        const int n0 = n_blk * TC_BN + static_cast<int>(rank) * (TC_BN / 2) + J.b_off_n;
        const int num_kb = J.sc.num_kb, b_off_k = J.b_off_k;
        const bool a_mn = J.a_mn != 0, b_mn = J.b_mn != 0;
        // the even CTA draws the next task while the last 16 K blocks of this
        // one are still to be loaded: the atomic's latency (the L2 is busy with
        // tile traffic) hides behind them
        const int draw_kb = rank == 0 ? (num_kb > 16 ? num_kb - 16 : 0) : -1;
        issued = true;
        if (a_mn)
          ok = b_mn ? dual_load_tile<true, true>(smem, full, empty, stage, phase, rank, mA, mB, m0, n0, b_off_k, num_kb,
                                                 draw_kb, task_ctr, next, have_next, abort_flag, status, timeout_ns)
                    : dual_load_tile<true, false>(smem, full, empty, stage, phase, rank, mA, mB, m0, n0, b_off_k,
                                                  num_kb, draw_kb, task_ctr, next, have_next, abort_flag, status,
                                                  timeout_ns);
        else
          ok = b_mn ? dual_load_tile<false, true>(smem, full, empty, stage, phase, rank, mA, mB, m0, n0, b_off_k,
                                                  num_kb, draw_kb, task_ctr, next, have_next, abort_flag, status,
                                                  timeout_ns)
                    : dual_load_tile<false, false>(smem, full, empty, stage, phase, rank, mA, mB, m0, n0, b_off_k,
                                                   num_kb, draw_kb, task_ctr, next, have_next, abort_flag, status,
                                                   timeout_ns);
      }
      if (*abort_flag && issued) {
        // completions land on the even CTA's barriers, which the odd CTA cannot
        // poll: give copies in flight a fixed, bounded time to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ pair MMA issuer (even CTA)
      int stage = 0, acc = 0, it = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      while (ok) {
        const int slot = it % DUAL_RING;
        const uint32_t rph = static_cast<uint32_t>(it / DUAL_RING) & 1u;
        if (!mbar_wait_cluster_bounded(&rfull[slot], rph, abort_flag, status, timeout_ns)) break;
        const int t = ring[slot];
        mbar_arrive(&rempty[slot]);
        ++it;
        if (t >= T) break;
        const PairJob J = job_copy(t >= T0, j0, j1);
        const bool a_mn = J.a_mn != 0, b_mn = J.b_mn != 0;
        const int num_kb = J.sc.num_kb;
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * TC_BN);
        issued = true;
        if (a_mn)
          ok = b_mn ? dual_mma_tile<true, true>(smem, full, empty, stage, phase, d_tmem, num_kb, abort_flag, status,
                                                timeout_ns)
                    : dual_mma_tile<true, false>(smem, full, empty, stage, phase, d_tmem, num_kb, abort_flag, status,
                                                 timeout_ns);
        else
          ok = b_mn ? dual_mma_tile<false, true>(smem, full, empty, stage, phase, d_tmem, num_kb, abort_flag, status,
                                                 timeout_ns)
                    : dual_mma_tile<false, false>(smem, full, empty, stage, phase, d_tmem, num_kb, abort_flag,
                                                  status, timeout_ns);
        if (!ok) break;
        umma_pair_commit_mc(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (issued) {
        // every pair MMA issued must be complete before TMEM is freed
        umma_pair_commit_mc(drain, 0x1);
        volatile int no_abort = 0;
        mbar_wait_bounded(drain, 0, &no_abort, nullptr, 0, timeout_ns);
      }
    }
  } else {
    // -------------------------------------------------- epilogue warps (both CTAs)
    const int sub = warp & 3;
    const int row = static_cast<int>(rank) * TC_BM + sub * 32 + lane;  // row within the 256-row tile
    const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
    int acc = 0, it = 0;
    uint32_t acc_phase = 0;
    Epi epi;
    while (true) {
      const int slot = it % DUAL_RING;
      const uint32_t rph = static_cast<uint32_t>(it / DUAL_RING) & 1u;
      const bool got = mbar_wait_cluster_bounded(&rfull[slot], rph, abort_flag, status, timeout_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&rempty[slot]);
        else
          mbar_arrive_cluster(mapa_shared(smem_u32(&rempty[slot]), 0));
      }
      ++it;
      if (t >= T) break;
      const bool second = t >= T0;
      const PairJob J = job_copy(second, j0, j1);
      typename Epi::Params ep;
      if (second)
        ep = ep1;
      else
        ep = ep0;
      int m_blk, n_blk;
      tc_task_of(J.sc, second ? t - T0 : t, m_blk, n_blk);
      if (!warp_wait(&tfull[acc], acc_phase, abort_flag, status, timeout_ns)) break;
      tc_fence_after();
      epi.begin_task(ep, J.sc, m_blk, row);
      epi.tile(ep, J.sc, tmem_base + lane_addr + static_cast<uint32_t>(acc * TC_BN), m_blk, n_blk, row, 0,
               TC_BN / 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      epi.end_task(ep, J.sc, m_blk, n_blk, row);
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal or read it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TC_TMEM_COLS);
}

}  // namespace gh
