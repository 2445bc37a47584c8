// CTA-pair variant of the tcgen05 GEMM core: a cluster of two CTAs on two
// SMs computes one 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256).
//
// Each CTA stages only its own 128 rows of A and its half (128 columns) of B
// per pipeline stage (32 KB), so the pair moves as few bytes from L2 per FLOP
// as a 256 x 256 tile on one SM, while each CTA keeps a double-buffered
// 128 x 256 accumulator in its own TMEM (the epilogue of tile i overlaps the
// MMAs of tile i+1).
//
//   both CTAs: warp 0 TMA producer (its A rows and B half; completion is
//              signalled on the even CTA's stage barrier), warps 2.. epilogue
//              (its 128 rows; frees the accumulator on the even CTA's barrier):
//              EG groups of four warps, group g taking every EG-th tile of the
//              pair in accumulator g (EG = 2 runs two tiles' epilogues at once
//              when one epilogue outlasts a tile's MMAs; every row's arithmetic
//              is the same either way)
//   even CTA : warp 1 issues the pair MMAs and commits them to both CTAs'
//              stage-free and accumulator-full barriers (multicast)
//   both CTAs: warp 1 allocates / frees TMEM collectively (cta_group::2)
//
// Waits are bounded as in tc_gemm_kernel; the cluster barriers at start and end
// are reached by every thread of both CTAs on every path.
#pragma once
#include "tc_gemm.cuh"

namespace gh {

struct TcPairCfg {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;        // 16 KB: this CTA's 128 rows
  static constexpr int B_BYTES = (TC_BN / 2) * TC_BK * 2;  // 16 KB: this CTA's 128 columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 7;  // 224 KB: the deepest pipeline that fits
  static constexpr int EPI_WARPS = 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
};

// threads of a pair kernel CTA with EG epilogue groups
constexpr int tc_pair_threads(int EG) { return 64 + 32 * TcPairCfg::EPI_WARPS * EG; }

template <bool A_MN, bool B_MN, class Epi, int EG = 1>
__global__ void __launch_bounds__(tc_pair_threads(EG), 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const TcSched sc, const int b_off_n, const int b_off_k, const typename Epi::Params ep,
                        int* status, const uint64_t timeout_ns) {
  using C = TcPairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: its peer
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  if (blockIdx.x == 0 && threadIdx.x == 0) Epi::on_entry(ep);  // before any wait that may abort
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
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
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
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      for (int task = cid; ok && task < sc.num_tasks; task += ncl) {
        int m_blk, ng;
        tc_task_of(sc, task, m_blk, ng);
        for (int nn = 0; ok && nn < sc.n_per_task; ++nn) {
          const int n_blk = ng * sc.n_per_task + nn;
          if (n_blk >= sc.num_n_blocks) break;
          const int m0 = m_blk * sc.m_step + static_cast<int>(rank) * TC_BM;
          const int n0 = n_blk * TC_BN + static_cast<int>(rank) * (TC_BN / 2) + b_off_n;
          for (int kb = 0; kb < sc.num_kb; ++kb) {
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) {
              ok = false;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
            const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
            uint8_t* sA = smem + stage * C::STAGE_BYTES;
            uint8_t* sB = sA + C::A_BYTES;
            const int k0 = kb * TC_BK;
            if (!A_MN) {
              tma_load_2d_pair(sA, &tmA, bar, k0, m0);
            } else {
              tma_load_2d_pair(sA, &tmA, bar, m0, k0);
              tma_load_2d_pair(sA + 8192, &tmA, bar, m0 + 64, k0);
            }
            if (!B_MN) {
              tma_load_2d_pair(sB, &tmB, bar, k0 + b_off_k, n0);
            } else {
              tma_load_2d_pair(sB, &tmB, bar, n0, k0 + b_off_k);
              tma_load_2d_pair(sB + 8192, &tmB, bar, n0 + 64, k0 + b_off_k);
            }
            issued = true;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && issued) {
        // completions land on the even CTA's barriers, which this CTA cannot
        // poll: give copies in flight a fixed, bounded time to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ pair MMA issuer (even CTA)
      constexpr uint32_t IDESC = idesc_bf16_f32(2 * TC_BM, TC_BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int task = cid; ok && task < sc.num_tasks; task += ncl) {
        int m_blk, ng;
        tc_task_of(sc, task, m_blk, ng);
        for (int nn = 0; ok && nn < sc.n_per_task; ++nn) {
          if (ng * sc.n_per_task + nn >= sc.num_n_blocks) break;
          if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * TC_BN);
          for (int kb = 0; kb < sc.num_kb; ++kb) {
            if (!mbar_wait_bounded(&full[stage], phase, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
            const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk) {
              const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                       : sdesc_sw128(a_base + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                       : sdesc_sw128(b_base + kk * 32, 16, 1024);
              umma_pair_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
            }
            issued = true;
            umma_pair_commit_mc(&empty[stage], 0x3);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_pair_commit_mc(&tfull[acc], 0x3);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
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
    // TMEM lane quadrant = warp id mod 4; group grp takes this pair's tasks
    // j = grp, grp + EG, ... (one tile each when EG > 1) in accumulator grp
    static_assert(EG == 1 || EG == 2, "one or two epilogue groups");
    const int sub = warp & 3;
    const int grp = EG == 1 ? 0 : (warp - 2) / TcPairCfg::EPI_WARPS;
    const int row = static_cast<int>(rank) * TC_BM + sub * 32 + lane;  // row within the 256-row tile
    const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
    int acc = grp;
    uint32_t acc_phase = 0;
    bool ok = true;
    Epi epi;
    int j = 0;
    for (int task = cid; ok && task < sc.num_tasks; task += ncl, ++j) {
      if (EG > 1 && j % EG != grp) continue;
      int m_blk, ng;
      tc_task_of(sc, task, m_blk, ng);
      epi.begin_task(ep, sc, m_blk, row);
      for (int nn = 0; ok && nn < sc.n_per_task; ++nn) {
        const int n_blk = ng * sc.n_per_task + nn;
        if (n_blk >= sc.num_n_blocks) break;
        if (!warp_wait(&tfull[acc], acc_phase, abort_flag, status, timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        epi.tile(ep, sc, tmem_base + lane_addr + static_cast<uint32_t>(acc * TC_BN), m_blk, n_blk, row, 0,
                 TC_BN / 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&tempty[acc]);
          else
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
        if (EG == 1) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;  // this group's accumulator, next use
        }
      }
      if (ok) epi.end_task(ep, sc, m_blk, ng, row);
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal or read it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TC_TMEM_COLS);
}

}  // namespace gh
