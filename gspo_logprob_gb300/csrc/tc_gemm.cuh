// Persistent, warp-specialised tcgen05 GEMM core with pluggable epilogues.
//
//   warp 0      : TMA producer (one thread) -- stages bf16 A/B tiles in shared memory
//   warp 1      : TMEM allocator + MMA issuer (one thread) -- tcgen05.mma M=128 N=256 K=16
//   warps 2..    : epilogue (4 warps per 128-row block; thread t owns TMEM lane /
//                  tile row t of its block)
//
// A CTA tile is MT x 128 rows by 256 columns.  With MT = 1 the accumulator is
// double-buffered in TMEM (2 x 256 fp32 columns) so the epilogue of tile i
// overlaps the MMAs of tile i+1; with MT = 2 both 128-row blocks multiply the
// same staged B tile (one B fill per 256 x 256 tile) into the two halves of
// TMEM.  Work is a list of tasks; a task is one row tile and n_per_task
// consecutive column blocks handed to one CTA in order, so an epilogue can
// carry state across the tiles of a task (the online log-sum-exp of a
// vocabulary split).  Tasks are rastered in groups of group_m row tiles
// (row fastest) for L2 reuse and dealt round-robin to gridDim.x persistent CTAs.
//
// Operand layouts (bf16, 128-byte swizzle, tiles 1024-byte aligned):
//   K-major A: TMA box {64 (K), 128 rows}; rows at 128 B, 8-row groups at 1024 B.
//   K-major B: TMA box {64 (K), 256 rows}.
//   MN-major A/B: boxes {64 (MN), 64 (K)} of 8 KB placed side by side along MN;
//   the descriptor's leading offset is the 8 KB MN-atom stride, the stride offset
//   the 1024 B step between 8-row K groups.
// Every pipeline wait is bounded (GH_DEV_TIMEOUT on expiry); on a timeout each
// role leaves its loop, in-flight copies and MMAs are waited for (bounded),
// and TMEM is freed before the CTA exits.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "grpo_head.h"
#include "ptx.cuh"

namespace gh {

constexpr int TC_BM = 128;   // rows per tcgen05.mma (TMEM lanes)
constexpr int TC_BN = 256;   // columns per tile
constexpr int TC_BK = 64;    // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB per 128-row A block
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;

// MT = 128-row MMA blocks per CTA tile (1: 128 x 256 tiles, double-buffered
// accumulator; 2: 256 x 256 tiles whose two row blocks share every staged B
// tile -- a third less shared-memory fill traffic per FLOP -- with a single
// 2 x 256-column accumulator and twice the epilogue warps).
// CG = epilogue warps per TMEM row (each takes 256 / CG of the tile's columns;
// more warps drain a single-buffered accumulator sooner).
template <int MT, int CG = 1>
struct TcCfg {
  static constexpr int STAGE_BYTES = MT * TC_A_BYTES + TC_B_BYTES;
  static constexpr int STAGES = MT == 1 ? 4 : 3;
  static constexpr int NUM_ACC = MT == 1 ? 2 : 1;
  static constexpr int EPI_WARPS = 4 * MT * CG;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
};

struct TcSched {
  int num_m_blocks;  // CTA row tiles (MT*128 rows loaded, m_step rows apart)
  int num_n_blocks;  // 256-wide column blocks
  int n_per_task;    // consecutive column blocks per task (the epilogue carries state across them)
  int num_kb;        // 64-deep K blocks
  int m_step;        // rows between consecutive row tiles: 64 (half tiles), 128 or 256
  int group_m;       // raster: tasks cover group_m row tiles (row fastest), then the next columns
  int num_ng;        // ceil(num_n_blocks / n_per_task)
  int num_tasks;     // num_m_blocks * num_ng
};

__device__ __forceinline__ void tc_task_of(const TcSched& sc, int task, int& m_blk, int& ng) {
  const int per_group = sc.group_m * sc.num_ng;
  const int g = task / per_group, r = task % per_group;
  const int gm = min(sc.group_m, sc.num_m_blocks - g * sc.group_m);
  m_blk = g * sc.group_m + r % gm;
  ng = r / gm;
}

// all lanes of the warp agree on the outcome of a bounded wait
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                          uint64_t tmo) {
  bool ok = mbar_wait_bounded(bar, parity, abort, status, GH_DEV_TIMEOUT, tmo);
  return __all_sync(0xffffffffu, ok);
}

template <int MT, int CG, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(TcCfg<MT, CG>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcSched sc, const int b_off_n, const int b_off_k, const typename Epi::Params ep,
                   int* status, const uint64_t timeout_ns) {
  using C = TcCfg<MT, CG>;
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
  if (blockIdx.x == 0 && threadIdx.x == 0) Epi::on_entry(ep);  // before any wait that may abort
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0, pend_par = 0;  // per stage: load issued and its phase parity
      bool ok = true;
      for (int task = blockIdx.x; ok && task < sc.num_tasks; task += gridDim.x) {
        int m_blk, ng;
        tc_task_of(sc, task, m_blk, ng);
        for (int nn = 0; ok && nn < sc.n_per_task; ++nn) {
          const int n_blk = ng * sc.n_per_task + nn;
          if (n_blk >= sc.num_n_blocks) break;
          const int m0 = m_blk * sc.m_step;
          const int n0 = n_blk * TC_BN + b_off_n;
          for (int kb = 0; kb < sc.num_kb; ++kb) {
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status, GH_DEV_TIMEOUT, timeout_ns)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
            uint8_t* sA = smem + stage * C::STAGE_BYTES;
            uint8_t* sB = sA + MT * TC_A_BYTES;
            const int k0 = kb * TC_BK;
#pragma unroll
            for (int q = 0; q < MT; ++q) {
              if (!A_MN) {
                tma_load_2d(sA + q * TC_A_BYTES, &tmA, &full[stage], k0, m0 + q * TC_BM);
              } else {
                tma_load_2d(sA + q * TC_A_BYTES, &tmA, &full[stage], m0 + q * TC_BM, k0);
                tma_load_2d(sA + q * TC_A_BYTES + 8192, &tmA, &full[stage], m0 + q * TC_BM + 64, k0);
              }
            }
            if (!B_MN) {
              tma_load_2d(sB, &tmB, &full[stage], k0 + b_off_k, n0);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) tma_load_2d(sB + q * 8192, &tmB, &full[stage], n0 + 64 * q, k0 + b_off_k);
            }
            pending |= 1u << stage;
            pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // let every copy this thread issued land before shared memory is released
        for (int s = 0; s < C::STAGES; ++s)
          if (pending & (1u << s)) {
            volatile int no_abort = 0;
            mbar_wait_bounded(&full[s], (pend_par >> s) & 1u, &no_abort, nullptr, 0, timeout_ns);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC = idesc_bf16_f32(TC_BM, TC_BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int task = blockIdx.x; ok && task < sc.num_tasks; task += gridDim.x) {
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
            const uint32_t b_base = a_base + MT * TC_A_BYTES;
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk) {
              const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                       : sdesc_sw128(b_base + kk * 32, 16, 1024);
#pragma unroll
              for (int q = 0; q < MT; ++q) {
                const uint32_t aq = a_base + q * TC_A_BYTES;
                const uint64_t ad = A_MN ? sdesc_sw128(aq + kk * 2048, 8192, 1024)
                                         : sdesc_sw128(aq + kk * 32, 16, 1024);
                umma_bf16(d_tmem + static_cast<uint32_t>(q * TC_BN), ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              }
            }
            issued = true;
            umma_commit(&empty[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(&tfull[acc]);
          if (C::NUM_ACC == 2) {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
          } else {
            acc_phase ^= 1u;
          }
        }
      }
      if (issued) {
        // every MMA issued must be complete before TMEM is freed (normally they
        // already are: the epilogue consumed each accumulator)
        umma_commit(drain);
        volatile int no_abort = 0;
        mbar_wait_bounded(drain, 0, &no_abort, nullptr, 0, timeout_ns);
      }
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int ew = warp - 2;
    const int grp = ew >> 2;
    const int q = grp / CG;     // which 128-row block of the tile
    const int cg = grp % CG;    // which share of the columns
    const int c_lo = cg * (TC_BN / 32 / CG), c_hi = c_lo + TC_BN / 32 / CG;
    const int sub = warp & 3;   // TMEM lane quarter this warp may access
    const int row = q * TC_BM + sub * 32 + lane;  // row within the CTA tile
    const uint32_t lane_addr = (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(q * TC_BN);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    Epi epi;
    for (int task = blockIdx.x; ok && task < sc.num_tasks; task += gridDim.x) {
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
        epi.tile(ep, sc, tmem_base + lane_addr + static_cast<uint32_t>(acc * TC_BN), m_blk, n_blk, row, c_lo, c_hi);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (C::NUM_ACC == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      if (ok) epi.end_task(ep, sc, m_blk, ng, row);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TC_TMEM_COLS);
}

// ============================================================================
// Epilogue 1: online fp32 (max, sumexp) over a vocabulary split + target gather.
// One task = (row block(s), split); the split's tiles are visited in increasing
// column order and merged into the running (m, s) of each row: per 32-column
// chunk, M = max(m, chunk max), s = s e^{m-M} + sum e^{z-M}.  Padded columns
// (>= V) are -inf and a chunk of only padding is skipped (identity (-inf, 0)).
// ============================================================================
struct EpiFwdLse {
  struct Params {
    int N, V;
    float* part_m;  // [splits, N]
    float* part_s;  // [splits, N]
    float* zy;      // [N]
    const int* targets;
    int col_offset;  // global vocabulary id of local column 0 (vocabulary shards)
  };
  static __device__ __forceinline__ void on_entry(const Params&) {}
  float m, s;
  int y, grow;
  bool valid;

  __device__ __forceinline__ void begin_task(const Params& p, const TcSched& sc, int m_blk, int row) {
    m = -INFINITY;
    s = 0.f;
    grow = m_blk * sc.m_step + row;
    valid = row < sc.m_step && grow < p.N;
    y = valid ? __ldg(p.targets + grow) - p.col_offset : -1;  // local column of the target
  }

  // needs the whole row (online state across its columns): CG must be 1
  __device__ __forceinline__ void tile(const Params& p, const TcSched&, uint32_t taddr, int, int n_blk, int, int, int) {
    float run_m = m, run_s = s;
    const int yy = y;
#pragma unroll 1
    for (int c = 0; c < TC_BN / 32; ++c) {
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      const int col0 = n_blk * TC_BN + c * 32;
      const int rel = yy - col0;
      if (rel >= 0 && rel < 32) {
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) z = (j == rel) ? v[j] : z;
        p.zy[grow] = z;  // rel in [0, 32) only for valid rows
      }
      if (col0 + 32 > p.V) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (col0 + j < p.V) ? v[j] : -INFINITY;
      }
      float cm0 = fmaxf(v[0], v[1]), cm1 = fmaxf(v[2], v[3]);
#pragma unroll
      for (int j = 4; j < 32; j += 4) {
        cm0 = fmaxf(cm0, fmaxf(v[j], v[j + 1]));
        cm1 = fmaxf(cm1, fmaxf(v[j + 2], v[j + 3]));
      }
      const float cmax = fmaxf(cm0, cm1);
      if (cmax != -INFINITY) {
        const float mnew = fmaxf(run_m, cmax);
        const float msc = mnew * LOG2E;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          a0 += ex2_approx(fmaf(v[j], LOG2E, -msc));
          a1 += ex2_approx(fmaf(v[j + 1], LOG2E, -msc));
          a2 += ex2_approx(fmaf(v[j + 2], LOG2E, -msc));
          a3 += ex2_approx(fmaf(v[j + 3], LOG2E, -msc));
        }
        run_s = run_s * ex2_approx((run_m - mnew) * LOG2E) + ((a0 + a1) + (a2 + a3));
        run_m = mnew;
      }
    }
    m = run_m;
    s = run_s;
  }

  __device__ __forceinline__ void end_task(const Params& p, const TcSched&, int, int split, int) {
    if (!valid) return;
    p.part_m[static_cast<size_t>(split) * p.N + grow] = m;
    p.part_s[static_cast<size_t>(split) * p.N + grow] = s;
  }
};

// ============================================================================
// Epilogue 2: dlogits.  G_ij = g coef_i (1[j = y_i] - exp(z_ij - LSE_i)) for the
// tile's columns, 0 at padded columns, rounded to bf16 (nearest even) into the
// block workspace G[N, ldg].
// ============================================================================
struct EpiDlogits {
  struct Params {
    int N, V;
    int vb0;  // first vocabulary column of this block
    int ldg;  // row stride of G (elements)
    const float* lse;
    const float* coef;
    const float* grad_out;  // device scalar or nullptr (1)
    const int* targets;
    int col_offset;  // global vocabulary id of local column 0 (vocabulary shards)
    __nv_bfloat16* G;
    int* zero_word;  // nullable: set to 0 on entry (the next launch's tile counter)
  };
  static __device__ __forceinline__ void on_entry(const Params& p) {
    if (p.zero_word) *p.zero_word = 0;
  }
  __device__ __forceinline__ void begin_task(const Params&, const TcSched&, int, int) {}
  __device__ __forceinline__ void end_task(const Params&, const TcSched&, int, int, int) {}

  __device__ __forceinline__ void tile(const Params& p, const TcSched& sc, uint32_t taddr, int m_blk, int n_blk,
                                       int row, int c_lo, int c_hi) {
    const int grow = m_blk * sc.m_step + row;
    const bool valid = grow < p.N;
    const float g = p.grad_out ? __ldg(p.grad_out) : 1.f;
    const float scale = valid ? g * __ldg(p.coef + grow) : 0.f;
    const float lse2 = valid ? __ldg(p.lse + grow) * LOG2E : 0.f;
    const int yy = valid ? __ldg(p.targets + grow) - p.col_offset : -1;
#pragma unroll 1
    for (int c = c_lo; c < c_hi; ++c) {
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      const int lcol = n_blk * TC_BN + c * 32;  // column within the block
      const int gcol = p.vb0 + lcol;
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float pr0 = (gcol + j < p.V) ? ex2_approx(fmaf(v[j], LOG2E, -lse2)) : 0.f;
        float pr1 = (gcol + j + 1 < p.V) ? ex2_approx(fmaf(v[j + 1], LOG2E, -lse2)) : 0.f;
        const float g0 = scale * (((gcol + j) == yy ? 1.f : 0.f) - pr0);
        const float g1 = scale * (((gcol + j + 1) == yy ? 1.f : 0.f) - pr1);
        __nv_bfloat162 h = __floats2bfloat162_rn(g0, g1);
        packed[j / 2] = *reinterpret_cast<uint32_t*>(&h);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.G + static_cast<size_t>(grow) * p.ldg + lcol);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
  }
};

// ============================================================================
// Epilogue 3: fp32 tile store for dH / dW.
//   mode 0: out32 = acc            mode 1: out32 += acc
//   mode 2: out16 = bf16(out32 + acc)   mode 3: out16 = bf16(acc)
// Rows >= M_valid and columns >= N_valid are not written.
// ============================================================================
struct EpiStore {
  struct Params {
    int M_valid, N_valid;
    int row_off;  // added to the tile row (vocabulary block start for dW)
    int ld;       // row stride of out (elements)
    int mode;
    float* out32;
    __nv_bfloat16* out16;
  };
  static __device__ __forceinline__ void on_entry(const Params&) {}
  __device__ __forceinline__ void begin_task(const Params&, const TcSched&, int, int) {}
  __device__ __forceinline__ void end_task(const Params&, const TcSched&, int, int, int) {}

  __device__ __forceinline__ void tile(const Params& p, const TcSched& sc, uint32_t taddr, int m_blk, int n_blk,
                                       int row, int c_lo, int c_hi) {
    const int lrow = m_blk * sc.m_step + row;
    const bool valid = lrow < p.M_valid;
    const size_t rbase = static_cast<size_t>(p.row_off + lrow) * p.ld;
#pragma unroll 1
    for (int c = c_lo; c < c_hi; ++c) {
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      const int col0 = n_blk * TC_BN + c * 32;
      if (!valid || col0 >= p.N_valid) continue;
      const bool fullc = col0 + 32 <= p.N_valid;
      if (p.mode <= 1) {
        float* dst = p.out32 + rbase + col0;
        if (fullc) {
          float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            if (p.mode == 1) {
              const float4 a = d4[q];
              o.x += a.x;
              o.y += a.y;
              o.z += a.z;
              o.w += a.w;
            }
            d4[q] = o;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < p.N_valid) dst[j] = (p.mode == 1 ? dst[j] : 0.f) + v[j];
        }
      } else {
        __nv_bfloat16* dst = p.out16 + rbase + col0;
        const float* prev = p.out32 + rbase + col0;
        if (fullc) {
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float a = v[j], b = v[j + 1];
            if (p.mode == 2) {
              a += prev[j];
              b += prev[j + 1];
            }
            __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            packed[j / 2] = *reinterpret_cast<uint32_t*>(&h);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < p.N_valid) dst[j] = __float2bfloat16_rn((p.mode == 2 ? prev[j] : 0.f) + v[j]);
        }
      }
    }
  }
};

}  // namespace gh
