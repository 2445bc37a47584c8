// fp32 path (exact fp32 FMA on the CUDA cores, no TF32): logits + online LSE,
// dlogits recompute and a plain tiled GEMM for dH / dW.
//
// Every logit z_ij is one fmaf chain over k = 0..D-1 in increasing order, so
// its value does not depend on the tiling.  Per 256-column vocabulary tile a
// warp owns 4 rows: lane l holds columns l + 32 j (j = 0..7); the tile max and
// the tile sum of exp(z - M) are formed lane-locally in j order and then by a
// xor butterfly (every lane ends with the same bits), and the running (m, s)
// of each row is updated tile by tile in column order.
#include <cuda_runtime.h>

#include "internal.h"

namespace gh {

namespace {

constexpr int F_ROWS = 32;   // rows per sub-block
constexpr int F_KC = 32;     // K chunk
constexpr int F_THREADS = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// z[r][j] for rows r0 + warp*4 + r and columns c0 + lane + 32 j of one 256-wide tile
__device__ __forceinline__ void f32_logits_tile(const float* __restrict__ H, const float* __restrict__ W, int N,
                                                int D, int V, int r0, int c0, float (*Hs)[F_KC],
                                                float (*Ws)[F_KC + 1], float z[4][8]) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 8; ++j) z[r][j] = 0.f;
  for (int k0 = 0; k0 < D; k0 += F_KC) {
    __syncthreads();
    for (int e = t; e < F_ROWS * F_KC; e += F_THREADS) {
      const int r = e / F_KC, k = e % F_KC;
      const int gr = r0 + r, gk = k0 + k;
      Hs[r][k] = (gr < N && gk < D) ? H[static_cast<size_t>(gr) * D + gk] : 0.f;
    }
    for (int e = t; e < 256 * F_KC; e += F_THREADS) {
      const int c = e / F_KC, k = e % F_KC;
      const int gc = c0 + c, gk = k0 + k;
      Ws[c][k] = (gc < V && gk < D) ? W[static_cast<size_t>(gc) * D + gk] : 0.f;
    }
    __syncthreads();
    const int kmax = (D - k0) < F_KC ? (D - k0) : F_KC;
    for (int k = 0; k < kmax; ++k) {
      float h[4], w[8];
#pragma unroll
      for (int r = 0; r < 4; ++r) h[r] = Hs[warp * 4 + r][k];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = Ws[lane + 32 * j][k];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) z[r][j] = fmaf(h[r], w[j], z[r][j]);
    }
  }
}

// grid: (num_row_groups, splits); each CTA walks the row group's 32-row
// sub-blocks and, for each, the split's vocabulary tiles in order.
__global__ void __launch_bounds__(F_THREADS) f32_fwd_kernel(const float* __restrict__ H, const float* __restrict__ W,
                                                           const int* __restrict__ targets, int N, int D, int V,
                                                           int row_tile, int col_offset, float* part_m,
                                                           float* part_s, float* zy) {
  __shared__ float Hs[F_ROWS][F_KC];
  __shared__ float Ws[256][F_KC + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  const int num_vt = (V + 255) / 256;
  const int t_begin = split * TILES_PER_SPLIT;
  const int t_end = min(num_vt, t_begin + TILES_PER_SPLIT);
  for (int sb = 0; sb < row_tile / F_ROWS; ++sb) {
    const int r0 = blockIdx.x * row_tile + sb * F_ROWS;
    if (r0 >= N) break;
    float m[4], s[4];
    int y[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      m[r] = -INFINITY;
      s[r] = 0.f;
      const int gr = r0 + warp * 4 + r;
      y[r] = gr < N ? targets[gr] - col_offset : -1;  // local column of the target
    }
    for (int vt = t_begin; vt < t_end; ++vt) {
      const int c0 = vt * 256;
      float z[4][8];
      f32_logits_tile(H, W, N, D, V, r0, c0, Hs, Ws, z);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int gr = r0 + warp * 4 + r;
        float lm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int col = c0 + lane + 32 * j;
          if (col == y[r] && gr < N) zy[gr] = z[r][j];
          if (col >= V) z[r][j] = -INFINITY;
          lm = fmaxf(lm, z[r][j]);
        }
        const float tmax = warp_max(lm);
        if (tmax == -INFINITY) continue;
        const float mnew = fmaxf(m[r], tmax);
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ls += expf(z[r][j] - mnew);
        const float tsum = warp_sum(ls);
        s[r] = (m[r] == -INFINITY ? 0.f : s[r] * expf(m[r] - mnew)) + tsum;
        m[r] = mnew;
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int gr = r0 + warp * 4 + r;
        if (gr < N) {
          part_m[static_cast<size_t>(split) * N + gr] = m[r];
          part_s[static_cast<size_t>(split) * N + gr] = s[r];
        }
      }
    }
  }
}

// grid: (ceil(N/32), width/256)
__global__ void __launch_bounds__(F_THREADS) f32_dlogits_kernel(const float* __restrict__ H,
                                                               const float* __restrict__ W,
                                                               const int* __restrict__ targets,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ coef,
                                                               const float* __restrict__ grad_out, int N, int D,
                                                               int V, int vb0, int ldg, int col_offset, float* G) {
  __shared__ float Hs[F_ROWS][F_KC];
  __shared__ float Ws[256][F_KC + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * F_ROWS;
  const int lc0 = blockIdx.y * 256;
  const int c0 = vb0 + lc0;
  float z[4][8];
  f32_logits_tile(H, W, N, D, V, r0, c0, Hs, Ws, z);
  const float g = grad_out ? *grad_out : 1.f;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int gr = r0 + warp * 4 + r;
    if (gr >= N) continue;
    const float sc = g * coef[gr];
    const float L = lse[gr];
    const int y = targets[gr] - col_offset;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = c0 + lane + 32 * j;
      const float p = col < V ? expf(z[r][j] - L) : 0.f;
      G[static_cast<size_t>(gr) * ldg + lc0 + lane + 32 * j] = sc * ((col == y ? 1.f : 0.f) - p);
    }
  }
}

constexpr int GT = 64, GK = 16;

__global__ void __launch_bounds__(256) f32_gemm_kernel(F32GemmArgs a) {
  __shared__ float As[GK][GT + 4];
  __shared__ float Bs[GK][GT + 4];
  const int t = threadIdx.x;
  const int tm = t / 16, tn = t % 16;  // 16 x 16 threads, 4 x 4 outputs each
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < a.K; k0 += GK) {
    __syncthreads();
    for (int e = t; e < GK * GT; e += 256) {
      int m, k;
      if (a.sak == 1) {
        k = e % GK;
        m = e / GK;
      } else {
        m = e % GT;
        k = e / GT;
      }
      const int gm = m0 + m, gk = k0 + k;
      As[k][m] = (gm < a.M && gk < a.K) ? a.A[gm * a.sam + gk * a.sak] : 0.f;
      int n, kb;
      if (a.sbn == 1) {
        n = e % GT;
        kb = e / GT;
      } else {
        kb = e % GK;
        n = e / GK;
      }
      const int gn = n0 + n, gkb = k0 + kb;
      Bs[kb][n] = (gn < a.Nn && gkb < a.K) ? a.B[gkb * a.sbk + gn * a.sbn] : 0.f;
    }
    __syncthreads();
    const int kmax = (a.K - k0) < GK ? (a.K - k0) : GK;
    for (int k = 0; k < kmax; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[k][tm + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[k][tn + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + tm + 16 * i;
    if (gm >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tn + 16 * j;
      if (gn >= a.Nn) continue;
      float* c = a.C + (static_cast<long long>(a.row_off) + gm) * a.ldc + gn;
      *c = a.accumulate ? (*c + acc[i][j]) : acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const F32FwdArgs& a, cudaStream_t st) {
  const int rt = (a.row_tile == 64 || a.row_tile == 256) ? a.row_tile : 128;
  const int splits = static_cast<int>(ceil_div(ceil_div(a.V, VTILE), TILES_PER_SPLIT));
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, rt)), static_cast<unsigned>(splits));
  if (a.N <= 0) return cudaSuccess;
  f32_fwd_kernel<<<grid, F_THREADS, 0, st>>>(a.H, a.W, a.targets, a.N, a.D, a.V, rt, a.col_offset, a.part_m, a.part_s,
                                              a.zy);
  return cudaGetLastError();
}

cudaError_t launch_dlogits_f32(const F32DlogitsArgs& a, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, F_ROWS)), static_cast<unsigned>(ceil_div(a.width, 256)));
  if (a.N <= 0) return cudaSuccess;
  f32_dlogits_kernel<<<grid, F_THREADS, 0, st>>>(a.H, a.W, a.targets, a.lse, a.coef, a.grad_out, a.N, a.D, a.V,
                                                  a.vb0, a.ldg, a.col_offset, a.G);
  return cudaGetLastError();
}

cudaError_t launch_gemm_f32(const F32GemmArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.Nn <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(ceil_div(a.Nn, GT)), static_cast<unsigned>(ceil_div(a.M, GT)));
  f32_gemm_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gh
