// fp32 path (exact fp32 FMA on the CUDA cores, no TF32): logits + per-tile
// (max, sum exp), dlogits recompute and the dH / dW GEMMs.
//
// Every logit z_ij is one fmaf chain over k = 0, 1, ... in increasing order,
// and every GEMM output is the left-to-right sum of such chains over fixed
// 512-long K slices (F32_SLICE), so no value depends on the tiling, on which
// CTA computes it or on how many slices run in parallel.  The kernels are register tiled: a thread keeps an 8 x 8
// block of outputs, operands are staged in shared memory (double buffered,
// the next K chunk is fetched into registers while the current one is used).
//
// Logits tile (forward and dlogits): 64 rows x 256 columns (one vocabulary
// tile) per 256-thread CTA.  Warp w owns rows 8w..8w+7; lane l owns columns
// 4l..4l+3 and 128+4l..128+4l+3.  A row's tile max and sum of exp(z - max) are
// formed lane-locally in column order and then by a xor butterfly, so every
// lane ends with the same bits whatever the row tile.
#include <cuda_runtime.h>

#include "internal.h"

namespace gh {

namespace {

constexpr int L_BM = 64, L_BN = 256, L_BK = 16, L_THREADS = 256;
constexpr int L_APAD = L_BM + 4;   // smem row stride of the H chunk (floats)
constexpr int L_BPAD = L_BN + 4;   // smem row stride of the W chunk (floats)

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

// four consecutive floats p[0..3] of a row of length `len` starting at column
// `c` (zero beyond len); vector load when aligned and in bounds
template <bool VEC>
__device__ __forceinline__ float4 load4(const float* __restrict__ row, int c, int len) {
  if (VEC && c + 3 < len) return __ldg(reinterpret_cast<const float4*>(row + c));
  float4 v;
  v.x = c < len ? __ldg(row + c) : 0.f;
  v.y = c + 1 < len ? __ldg(row + c + 1) : 0.f;
  v.z = c + 2 < len ? __ldg(row + c + 2) : 0.f;
  v.w = c + 3 < len ? __ldg(row + c + 3) : 0.f;
  return v;
}

// ROWS x 256 logits tile of a CTA of ROWS * 4 threads (64: 256 threads, the
// default; 32: 128 threads, for small dlogits grids)
template <int ROWS>
struct LogitsSmem {
  float A[2][L_BK][ROWS + 4];  // H chunk, k-major: A[k][row]
  float B[2][L_BK][L_BPAD];    // W chunk, k-major: B[k][col]
};

// Column of output j (0..7) of lane l within the 256-wide tile.
__device__ __forceinline__ int lcol(int lane, int j) { return (j < 4 ? 4 * lane : 128 + 4 * lane) + (j & 3); }

// z[r][j] = sum_k H[r0 + 8w + r, k] W[c0 + lcol(lane, j), k] (zero for rows >= N
// or columns >= V).  Thread t fetches one float4 of H (row t/4, k 4(t%4)) and
// QB of W (column (t + THREADS q)/4) per K chunk.
template <bool VEC, int ROWS = L_BM>
__device__ __forceinline__ void logits_tile(const float* __restrict__ H, const float* __restrict__ W, int N, int D,
                                            int V, int r0, int c0, LogitsSmem<ROWS>& sm, float z[8][8]) {
  constexpr int THREADS = ROWS * 4;
  constexpr int QB = L_BN * 4 / THREADS;  // float4 of the W chunk per thread
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int j = 0; j < 8; ++j) z[r][j] = 0.f;
  const int ar = t >> 2, akq = (t & 3) * 4;
  const int agr = r0 + ar;
  const float* hrow = H + static_cast<size_t>(agr < N ? agr : 0) * D;
  const float* wrow[QB];
  int bc[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    bc[q] = (t + THREADS * q) >> 2;
    const int gc = c0 + bc[q];
    wrow[q] = W + static_cast<size_t>(gc < V ? gc : 0) * D;
  }
  const bool arow_ok = agr < N;
  bool bcol_ok[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) bcol_ok[q] = c0 + bc[q] < V;

  float4 pa, pb[QB];
  auto fetch = [&](int k0) {
    pa = arow_ok ? load4<VEC>(hrow, k0 + akq, D) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QB; ++q)
      pb[q] = bcol_ok[q] ? load4<VEC>(wrow[q], k0 + akq, D) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto stash = [&](int buf) {
    sm.A[buf][akq + 0][ar] = pa.x;
    sm.A[buf][akq + 1][ar] = pa.y;
    sm.A[buf][akq + 2][ar] = pa.z;
    sm.A[buf][akq + 3][ar] = pa.w;
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      sm.B[buf][akq + 0][bc[q]] = pb[q].x;
      sm.B[buf][akq + 1][bc[q]] = pb[q].y;
      sm.B[buf][akq + 2][bc[q]] = pb[q].z;
      sm.B[buf][akq + 3][bc[q]] = pb[q].w;
    }
  };

  const int nk = (D + L_BK - 1) / L_BK;
  __syncthreads();  // the previous tile's readers of sm are done
  fetch(0);
  stash(0);
  __syncthreads();
  for (int kc = 0; kc < nk; ++kc) {
    const int buf = kc & 1;
    if (kc + 1 < nk) fetch((kc + 1) * L_BK);
#pragma unroll
    for (int k = 0; k < L_BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sm.A[buf][k][warp * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sm.A[buf][k][warp * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sm.B[buf][k][4 * lane]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sm.B[buf][k][128 + 4 * lane]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) z[r][j] = fmaf(a[r], b[j], z[r][j]);
    }
    if (kc + 1 < nk) {
      stash(buf ^ 1);
      __syncthreads();
    }
  }
}

// grid: (ceil(N / row_tile), vocabulary tiles).  A CTA walks its row tile in
// 64-row sub-blocks; for each row it writes the tile's (max, sum exp(z - max))
// as the split partial and, where the target falls in the tile, z_y.
template <bool VEC>
__global__ void __launch_bounds__(L_THREADS, 2) f32_fwd_kernel(const float* __restrict__ H,
                                                              const float* __restrict__ W,
                                                              const int* __restrict__ targets, int N, int D, int V,
                                                              int row_tile, int col_offset, float* part_m,
                                                              float* part_s, float* zy) {
  __shared__ __align__(16) LogitsSmem<L_BM> sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  const int c0 = split * L_BN;
  for (int sb = 0; sb < row_tile / L_BM; ++sb) {
    const int r0 = blockIdx.x * row_tile + sb * L_BM;
    if (r0 >= N) break;
    float z[8][8];
    logits_tile<VEC>(H, W, N, D, V, r0, c0, sm, z);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int gr = r0 + warp * 8 + r;
      const int y = gr < N ? __ldg(targets + gr) - col_offset : -1;  // local column of the target
      float lm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int col = c0 + lcol(lane, j);
        if (col == y) zy[gr] = z[r][j];
        if (col >= V) z[r][j] = -INFINITY;
        lm = fmaxf(lm, z[r][j]);
      }
      const float tmax = warp_max(lm);
      float tsum = 0.f;
      if (tmax != -INFINITY) {
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ls += expf(z[r][j] - tmax);
        tsum = warp_sum(ls);
      }
      if (lane == 0 && gr < N) {
        part_m[static_cast<size_t>(split) * N + gr] = tmax;
        part_s[static_cast<size_t>(split) * N + gr] = tsum;
      }
    }
  }
}

// grid: (ceil(N / ROWS), width / 256).  G[i, lc] = g coef_i (1[col = y_i] - exp(z - LSE_i))
// for the block's local column lc (0 at padded columns).
template <bool VEC, int ROWS>
__global__ void __launch_bounds__(ROWS * 4, 2) f32_dlogits_kernel(
    const float* __restrict__ H, const float* __restrict__ W, const int* __restrict__ targets,
    const float* __restrict__ lse, const float* __restrict__ coef, const float* __restrict__ grad_out, int N, int D,
    int V, int vb0, int ldg, int col_offset, float* G) {
  __shared__ __align__(16) LogitsSmem<ROWS> sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * ROWS;
  const int lc0 = blockIdx.y * L_BN;
  const int c0 = vb0 + lc0;
  float z[8][8];
  logits_tile<VEC, ROWS>(H, W, N, D, V, r0, c0, sm, z);
  const float g = grad_out ? *grad_out : 1.f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int gr = r0 + warp * 8 + r;
    if (gr >= N) continue;
    const float sc = g * coef[gr];
    const float L = lse[gr];
    const int y = targets[gr] - col_offset;
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = c0 + lcol(lane, j);
      const float p = col < V ? expf(z[r][j] - L) : 0.f;
      o[j] = sc * ((col == y ? 1.f : 0.f) - p);
    }
    float* grow = G + static_cast<size_t>(gr) * ldg + lc0;
    *reinterpret_cast<float4*>(grow + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(grow + 128 + 4 * lane) = make_float4(o[4], o[5], o[6], o[7]);
  }
}

// ---------------------------------------------------------------- GEMM
// C[row_off + m, n] (+)= sum_k A(m, k) B(k, n) with B n-contiguous (B(k, n) =
// B[k sbk + n]) and A either k-contiguous (A(m, k) = A[m sam + k]: dH = G W)
// or m-contiguous (A(m, k) = A[m + k sak]: dW = G^T H).  A TILE x TILE output
// tile per CTA of (TILE / RPT)^2 threads, each owning RPT x RPT outputs:
// rows 4tr.. (and TILE/2 + 4tr.. when RPT = 8), columns alike.  Neither the
// tile nor the outputs per thread change any output's arithmetic.
constexpr int G_BK = 16;

template <int TILE, int RPT, bool A_KCONTIG, bool VEC>
__global__ void __launch_bounds__((TILE / RPT) * (TILE / RPT), 2) f32_gemm_kernel(F32GemmArgs a) {
  constexpr int THREADS = (TILE / RPT) * (TILE / RPT);
  constexpr int TPR = TILE / RPT;      // threads per row of the thread grid
  constexpr int Q = TILE * 4 / THREADS;  // float4 of each operand chunk per thread
  constexpr int F4R = TILE / 4;        // float4 per k-row of an MN-contiguous chunk
  constexpr int PAD = TILE + 4;
  static_assert(RPT == 4 || RPT == 8, "4 x 4 or 8 x 8 outputs per thread");
  __shared__ __align__(16) float As[2][G_BK][PAD];
  __shared__ __align__(16) float Bs[2][G_BK][PAD];
  const int t = threadIdx.x;
  const int tr = t / TPR, tc = t % TPR;
  const int m0 = blockIdx.y * TILE, n0 = blockIdx.x * TILE;
  // output i of the thread's RPT rows (columns alike): 4tr + i, and with 8 per
  // thread the second four at TILE / 2 + 4tr
  float acc[RPT][RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int j = 0; j < RPT; ++j) acc[i][j] = 0.f;

  float4 pa[Q], pb[Q];
  // A chunk: TILE x 16.  k-contiguous: element e = t + THREADS q -> row e/4,
  // k 4(e%4).  m-contiguous: e -> k e/F4R, rows 4(e%F4R)..
  auto fetch = [&](int k0, int k_end) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = t + THREADS * q;
      if (A_KCONTIG) {
        const int m = e >> 2, kq = (e & 3) * 4;
        const int gm = m0 + m;
        pa[q] = gm < a.M ? load4<VEC>(a.A + static_cast<long long>(gm) * a.sam, k0 + kq, k_end)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const int k = e / F4R, mq = (e % F4R) * 4;
        const int gk = k0 + k;
        pa[q] = gk < k_end ? load4<VEC>(a.A + static_cast<long long>(gk) * a.sak, m0 + mq, a.M)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const int k = e / F4R, nq = (e % F4R) * 4;
      const int gk = k0 + k;
      pb[q] = gk < k_end ? load4<VEC>(a.B + static_cast<long long>(gk) * a.sbk, n0 + nq, a.Nn)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = t + THREADS * q;
      if (A_KCONTIG) {
        const int m = e >> 2, kq = (e & 3) * 4;
        As[buf][kq + 0][m] = pa[q].x;
        As[buf][kq + 1][m] = pa[q].y;
        As[buf][kq + 2][m] = pa[q].z;
        As[buf][kq + 3][m] = pa[q].w;
      } else {
        const int k = e / F4R, mq = (e % F4R) * 4;
        *reinterpret_cast<float4*>(&As[buf][k][mq]) = pa[q];
      }
      const int k = e / F4R, nq = (e % F4R) * 4;
      *reinterpret_cast<float4*>(&Bs[buf][k][nq]) = pb[q];
    }
  };

  // Slices [s_beg, s_end): all of them inside this CTA, or slice slice0 +
  // blockIdx.z of a parallel wave.  Loads past k_end read 0.
  const bool wave = a.scratch != nullptr;
  const int nslices = a.K > 0 ? (a.K + F32_SLICE - 1) / F32_SLICE : 1;
  const int s_beg = wave ? a.slice0 + static_cast<int>(blockIdx.z) : 0;
  const int s_end = wave ? s_beg + 1 : nslices;
  const int k_beg = s_beg * F32_SLICE;
  const int k_end = min(a.K, s_end * F32_SLICE);
  constexpr int CPS = F32_SLICE / G_BK;  // K chunks per slice
  static_assert(F32_SLICE % G_BK == 0, "slices are whole K chunks");
  const int nk = k_end > k_beg ? (k_end - k_beg + G_BK - 1) / G_BK : 1;

  // slice s finished: C = p_0 (first slice, no accumulate) or C + p_s; in a
  // parallel wave the partial goes to this slice's scratch slab instead
  auto flush = [&](int s) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int gm = m0 + (i < 4 ? 4 * tr : TILE / 2 + 4 * tr) + (i & 3);
      if (gm >= a.M) continue;
      float* crow = wave ? a.scratch + (static_cast<long long>(blockIdx.z) * a.M + gm) * a.Nn
                         : a.C + (static_cast<long long>(a.row_off) + gm) * a.ldc;
      const bool add = !wave && (s > 0 || a.accumulate);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const int gn = n0 + (j < 4 ? 4 * tc : TILE / 2 + 4 * tc) + (j & 3);
        if (gn >= a.Nn) continue;
        crow[gn] = add ? crow[gn] + acc[i][j] : acc[i][j];
      }
    }
  };

  fetch(k_beg, k_end);
  stash(0);
  __syncthreads();
  for (int kc = 0; kc < nk; ++kc) {
    const int buf = kc & 1;
    if (kc + 1 < nk) fetch(k_beg + (kc + 1) * G_BK, k_end);
#pragma unroll
    for (int k = 0; k < G_BK; ++k) {
      if constexpr (RPT == 8) {
        const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][4 * tr]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][TILE / 2 + 4 * tr]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][4 * tc]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][TILE / 2 + 4 * tc]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      } else {
        const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][4 * tr]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][4 * tc]);
        const float av[4] = {a0.x, a0.y, a0.z, a0.w};
        const float bv[4] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
    }
    if ((kc + 1) % CPS == 0 || kc + 1 == nk) {
      flush(s_beg + kc / CPS);
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < RPT; ++j) acc[i][j] = 0.f;
    }
    if (kc + 1 < nk) {
      stash(buf ^ 1);
      __syncthreads();
    }
  }
}

// One parallel wave of `count` slices starting at slice0, added to C in slice
// order: C = (first slice and no accumulate ? p_0 : C + p_0) + p_1 + ...
__global__ void __launch_bounds__(256) f32_slice_reduce_kernel(F32GemmArgs a, int count) {
  const long long total = static_cast<long long>(a.M) * a.Nn;
  const bool start = a.slice0 == 0 && !a.accumulate;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long m = i / a.Nn, n = i % a.Nn;
    float* c = a.C + (a.row_off + m) * a.ldc + n;
    float v = start ? a.scratch[i] : *c + a.scratch[i];
    for (int z = 1; z < count; ++z) v += a.scratch[z * total + i];
    *c = v;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_fwd_f32(const F32FwdArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  const int rt = (a.row_tile == 128 || a.row_tile == 256) ? a.row_tile : L_BM;
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, rt)), static_cast<unsigned>(ceil_div(a.V, VTILE)));
  const bool vec = a.D % 4 == 0 && aligned16(a.H) && aligned16(a.W);
  if (vec)
    f32_fwd_kernel<true><<<grid, L_THREADS, 0, st>>>(a.H, a.W, a.targets, a.N, a.D, a.V, rt, a.col_offset, a.part_m,
                                                      a.part_s, a.zy);
  else
    f32_fwd_kernel<false><<<grid, L_THREADS, 0, st>>>(a.H, a.W, a.targets, a.N, a.D, a.V, rt, a.col_offset,
                                                       a.part_m, a.part_s, a.zy);
  return cudaGetLastError();
}

template <int ROWS>
static void dlogits_f32_launch(const F32DlogitsArgs& a, bool vec, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, ROWS)), static_cast<unsigned>(a.width / L_BN));
  if (vec)
    f32_dlogits_kernel<true, ROWS><<<grid, ROWS * 4, 0, st>>>(a.H, a.W, a.targets, a.lse, a.coef, a.grad_out, a.N,
                                                               a.D, a.V, a.vb0, a.ldg, a.col_offset, a.G);
  else
    f32_dlogits_kernel<false, ROWS><<<grid, ROWS * 4, 0, st>>>(a.H, a.W, a.targets, a.lse, a.coef, a.grad_out, a.N,
                                                                a.D, a.V, a.vb0, a.ldg, a.col_offset, a.G);
}

cudaError_t launch_dlogits_f32(const F32DlogitsArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  if (a.width % L_BN != 0 || a.ldg % 4 != 0 || !aligned16(a.G)) return cudaErrorInvalidValue;
  const bool vec = a.D % 4 == 0 && aligned16(a.H) && aligned16(a.W);
  // 32-row tiles (twice the CTAs) when 64-row tiles would leave SMs idle; the
  // tile changes no value
  if (ceil_div(a.N, L_BM) * (a.width / L_BN) < 152)
    dlogits_f32_launch<32>(a, vec, st);
  else
    dlogits_f32_launch<L_BM>(a, vec, st);
  return cudaGetLastError();
}

// Output tile of an M x Nn fp32 GEMM: 128 x 128 (256 threads, 8 x 8 outputs
// each) unless that leaves fewer CTAs than a GB300 has SMs (152; a constant,
// so nothing here depends on the machine), then 64 x 64 (256 threads, 4 x 4
// outputs each: four times the warps on a small output).
static int gemm_f32_tile(long long M, long long Nn) {
  return ceil_div(M, 128) * ceil_div(Nn, 128) < 152 ? 64 : 128;
}

int gemm_f32_par(long long M, long long Nn, long long K, size_t scratch_bytes) {
  // about 304 CTAs (two on each of a GB300's 152 SMs), at most one per slice,
  // within the scratch; constants, so workspace sizes do not depend on the
  // machine that asks
  const long long slices = K > 0 ? ceil_div(K, F32_SLICE) : 1;
  const int tile = gemm_f32_tile(M, Nn);
  const long long tiles = ceil_div(M, tile) * ceil_div(Nn, tile);
  const long long want = 304;
  if (slices <= 1 || tiles <= 0 || tiles >= want || M <= 0 || Nn <= 0) return 1;
  long long p = ceil_div(want, tiles);
  p = p < slices ? p : slices;
  const long long fit = static_cast<long long>(scratch_bytes / (static_cast<size_t>(M) * Nn * 4));
  p = p < fit ? p : fit;
  return p > 1 ? static_cast<int>(p) : 1;
}

template <int TILE, int RPT>
static void gemm_f32_launch(const F32GemmArgs& a, unsigned count, bool kc, bool vec, cudaStream_t st) {
  constexpr int THREADS = (TILE / RPT) * (TILE / RPT);
  dim3 grid(static_cast<unsigned>(ceil_div(a.Nn, TILE)), static_cast<unsigned>(ceil_div(a.M, TILE)), count);
  if (kc) {
    if (vec)
      f32_gemm_kernel<TILE, RPT, true, true><<<grid, THREADS, 0, st>>>(a);
    else
      f32_gemm_kernel<TILE, RPT, true, false><<<grid, THREADS, 0, st>>>(a);
  } else {
    if (vec)
      f32_gemm_kernel<TILE, RPT, false, true><<<grid, THREADS, 0, st>>>(a);
    else
      f32_gemm_kernel<TILE, RPT, false, false><<<grid, THREADS, 0, st>>>(a);
  }
}

cudaError_t launch_gemm_f32(const F32GemmArgs& a0, cudaStream_t st) {
  if (a0.M <= 0 || a0.Nn <= 0) return cudaSuccess;
  if (a0.sbn != 1 || (a0.sak != 1 && a0.sam != 1)) return cudaErrorInvalidValue;
  const int slices = a0.K > 0 ? static_cast<int>(ceil_div(a0.K, F32_SLICE)) : 1;
  F32GemmArgs a = a0;
  a.slice0 = 0;
  int par = a.par < slices ? a.par : slices;
  if (par <= 1 || !a.scratch) {
    par = 1;
    a.scratch = nullptr;
  }
  const bool kc = a.sak == 1;
  const long long lda = kc ? a.sam : a.sak;
  const bool vec = aligned16(a.A) && aligned16(a.B) && lda % 4 == 0 && a.sbk % 4 == 0;
  const int tile = gemm_f32_tile(a.M, a.Nn);
  const long long total = static_cast<long long>(a.M) * a.Nn;
  const unsigned rblocks = static_cast<unsigned>(ceil_div(total, 256) < 4096 ? ceil_div(total, 256) : 4096);
  bool first = true;
  for (int s0 = 0; s0 < (par > 1 ? slices : 1); s0 += par) {
    const int count = par > 1 ? (slices - s0 < par ? slices - s0 : par) : 1;
    a.slice0 = s0;
    if (tile == 64)
      gemm_f32_launch<64, 4>(a, static_cast<unsigned>(count), kc, vec, st);
    else
      gemm_f32_launch<128, 8>(a, static_cast<unsigned>(count), kc, vec, st);
    if (!first) count_extra_launch();
    first = false;
    if (par > 1) {
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      f32_slice_reduce_kernel<<<rblocks, 256, 0, st>>>(a, count);
      count_extra_launch();
    }
  }
  return cudaGetLastError();
}

}  // namespace gh
