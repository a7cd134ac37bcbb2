// Float32 FMA tile GEMM used by the factorisation updates: C = beta*C + alpha*A*B.
//
// 128x128 output tile per CTA, 256 threads, each thread an 8x8 sub-tile (two 4x4 quads
// in each direction so that shared-memory reads are float4 and conflict-free), K staged
// through shared memory 16 at a time.  Operand layouts are template parameters:
//   A_MK: A(i, k) = A[i*lda + k]   else A(i, k) = A[k*lda + i]
//   B_NK: B(k, j) = B[j*ldb + k]   else B(k, j) = B[k*ldb + j]
// LOWER: only tiles with tile_row >= tile_col are computed (blockIdx.x enumerates them)
// and only entries with i >= j are written.
#pragma once

#include "common.cuh"

namespace gptq {

struct GemmArgs {
  float* C;
  int ldc;
  const float* A;
  int lda;
  const float* B;
  int ldb;
  int M, N, K;
  float alpha;
  float beta;  // 0 or 1
};

constexpr int kGemmTile = 128;
constexpr int kGemmK = 16;

template <bool A_MK, bool B_NK, bool LOWER>
__global__ void __launch_bounds__(256) gemm_tile_kernel(const GemmArgs g) {
  __shared__ __align__(16) float sa[kGemmK][kGemmTile + 4];
  __shared__ __align__(16) float sb[kGemmK][kGemmTile + 4];
  int bi, bj;
  if (LOWER) {
    int rem = blockIdx.x;
    bi = 0;
    while (rem > bi) { rem -= bi + 1; ++bi; }
    bj = rem;
  } else {
    bi = blockIdx.y;
    bj = blockIdx.x;
  }
  const int i0 = bi * kGemmTile, j0 = bj * kGemmTile;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[8][8];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[u][v] = 0.0f;

  // Register prefetch: the next K chunk's global loads are in flight while the current
  // chunk is multiplied out of shared memory.
  constexpr int PER = kGemmK * kGemmTile / 256;  // elements per thread per operand
  float ra[PER], rb[PER];
  auto load = [&](int k0) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = threadIdx.x + p * 256;
      int kk, ii;
      if (A_MK) { ii = e / kGemmK; kk = e % kGemmK; } else { kk = e / kGemmTile; ii = e % kGemmTile; }
      const int i = i0 + ii, k = k0 + kk;
      float v = 0.0f;
      if (i < g.M && k < g.K)
        v = A_MK ? g.A[static_cast<size_t>(i) * g.lda + k] : g.A[static_cast<size_t>(k) * g.lda + i];
      ra[p] = v;
      int jj;
      if (B_NK) { jj = e / kGemmK; kk = e % kGemmK; } else { kk = e / kGemmTile; jj = e % kGemmTile; }
      const int j = j0 + jj, k2 = k0 + kk;
      float w = 0.0f;
      if (j < g.N && k2 < g.K)
        w = B_NK ? g.B[static_cast<size_t>(j) * g.ldb + k2] : g.B[static_cast<size_t>(k2) * g.ldb + j];
      rb[p] = w;
    }
  };
  load(0);
  for (int k0 = 0; k0 < g.K; k0 += kGemmK) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = threadIdx.x + p * 256;
      if (A_MK) sa[e % kGemmK][e / kGemmK] = ra[p]; else sa[e / kGemmTile][e % kGemmTile] = ra[p];
      if (B_NK) sb[e % kGemmK][e / kGemmK] = rb[p]; else sb[e / kGemmTile][e % kGemmTile] = rb[p];
    }
    __syncthreads();
    if (k0 + kGemmK < g.K) load(k0 + kGemmK);
#pragma unroll
    for (int kk = 0; kk < kGemmK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sa[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sa[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sb[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sb[kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = i0 + (u < 4 ? ty * 4 + u : 64 + ty * 4 + u - 4);
    if (i >= g.M) continue;
    float* crow = g.C + static_cast<size_t>(i) * g.ldc;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int j = j0 + (v < 4 ? tx * 4 + v : 64 + tx * 4 + v - 4);
      if (j >= g.N || (LOWER && j > i)) continue;
      const float prod = g.alpha * acc[u][v];
      crow[j] = (g.beta != 0.0f) ? crow[j] + prod : prod;
    }
  }
}

// Launches gemm_tile_kernel over every output tile (or the lower tiles).
template <bool A_MK, bool B_NK, bool LOWER>
void launch_gemm_tile(int kind, const GemmArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return;
  const int tm = static_cast<int>(ceil_div(g.M, kGemmTile));
  const int tn = static_cast<int>(ceil_div(g.N, kGemmTile));
  auto kfn = gemm_tile_kernel<A_MK, B_NK, LOWER>;
  if (LOWER) {
    GPTQ_LAUNCH(kind, s, kfn, tm * (tm + 1) / 2, 256, 0, g);
  } else {
    GPTQ_LAUNCH(kind, s, kfn, dim3(tn, tm), 256, 0, g);
  }
}

}  // namespace gptq
