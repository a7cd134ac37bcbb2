// Hessian accumulation, float32-FMA path and the split reduction.
//
// H <- beta H + alpha X^T X with alpha = 2/(n+t), beta = n/(n+t): the streaming hook of
// "GPTQ Architecture, in depth", "The algorithm in code" (HessianHook), H = 2XX^T of
// "Same Ruler, Smarter Placement: GPTQ", section 1.4.  The token axis is split into S
// ranges; each range's X^T X lands in its own partial P[s] (d x d, upper 128-tiles), and
// gptq_syrk_reduce folds the partials into H in a fixed order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int kTile = 64;   // output tile edge
constexpr int kStep = 16;   // tokens per shared-memory stage

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// One CTA per (64x64 tile in the upper 128-tile triangle, token split).  blockIdx.x
// enumerates tile pairs (I, J) of 64-tiles with I/2 <= J/2; blockIdx.y is the split.
template <typename T>
__global__ void __launch_bounds__(256) syrk_simt_kernel(const T* __restrict__ X, int64_t ntok,
                                                        int d, int64_t tok_per_split,
                                                        float* __restrict__ P) {
  const int nt = (d + kTile - 1) / kTile;
  // decode the tile pair from blockIdx.x: walk column tiles J
  int rem = blockIdx.x, J = 0, I = 0;
  for (J = 0; J < nt; ++J) {
    int cnt = min(2 * (J / 2) + 2, nt);  // I in [0, min(2*(J/2)+1, nt-1)]
    if (rem < cnt) { I = rem; break; }
    rem -= cnt;
  }
  const int i0 = I * kTile, j0 = J * kTile;
  const int64_t t_begin = (int64_t)blockIdx.y * tok_per_split;
  const int64_t t_end = min(ntok, t_begin + tok_per_split);
  float* Ps = P + (size_t)blockIdx.y * d * d;

  __shared__ __align__(16) float sa[kStep][kTile];
  __shared__ __align__(16) float sb[kStep][kTile];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kStep) {
    // 16 tokens x 64 columns for each operand; 256 threads x 4 elements
    for (int e = threadIdx.x; e < kStep * kTile; e += 256) {
      int r = e / kTile, c = e % kTile;
      int64_t t = t0 + r;
      float va = 0.f, vb = 0.f;
      if (t < t_end) {
        if (i0 + c < d) va = to_f32(X[t * d + i0 + c]);
        if (j0 + c < d) vb = to_f32(X[t * d + j0 + c]);
      }
      sa[r][c] = va;
      sb[r][c] = vb;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kStep; ++k) {
      float4 a = *reinterpret_cast<const float4*>(&sa[k][ty * 4]);
      float4 b = *reinterpret_cast<const float4*>(&sb[k][tx * 4]);
      float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    int i = i0 + ty * 4 + u;
    if (i >= d) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      int j = j0 + tx * 4 + v;
      if (j < d) Ps[(size_t)i * d + j] = acc[u][v];
    }
  }
}

// H[i, j] = beta * H[i, j] + alpha * sum_s P[s][i, j] over the upper 128-tile region.
// One CTA row per i, float4 along j (d % 4 == 0).
__global__ void syrk_reduce_kernel(float* __restrict__ H, const float* __restrict__ P, int d,
                                   int splits, float alpha, float beta, int overwrite) {
  const int i = blockIdx.y;
  const int jstart = (i / 128) * 128;
  const int j = jstart + 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (j >= d) return;
  const size_t off = (size_t)i * d + j;
  float4 acc = *reinterpret_cast<const float4*>(P + off);
  for (int s = 1; s < splits; ++s) {
    float4 p = *reinterpret_cast<const float4*>(P + (size_t)s * d * d + off);
    acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
  }
  float4 h;
  if (overwrite) {
    h = make_float4(alpha * acc.x, alpha * acc.y, alpha * acc.z, alpha * acc.w);
  } else {
    h = *reinterpret_cast<const float4*>(H + off);
    h.x = beta * h.x + alpha * acc.x;
    h.y = beta * h.y + alpha * acc.y;
    h.z = beta * h.z + alpha * acc.z;
    h.w = beta * h.w + alpha * acc.w;
  }
  *reinterpret_cast<float4*>(H + off) = h;
}

// H[i][j] = factor * H[i][j] on the upper 128-tile triangle (zeros when factor == 0, so
// that a partial of no tokens contributes nothing whatever H held); same indexing as the
// reduction, 16-byte accesses.
__global__ void hessian_rescale_kernel(float* __restrict__ H, int d, float factor) {
  const int i = blockIdx.y;
  const int jstart = (i / 128) * 128;
  const int j = jstart + 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (j >= d) return;
  float4* p = reinterpret_cast<float4*>(H + (size_t)i * d + j);
  float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
  if (factor != 0.0f) {
    h = *p;
    h.x *= factor; h.y *= factor; h.z *= factor; h.w *= factor;
  }
  *p = h;
}

}  // namespace

void launch_hessian_rescale(float* H, int d, float factor, cudaStream_t s) {
  dim3 grid((unsigned)ceil_div(d / 4, 256), d);
  GPTQ_LAUNCH(GPTQ_K_HESSIAN_RESCALE, s, hessian_rescale_kernel, grid, 256, 0, H, d, factor);
}

int syrk_simt_tiles(int d) {
  int nt = (d + kTile - 1) / kTile, n = 0;
  for (int J = 0; J < nt; ++J) n += (2 * (J / 2) + 2 < nt) ? 2 * (J / 2) + 2 : nt;
  return n;
}

void launch_syrk_simt(const void* X, bool bf16, int64_t ntok, int d, int splits,
                      int64_t tok_per_split, float* P, cudaStream_t s) {
  dim3 grid(syrk_simt_tiles(d), splits);
  if (bf16) {
    GPTQ_LAUNCH(GPTQ_K_SYRK_SIMT, s, syrk_simt_kernel<__nv_bfloat16>, grid, 256, 0,
                static_cast<const __nv_bfloat16*>(X), ntok, d, tok_per_split, P);
  } else {
    GPTQ_LAUNCH(GPTQ_K_SYRK_SIMT, s, syrk_simt_kernel<float>, grid, 256, 0,
                static_cast<const float*>(X), ntok, d, tok_per_split, P);
  }
}

void launch_syrk_reduce(float* H, const float* P, int d, int splits, float alpha, float beta,
                        bool overwrite, cudaStream_t s) {
  int threads = 128;
  dim3 grid((unsigned)ceil_div(d / 4, threads), d);
  GPTQ_LAUNCH(GPTQ_K_SYRK_REDUCE, s, syrk_reduce_kernel, grid, threads, 0, H, P, d, splits,
              alpha, beta, overwrite ? 1 : 0);
}

}  // namespace gptq
