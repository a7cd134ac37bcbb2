// gptq_prepare kernels: dead-column fix, act-order ranking, symmetric gather with
// damping, and the inverse Cholesky factor.
//
// What is computed ("GPTQ Architecture, in depth", "The algorithm in code"; "Same Ruler,
// Smarter Placement: GPTQ", sections 1.6, 1.7, 1.9):
//   dead = diag(H) == 0 -> H_jj = 1;  perm = argsort(diag, descending, stable);
//   H_damp = H[perm][:, perm] + lambda I, lambda = damp * mean(diag);
//   U upper with H_damp^-1 = U^T U.
// How U is reached differs from the pages' four steps (chol, cholesky_inverse, chol):
// with J the index reversal, U = J chol(J H_damp J)^-1 J, one Cholesky factorisation and
// one triangular inverse (2d^3/3 flops instead of 4d^3/3).  The gather writes
// Hr = J H_damp J directly, so both factorisations run on Hr and the last kernel
// reverses the inverse into U.
#include "common.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int NB = 64;  // panel width of the blocked factorisation and inverse

// ---------------------------------------------------------------- diagonal statistics

// One CTA of 1024 threads.  diag_fixed[j] = H_jj or 1 for a dead channel; lam = damp *
// mean(diag_fixed) (summed in double in a fixed order).
__global__ void __launch_bounds__(1024) prep_diag_kernel(const float* __restrict__ H, int d,
                                                         float damp, uint8_t* __restrict__ dead,
                                                         float* __restrict__ diag_fixed,
                                                         float* __restrict__ lam_out,
                                                         DevStatus* st) {
  __shared__ double part[1024];
  double s = 0.0;
  for (int j = threadIdx.x; j < d; j += 1024) {
    float h = H[static_cast<size_t>(j) * d + j];
    if (!isfinite(h)) dev_fail(st, GPTQ_ERR_NONFINITE, j + 1);
    uint8_t is_dead = (h == 0.0f) ? 1 : 0;
    float f = is_dead ? 1.0f : h;
    dead[j] = is_dead;
    diag_fixed[j] = f;
    s += static_cast<double>(f);
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *lam_out = static_cast<float>(static_cast<double>(damp) * part[0] / d);
}

// ---------------------------------------------------------------- act-order ranking

// rank[j] = #{k : diag[k] > diag[j] or (diag[k] == diag[j] and k < j)}; perm[rank] = j.
// This is the stable descending order of "GPTQ > ActOrder" with ties by index.
__global__ void __launch_bounds__(256) prep_rank_kernel(const float* __restrict__ diag, int d,
                                                        int actorder, int32_t* __restrict__ perm) {
  __shared__ float tile[2048];
  const int j = blockIdx.x * 256 + threadIdx.x;
  const float dj = (j < d) ? diag[j] : 0.0f;
  int rank = 0;
  if (!actorder) {
    if (j < d) perm[j] = j;
    return;
  }
  for (int k0 = 0; k0 < d; k0 += 2048) {
    const int n = min(2048, d - k0);
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += 256) tile[t] = diag[k0 + t];
    __syncthreads();
    if (j < d) {
      for (int t = 0; t < n; ++t) {
        const float dk = tile[t];
        rank += (dk > dj) || (dk == dj && k0 + t < j);
      }
    }
  }
  if (j < d) perm[rank] = j;
}

// ---------------------------------------------------------------- symmetric copy

// S[i][j] = H[min(i,j)][max(i,j)] (strict upper triangle of H is authoritative).
// 32x32 tiles, 32x8 threads; the lower half is read through a shared-memory transpose.
__global__ void __launch_bounds__(256) prep_mirror_kernel(const float* __restrict__ H, int d,
                                                          float* __restrict__ S, DevStatus* st) {
  __shared__ float t[32][33];
  const int bi = blockIdx.y, bj = blockIdx.x;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  // read the source tile (bi', bj') = upper one of (bi, bj) / (bj, bi)
  const int si = min(bi, bj), sj = max(bi, bj);
  for (int r = ty; r < 32; r += 8) {
    const int i = si * 32 + r, j = sj * 32 + tx;
    float v = 0.0f;
    if (i < d && j < d) {
      v = H[static_cast<size_t>(i) * d + j];
      if (i <= j && !isfinite(v)) dev_fail(st, GPTQ_ERR_NONFINITE, 0);
    }
    t[r][tx] = v;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int i = bi * 32 + r, j = bj * 32 + tx;
    if (i >= d || j >= d) continue;
    float v;
    if (bi < bj) v = t[r][tx];
    else if (bi > bj) v = t[tx][r];
    else v = (r <= tx) ? t[r][tx] : t[tx][r];
    S[static_cast<size_t>(i) * d + j] = v;
  }
}

// ---------------------------------------------------------------- reversed gather

// Hr[a][b] = S[p][q] with p = perm[d-1-a], q = perm[d-1-b], for b <= a; the diagonal gets
// the dead fix (1) and + lambda.  One CTA per row a; the source row is staged in shared
// memory (d floats).
__global__ void __launch_bounds__(256) prep_gather_kernel(const float* __restrict__ S, int d,
                                                          const int32_t* __restrict__ perm,
                                                          const uint8_t* __restrict__ dead,
                                                          const float* __restrict__ lam,
                                                          float* __restrict__ Hr) {
  extern __shared__ float row[];
  const int a = blockIdx.x;
  const int p = perm[d - 1 - a];
  const float* src = S + static_cast<size_t>(p) * d;
  for (int j = threadIdx.x; j < d; j += 256) row[j] = src[j];
  __syncthreads();
  float* dst = Hr + static_cast<size_t>(a) * d;
  const float l = *lam;
  for (int b = threadIdx.x; b <= a; b += 256) {
    const int q = perm[d - 1 - b];
    float v = row[q];
    if (b == a) v = (dead[p] ? 1.0f : v) + l;
    dst[b] = v;
  }
}

// ---------------------------------------------------------------- blocked Cholesky

// Factor the NB x NB diagonal block at (k, k) in place (lower).  One CTA.
__global__ void __launch_bounds__(256) potf2_kernel(float* __restrict__ A, int d, int k,
                                                    DevStatus* st, int32_t info_base) {
  __shared__ float s[NB][NB + 1];
  __shared__ int bad;
  if (st->code != 0) return;
  const int nb = min(NB, d - k);
  for (int e = threadIdx.x; e < NB * NB; e += 256) {
    const int r = e / NB, c = e % NB;
    s[r][c] = (r < nb && c <= r) ? A[static_cast<size_t>(k + r) * d + k + c] : 0.0f;
  }
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int c = 0; c < nb; ++c) {
    if (threadIdx.x == 0) {
      const float piv = s[c][c];
      if (!(piv > 0.0f) || !isfinite(piv)) {
        bad = 1;
        dev_fail(st, GPTQ_ERR_NOT_PD, info_base - (k + c));
      } else {
        s[c][c] = sqrtf(piv);
      }
    }
    __syncthreads();
    if (bad) return;
    const float inv = 1.0f / s[c][c];
    for (int r = c + 1 + threadIdx.x; r < nb; r += 256) s[r][c] *= inv;
    __syncthreads();
    const int m = nb - c - 1;
    for (int e = threadIdx.x; e < m * m; e += 256) {
      const int r = c + 1 + e / m, cc = c + 1 + e % m;
      if (cc <= r) s[r][cc] -= s[r][c] * s[cc][c];
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < nb * nb; e += 256) {
    const int r = e / nb, c = e % nb;
    if (c <= r) A[static_cast<size_t>(k + r) * d + k + c] = s[r][c];
  }
}

// Panel below the diagonal block: L[r, k:k+NB] = A[r, k:k+NB] L_kk^-T, one thread per row.
__global__ void __launch_bounds__(128) trsm_panel_kernel(float* __restrict__ A, int d, int k,
                                                         const DevStatus* st) {
  __shared__ float l[NB][NB + 1];
  __shared__ float inv[NB];
  if (st->code != 0) return;
  for (int e = threadIdx.x; e < NB * NB; e += 128) {
    const int r = e / NB, c = e % NB;
    l[r][c] = (c <= r) ? A[static_cast<size_t>(k + r) * d + k + c] : 0.0f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < NB; c += 128) inv[c] = 1.0f / l[c][c];
  __syncthreads();
  const int r = k + NB + blockIdx.x * 128 + threadIdx.x;
  if (r >= d) return;
  float* row = A + static_cast<size_t>(r) * d + k;
  float x[NB];
#pragma unroll
  for (int c = 0; c < NB; c += 4) {
    float4 v = *reinterpret_cast<const float4*>(row + c);
    x[c] = v.x; x[c + 1] = v.y; x[c + 2] = v.z; x[c + 3] = v.w;
  }
#pragma unroll
  for (int c = 0; c < NB; ++c) {
#pragma unroll
    for (int cp = 0; cp < c; ++cp) x[c] = fmaf(-x[cp], l[c][cp], x[c]);
    x[c] *= inv[c];
  }
#pragma unroll
  for (int c = 0; c < NB; c += 4)
    *reinterpret_cast<float4*>(row + c) = make_float4(x[c], x[c + 1], x[c + 2], x[c + 3]);
}

// C[i][j] -= sum_c A1[i][c] * A2[j][c] over a 64x64 tile, K = NB.  Shared by the
// Cholesky trailing update (A1 = A2 = panel, lower tiles) and the triangular-inverse
// update.  Operands are staged transposed: sa[c][i], sb[c][j].
struct TileOperands {
  float sa[NB][68];
  float sb[NB][68];
};

__device__ __forceinline__ void tile_update(TileOperands& t, int tx, int ty, float (&acc)[4][4]) {
#pragma unroll 8
  for (int c = 0; c < NB; ++c) {
    const float4 a = *reinterpret_cast<const float4*>(&t.sa[c][ty * 4]);
    const float4 b = *reinterpret_cast<const float4*>(&t.sb[c][tx * 4]);
    const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
}

// Trailing update of the Cholesky: A[i][j] -= L[i][k:k+NB] . L[j][k:k+NB] for
// k+NB <= j <= i.  blockIdx.x enumerates 64-tiles (bi >= bj) of the trailing matrix.
__global__ void __launch_bounds__(256) potrf_update_kernel(float* __restrict__ A, int d, int k,
                                                           const DevStatus* st) {
  __shared__ TileOperands t;
  if (st->code != 0) return;
  const int base = k + NB;
  int rem = blockIdx.x, bi = 0;
  while (rem > bi) { rem -= bi + 1; ++bi; }
  const int bj = rem;
  const int i0 = base + bi * 64, j0 = base + bj * 64;
  for (int e = threadIdx.x; e < 64 * NB; e += 256) {
    const int r = e / NB, c = e % NB;
    t.sa[c][r] = (i0 + r < d) ? A[static_cast<size_t>(i0 + r) * d + k + c] : 0.0f;
    t.sb[c][r] = (j0 + r < d) ? A[static_cast<size_t>(j0 + r) * d + k + c] : 0.0f;
  }
  __syncthreads();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  tile_update(t, tx, ty, acc);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= d) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j <= i) A[static_cast<size_t>(i) * d + j] -= acc[u][v];
    }
  }
}

// ---------------------------------------------------------------- triangular inverse

// Xb (lower part) = 0 before the inverse.
__global__ void zero_lower_kernel(float* __restrict__ X, int d) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j <= i && i < d) X[static_cast<size_t>(i) * d + j] = 0.0f;
}

// Block row i of X = L^-1: X[rows of block i][c] = L_ii^-1 R[rows of block i][c] for
// every c < (i+1) NB, one thread per column; inside the diagonal block R is the
// identity, left of it R holds what the updates accumulated.
__global__ void __launch_bounds__(128) trtri_rows_kernel(const float* __restrict__ L,
                                                         float* __restrict__ X, int d, int i0,
                                                         const DevStatus* st) {
  __shared__ float l[NB][NB + 1];
  __shared__ float inv[NB];
  if (st->code != 0) return;
  const int nb = min(NB, d - i0);
  for (int e = threadIdx.x; e < NB * NB; e += 128) {
    const int r = e / NB, c = e % NB;
    l[r][c] = (r < nb && c <= r) ? L[static_cast<size_t>(i0 + r) * d + i0 + c] : 0.0f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < NB; c += 128) inv[c] = (c < nb) ? 1.0f / l[c][c] : 0.0f;
  __syncthreads();
  const int c = blockIdx.x * 128 + threadIdx.x;
  if (c >= i0 + nb) return;
  float y[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    float v;
    if (c >= i0) v = (c - i0 == r) ? 1.0f : 0.0f;
    else v = (r < nb) ? X[static_cast<size_t>(i0 + r) * d + c] : 0.0f;
    y[r] = v;
  }
#pragma unroll
  for (int r = 0; r < NB; ++r) {
#pragma unroll
    for (int rp = 0; rp < r; ++rp) y[r] = fmaf(-l[r][rp], y[rp], y[r]);
    y[r] *= inv[r];
  }
  // inside the diagonal block the entries above its diagonal come out as exact zeros;
  // they are written too because the update reads the whole block row
#pragma unroll
  for (int r = 0; r < NB; ++r)
    if (r < nb) X[static_cast<size_t>(i0 + r) * d + c] = y[r];
}

// X[r][c] -= sum_t L[r][i0+t] X[i0+t][c] for r >= i0+NB, c < i0+NB (64x64 tiles).
__global__ void __launch_bounds__(256) trtri_update_kernel(const float* __restrict__ L,
                                                           float* __restrict__ X, int d, int i0,
                                                           const DevStatus* st) {
  __shared__ TileOperands t;
  if (st->code != 0) return;
  const int r0 = i0 + NB + blockIdx.y * 64;
  const int c0 = blockIdx.x * 64;
  for (int e = threadIdx.x; e < 64 * NB; e += 256) {
    const int r = e / NB, c = e % NB;
    t.sa[c][r] = (r0 + r < d) ? L[static_cast<size_t>(r0 + r) * d + i0 + c] : 0.0f;
    // sb[t][col] = X[i0 + t][c0 + col]
    const int tt = e / 64, col = e % 64;
    t.sb[tt][col] = (c0 + col < i0 + NB) ? X[static_cast<size_t>(i0 + tt) * d + c0 + col] : 0.0f;
  }
  __syncthreads();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  tile_update(t, tx, ty, acc);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = r0 + ty * 4 + u;
    if (r >= d) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c = c0 + tx * 4 + v;
      if (c < i0 + NB) X[static_cast<size_t>(r) * d + c] -= acc[u][v];
    }
  }
}

// U[i][j] = X[d-1-i][d-1-j] for j >= i, 0 below the diagonal.
__global__ void reverse_kernel(const float* __restrict__ X, int d, float* __restrict__ U) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= d) return;
  U[static_cast<size_t>(i) * d + j] =
      (j >= i) ? X[static_cast<size_t>(d - 1 - i) * d + (d - 1 - j)] : 0.0f;
}

}  // namespace

void launch_prepare(const float* H, int d, float damp, int actorder, int32_t* perm,
                    uint8_t* dead, float* U, float* S, float* Hr, float* diag_fixed,
                    float* lam, DevStatus* st, cudaStream_t s) {
  GPTQ_LAUNCH(GPTQ_K_PREP_DIAG, s, prep_diag_kernel, 1, 1024, 0, H, d, damp, dead, diag_fixed,
              lam, st);
  GPTQ_LAUNCH(GPTQ_K_PREP_RANK, s, prep_rank_kernel, (unsigned)ceil_div(d, 256), 256, 0,
              diag_fixed, d, actorder, perm);
  const unsigned t32 = (unsigned)ceil_div(d, 32);
  GPTQ_LAUNCH(GPTQ_K_PREP_MIRROR, s, prep_mirror_kernel, dim3(t32, t32), 256, 0, H, d, S, st);
  const size_t row_smem = static_cast<size_t>(d) * sizeof(float);
  static size_t attr_smem = 0;
  if (row_smem > 48 * 1024 && row_smem > attr_smem) {
    GPTQ_CUDA(cudaFuncSetAttribute(prep_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(row_smem)));
    attr_smem = row_smem;
  }
  GPTQ_LAUNCH(GPTQ_K_PREP_GATHER, s, prep_gather_kernel, d, 256, row_smem, S, d, perm, dead, lam,
              Hr);

  // Cholesky of Hr (lower, in place).  A failing pivot at reversed position a reports
  // processing position d - a (1-based).
  for (int k = 0; k < d; k += NB) {
    GPTQ_LAUNCH(GPTQ_K_POTRF_PANEL, s, potf2_kernel, 1, 256, 0, Hr, d, k, st, d);
    const int rest = d - k - NB;
    if (rest <= 0) break;
    GPTQ_LAUNCH(GPTQ_K_POTRF_TRSM, s, trsm_panel_kernel, (unsigned)ceil_div(rest, 128), 128, 0,
                Hr, d, k, st);
    const int T = static_cast<int>(ceil_div(rest, 64));
    GPTQ_LAUNCH(GPTQ_K_POTRF_UPDATE, s, potrf_update_kernel, T * (T + 1) / 2, 256, 0, Hr, d, k,
                st);
  }

  // X = Hr^-1 (lower) into S, then U = J X J.
  {
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_TRTRI_UPDATE, s, zero_lower_kernel, grid, 256, 0, S, d);
  }
  for (int i0 = 0; i0 < d; i0 += NB) {
    const int ncols = (i0 + NB < d) ? i0 + NB : d;
    GPTQ_LAUNCH(GPTQ_K_TRTRI_DIAG, s, trtri_rows_kernel, (unsigned)ceil_div(ncols, 128), 128, 0,
                Hr, S, d, i0, st);
    const int rest = d - i0 - NB;
    if (rest <= 0) break;
    dim3 grid((unsigned)ceil_div(i0 + NB, 64), (unsigned)ceil_div(rest, 64));
    GPTQ_LAUNCH(GPTQ_K_TRTRI_UPDATE, s, trtri_update_kernel, grid, 256, 0, Hr, S, d, i0, st);
  }
  {
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_PREP_REVERSE, s, reverse_kernel, grid, 256, 0, S, d, U);
  }
}

}  // namespace gptq
