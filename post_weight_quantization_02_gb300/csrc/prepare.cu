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
#include "gemm_simt.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;  // panel width of the blocked factorisation and inverse

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

// Factor the NB x NB diagonal block at (k, k) in place (lower).  One CTA of NB threads;
// thread r holds row r in registers.  Right-looking with a rolling register window: at
// step c the window holds the row's columns c .. NB-1 in w[0 ..], so the pivot column is
// always w[0] and every register index is static; the update writes each compensated
// column one slot down.  Per step: the pivot's owner publishes it, every later row
// publishes l_rc, and all rows update.
__global__ void __launch_bounds__(NB) chol_diag_kernel(float* __restrict__ A, int d, int k,
                                                       DevStatus* st, int32_t info_base) {
  __shared__ __align__(16) float col[NB + 4];
  __shared__ float piv_s;
  if (st->code != 0) return;
  const int nb = min(NB, d - k);
  const int r = threadIdx.x;
  float w[NB];
  const float* arow = A + static_cast<size_t>(k + (r < nb ? r : 0)) * d + k;
#pragma unroll
  for (int j = 0; j < NB; j += 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nb && j < nb) v = *reinterpret_cast<const float4*>(arow + j);
    w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
  }
  float lrow_c = 0.0f;  // this row's finished entry of the current column
#pragma unroll 1
  for (int c = 0; c < nb; ++c) {
    if (r == c) piv_s = w[0];
    __syncthreads();
    const float piv = piv_s;
    if (!(piv > 0.0f) || !isfinite(piv)) {
      if (r == 0) dev_fail(st, GPTQ_ERR_NOT_PD, info_base - (k + c));
      return;
    }
    const float sq = sqrtf(piv);
    if (r >= c) {
      lrow_c = (r == c) ? sq : w[0] / sq;
      if (r < nb) A[static_cast<size_t>(k + r) * d + k + c] = lrow_c;
    }
    // col[j'] = l_{c+1+j', c}
    if (r > c) col[r - c - 1] = lrow_c;
    __syncthreads();
    if (r > c) {
#pragma unroll
      for (int j = 0; j < NB - 1; j += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(col + j);
        w[j] = fmaf(-lrow_c, l4.x, w[j + 1]);
        if (j + 1 < NB - 1) w[j + 1] = fmaf(-lrow_c, l4.y, w[j + 2]);
        if (j + 2 < NB - 1) w[j + 2] = fmaf(-lrow_c, l4.z, w[j + 3]);
        if (j + 3 < NB - 1) w[j + 3] = fmaf(-lrow_c, l4.w, w[j + 4 < NB ? j + 4 : NB - 1]);
      }
    }
  }
}

// Forward substitution L y = b for one right-hand side per thread, L = the NB x NB lower
// factor at (k, k).  Used twice:
//   panel (ident == 0): b = row r of A[k+NB:, k:k+NB]; y overwrites it, giving
//                        L[r, k:k+NB] = A[r, k:k+NB] L_kk^-T;
//   inverse (ident == 1): b = e_c for c = threadIdx.x, one CTA per diagonal block
//                        (blockIdx.x), y = column c of L_bb^-1 written to DI[b].
// Right-looking with the same rolling register window as the factorisation; column t of
// L below its diagonal is staged in shared memory as lt[t][j'] = L[t+1+j'][t].
__global__ void __launch_bounds__(NB) trsv_rows_kernel(float* __restrict__ A, int d, int k,
                                                       int ident, float* __restrict__ DI,
                                                       const DevStatus* st) {
  extern __shared__ __align__(16) float smem_f[];
  float(*lt)[NB] = reinterpret_cast<float(*)[NB]>(smem_f);
  float* inv = smem_f + NB * NB;
  if (st->code != 0) return;
  const int kb = ident ? blockIdx.x * NB : k;
  const int nb = min(NB, d - kb);
  for (int e = threadIdx.x; e < NB * NB; e += NB) {
    const int t = e / NB, j = e % NB;   // lt[t][j] = L[t+1+j][t]
    lt[t][j] = (t < nb && t + 1 + j < nb) ? A[static_cast<size_t>(kb + t + 1 + j) * d + kb + t] : 0.0f;
  }
  for (int t = threadIdx.x; t < NB; t += NB)
    inv[t] = (t < nb) ? 1.0f / A[static_cast<size_t>(kb + t) * d + kb + t] : 1.0f;
  __syncthreads();
  float w[NB];
  float* yrow = nullptr;
  if (ident) {
#pragma unroll
    for (int j = 0; j < NB; ++j) w[j] = (j == static_cast<int>(threadIdx.x)) ? 1.0f : 0.0f;
  } else {
    const int r = k + NB + blockIdx.x * NB + threadIdx.x;
    if (r >= d) return;
    yrow = A + static_cast<size_t>(r) * d + k;
#pragma unroll
    for (int j = 0; j < NB; j += 4) {
      const float4 v = *reinterpret_cast<const float4*>(yrow + j);
      w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
    }
  }
  float* dcol = ident ? DI + static_cast<size_t>(blockIdx.x) * NB * NB + threadIdx.x : nullptr;
#pragma unroll 1
  for (int t = 0; t < NB; ++t) {
    const float y = w[0] * inv[t];
    if (ident) dcol[static_cast<size_t>(t) * NB] = y;
    else yrow[t] = y;
    const float* l = lt[t];
#pragma unroll
    for (int j = 0; j < NB - 1; j += 4) {
      const float4 l4 = *reinterpret_cast<const float4*>(l + j);
      w[j] = fmaf(-y, l4.x, w[j + 1]);
      if (j + 1 < NB - 1) w[j + 1] = fmaf(-y, l4.y, w[j + 2]);
      if (j + 2 < NB - 1) w[j + 2] = fmaf(-y, l4.z, w[j + 3]);
      if (j + 3 < NB - 1) w[j + 3] = fmaf(-y, l4.w, w[j + 4 < NB ? j + 4 : NB - 1]);
    }
  }
}

// S = I (the right-hand side of L X = I; updates accumulate into it).
__global__ void identity_kernel(float* __restrict__ S, int d) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < d) S[static_cast<size_t>(i) * d + j] = (i == j) ? 1.0f : 0.0f;
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
                    float* lam, float* DI, DevStatus* st, cudaStream_t s) {
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

  // Cholesky of Hr (lower, in place), NB-wide panels.  A failing pivot at reversed
  // position a reports processing position d - a (1-based).
  const int trsv_smem = (NB * NB + NB) * static_cast<int>(sizeof(float));
  static bool trsv_attr = false;
  if (!trsv_attr) {
    GPTQ_CUDA(cudaFuncSetAttribute(trsv_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   trsv_smem));
    trsv_attr = true;
  }
  for (int k = 0; k < d; k += NB) {
    GPTQ_LAUNCH(GPTQ_K_POTRF_PANEL, s, chol_diag_kernel, 1, NB, 0, Hr, d, k, st, d);
    const int rest = d - k - NB;
    if (rest <= 0) break;
    GPTQ_LAUNCH(GPTQ_K_POTRF_TRSM, s, trsv_rows_kernel, (unsigned)ceil_div(rest, NB), NB, trsv_smem,
                Hr, d, k, 0, DI, st);
    GemmArgs upd{Hr + static_cast<size_t>(k + NB) * d + k + NB, d,
                 Hr + static_cast<size_t>(k + NB) * d + k, d,
                 Hr + static_cast<size_t>(k + NB) * d + k, d, rest, rest, NB, -1.0f, 1.0f};
    launch_gemm_tile<true, true, true>(GPTQ_K_POTRF_UPDATE, upd, s);
  }
  // inverses of all diagonal blocks at once
  GPTQ_LAUNCH(GPTQ_K_TRTRI_DIAG, s, trsv_rows_kernel, (unsigned)ceil_div(d, NB), NB, trsv_smem, Hr,
              d, 0, 1, DI, st);

  // X = Hr^-1 (lower) into S: block rows in order, X[i] = DI[i] R[i], then the later rows'
  // right-hand sides lose L[r, i] X[i].  Then U = J X J.
  {
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_TRTRI_UPDATE, s, identity_kernel, grid, 256, 0, S, d);
  }
  for (int i0 = 0; i0 < d; i0 += NB) {
    const int nbi = (d - i0 < NB) ? d - i0 : NB;
    const float* DIi = DI + static_cast<size_t>(i0 / NB) * NB * NB;
    GemmArgs rows{S + static_cast<size_t>(i0) * d, d, DIi, NB, S + static_cast<size_t>(i0) * d, d,
                  nbi, i0 + nbi, nbi, 1.0f, 0.0f};
    launch_gemm_tile<true, false, false>(GPTQ_K_TRTRI_DIAG, rows, s);
    const int rest = d - i0 - NB;
    if (rest <= 0) break;
    GemmArgs upd{S + static_cast<size_t>(i0 + NB) * d, d, Hr + static_cast<size_t>(i0 + NB) * d + i0,
                 d, S + static_cast<size_t>(i0) * d, d, rest, i0 + NB, NB, -1.0f, 1.0f};
    launch_gemm_tile<true, false, false>(GPTQ_K_TRTRI_UPDATE, upd, s);
  }
  {
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_PREP_REVERSE, s, reverse_kernel, grid, 256, 0, S, d, U);
  }
}

}  // namespace gptq
