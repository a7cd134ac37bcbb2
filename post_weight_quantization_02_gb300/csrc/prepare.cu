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

// Layout of one factorised diagonal block for the quad triangular solves: for step t
// (column t of L_kk) and lane u of a group of eight, 16 coefficients
//   LL[t][u][i] = L_kk[c][t], c = 8(i + t/8 + (t%8 == 7)) + u, if t < c < nb, else 0,
// (padded to 20), then the 128 reciprocals 1/L_kk[t][t].  Same shape as the column
// loop's layout of U.
constexpr int QL = 8, WL = NB / QL, LSTR = WL + 4, RSTR = QL * LSTR, RPT = 128 / QL;
constexpr int kLLFloats = NB * RSTR + NB;
static_assert(kLLFloats == kLoopUblkFloats, "workspace sizing of the solve layout");

// Factor the NB x NB diagonal block at (k, k) in place (lower), then write its solve
// layout LL.  One CTA of 512 threads, recursively by 32-column sub-panels c0:
//   1. warp 0 factors the 32 x 32 diagonal sub-block in registers (lane = row; the pivot
//      column is broadcast with shuffles);
//   2. 96 threads solve the rows below it, x S^T = a, one row per thread in registers;
//   3. the rest of the block takes L[r][j] -= sum_t L[r][c0+t] L[j][c0+t], one 4 x 4
//      register tile per thread over the lower tiles, float4 shared-memory reads.
constexpr int DSTR = NB + 4;  // row stride of the staged block (16-byte aligned rows)
__global__ void __launch_bounds__(512) chol_diag_kernel(float* __restrict__ A, int d, int k,
                                                        float* __restrict__ LL, DevStatus* st,
                                                        int32_t info_base) {
  extern __shared__ __align__(16) float smem_f[];
  float* L = smem_f;               // [NB][DSTR]
  __shared__ float sinv[32];
  __shared__ int bad;
  if (st->code != 0) return;
  const int nb = min(NB, d - k);
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  {
    float v[NB * NB / 512];
#pragma unroll
    for (int p = 0; p < NB * NB / 512; ++p) {
      const int e = tid + p * 512, r = e / NB, c = e % NB;
      v[p] = (r < nb && c <= r) ? A[static_cast<size_t>(k + r) * d + k + c] : (r == c ? 1.0f : 0.0f);
    }
#pragma unroll
    for (int p = 0; p < NB * NB / 512; ++p) {
      const int e = tid + p * 512;
      L[(e / NB) * DSTR + e % NB] = v[p];  // identity past a ragged end
    }
  }
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int c0 = 0; c0 < NB; c0 += 32) {
    // 1. the 32 x 32 diagonal sub-block
    if (warp == 0) {
      // rolling window: at step c, w[0] is this row's column c (static register indices)
      float* lrow = L + (c0 + lane) * DSTR + c0;
      float w[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = (j <= lane) ? lrow[j] : 0.0f;
      int badc = -1;
#pragma unroll 1
      for (int c = 0; c < 32; ++c) {
        const float piv = __shfl_sync(0xffffffffu, w[0], c);
        if (badc < 0 && (!(piv > 0.0f) || !isfinite(piv))) badc = c;
        const float l = sqrtf(piv);
        const float il = 1.0f / l;
        const float lc = (lane == c) ? l : ((lane > c) ? w[0] * il : 0.0f);
        if (lane >= c) lrow[c] = lc;
        if (lane == c) sinv[c] = il;
#pragma unroll
        for (int j = 0; j < 31; ++j) {
          const float lx = __shfl_sync(0xffffffffu, lc, (c + 1 + j) & 31);
          w[j] = fmaf(-lc, lx, w[j + 1]);
        }
      }
      if (lane == 0 && badc >= 0 && c0 + badc < nb) {
        bad = 1;
        dev_fail(st, GPTQ_ERR_NOT_PD, info_base - (k + c0 + badc));
      }
    }
    __syncthreads();
    if (bad) return;
    // 2. rows below the sub-block: x_c = (a_c - sum_{t<c} x_t S[c][t]) / S[c][c]
    if (tid < NB - c0 - 32) {
      float* xrow = L + (c0 + 32 + tid) * DSTR + c0;
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(xrow + j);
        x[j] = v.x; x[j + 1] = v.y; x[j + 2] = v.z; x[j + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float* srow = L + (c0 + c) * DSTR + c0;
        float acc = x[c];
#pragma unroll
        for (int t = 0; t < c; ++t) acc = fmaf(-x[t], srow[t], acc);
        x[c] = acc * sinv[c];
      }
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(xrow + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
    }
    __syncthreads();
    // 3. the rest of the block, lower 4 x 4 tiles
    const int m2 = NB - c0 - 32;
    const int T = m2 / 4;
    for (int tile = tid; tile < T * (T + 1) / 2; tile += 512) {
      int ti = 0, rem = tile;
      while (rem > ti) { rem -= ti + 1; ++ti; }
      const int tj = rem;
      const int r0 = c0 + 32 + 4 * ti, j0 = c0 + 32 + 4 * tj;
      float acc[4][4] = {};
#pragma unroll
      for (int t = 0; t < 32; t += 4) {
        float4 ra[4], rb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ra[u] = *reinterpret_cast<const float4*>(L + (r0 + u) * DSTR + c0 + t);
          rb[u] = *reinterpret_cast<const float4*>(L + (j0 + u) * DSTR + c0 + t);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            acc[u][v] += ra[u].x * rb[v].x + ra[u].y * rb[v].y + ra[u].z * rb[v].z +
                         ra[u].w * rb[v].w;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v)
          if (j0 + v <= r0 + u) L[(r0 + u) * DSTR + j0 + v] -= acc[u][v];
    }
    __syncthreads();
  }
#pragma unroll 4
  for (int e = tid; e < nb * nb; e += 512) {
    const int r = e / nb, c = e % nb;
    if (c <= r) A[static_cast<size_t>(k + r) * d + k + c] = L[r * DSTR + c];
  }
  float* out = LL + static_cast<size_t>(k / NB) * kLLFloats;
#pragma unroll 4
  for (int e = tid; e < NB * RSTR; e += 512) {
    const int t = e / RSTR, uu = (e % RSTR) / LSTR, i = e % LSTR;
    const int c = QL * (i + t / QL + ((t % QL) == QL - 1 ? 1 : 0)) + uu;
    out[e] = (i < WL && t < nb && c > t && c < nb) ? L[c * DSTR + t] : 0.0f;
  }
  for (int t = tid; t < NB; t += 512) out[NB * RSTR + t] = (t < nb) ? 1.0f / L[t * DSTR + t] : 1.0f;
}

// Forward substitution L_bb y = b, one right-hand side per group of QL = 8 lanes (lane u
// owns unknowns 8i+u; a 16-register window slides as in the column loop).
//   panel (ident == 0): b = row r of A[k+NB:, k:k+NB], y overwrites it, giving
//                       L[r, k:k+NB] = A[r, k:k+NB] L_kk^-T;
//   inverse (ident == 1): b = e_c for 16 values of c per CTA (blockIdx.x = 8*(block -
//                       k/NB) + part), y = column c of L_bb^-1, written to DI[block].
__global__ void __launch_bounds__(128) trsv_quad_kernel(float* __restrict__ A, int d, int k,
                                                        int ident, const float* __restrict__ LLall,
                                                        float* __restrict__ DI,
                                                        const DevStatus* st) {
  extern __shared__ __align__(16) float smem_f[];
  float* ys = smem_f + kLLFloats;  // [NB][RPT] staged results
  if (st->code != 0) return;
  const int blk = ident ? k / NB + blockIdx.x / QL : k / NB;
  const int part = ident ? blockIdx.x % QL : 0;
  const int kb = blk * NB;
  const int nb = min(NB, d - kb);
  {
    const float4* src = reinterpret_cast<const float4*>(LLall + static_cast<size_t>(blk) * kLLFloats);
    float4* dst = reinterpret_cast<float4*>(smem_f);
    for (int e = threadIdx.x; e < kLLFloats / 4; e += 128) {
      const uint32_t s_addr = static_cast<uint32_t>(__cvta_generic_to_shared(dst + e));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s_addr), "l"(src + e) : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  const float* lay = smem_f;
  const float* rinv = smem_f + NB * RSTR;
  const int lane = threadIdx.x % 32, u = lane % QL, qbase = lane & ~(QL - 1);
  const int rl = threadIdx.x / QL;  // 0..RPT-1
  float w[WL];
  int nrows;
  size_t row0;
  if (ident) {
    const int c = part * RPT + rl;
#pragma unroll
    for (int i = 0; i < WL; ++i) w[i] = (QL * i + u == c) ? 1.0f : 0.0f;
    nrows = RPT;
    row0 = 0;
  } else {
    const int rbase = k + NB + blockIdx.x * RPT;
    nrows = min(RPT, d - rbase);
    row0 = static_cast<size_t>(rbase);
    const float* arow = A + static_cast<size_t>(rbase + (rl < nrows ? rl : 0)) * d + k;
#pragma unroll
    for (int i = 0; i < WL; ++i) w[i] = (rl < nrows) ? arow[QL * i + u] : 0.0f;
  }
  const int ngroups = (nb + QL - 1) / QL;
#pragma unroll 1
  for (int g = 0; g < ngroups; ++g) {
#pragma unroll
    for (int o = 0; o < QL; ++o) {
      const int t = QL * g + o;
      const float y = __shfl_sync(0xffffffffu, w[0] * rinv[t], qbase + o);
      if (u == o) ys[t * RPT + rl] = y;
      const float* l = lay + t * RSTR + u * LSTR;
      if (o < QL - 1) {
#pragma unroll
        for (int i = 0; i < WL; i += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(l + i);
          w[i] = fmaf(-y, l4.x, w[i]);
          w[i + 1] = fmaf(-y, l4.y, w[i + 1]);
          w[i + 2] = fmaf(-y, l4.z, w[i + 2]);
          w[i + 3] = fmaf(-y, l4.w, w[i + 3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < WL; i += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(l + i);
          w[i] = fmaf(-y, l4.x, w[i + 1]);
          w[i + 1] = fmaf(-y, l4.y, w[i + 2]);
          w[i + 2] = fmaf(-y, l4.z, w[i + 3]);
          if (i + 3 < WL - 1) w[i + 3] = fmaf(-y, l4.w, w[i + 4 < WL ? i + 4 : WL - 1]);
        }
      }
    }
  }
  __syncthreads();
  if (ident) {
    // DI[blk][t][c] for the CTA's RPT columns c, all NB rows t (zeros above the diagonal
    // come out of the substitution exactly); identity past a ragged end
    float* dout = DI + static_cast<size_t>(blk) * NB * NB + part * RPT;
    for (int e = threadIdx.x; e < NB * RPT; e += 128) {
      const int t = e / RPT, j = e % RPT;
      dout[static_cast<size_t>(t) * NB + j] = (t < nb) ? ys[e] : (t == part * RPT + j ? 1.0f : 0.0f);
    }
  } else {
    for (int e = threadIdx.x; e < nrows * NB; e += 128) {
      const int j = e / NB, t = e % NB;
      if (t < nb) A[(row0 + j) * d + k + t] = ys[t * RPT + j];
    }
  }
}

// S = I (the right-hand side of L X = I; updates accumulate into it).
__global__ void identity_kernel(float* __restrict__ S, int d) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < d) S[static_cast<size_t>(i) * d + j] = (i == j) ? 1.0f : 0.0f;
}

// U[i][j] = X[d-1-i][d-1-j] = Y[d-1-j][d-1-i] for j >= i, 0 below the diagonal; 32x32
// tiles transposed through shared memory.
__global__ void reverse_transpose_kernel(const float* __restrict__ Y, int d, float* __restrict__ U) {
  __shared__ float t[32][33];
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
  for (int jj = threadIdx.y; jj < 32; jj += 8) {
    const int j = j0 + jj, ii = threadIdx.x, i = i0 + ii;
    t[jj][ii] = (i < d && j < d) ? Y[static_cast<size_t>(d - 1 - j) * d + (d - 1 - i)] : 0.0f;
  }
  __syncthreads();
  for (int ii = threadIdx.y; ii < 32; ii += 8) {
    const int i = i0 + ii, jj = threadIdx.x, j = j0 + jj;
    if (i < d && j < d) U[static_cast<size_t>(i) * d + j] = (j >= i) ? t[jj][ii] : 0.0f;
  }
}

}  // namespace

void launch_prepare(const float* H, int d, float damp, int actorder, int32_t* perm,
                    uint8_t* dead, float* U, float* S, float* Hr, float* diag_fixed,
                    float* lam, float* DI, float* LL, DevStatus* st, cudaStream_t s) {
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

  // Cholesky of Hr (lower, in place) by NB-wide panels on stream A, and the inverse of
  // the factor on stream B: block column k of the inverse needs only L's first k+1 block
  // columns, so it runs as soon as panel k is final, overlapping the (latency-bound)
  // factorisation of the next panels.  A failing pivot at reversed position a reports
  // processing position d - a (1-based).
  //
  // The inverse X = L^-1 is kept transposed as Y = X^T in S so that both GEMM operands
  // are K-major: block column i of Y is Y[:, i] = R DI[i]^T (R = the accumulated right-
  // hand side, initially I), after which every later block column loses
  // Y[:, i] L[r, i]^T.  Finally U = J X J = (J Y J)^T.
  const int trsv_smem = (kLLFloats + NB * RPT) * static_cast<int>(sizeof(float));
  const int diag_smem = NB * DSTR * static_cast<int>(sizeof(float));
  static bool attrs = false;
  if (!attrs) {
    GPTQ_CUDA(cudaFuncSetAttribute(chol_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   diag_smem));
    GPTQ_CUDA(cudaFuncSetAttribute(trsv_quad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   trsv_smem));
    attrs = true;
  }
  CUtensorMap mHr, mS, mDI;
  make_gemm_map(&mHr, Hr, d, d, d);
  make_gemm_map(&mS, S, d, d, d);
  make_gemm_map(&mDI, DI, static_cast<int>(ceil_div(d, NB)) * NB, NB, NB);
  {
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_TRTRI_UPDATE, s, identity_kernel, grid, 256, 0, S, d);
  }
  const int nblk = static_cast<int>(ceil_div(d, NB));
  AuxStreams& aux = aux_streams(nblk + 2);
  cudaStream_t sa = aux.a, sb = aux.b;
  GPTQ_CUDA(cudaEventRecord(aux.ev[nblk], s));
  GPTQ_CUDA(cudaStreamWaitEvent(sa, aux.ev[nblk], 0));
  GPTQ_CUDA(cudaStreamWaitEvent(sb, aux.ev[nblk], 0));
  for (int k = 0; k < d; k += NB) {
    const int kb = k / NB;
    const int rest = d - k - NB;
    GPTQ_LAUNCH(GPTQ_K_POTRF_PANEL, sa, chol_diag_kernel, 1, 512, diag_smem, Hr, d, k, LL, st, d);
    if (rest > 0) {
      GPTQ_LAUNCH(GPTQ_K_POTRF_TRSM, sa, trsv_quad_kernel, (unsigned)ceil_div(rest, RPT), 128,
                  trsv_smem, Hr, d, k, 0, LL, DI, st);
    }
    GPTQ_CUDA(cudaEventRecord(aux.ev[kb], sa));
    if (rest > 0) {
      // trailing update, lower tiles: Hr[k+NB+i][k+NB+j] -= L[k+NB+i, panel] . L[k+NB+j, panel]
      launch_gemm_tf32x3(GPTQ_K_POTRF_UPDATE, mHr, k + NB, k, mHr, k + NB, k,
                         Hr + static_cast<size_t>(k + NB) * d + k + NB, d, rest, rest, -1.0f,
                         1.0f, true, st, sa);
    }
    // inverse, block column kb, on stream B once panel kb is final
    GPTQ_CUDA(cudaStreamWaitEvent(sb, aux.ev[kb], 0));
    const int nbi = (d - k < NB) ? d - k : NB;
    GPTQ_LAUNCH(GPTQ_K_TRTRI_DIAG, sb, trsv_quad_kernel, (unsigned)QL, 128, trsv_smem, Hr, d, k, 1,
                LL, DI, st);
    // Y[c][k+t] = sum_j Y[c][k+j] DI[kb][t][j], rows c < k + nbi
    launch_gemm_tf32x3(GPTQ_K_TRTRI_DIAG, mS, 0, k, mDI, k, 0, S + k, d, k + nbi, nbi, 1.0f, 0.0f,
                       false, st, sb);
    if (rest > 0) {
      // Y[c][r] -= sum_j Y[c][k+j] L[r][k+j], c < k + NB <= r
      launch_gemm_tf32x3(GPTQ_K_TRTRI_UPDATE, mS, 0, k, mHr, k + NB, k, S + k + NB, d, k + NB,
                         rest, -1.0f, 1.0f, false, st, sb);
    }
  }
  GPTQ_CUDA(cudaEventRecord(aux.ev[nblk + 1], sb));
  GPTQ_CUDA(cudaStreamWaitEvent(s, aux.ev[nblk + 1], 0));
  GPTQ_CUDA(cudaEventRecord(aux.ev[nblk], sa));
  GPTQ_CUDA(cudaStreamWaitEvent(s, aux.ev[nblk], 0));
  {
    dim3 grid((unsigned)ceil_div(d, 32), (unsigned)ceil_div(d, 32));
    GPTQ_LAUNCH(GPTQ_K_PREP_REVERSE, s, reverse_transpose_kernel, grid, dim3(32, 8), 0, S, d, U);
  }
}

}  // namespace gptq
