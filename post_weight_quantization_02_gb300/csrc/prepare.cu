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
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;    // panel width of the blocked factorisation and inverse
constexpr int NBS = kSuperpanel;  // superpanel: panels whose update of later columns is grouped
// Superpanels pay off where the trailing matrix is large: below this width the prepare is
// a short latency chain, and the superpanel updates would lengthen it.
constexpr int kSuperpanelFrom = 8192;

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
  // four strided loads in flight per thread; the sum keeps the order j, j + 1024, ...
  for (int j0 = threadIdx.x; j0 < d; j0 += 4 * 1024) {
    float hv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q * 1024;
      hv[q] = (j < d) ? H[static_cast<size_t>(j) * d + j] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q * 1024;
      if (j >= d) break;
      const float h = hv[q];
      if (!isfinite(h)) dev_fail(st, GPTQ_ERR_NONFINITE, j + 1);
      const uint8_t is_dead = (h == 0.0f) ? 1 : 0;
      const float f = is_dead ? 1.0f : h;
      dead[j] = is_dead;
      diag_fixed[j] = f;
      s += static_cast<double>(f);
    }
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
// This is the stable descending order of "GPTQ > ActOrder" with ties by index.  One warp
// per j: the lanes count over interleaved k (coalesced reads of diag, which stays in L1)
// and the warp sums the counts.
__global__ void __launch_bounds__(256) prep_rank_kernel(const float* __restrict__ diag, int d,
                                                        int actorder, int32_t* __restrict__ perm) {
  const int j = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (j >= d) return;
  if (!actorder) {
    if (lane == 0) perm[j] = j;
    return;
  }
  const float dj = diag[j];
  unsigned cnt = 0;
  for (int k = lane; k < d; k += 32) {
    const float dk = diag[k];
    cnt += (dk > dj) || (dk == dj && k < j);
  }
  const unsigned rank = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) perm[rank] = j;
}

// ---------------------------------------------------------------- symmetric copy

// S[i][j] = H[min(i,j)][max(i,j)] (strict upper triangle of H is authoritative).
// 32x32 tiles, 256 threads; each thread moves one 16-byte piece of a row in and one out,
// and the lower half is read through a shared-memory transpose (row stride 33: the
// scalar stores and the transposed reads both hit 32 different banks).
__global__ void __launch_bounds__(256) prep_mirror_kernel(const float* __restrict__ H, int d,
                                                          float* __restrict__ S, DevStatus* st) {
  __shared__ float t[32][33];
  const int bi = blockIdx.y, bj = blockIdx.x;
  const int r = threadIdx.x / 8, c = (threadIdx.x % 8) * 4;
  // read the source tile (bi', bj') = upper one of (bi, bj) / (bj, bi)
  const int si = min(bi, bj), sj = max(bi, bj);
  {
    const int i = si * 32 + r, j = sj * 32 + c;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < d && j < d) {  // d is a multiple of 8: a row piece is whole or absent
      v = *reinterpret_cast<const float4*>(H + static_cast<size_t>(i) * d + j);
      const bool upper = i <= j + 3;  // some of the piece is on or above the diagonal
      if (upper && !(isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w))) {
        // only entries on or above the diagonal are authoritative
        const float e[4] = {v.x, v.y, v.z, v.w};
        for (int q = 0; q < 4; ++q)
          if (i <= j + q && !isfinite(e[q])) dev_fail(st, GPTQ_ERR_NONFINITE, 0);
      }
    }
    t[r][c] = v.x; t[r][c + 1] = v.y; t[r][c + 2] = v.z; t[r][c + 3] = v.w;
  }
  __syncthreads();
  const int i = bi * 32 + r, j = bj * 32 + c;
  if (i >= d || j >= d) return;
  float e[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int cc = c + q;
    if (bi < bj) e[q] = t[r][cc];
    else if (bi > bj) e[q] = t[cc][r];
    else e[q] = (r <= cc) ? t[r][cc] : t[cc][r];
  }
  *reinterpret_cast<float4*>(S + static_cast<size_t>(i) * d + j) = make_float4(e[0], e[1], e[2], e[3]);
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

// ------------------------------------------------------ diagonal block: factor, inverse

// One CTA of 512 threads factors the NB x NB diagonal block at (k, k) of A (lower) and
// writes the inverse of its factor, V = L_kk^-1, densely to DI[k/NB] (row-major, exact
// zeros above the diagonal, identity past a ragged end).  The factor itself stays in
// shared memory: the panel below it is solved against V by a GEMM, and the inverse of
// the whole factor is assembled from the V blocks.
//
// Factor, right-looking by 32-column sub-panels s (columns c0 = 32 s ..):
//   P1. warp 0 factors the 32 x 32 diagonal sub-block, lane = row, columns in registers.
//       Column c: l_cc = sqrt(p), l_rc = a_rc / l_cc, through one reciprocal square root
//       of the pivot p; the column is published in shared memory (ST[c][r] = l_rc,
//       ST[c][c] = 1/l_cc) and every row subtracts l_rc l_jc from its entries j > c.  The
//       next pivot only needs row c+1's own l_{c+1,c}, so it is formed first and the
//       broadcast stays off the pivot chain; the pivots are checked after the column loop.
//   P2. the rows below solve x S^T = a right-looking, one row per thread (x_c = acc_c /
//       l_cc, then acc_j -= x_c l_jc for j > c), and also store the solved panel
//       transposed (XT).
//   P3. the rank-32 update of the rest of the block, L[r][j] -= sum_t L[r][c0+t] L[j][c0+t]
//       (j <= r): one warp per 32 rows x 16 columns, lane = row; each lane holds its own
//       panel row in registers and the 16 columns' panel values are read from XT with
//       warp-wide broadcast loads.  With one sub-panel of look-ahead: the next sub-panel's
//       columns first (P3a), the columns after it (P3b) while warp 0 runs the next P1.
// Inverse, by 32 x 32 blocks (block indices), interleaved with the factor: V_ss = L_ss^-1
// (forward substitution, lane = column, on a spare warp next to P2) replaces L_ss, and
// then the row block V_sj = -V_ss sum_{t=j}^{s-1} L_st V_tj (j < s): each warp forms
// 32 x 16 of the sum in registers (own L row times broadcast V rows) on the spare warps
// beside P1(s), when every input is final, and leaves it in a private buffer; beside
// P2(s), V_sj = L_ss^-1 (-sum) is solved by forward substitution like V_ss itself.
// Shared memory (about 120 KB; the launch asks for a whole SM's worth so that the CTA runs
// alone on its SM): the staged block L, whose free upper 32 x 32 blocks hold the
// published columns; the six V_ij below the diagonal; XT; six private 32 x 16 buffers.
constexpr int DSTR = NB + 4;       // row stride of the staged block (16-byte rows)
constexpr int SB = 32;             // sub-panel width
constexpr int NSB = NB / SB;
constexpr int VSTR = SB + 4;       // row stride of an off-diagonal V block
constexpr int XSTR = NB - SB + 4;  // row stride of XT (up to 96 rows below a sub-panel)
constexpr int TBSTR = 16 + 4;      // row stride of a private 32 x 16 buffer
constexpr int NTB = 6;             // private buffers (inverse tasks of one step)
constexpr int kNVoff = NSB * (NSB - 1) / 2;
constexpr int kDiagSmemFloats = NB * DSTR + kNVoff * SB * VSTR + SB * XSTR + NTB * SB * TBSTR;

// the free upper block that holds sub-panel s's published columns
__device__ __forceinline__ float* st_slot(float* L, int s) {
  const int bi = s < 3 ? 0 : 1, bj = s < 3 ? s + 1 : 2;
  return L + (SB * bi) * DSTR + SB * bj;
}
__device__ __forceinline__ int voff_index(int i, int j) { return i * (i - 1) / 2 + j; }

// P3 task: rows r0 + lane, columns j0 .. j0 + 15 (entries j <= r) lose
// sum_t L[r][c0 + t] XT[t][j - (c0 + SB)].
__device__ __forceinline__ void rank32_task(float* L, const float* XT, int c0, int r0, int j0,
                                            int lane) {
  const int r = r0 + lane;
  float xr[SB];
  {
    const float* xrow = L + r * DSTR + c0;
#pragma unroll
    for (int t = 0; t < SB; t += 4) {
      const float4 v = *reinterpret_cast<const float4*>(xrow + t);
      xr[t] = v.x; xr[t + 1] = v.y; xr[t + 2] = v.z; xr[t + 3] = v.w;
    }
  }
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
  const float* xt = XT + (j0 - c0 - SB);
#pragma unroll
  for (int t = 0; t < SB; ++t) {
#pragma unroll
    for (int q = 0; q < 16; q += 4) {
      const float4 v = *reinterpret_cast<const float4*>(xt + t * XSTR + q);
      acc[q] = fmaf(xr[t], v.x, acc[q]);
      acc[q + 1] = fmaf(xr[t], v.y, acc[q + 1]);
      acc[q + 2] = fmaf(xr[t], v.z, acc[q + 2]);
      acc[q + 3] = fmaf(xr[t], v.w, acc[q + 3]);
    }
  }
  float* lrow = L + r * DSTR + j0;
#pragma unroll
  for (int q = 0; q < 16; q += 4) {
    float4 v = *reinterpret_cast<float4*>(lrow + q);
    if (j0 + q <= r) v.x -= acc[q];
    if (j0 + q + 1 <= r) v.y -= acc[q + 1];
    if (j0 + q + 2 <= r) v.z -= acc[q + 2];
    if (j0 + q + 3 <= r) v.w -= acc[q + 3];
    *reinterpret_cast<float4*>(lrow + q) = v;
  }
}

// Inverse row block s, first half (one warp, lane = row):
//   T_j[:, 16h .. 16h + 15] = sum_{t=j}^{s-1} L_st V_tj[:, same]
// (all of it final once sub-panel s - 1 is done, so it runs beside P1(s)), into the
// private buffer Tw of slot 2 j + h.  The second half, V_sj = L_ss^-1 (-T_j), is a
// forward substitution beside P2(s).
__device__ __forceinline__ void inv_sum_task(const float* L, const float* Voff, float* Tw, int s,
                                             int j, int h, int lane) {
  const int r = SB * s + lane;
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
  for (int tb = j; tb < s; ++tb) {
    const float* vb = (tb == j) ? L + (SB * j) * DSTR + SB * j + 16 * h
                                : Voff + voff_index(tb, j) * SB * VSTR + 16 * h;
    const int vs = (tb == j) ? DSTR : VSTR;
    float lv[SB];
    const float* lrow = L + r * DSTR + SB * tb;
#pragma unroll
    for (int t = 0; t < SB; t += 4) {
      const float4 v = *reinterpret_cast<const float4*>(lrow + t);
      lv[t] = v.x; lv[t + 1] = v.y; lv[t + 2] = v.z; lv[t + 3] = v.w;
    }
#pragma unroll
    for (int t = 0; t < SB; ++t) {
#pragma unroll
      for (int q = 0; q < 16; q += 4) {
        const float4 v = *reinterpret_cast<const float4*>(vb + t * vs + q);
        acc[q] = fmaf(lv[t], v.x, acc[q]);
        acc[q + 1] = fmaf(lv[t], v.y, acc[q + 1]);
        acc[q + 2] = fmaf(lv[t], v.z, acc[q + 2]);
        acc[q + 3] = fmaf(lv[t], v.w, acc[q + 3]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 16; q += 4)
    *reinterpret_cast<float4*>(Tw + lane * TBSTR + q) =
        make_float4(acc[q], acc[q + 1], acc[q + 2], acc[q + 3]);
}

__global__ void __launch_bounds__(512) chol_inv_diag_kernel(const float* __restrict__ A, int d,
                                                            int k, float* __restrict__ DI,
                                                            DevStatus* st, int32_t info_base) {
  extern __shared__ __align__(16) float smem_f[];
  float* L = smem_f;                  // [NB][DSTR]
  float* Voff = L + NB * DSTR;        // [6][SB][VSTR]
  float* XT = Voff + kNVoff * SB * VSTR;  // [SB][XSTR]
  float* Tbuf = XT + SB * XSTR;       // [NTB][SB][TBSTR]
  __shared__ int bad;
  griddep_launch_dependents();
  griddep_wait();
  const int nb = min(NB, d - k);  // a multiple of 8
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  // every load of the block in flight at once, with the status word
  constexpr int NLD = NB * NB / 4 / 512;
  float4 vin[NLD];
#pragma unroll
  for (int p = 0; p < NLD; ++p) {
    const int e4 = tid + p * 512, r = e4 / (NB / 4), c = (e4 % (NB / 4)) * 4;
    vin[p] = (r < nb && c < nb && c <= r)
                 ? *reinterpret_cast<const float4*>(A + static_cast<size_t>(k + r) * d + k + c)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (st->code != 0) return;
#pragma unroll
  for (int p = 0; p < NLD; ++p) {
    const int e4 = tid + p * 512, r = e4 / (NB / 4), c = (e4 % (NB / 4)) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nb && c < nb) {
      v = vin[p];
      if (c + 1 > r) v.y = 0.0f;
      if (c + 2 > r) v.z = 0.0f;
      if (c + 3 > r) v.w = 0.0f;
      if (c > r) v.x = 0.0f;
    } else if (r >= nb && r >= c && r < c + 4) {  // identity past a ragged end
      (&v.x)[r - c] = 1.0f;
    }
    *reinterpret_cast<float4*>(L + r * DSTR + c) = v;
  }
  if (tid == 0) bad = 0;
  __syncthreads();

  for (int s = 0; s < NSB; ++s) {
    const int c0 = s * SB;
    float* STs = st_slot(L, s);  // STs[c * DSTR + j] = l_{c0+j, c0+c} (j > c), 1/l_cc (j = c)
    // [A] P1(s) on warp 0; P3b of sub-panel s - 1 on the other warps
    if (warp == 0) {
      const float* lrow = L + (c0 + lane) * DSTR + c0;
      float w[SB];
#pragma unroll
      for (int j = 0; j < SB; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(lrow + j);
        w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
      }
      float il_own = 1.0f;
      float piv = __shfl_sync(0xffffffffu, w[0], 0);
#pragma unroll
      for (int c = 0; c < SB; ++c) {
        const float il = rsqrtf(piv);
        const float lc = (lane == c) ? piv * il : w[c] * il;
        if (lane == c) il_own = il;
        STs[c * DSTR + lane] = (lane > c) ? lc : ((lane == c) ? il : 0.0f);
        if (c + 1 < SB) piv = __shfl_sync(0xffffffffu, fmaf(-lc, lc, w[c + 1]), c + 1);
        __syncwarp();
#pragma unroll
        for (int j4 = ((c + 1) / 4) * 4; j4 < SB; j4 += 4) {
          const float4 v = *reinterpret_cast<const float4*>(STs + c * DSTR + j4);
          if (j4 > c) w[j4] = fmaf(-lc, v.x, w[j4]);
          if (j4 + 1 > c) w[j4 + 1] = fmaf(-lc, v.y, w[j4 + 1]);
          if (j4 + 2 > c) w[j4 + 2] = fmaf(-lc, v.z, w[j4 + 2]);
          if (j4 + 3 > c) w[j4 + 3] = fmaf(-lc, v.w, w[j4 + 3]);
        }
      }
      // a pivot that is not positive and finite gives a reciprocal root that is not either
      const unsigned badmask =
          __ballot_sync(0xffffffffu, !(il_own > 0.0f && il_own < INFINITY) && c0 + lane < nb);
      if (lane == 0 && badmask != 0u) {
        bad = 1;
        dev_fail(st, GPTQ_ERR_NOT_PD, info_base - (k + c0 + __ffs(badmask) - 1));
      }
    } else {
      // P3b of sub-panel s - 1 (rows and columns >= c0 + SB; its XT is still in place),
      // then the sums of the inverse's row block s, on warps 1 .. 15
      const int np3b = (s == 1) ? 6 : (s == 2) ? 2 : 0;
      for (int task = warp - 1; task < np3b + 2 * s; task += 15) {
        if (task < np3b) {
          int g = 0;
          while ((g + 1) * (g + 2) <= task) ++g;
          const int h = task - g * (g + 1);
          rank32_task(L, XT, c0 - SB, c0 + SB + SB * g, c0 + SB + 16 * h, lane);
        } else {
          const int it = task - np3b;  // slot 2 j + h
          inv_sum_task(L, Voff, Tbuf + it * SB * TBSTR, s, it / 2, it % 2, lane);
        }
      }
    }
    __syncthreads();
    if (bad) return;
    // [B] P2(s) on the threads of the rows below; V_ss and row block s of V beside it
    const int m2 = NB - c0 - SB;
    if (tid < m2) {
      float* xrow = L + (c0 + SB + tid) * DSTR + c0;
      float x[SB];
#pragma unroll
      for (int j = 0; j < SB; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(xrow + j);
        x[j] = v.x; x[j + 1] = v.y; x[j + 2] = v.z; x[j + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < SB; ++c) {
        const float* srow = STs + c * DSTR;
        const float xc = x[c] * srow[c];
        x[c] = xc;
#pragma unroll
        for (int j4 = ((c + 1) / 4) * 4; j4 < SB; j4 += 4) {
          const float4 v = *reinterpret_cast<const float4*>(srow + j4);
          if (j4 > c) x[j4] = fmaf(-xc, v.x, x[j4]);
          if (j4 + 1 > c) x[j4 + 1] = fmaf(-xc, v.y, x[j4 + 1]);
          if (j4 + 2 > c) x[j4 + 2] = fmaf(-xc, v.z, x[j4 + 2]);
          if (j4 + 3 > c) x[j4 + 3] = fmaf(-xc, v.w, x[j4 + 3]);
        }
      }
#pragma unroll
      for (int j = 0; j < SB; j += 4)
        *reinterpret_cast<float4*>(xrow + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
#pragma unroll
      for (int t = 0; t < SB; ++t) XT[t * XSTR + tid] = x[t];
    }
    // V_ss (warp 15) and the row block V_sj = L_ss^-1 (-T_j), j < s (one warp per j, on
    // the warps after P2's), by forward substitution with lane = column
    const int wv = m2 / SB;  // first warp after P2's
    const bool vss = (warp == 15);
    const bool vsj = (warp >= wv && warp < wv + s);
    if (vss || vsj) {
      const int j = warp - wv;
      const float* tcol = Tbuf + (2 * j + lane / 16) * SB * TBSTR + lane % 16;
      float y[SB];
#pragma unroll
      for (int t = 0; t < SB; ++t) y[t] = vss ? ((t == lane) ? 1.0f : 0.0f) : -tcol[t * TBSTR];
#pragma unroll
      for (int t = 0; t < SB; ++t) {
        const float* srow = STs + t * DSTR;
        const float yt = y[t] * srow[t];
        y[t] = yt;
#pragma unroll
        for (int j4 = ((t + 1) / 4) * 4; j4 < SB; j4 += 4) {
          const float4 v = *reinterpret_cast<const float4*>(srow + j4);
          if (j4 > t) y[j4] = fmaf(-yt, v.x, y[j4]);
          if (j4 + 1 > t) y[j4 + 1] = fmaf(-yt, v.y, y[j4 + 1]);
          if (j4 + 2 > t) y[j4 + 2] = fmaf(-yt, v.z, y[j4 + 2]);
          if (j4 + 3 > t) y[j4 + 3] = fmaf(-yt, v.w, y[j4 + 3]);
        }
      }
      // V_ss replaces L_ss; V_sj goes to its off-diagonal block
      float* vcol = vss ? L + c0 * DSTR + c0 + lane : Voff + voff_index(s, j) * SB * VSTR + lane;
      const int vstride = vss ? DSTR : VSTR;
#pragma unroll
      for (int t = 0; t < SB; ++t) vcol[t * vstride] = y[t];
    }
    __syncthreads();
    // [C] P3a(s): columns c0 + SB .. c0 + 2 SB, rows below
    const int n3a = (s < NSB - 1) ? 2 * (NSB - 1 - s) : 0;
    for (int task = warp; task < n3a; task += 16)
      rank32_task(L, XT, c0, c0 + SB + SB * (task / 2), c0 + SB + 16 * (task % 2), lane);
    __syncthreads();
  }

  float* dout = DI + static_cast<size_t>(k / NB) * NB * NB;
#pragma unroll
  for (int p = 0; p < NB * NB / 4 / 512; ++p) {
    const int e4 = tid + p * 512, r = e4 / (NB / 4), c = (e4 % (NB / 4)) * 4;
    const int bi = r / SB, bj = c / SB;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bi == bj) {
      v = *reinterpret_cast<const float4*>(L + r * DSTR + c);
    } else if (bi > bj) {
      v = *reinterpret_cast<const float4*>(Voff + voff_index(bi, bj) * SB * VSTR +
                                           (r % SB) * VSTR + c % SB);
    }
    *reinterpret_cast<float4*>(dout + r * NB + c) = v;
  }
}

// S = I (the right-hand side of L X = I; updates accumulate into it).
__global__ void identity_kernel(float* __restrict__ S, int d) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < d) S[static_cast<size_t>(i) * d + j] = (i == j) ? 1.0f : 0.0f;
}

// U[i][j] = X[d-1-i][d-1-j] = Y[d-1-j][d-1-i] for j >= i, 0 below the diagonal.  64x64
// tiles transposed through shared memory with 16-byte global accesses (d a multiple of 8,
// so a 4-float piece is wholly inside the matrix or wholly outside): tile row jj reads
// Y[d-1-(j0+jj)] at columns d-64-i0 .. d-1-i0, which hold i = i0+63 .. i0 in reverse.
__global__ void __launch_bounds__(256) reverse_transpose_kernel(const float* __restrict__ Y,
                                                                int d, float* __restrict__ U) {
  __shared__ float t[64][65];  // t[j - j0][i - i0]
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  const bool below = j0 + 63 < i0;  // a tile of zeros: nothing to read
  if (!below) {
    const int cbase = d - 64 - i0;
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      const int jj = e / 16, k = e % 16;
      const int j = j0 + jj, c = cbase + 4 * k;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < d && c >= 0)
        v = *reinterpret_cast<const float4*>(Y + static_cast<size_t>(d - 1 - j) * d + c);
      const int ii = d - 1 - i0 - c;  // the tile column of v.x; v.y .. v.w go down from it
      if (ii < 64) t[jj][ii] = v.x;
      if (ii - 1 >= 0 && ii - 1 < 64) t[jj][ii - 1] = v.y;
      if (ii - 2 >= 0 && ii - 2 < 64) t[jj][ii - 2] = v.z;
      if (ii - 3 >= 0 && ii - 3 < 64) t[jj][ii - 3] = v.w;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * 16; e += 256) {
    const int ii = e / 16, k = e % 16;
    const int i = i0 + ii, j = j0 + 4 * k;
    if (i >= d || j >= d) continue;
    float4 v;
    v.x = (!below && j >= i) ? t[4 * k][ii] : 0.0f;
    v.y = (!below && j + 1 >= i) ? t[4 * k + 1][ii] : 0.0f;
    v.z = (!below && j + 2 >= i) ? t[4 * k + 2][ii] : 0.0f;
    v.w = (!below && j + 3 >= i) ? t[4 * k + 3][ii] : 0.0f;
    *reinterpret_cast<float4*>(U + static_cast<size_t>(i) * d + j) = v;
  }
}

}  // namespace

void launch_prepare(const float* H, int d, float damp, int actorder, int32_t* perm,
                    uint8_t* dead, float* U, float* S, float* Hr, float* diag_fixed,
                    float* lam, float* DI, float* Lo, DevStatus* st, cudaStream_t s) {
  GPTQ_LAUNCH(GPTQ_K_PREP_DIAG, s, prep_diag_kernel, 1, 1024, 0, H, d, damp, dead, diag_fixed,
              lam, st);
  GPTQ_LAUNCH(GPTQ_K_PREP_RANK, s, prep_rank_kernel, (unsigned)ceil_div(d, 8), 256, 0,
              diag_fixed, d, actorder, perm);
  const unsigned t32 = (unsigned)ceil_div(d, 32);
  GPTQ_LAUNCH(GPTQ_K_PREP_MIRROR, s, prep_mirror_kernel, dim3(t32, t32), 256, 0, H, d, S, st);
  const size_t row_smem = static_cast<size_t>(d) * sizeof(float);
  ensure_dynamic_smem(prep_gather_kernel, static_cast<int>(row_smem));
  GPTQ_LAUNCH(GPTQ_K_PREP_GATHER, s, prep_gather_kernel, d, 256, row_smem, S, d, perm, dead, lam,
              Hr);

  // Cholesky of Hr (lower, in place) by NB-wide panels, right-looking with one panel of
  // look-ahead, the panels grouped into superpanels of nbs columns (NBS on wide layers,
  // the whole matrix below kSuperpanelFrom).  Stream A carries the critical chain: factor
  // and invert the diagonal block, solve the panel below it, apply the panel's update to
  // the next block column only (the near update).  Stream C applies the rest of the
  // panel's update inside its superpanel (the far update) behind it.  Ordering: block
  // column kb is final once the near update of kb - 1 (stream A, in order) and the far
  // update of kb - 2 have run; the near update of kb writes block column kb + 1, which the
  // far update of kb - 1 also writes, so it waits for that one.  At a superpanel's end its
  // panels' update of every later column is applied at once (K = the superpanel's width):
  // the next superpanel's columns on stream A, the rest on stream C, each after the
  // previous superpanel's far update that wrote the same columns.  A failing pivot at
  // reversed position a reports processing position d - a (1-based).
  //
  // Stream B inverts the factor meanwhile: block column kb of the inverse needs only L's
  // first kb + 1 block columns, so it runs as soon as panel kb is final.  The inverse
  // X = L^-1 is kept transposed as Y = X^T in S so that both GEMM operands are K-major:
  // block column i of Y is Y[:, i] = R DI[i]^T (R = the accumulated right-hand side,
  // initially I), after which every later block column loses Y[:, i] L[r, i]^T (inside
  // the superpanel per panel, past it once per superpanel).  Finally U = J X J =
  // (J Y J)^T.
  // The diagonal block's CTA asks for all of an SM's shared memory, so that no GEMM CTA
  // of the other streams shares its SM: its chain of dependent steps runs about 15 %
  // slower beside one.
  // (the block's limit covers its static shared memory too)
  int dev = 0, smem_optin = 0;
  GPTQ_CUDA(cudaGetDevice(&dev));
  GPTQ_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  cudaFuncAttributes diag_attr;
  GPTQ_CUDA(cudaFuncGetAttributes(&diag_attr, chol_inv_diag_kernel));
  const int diag_smem = std::max(kDiagSmemFloats * static_cast<int>(sizeof(float)),
                                 smem_optin - static_cast<int>(diag_attr.sharedSizeBytes));
  ensure_dynamic_smem(chol_inv_diag_kernel, diag_smem);
  CUtensorMap mHr, mS, mDI, mLo[2];
  make_gemm_map(&mHr, Hr, d, d, d);
  make_gemm_map(&mS, S, d, d, d);
  make_gemm_map(&mDI, DI, static_cast<int>(ceil_div(d, NB)) * NB, NB, NB);
  // lo parts (x - tf32(x)) of a superpanel's columns, two buffers [d][NBS] that
  // alternate between superpanels: rows past the superpanel from L (Hr), rows before it
  // from the inverse (S)
  for (int b = 0; b < 2; ++b) make_gemm_map(&mLo[b], Lo + static_cast<size_t>(b) * d * NBS, d, NBS, NBS);
  const int nblk = static_cast<int>(ceil_div(d, NB));
  // superpanel width: NBS on wide layers, the whole matrix (no superpanel updates) below
  const int nbs = (d >= kSuperpanelFrom) ? NBS : static_cast<int>(ceil_div(d, NB)) * NB;
  const int nsp = static_cast<int>(ceil_div(d, nbs));
  AuxStreams& aux = aux_streams(2 * nblk + 3 * nsp + 3);
  cudaStream_t sa = aux.a, sb = aux.b, sc = aux.c;
  cudaEvent_t* ev_panel = aux.ev.data();             // [nblk] panel kb factored and solved
  cudaEvent_t* ev_far = ev_panel + nblk;             // [nblk] panel kb's far update applied
  cudaEvent_t* ev_spfar = ev_far + nblk;             // [nsp] superpanel's far update applied
  cudaEvent_t* ev_lo = ev_spfar + nsp;               // [nsp] its lo parts of L written
  cudaEvent_t* ev_sptri = ev_lo + nsp;               // [nsp] its inverse update applied
  cudaEvent_t ev_fork = ev_sptri[nsp], ev_b = ev_sptri[nsp + 1], ev_c = ev_sptri[nsp + 2];
  std::vector<char> far_done(nblk, 0), spfar_done(nsp, 0), sptri_done(nsp, 0);
  GPTQ_CUDA(cudaEventRecord(ev_fork, s));
  GPTQ_CUDA(cudaStreamWaitEvent(sa, ev_fork, 0));
  GPTQ_CUDA(cudaStreamWaitEvent(sb, ev_fork, 0));
  GPTQ_CUDA(cudaStreamWaitEvent(sc, ev_fork, 0));
  {
    // S = I on stream B, where the inverse needs it first (the gather has read S)
    dim3 grid((unsigned)ceil_div(d, 256), d);
    GPTQ_LAUNCH(GPTQ_K_TRTRI_UPDATE, sb, identity_kernel, grid, 256, 0, S, d);
  }
  for (int kb = 0; kb < nblk; ++kb) {
    const int k = kb * NB;
    const int rest = d - k - NB;
    const int sp = k / nbs;
    const int sp0 = sp * nbs;                              // this panel's superpanel
    const int sp_end = (d - sp0 < nbs) ? d : sp0 + nbs;
    const int in_sp = sp_end - (k + NB);                   // its columns after this panel
    // Block column kb is complete once the near update of panel kb - 1 is (that update
    // waited for the far update of panel kb - 2, the last panel-level update of block
    // column kb), and, for the first panel of a superpanel, once the near update of the
    // previous superpanel is (which waited for the far update of the one before it).
    // The factor's critical chain (diagonal block, panel solve, near update) runs on
    // stream A as programmatic dependents, each launched during the kernel before it.
    GPTQ_LAUNCH_PDL(GPTQ_K_POTRF_PANEL, sa, chol_inv_diag_kernel, 1, 512, diag_smem, Hr, d, k,
                    DI, st, d);
    if (rest > 0) {
      // the panel below, in place: L[r, k:k+NB] = A[r, k:k+NB] L_kk^-T (rows r >= k + NB;
      // each CTA owns whole rows, loaded before it writes them)
      launch_gemm_tf32x3(GPTQ_K_POTRF_TRSM, mHr, k + NB, k, mDI, k, 0, NB,
                         Hr + static_cast<size_t>(k + NB) * d + k, d, rest, NB, 1.0f, 0.0f,
                         false, st, sa, true);
    }
    if (in_sp > 0) {
      // near update, block column kb + 1 (inside the superpanel), every row below it:
      // Hr[r][k+NB+j] -= L[r, panel] . L[k+NB+j, panel] (whole tiles; the entries it
      // changes above the diagonal are never read).  It adds into block column kb + 1
      // after the far update of panel kb - 1 has, so that every entry receives its
      // updates in panel order.
      if (kb >= 1 && far_done[kb - 1]) GPTQ_CUDA(cudaStreamWaitEvent(sa, ev_far[kb - 1], 0));
      launch_gemm_tf32x3(GPTQ_K_POTRF_UPDATE, mHr, k + NB, k, mHr, k + NB, k, NB,
                         Hr + static_cast<size_t>(k + NB) * d + k + NB, d, rest,
                         in_sp < NB ? in_sp : NB, -1.0f, 1.0f, false, st, sa, true);
    }
    // panel kb is final (recorded after the near update, which keeps this stream's
    // kernel-to-kernel steps free of other stream operations where it can)
    GPTQ_CUDA(cudaEventRecord(ev_panel[kb], sa));
    if (in_sp > NB) {
      // far update inside the superpanel, on stream C: block columns kb + 2 .. its end,
      // every row below them (the triangle of those columns and whole rows beneath)
      GPTQ_CUDA(cudaStreamWaitEvent(sc, ev_panel[kb], 0));
      launch_gemm_tf32x3(GPTQ_K_POTRF_UPDATE, mHr, k + 2 * NB, k, mHr, k + 2 * NB, k, NB,
                         Hr + static_cast<size_t>(k + 2 * NB) * d + k + 2 * NB, d, rest - NB,
                         in_sp - NB, -1.0f, 1.0f, true, st, sc, false);
      GPTQ_CUDA(cudaEventRecord(ev_far[kb], sc));
      far_done[kb] = 1;
    }
    const bool sp_last = (k + NB >= sp_end);
    if (sp_last && sp_end < d) {
      // The superpanel's panels are factored and solved: every later column receives the
      // superpanel's update at once, A[r][c] -= L[r, sp] . L[c, sp] with K = its width (the
      // same sum as one update per panel, grouped).  The next superpanel's columns (every
      // row below them) on stream A, which that superpanel's panels need next; the columns
      // past it on stream C.  Each adds into columns that the previous superpanel's far
      // update also wrote, after it.
      const int spw = sp_end - sp0;
      const int nxt = (d - sp_end < nbs) ? d - sp_end : nbs;
      const int lb = sp % 2;  // this superpanel's lo buffer
      float* lo = Lo + static_cast<size_t>(lb) * d * NBS;
      // the lo parts of L[sp_end:, sp] (final since the last panel solve); the buffer was
      // last read by the far and inverse updates of superpanel sp - 2 (the far one is
      // already ordered before this stream by the wait below of sp - 1's near update)
      if (sp >= 2 && sptri_done[sp - 2]) GPTQ_CUDA(cudaStreamWaitEvent(sa, ev_sptri[sp - 2], 0));
      if (sp >= 1 && spfar_done[sp - 1]) GPTQ_CUDA(cudaStreamWaitEvent(sa, ev_spfar[sp - 1], 0));
      launch_split_lo(Hr + static_cast<size_t>(sp_end) * d + sp0, d, d - sp_end, spw,
                      lo + static_cast<size_t>(sp_end) * NBS, NBS, sa);
      GPTQ_CUDA(cudaEventRecord(ev_lo[sp], sa));
      launch_gemm_tf32x3_presplit(GPTQ_K_POTRF_UPDATE, mHr, sp_end, sp0, mLo[lb], sp_end, 0, mHr,
                                  sp_end, sp0, mLo[lb], sp_end, 0, spw,
                                  Hr + static_cast<size_t>(sp_end) * d + sp_end, d, d - sp_end,
                                  nxt, -1.0f, 1.0f, true, st, sa, false);
      const int far = d - sp_end - nxt;
      if (far > 0) {
        GPTQ_CUDA(cudaStreamWaitEvent(sc, ev_lo[sp], 0));
        launch_gemm_tf32x3_presplit(GPTQ_K_POTRF_UPDATE, mHr, sp_end + nxt, sp0, mLo[lb],
                                    sp_end + nxt, 0, mHr, sp_end + nxt, sp0, mLo[lb], sp_end + nxt,
                                    0, spw, Hr + static_cast<size_t>(sp_end + nxt) * d + sp_end + nxt,
                                    d, far, far, -1.0f, 1.0f, true, st, sc, false);
        GPTQ_CUDA(cudaEventRecord(ev_spfar[sp], sc));
        spfar_done[sp] = 1;
      }
    }
    // inverse, block column kb, on stream B once panel kb is final
    GPTQ_CUDA(cudaStreamWaitEvent(sb, ev_panel[kb], 0));
    const int nbi = (d - k < NB) ? d - k : NB;
    // Y[c][k+t] = sum_j Y[c][k+j] DI[kb][t][j], rows c < k + nbi
    launch_gemm_tf32x3(GPTQ_K_TRTRI_DIAG, mS, 0, k, mDI, k, 0, NB, S + k, d, k + nbi, nbi, 1.0f,
                       0.0f, false, st, sb, false);
    if (in_sp > 0) {
      // Y[c][r] -= sum_j Y[c][k+j] L[r][k+j], c < k + NB <= r < the superpanel's end
      launch_gemm_tf32x3(GPTQ_K_TRTRI_UPDATE, mS, 0, k, mHr, k + NB, k, NB, S + k + NB, d,
                         k + NB, in_sp, -1.0f, 1.0f, false, st, sb, false);
    }
    if (sp_last && sp_end < d) {
      // the superpanel's share at once: Y[c][r] -= sum_{j in sp} Y[c][j] L[r][j],
      // c < sp_end <= r (rows c past a block column's end hold exact zeros there).  The
      // lo parts of Y[:sp_end, sp] go to rows 0 .. sp_end of the superpanel's buffer, once
      // the far update of superpanel sp - 2, which read those rows, is done; the lo parts
      // of L come from stream A.
      const int lb = sp % 2;
      float* lo = Lo + static_cast<size_t>(lb) * d * NBS;
      if (sp >= 2 && spfar_done[sp - 2]) GPTQ_CUDA(cudaStreamWaitEvent(sb, ev_spfar[sp - 2], 0));
      launch_split_lo(S + sp0, d, sp_end, sp_end - sp0, lo, NBS, sb);
      GPTQ_CUDA(cudaStreamWaitEvent(sb, ev_lo[sp], 0));
      launch_gemm_tf32x3_presplit(GPTQ_K_TRTRI_UPDATE, mS, 0, sp0, mLo[lb], 0, 0, mHr, sp_end, sp0,
                                  mLo[lb], sp_end, 0, sp_end - sp0, S + sp_end, d, sp_end,
                                  d - sp_end, -1.0f, 1.0f, false, st, sb, false);
      GPTQ_CUDA(cudaEventRecord(ev_sptri[sp], sb));
      sptri_done[sp] = 1;
    }
  }
  GPTQ_CUDA(cudaEventRecord(ev_b, sb));
  GPTQ_CUDA(cudaStreamWaitEvent(s, ev_b, 0));
  GPTQ_CUDA(cudaEventRecord(ev_c, sc));
  GPTQ_CUDA(cudaStreamWaitEvent(s, ev_c, 0));
  GPTQ_CUDA(cudaEventRecord(ev_fork, sa));
  GPTQ_CUDA(cudaStreamWaitEvent(s, ev_fork, 0));
  {
    dim3 grid((unsigned)ceil_div(d, 64), (unsigned)ceil_div(d, 64));
    GPTQ_LAUNCH(GPTQ_K_PREP_REVERSE, s, reverse_transpose_kernel, grid, 256, 0, S, d, U);
  }
}

}  // namespace gptq
