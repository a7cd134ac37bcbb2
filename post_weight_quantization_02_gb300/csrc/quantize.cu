// gptq_quantize_layer kernels: permuted working copy of W, group fit, the column loop,
// packing and the loss sum (the lazy update's tensor-core kernel is in lazy_tc.cu).
//
// Method ("GPTQ Architecture, in depth", "The algorithm in code" and "Packing, tooling
// and serving"; "Same Ruler, Smarter Placement: GPTQ", sections 1.5 and 1.8):
//   for each block [i1, i2) of 128 columns in processing order:
//     for q in block: fit (s, z) at a group start on the current W[:, q:q+g];
//       code = clamp(round(w_q / s) + z, lowest, maxq); what = s (code - z);
//       e = (w_q - what) / U_qq; W[:, q+1:i2] -= e U[q, q+1:i2]; Err[:, q-i1] = e
//     W[:, i2:] -= Err U[i1:i2, i2:]          (the lazy update)
// The lazy update is deferred in two levels (same product, fewer passes over W): after a
// block only the rest of its 1024-column superblock, after the superblock every later
// column.  Layouts in the workspace: Wp [m][d] float32 (processing order), codesT [d][m]
// uint8 (column-major codes, so that a step's codes are one coalesced row), the
// superblock's errors as bf16 halves ehi/elo [1024][m] (e = hi + lo), U's bf16 halves
// [d][d], the loop's
// per-block layout of U, zeros [G][m] int32, loss_rows [m] float64 and pos [d] int32
// (the inverse permutation).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int BLK = 128;   // columns per block of the loop

// ---------------------------------------------------------------- permuted copy

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// 16 bytes of a row of W as float32 values (8 bf16 or 4 float32 elements).
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* v) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* v) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);             // bf16 -> float32 is exact
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

// Wp[r][k] = dead[perm[k]] ? 0 : W[r][perm[k]]; loss_rows[r] = 0.  One CTA per row: the
// source row is read with 16-byte loads into shared memory (dead columns zeroed there),
// then written in processing order with 16-byte stores (d is a multiple of 32; W and Wp
// are 16-byte aligned).
template <typename T>
__global__ void __launch_bounds__(256) gather_w_kernel(const T* __restrict__ W, int d,
                                                       const int32_t* __restrict__ perm,
                                                       const uint8_t* __restrict__ dead,
                                                       float* __restrict__ Wp,
                                                       double* __restrict__ loss_rows,
                                                       DevStatus* st) {
  extern __shared__ float srow[];
  constexpr int VN = Vec16<T>::N;
  const int r = blockIdx.x;
  const T* src = W + static_cast<size_t>(r) * d;
  bool bad = false;
  for (int j = threadIdx.x * VN; j < d; j += 256 * VN) {
    float v[VN];
    Vec16<T>::load(src + j, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) {
      bad |= !isfinite(v[i]);
      if (dead != nullptr && dead[j + i]) v[i] = 0.0f;
      srow[j + i] = v[i];
    }
  }
  if (bad) dev_fail(st, GPTQ_ERR_NONFINITE, r + 1);
  __syncthreads();
  float4* dst = reinterpret_cast<float4*>(Wp + static_cast<size_t>(r) * d);
  for (int k4 = threadIdx.x; k4 < d / 4; k4 += 256) {
    int4 p = make_int4(4 * k4, 4 * k4 + 1, 4 * k4 + 2, 4 * k4 + 3);
    if (perm != nullptr) {  // the caller's perm need not be 16-byte aligned
      const int32_t* pp = perm + 4 * k4;
      p = make_int4(pp[0], pp[1], pp[2], pp[3]);
    }
    dst[k4] = make_float4(srow[p.x], srow[p.y], srow[p.z], srow[p.w]);
  }
  if (threadIdx.x == 0) loss_rows[r] = 0.0;
}

// pos[perm[k]] = k; g_idx[c] = pos[c] / group (0 for group == -1), or c / group with
// static groups (fixed in the original order).
__global__ void gidx_kernel(const int32_t* __restrict__ perm, int d, int group, int static_groups,
                            int32_t* __restrict__ pos, int32_t* __restrict__ g_idx) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= d) return;
  const int c = perm ? perm[k] : k;
  pos[c] = k;
  g_idx[c] = (group == -1) ? 0 : (static_groups ? c : k) / group;
}

// ---------------------------------------------------------------- group fit

struct Grid {
  int bits;
  int sym;
  float maxq;
  float lowest;
  float zfix;
};

// w / s as the reciprocal product with one residual correction: within one ulp of the
// IEEE quotient (the two differ only where w / s sits on a rounding boundary of the
// quotient itself, far inside the near-tie band the parity check allows).
__device__ __forceinline__ float div_by_scale(float w, float s, float rs) {
  const float v0 = w * rs;
  const float r = fmaf(-v0, s, w);
  return fmaf(r, rs, v0);
}

// Scale and zero of one row of a group from its min / max (or max |w|), float32.
__device__ __forceinline__ void fit_from_range(const Grid& g, float mn, float mx, float amax,
                                               float& s, float& z) {
  if (g.sym) {
    s = fmaxf(__fdiv_rn(amax, static_cast<float>((1 << (g.bits - 1)) - 1)), 1e-8f);
    z = g.zfix;
  } else {
    const float lo = fminf(mn, 0.0f), hi = fmaxf(mx, 0.0f);
    s = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), g.maxq), 1e-8f);
    z = rintf(__fdiv_rn(-lo, s));
  }
}

// Fit on Wp[r][q0 : q0+len) for every row, one warp per row (warp-shuffle min / max).
// Used for groups wider than a block and for group = -1 (one group over the row).
__global__ void __launch_bounds__(256) fit_kernel(const float* __restrict__ Wp, int m, int d,
                                                  int q0, int len, Grid g, int gi,
                                                  float* __restrict__ scales,
                                                  int32_t* __restrict__ zeros) {
  const int r = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= m) return;
  const float* row = Wp + static_cast<size_t>(r) * d + q0;
  float mn = INFINITY, mx = -INFINITY, am = 0.0f;
  for (int j = lane; j < len; j += 32) {
    const float v = row[j];
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
    am = fmaxf(am, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  }
  if (lane == 0) {
    float s, z;
    fit_from_range(g, mn, mx, am, s, z);
    scales[static_cast<size_t>(gi) * m + r] = s;
    zeros[static_cast<size_t>(gi) * m + r] = static_cast<int32_t>(z);
  }
}

// Static groups ("GPTQ Architecture, in depth", "Groups, act-order and other knobs":
// groups fixed in the original order before permuting): scale and zero of every row and
// original group [gi*group, (gi+1)*group) from W after the dead fix, before the loop.
// One warp per row (warp-shuffle min / max).
template <typename T>
__global__ void __launch_bounds__(256) static_fit_kernel(const T* __restrict__ W,
                                                         const uint8_t* __restrict__ dead,
                                                         int m, int d, int group, Grid g,
                                                         float* __restrict__ scales,
                                                         int32_t* __restrict__ zeros) {
  const int r = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= m) return;
  const T* row = W + static_cast<size_t>(r) * d;
  const int G = (d + group - 1) / group;
  for (int gi = 0; gi < G; ++gi) {
    const int c1 = min(d, (gi + 1) * group);
    float mn = INFINITY, mx = -INFINITY, am = 0.0f;
    for (int c = gi * group + lane; c < c1; c += 32) {
      float v = ldf(row + c);
      if (dead != nullptr && dead[c]) v = 0.0f;
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
      am = fmaxf(am, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    }
    if (lane == 0) {
      float sc, z;
      fit_from_range(g, mn, mx, am, sc, z);
      scales[static_cast<size_t>(gi) * m + r] = sc;
      zeros[static_cast<size_t>(gi) * m + r] = static_cast<int32_t>(z);
    }
  }
}

// ---------------------------------------------------------------- the column loop

// 16-byte asynchronous global -> shared copy.
__device__ __forceinline__ void cp_async16(float4* dst, const float4* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// 4-byte asynchronous global -> shared copy.
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

// The column loop gives each output row LPR lanes; lane t holds the block's LW = 128 / LPR
// columns LW t .. LW t + LW - 1 in registers for the whole block.  Sub-block b (columns
// LW b ..) is quantised by lane b, column after column: the owner rounds its column,
// broadcasts the error e to the row's lanes, and every lane subtracts e U[q][c] from its
// columns (U is laid out with zeros at c <= q, so the same LW FMAs serve the owner, the
// lanes after it and, as no-ops, the lanes before it).  The owner forms its next column's
// value from its own e before the broadcast returns, which keeps the shuffle off the
// column chain.  The U rows are read with loads that the LPR lane positions share across
// the warp:
//   Ulay[b][q][t][j] = U[i1+q][i1+LW t+j] if q < LW t+j < nb else 0
// (j < LW, padded by 4 floats per lane position so the positions hit different banks),
// followed by the 128 reciprocals 1/U[i1+q][i1+q].
constexpr int LPR = kLoopLanesPerRow;          // lanes per row
constexpr int LW = BLK / LPR;                  // columns per lane
constexpr int LSTR = LW + 4;                   // padded lane stride
constexpr int UROW = LPR * LSTR;               // floats per row q of the layout
constexpr int kUlayFloats = BLK * UROW + BLK;
constexpr int LOOP_THREADS = 128;
constexpr int RPC = LOOP_THREADS / LPR;        // rows per CTA
static_assert(RPC % 16 == 0, "the loop's write-out stores 16 output rows per 16 bytes");
static_assert(kUlayFloats == kLoopUblkFloats, "workspace sizing of the loop's U layout");

__global__ void ulayout_kernel(const float* __restrict__ U, int d, float* __restrict__ Ulay) {
  const int b = blockIdx.x, q = blockIdx.y;
  const int i1 = b * BLK;
  const int nb = min(BLK, d - i1);
  float* out = Ulay + static_cast<size_t>(b) * kUlayFloats;
  const float* urow = U + static_cast<size_t>(i1 + (q < nb ? q : 0)) * d + i1;
  for (int e = threadIdx.x; e < UROW; e += blockDim.x) {
    const int t = e / LSTR, j = e % LSTR;
    const int c = LW * t + j;
    out[q * UROW + e] = (j < LW && q < nb && c > q && c < nb) ? urow[c] : 0.0f;
  }
  if (threadIdx.x == 0) out[BLK * UROW + q] = (q < nb) ? 1.0f / urow[q] : 1.0f;
}

struct LoopArgs {
  float* Wp;
  const float* Ulay;
  int m, d;
  int i1, nb;          // block start and width (nb <= 128)
  int group;           // in-kernel fit width (16, 32, 64 or 128), or 0: fitted outside
  int gi_outer;        // group index of the outside fit (group -1 or wide groups)
  int static_group;    // static groups: the group width (column q uses perm[q] / it), else 0
  const int32_t* perm; // processing order (static groups), may be null
  Grid g;
  float* scales;       // [G][m]
  int32_t* zeros;      // [G][m]
  uint8_t* codesT;     // [d][m]
  __nv_bfloat16* ehi;  // [128][m] rows of the superblock's [1024][m]: e = hi + lo, bf16
  __nv_bfloat16* elo;
  double* loss_rows;   // [m]
};

// Group fit at column J of the lane's window: over w[J .. J+group) when a group is
// narrower than the window, else over the whole window combined across the group's
// group / LW lanes (xor shuffles), masking columns past the block's end.
template <int J>
__device__ __forceinline__ void fit_lanes(const float (&w)[LW], int group, int t, int nb,
                                          const Grid& gr, float& s, float& z) {
  float mn = INFINITY, mx = -INFINITY, am = 0.0f;
  const int lo = (group < LW) ? J : 0, hi = (group < LW) ? J + group : LW;
#pragma unroll
  for (int i = 0; i < LW; ++i) {
    if (i >= lo && i < hi && LW * t + i < nb) {
      mn = fminf(mn, w[i]);
      mx = fmaxf(mx, w[i]);
      am = fmaxf(am, fabsf(w[i]));
    }
  }
#pragma unroll
  for (int o = 1; o < LPR; o <<= 1) {
    if (o * LW < group) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    }
  }
  fit_from_range(gr, mn, mx, am, s, z);
}

// One column q = LW b + J of sub-block b: fit at a group start, round the owner's value
// wq, broadcast e, update every lane's window.  The owner's code and error stay in
// registers (code_r[J], e_r[J]) until the sub-block ends, so a column is one branch-free
// stretch of code that the compiler can overlap with the next column's rounding.
// Returns the owner's next column value.
template <bool STATIC, int J>
__device__ __forceinline__ float loop_column(float (&w)[LW], float (&code_r)[LW],
                                             float (&e_r)[LW], float wq, int b, int t, int gb,
                                             bool active, int r, const LoopArgs& a,
                                             const float* __restrict__ ulay,
                                             const float* __restrict__ urinv,
                                             const float* __restrict__ szr, float& s,
                                             float& z, float& rs, float& loss) {
  const int q = LW * b + J;
  if constexpr (STATIC) {
    // static groups: this column's grid was fitted before the loop (scale, zero, 1/scale
    // of the row's group, staged per column)
    s = szr[q * RPC];
    z = szr[(BLK + q) * RPC];
    rs = szr[(2 * BLK + q) * RPC];
  } else if constexpr (J % 16 == 0) {
    // groups (16 .. 128 columns) start only at window positions that are multiples of 16
    if (a.group > 0 && (q % a.group) == 0) {
      fit_lanes<J>(w, a.group, t, a.nb, a.g, s, z);
      rs = __frcp_rn(s);
      wq = w[J];  // the fit saw the settled window
      if (active && t == b) {
        const int gi = (a.i1 + q) / a.group;
        a.scales[static_cast<size_t>(gi) * a.m + r] = s;
        a.zeros[static_cast<size_t>(gi) * a.m + r] = static_cast<int32_t>(z);
      }
    }
  }
  const float v = div_by_scale(wq, s, rs);
  const float code = fminf(fmaxf(rintf(v) + z, a.g.lowest), a.g.maxq);
  const float what = s * (code - z);
  const float e_own = (wq - what) * urinv[q];
  const float* u = ulay + q * UROW + t * LSTR;
  // the owner's next column from its own error (the broadcast update below computes the
  // same value with the same fma)
  float wnext = 0.0f;
  if constexpr (J + 1 < LW) wnext = fmaf(-e_own, u[J + 1], w[J + 1]);
  const float e = __shfl_sync(0xffffffffu, e_own, gb + b);
  code_r[J] = code;
  e_r[J] = e;
  loss = fmaf((t == b && q < a.nb) ? 0.5f * e : 0.0f, e, loss);
#pragma unroll
  for (int i = 0; i < LW; i += 4) {
    const float4 u4 = *reinterpret_cast<const float4*>(u + i);
    w[i] = fmaf(-e, u4.x, w[i]);
    w[i + 1] = fmaf(-e, u4.y, w[i + 1]);
    w[i + 2] = fmaf(-e, u4.z, w[i + 2]);
    w[i + 3] = fmaf(-e, u4.w, w[i + 3]);
  }
  return wnext;
}

template <bool STATIC, int J>
__device__ __forceinline__ void loop_columns(float (&w)[LW], float (&code_r)[LW],
                                             float (&e_r)[LW], float& wq, int b, int t, int gb,
                                             bool active, int r, const LoopArgs& a,
                                             const float* __restrict__ ulay,
                                             const float* __restrict__ urinv,
                                             const float* __restrict__ szr, float& s,
                                             float& z, float& rs, float& loss) {
  wq = loop_column<STATIC, J>(w, code_r, e_r, wq, b, t, gb, active, r, a, ulay, urinv, szr, s,
                              z, rs, loss);
  if constexpr (J + 1 < LW)
    loop_columns<STATIC, J + 1>(w, code_r, e_r, wq, b, t, gb, active, r, a, ulay, urinv, szr,
                                s, z, rs, loss);
}

// Shared memory of the loop: the U layout, the staging of codes and bf16 error halves,
// and with static groups the per-column scale, zero and reciprocal of each row.
constexpr int kLoopSmemDynamic = kUlayFloats * 4 + BLK * RPC * (1 + 2 + 2);
constexpr int kLoopSmemStatic = kLoopSmemDynamic + 3 * BLK * RPC * 4 + BLK * 4;

template <bool STATIC>
__global__ void __launch_bounds__(LOOP_THREADS) column_loop_kernel(const LoopArgs a) {
  extern __shared__ __align__(16) float smem_f[];
  const float* ulay = smem_f;
  const float* urinv = smem_f + BLK * UROW;
  // the block's codes and bf16 error halves, staged so that the global writes are whole
  // rows of RPC consecutive output rows
  uint8_t* codes_s = reinterpret_cast<uint8_t*>(smem_f + kUlayFloats);               // [128][RPC]
  __nv_bfloat16* ehi_s = reinterpret_cast<__nv_bfloat16*>(codes_s + BLK * RPC);      // [128][RPC]
  __nv_bfloat16* elo_s = ehi_s + BLK * RPC;                                          // [128][RPC]
  float* sz_s = reinterpret_cast<float*>(elo_s + BLK * RPC);  // static: [3][128][RPC], [128]
  const int i1 = a.i1, nb = a.nb;
  // the lazy update after this kernel is launched as its programmatic dependent: let it
  // set up while this block's loop runs (it waits for this grid before touching memory).
  // This kernel itself is an ordinary launch (launched as a dependent, its CTAs would
  // crowd onto the SMs a small update leaves free), so the wait returns at once.
  griddep_launch_dependents();
  griddep_wait();
  {
    const float4* src = reinterpret_cast<const float4*>(a.Ulay + static_cast<size_t>(i1 / BLK) * kUlayFloats);
    float4* dst = reinterpret_cast<float4*>(smem_f);
    for (int e = threadIdx.x; e < kUlayFloats / 4; e += blockDim.x) cp_async16(dst + e, src + e);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const int lane = threadIdx.x % 32;
  const int t = lane % LPR;
  const int gb = lane & ~(LPR - 1);
  const int rl = threadIdx.x / LPR;  // row within the CTA
  const int r = blockIdx.x * RPC + rl;
  const bool active = r < a.m;
  float w[LW];
  {
    const float* wrow = a.Wp + static_cast<size_t>(active ? r : 0) * a.d + i1 + LW * t;
#pragma unroll
    for (int j = 0; j < LW; j += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && LW * t + j < nb) v = *reinterpret_cast<const float4*>(wrow + j);
      w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
    }
  }
  float s = 1.0f, z = 0.0f;
  if constexpr (STATIC) {
    // each column's grid: the row's scale and zero of the original column's group.  The
    // columns' groups go to shared memory first (one load per thread), then every
    // thread gathers its row's scales and zeros with many loads in flight.
    static_assert(LOOP_THREADS == BLK && RPC == 32, "static-group staging layout");
    int* gcol_s = reinterpret_cast<int*>(sz_s + 3 * BLK * RPC);  // [128]
    {
      const int q = threadIdx.x;
      gcol_s[q] = (q < nb) ? (a.perm ? a.perm[i1 + q] : i1 + q) / a.static_group : 0;
    }
    __syncthreads();
    const int r0 = blockIdx.x * RPC;
    const int j = threadIdx.x % RPC;            // row within the CTA
    const bool row_ok = r0 + j < a.m;
    constexpr int QS = LOOP_THREADS / RPC;      // columns per pass
    // asynchronous 4-byte copies (the zero's int32 bits for now), in flight with the U
    // layout's; padding columns and rows take s = 1, z = 0
    for (int q = threadIdx.x / RPC; q < BLK; q += QS) {
      float* sd = sz_s + q * RPC + j;
      float* zd = sz_s + (BLK + q) * RPC + j;
      if (q < nb && row_ok) {
        const size_t o = static_cast<size_t>(gcol_s[q]) * a.m + r0 + j;
        cp_async4(sd, a.scales + o);
        cp_async4(zd, reinterpret_cast<const float*>(a.zeros + o));
      } else {
        *sd = 1.0f;
        *reinterpret_cast<int32_t*>(zd) = 0;
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  } else if (a.group == 0 && active) {
    s = a.scales[static_cast<size_t>(a.gi_outer) * a.m + r];
    z = static_cast<float>(a.zeros[static_cast<size_t>(a.gi_outer) * a.m + r]);
  }
  float rs = __frcp_rn(s);
  // the row's loss total so far, read now so that the read is off the block's tail
  const double loss_prev = (active && t == 0) ? a.loss_rows[r] : 0.0;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if constexpr (STATIC) {
    // zeros to float and the scales' reciprocals, in place
    for (int e = threadIdx.x; e < BLK * RPC; e += blockDim.x) {
      const float sv = sz_s[e];
      sz_s[BLK * RPC + e] = static_cast<float>(reinterpret_cast<const int32_t*>(sz_s)[BLK * RPC + e]);
      sz_s[2 * BLK * RPC + e] = __frcp_rn(sv);
    }
    __syncthreads();
  }
  // a block's share of the loss (at most 32 terms per lane) is summed in float32 and
  // added to the row's float64 total once per block; FP64 arithmetic inside the step
  // chain would serialise on this part's low FP64 rate
  float loss = 0.0f;
#pragma unroll 1
  for (int b = 0; b < LPR; ++b) {
    if (LW * b >= nb) break;
    // the owner's first column, settled by every earlier column's update
    float wq = w[0];
    float code_r[LW], e_r[LW];
    loop_columns<STATIC, 0>(w, code_r, e_r, wq, b, t, gb, active, r, a, ulay, urinv, sz_s + rl,
                            s, z, rs, loss);
    if (t == b) {
#pragma unroll
      for (int j = 0; j < LW; ++j) {
        const int q = LW * b + j;
        const __nv_bfloat16 eh = __float2bfloat16_rn(e_r[j]);
        codes_s[q * RPC + rl] = static_cast<uint8_t>(code_r[j]);
        ehi_s[q * RPC + rl] = eh;
        elo_s[q * RPC + rl] = __float2bfloat16_rn(e_r[j] - __bfloat162float(eh));
      }
    }
  }
  // each lane accumulated the loss of the columns it owns
  loss += __shfl_xor_sync(0xffffffffu, loss, 1);
  loss += __shfl_xor_sync(0xffffffffu, loss, 2);
  if (active && t == 0) a.loss_rows[r] = loss_prev + static_cast<double>(loss);
  __syncthreads();
  const int r0 = blockIdx.x * RPC;
  const int nrows = min(RPC, a.m - r0);
  if (nrows == RPC && a.m % 16 == 0) {
    // whole rows of RPC outputs, 16 bytes per store (every row start is 16-byte aligned)
    constexpr int CV = RPC / 16, EV = RPC / 8;
    for (int e = threadIdx.x; e < nb * CV; e += blockDim.x) {
      const int q = e / CV, v = e % CV;
      reinterpret_cast<uint4*>(a.codesT + static_cast<size_t>(i1 + q) * a.m + r0)[v] =
          reinterpret_cast<const uint4*>(codes_s + q * RPC)[v];
    }
    for (int e = threadIdx.x; e < nb * EV; e += blockDim.x) {
      const int q = e / EV, v = e % EV;
      reinterpret_cast<uint4*>(a.ehi + static_cast<size_t>(q) * a.m + r0)[v] =
          reinterpret_cast<const uint4*>(ehi_s + q * RPC)[v];
      reinterpret_cast<uint4*>(a.elo + static_cast<size_t>(q) * a.m + r0)[v] =
          reinterpret_cast<const uint4*>(elo_s + q * RPC)[v];
    }
  } else {
    for (int e = threadIdx.x; e < nb * RPC; e += blockDim.x) {
      const int q = e / RPC, j = e % RPC;
      if (j < nrows) {
        a.codesT[static_cast<size_t>(i1 + q) * a.m + r0 + j] = codes_s[e];
        a.ehi[static_cast<size_t>(q) * a.m + r0 + j] = ehi_s[e];
        a.elo[static_cast<size_t>(q) * a.m + r0 + j] = elo_s[e];
      }
    }
  }
}

// ---------------------------------------------------------------- packing

// Word `wi` of a little-endian bit stream whose value k is get(k) (bits wide).
template <typename Get>
__device__ __forceinline__ uint32_t stream_word(int wi, int bits, Get get) {
  const int b0 = wi * 32;
  const int k_first = b0 / bits, k_last = (b0 + 31) / bits;
  uint32_t word = 0;
  for (int k = k_first; k <= k_last; ++k) {
    const uint32_t v = get(k);
    const int shift = k * bits - b0;
    word |= (shift >= 0) ? (v << shift) : (v >> (-shift));
  }
  return word;
}

// qweight[wi][r]: codes of row r in original column order, packed along d.  A thread
// packs word wi of 16 consecutive rows: it reads each code row it needs (codesT[pos[k]]
// at those 16 rows) with one 16-byte load and writes the 16 words with four 16-byte
// stores (m is a multiple of 32; qweight is 16-byte aligned).
__global__ void pack_qweight_kernel(const uint8_t* __restrict__ codesT,
                                    const int32_t* __restrict__ pos, int m, int d, int bits,
                                    int32_t* __restrict__ qweight) {
  const int r0 = 16 * (blockIdx.x * blockDim.x + threadIdx.x);
  const int wi = blockIdx.y;
  if (r0 >= m) return;
  uint32_t word[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) word[j] = 0;
  const int b0 = wi * 32;
  const int k_first = b0 / bits, k_last = (b0 + 31) / bits;
  for (int k = k_first; k <= k_last && k < d; ++k) {
    const uint4 c = *reinterpret_cast<const uint4*>(codesT + static_cast<size_t>(pos[k]) * m + r0);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    const int shift = k * bits - b0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t v = (cw[j / 4] >> (8 * (j % 4))) & 0xFFu;
      word[j] |= (shift >= 0) ? (v << shift) : (v >> (-shift));
    }
  }
  uint4* out = reinterpret_cast<uint4*>(qweight + static_cast<size_t>(wi) * m + r0);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    out[q] = make_uint4(word[4 * q], word[4 * q + 1], word[4 * q + 2], word[4 * q + 3]);
}

// The same with 4-byte stores, for a qweight that is not 16-byte aligned.
__global__ void pack_qweight_unaligned_kernel(const uint8_t* __restrict__ codesT,
                                              const int32_t* __restrict__ pos, int m, int d,
                                              int bits, int32_t* __restrict__ qweight) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const int wi = blockIdx.y;
  if (r >= m) return;
  const uint32_t word = stream_word(wi, bits, [&](int k) -> uint32_t {
    return codesT[static_cast<size_t>(pos[k]) * m + r];
  });
  qweight[static_cast<size_t>(wi) * m + r] = static_cast<int32_t>(word);
}

// qzeros[gi][wi]: zero points of group gi packed along d_out.
__global__ void pack_qzeros_kernel(const int32_t* __restrict__ zeros, int m, int G, int bits,
                                   int32_t* __restrict__ qzeros) {
  const int nw = m * bits / 32;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= G * nw) return;
  const int gi = idx / nw, wi = idx % nw;
  const int32_t* zr = zeros + static_cast<size_t>(gi) * m;
  const uint32_t word = stream_word(wi, bits, [&](int k) -> uint32_t {
    return static_cast<uint32_t>(zr[k]);
  });
  qzeros[idx] = static_cast<int32_t>(word);
}

// *loss = sum of loss_rows in a fixed order (one CTA).
__global__ void __launch_bounds__(1024) loss_sum_kernel(const double* __restrict__ rows, int m,
                                                        double* __restrict__ loss) {
  __shared__ double part[1024];
  double s = 0.0;
  for (int r = threadIdx.x; r < m; r += 1024) s += rows[r];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = part[0];
}

}  // namespace

// ---------------------------------------------------------------- host side

void launch_quantize(const QuantArgs& q, cudaStream_t s) {
  const int m = q.m, d = q.d;
  Grid g;
  g.bits = q.bits;
  g.sym = q.sym;
  g.maxq = static_cast<float>((1 << q.bits) - 1);
  g.lowest = q.sym ? 1.0f : 0.0f;
  g.zfix = static_cast<float>(1 << (q.bits - 1));

  const bool stat = q.static_groups && q.group > 0;  // with group -1 both modes coincide
  GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gidx_kernel, (unsigned)ceil_div(d, 256), 256, 0, q.perm,
              d, q.group, stat ? 1 : 0, q.pos, q.g_idx);
  if (stat && m > 0) {
    // every group's grid, fitted before the loop on W after the dead fix (original order)
    if (q.w_bf16) {
      GPTQ_LAUNCH(GPTQ_K_QUANT_FIT, s, static_fit_kernel<__nv_bfloat16>, (unsigned)ceil_div(m, 8),
                  256, 0, static_cast<const __nv_bfloat16*>(q.W), q.dead, m, d, q.group, g,
                  q.scales, q.zeros);
    } else {
      GPTQ_LAUNCH(GPTQ_K_QUANT_FIT, s, static_fit_kernel<float>, (unsigned)ceil_div(m, 8), 256, 0,
                  static_cast<const float*>(q.W), q.dead, m, d, q.group, g, q.scales, q.zeros);
    }
  }
  if (m > 0) {
    const size_t row_smem = static_cast<size_t>(d) * sizeof(float);
    if (q.w_bf16) {
      ensure_dynamic_smem(gather_w_kernel<__nv_bfloat16>, static_cast<int>(row_smem));
      GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gather_w_kernel<__nv_bfloat16>, m, 256, row_smem,
                  static_cast<const __nv_bfloat16*>(q.W), d, q.perm, q.dead, q.Wp, q.loss_rows,
                  q.st);
    } else {
      ensure_dynamic_smem(gather_w_kernel<float>, static_cast<int>(row_smem));
      GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gather_w_kernel<float>, m, 256, row_smem,
                  static_cast<const float*>(q.W), d, q.perm, q.dead, q.Wp, q.loss_rows, q.st);
    }

    GPTQ_LAUNCH(GPTQ_K_QUANT_SPLIT, s, ulayout_kernel, dim3((unsigned)ceil_div(d, BLK), BLK), 128,
                0, q.U, d, q.Ublk);
    launch_usplit(q.U, d, q.uhi, q.ulo, s);
    const LazyMaps maps = make_lazy_maps(q.ehi, q.elo, kErrRows, q.uhi, q.ulo, q.Wp, m, d);
    ensure_dynamic_smem(column_loop_kernel<false>, kLoopSmemDynamic);
    ensure_dynamic_smem(column_loop_kernel<true>, kLoopSmemStatic);
    const bool inblock_fit = !stat && q.group > 0 && q.group <= BLK;
    // Deferred updates in two levels: superblocks of kErrRows columns, unless a group that
    // starts inside a superblock would reach past its end (its fit must see every earlier
    // block's update), in which case every block is its own superblock.
    const bool groups_nest = stat || q.group == -1 || q.group <= BLK ||
                             kErrRows % q.group == 0 || q.group % kErrRows == 0;
    const int sb_cols = groups_nest ? kErrRows : BLK;
    // The far update of superblock S (every later column) is one launch on the call's
    // stream over the whole GPU: on wide layers it is most of the update's work, and a
    // share of the SMs beside the next superblock's column loop left it on the critical
    // path.  Every W element receives its updates in the sequential order of the blocks.
    for (int s0 = 0; s0 < d; s0 += sb_cols) {
      const int s1 = (d - s0 < sb_cols) ? d : s0 + sb_cols;
      for (int i1 = s0; i1 < s1; i1 += BLK) {
        const int nb = (d - i1 < BLK) ? d - i1 : BLK;
        LoopArgs a;
        a.Wp = q.Wp;
        a.Ulay = q.Ublk;
        a.m = m;
        a.d = d;
        a.i1 = i1;
        a.nb = nb;
        a.group = inblock_fit ? q.group : 0;
        a.gi_outer = 0;
        a.static_group = stat ? q.group : 0;
        a.perm = q.perm;
        a.g = g;
        a.scales = q.scales;
        a.zeros = q.zeros;
        a.codesT = q.codesT;
        a.ehi = q.ehi + static_cast<size_t>(i1 - s0) * m;
        a.elo = q.elo + static_cast<size_t>(i1 - s0) * m;
        a.loss_rows = q.loss_rows;
        if (!inblock_fit && !stat) {
          const bool start = (q.group == -1) ? (i1 == 0) : (i1 % q.group == 0);
          const int gi = (q.group == -1) ? 0 : i1 / q.group;
          if (start) {
            const int len = (q.group == -1) ? d : ((d - i1 < q.group) ? d - i1 : q.group);
            GPTQ_LAUNCH(GPTQ_K_QUANT_FIT, s, fit_kernel, (unsigned)ceil_div(m, 8), 256, 0, q.Wp,
                        m, d, i1, len, g, gi, q.scales, q.zeros);
          }
          a.gi_outer = gi;
        }
        if (stat) {
          GPTQ_LAUNCH(GPTQ_K_QUANT_LOOP, s, column_loop_kernel<true>, (unsigned)ceil_div(m, RPC),
                      LOOP_THREADS, kLoopSmemStatic, a);
        } else {
          GPTQ_LAUNCH(GPTQ_K_QUANT_LOOP, s, column_loop_kernel<false>, (unsigned)ceil_div(m, RPC),
                      LOOP_THREADS, kLoopSmemDynamic, a);
        }
        // near: the rest of the superblock, W[:, i2:s1] -= Err_block U[i1:i2, i2:s1]
        if (i1 + nb < s1) launch_lazy_tc(maps, i1 - s0, i1, nb, i1 + nb, s1, q.st, s, 0);
      }
      if (s1 >= d) break;
      // far: every later column, W[:, s1:] -= Err_superblock U[s0:s1, s1:]
      launch_lazy_tc(maps, 0, s0, s1 - s0, s1, d, q.st, s, 0);
    }
    if (reinterpret_cast<uintptr_t>(q.qweight) % 16 == 0) {
      dim3 gq((unsigned)ceil_div(m, 16 * 64), static_cast<unsigned>(q.bits * d / 32));
      GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, pack_qweight_kernel, gq, 64, 0, q.codesT, q.pos, m, d,
                  q.bits, q.qweight);
    } else {
      dim3 gq((unsigned)ceil_div(m, 128), static_cast<unsigned>(q.bits * d / 32));
      GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, pack_qweight_unaligned_kernel, gq, 128, 0, q.codesT,
                  q.pos, m, d, q.bits, q.qweight);
    }
    const int nz = q.G * (m * q.bits / 32);
    GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, pack_qzeros_kernel, (unsigned)ceil_div(nz, 256), 256, 0,
                q.zeros, m, q.G, q.bits, q.qzeros);
  }
  GPTQ_LAUNCH(GPTQ_K_QUANT_LOSS, s, loss_sum_kernel, 1, 1024, 0, q.loss_rows, m, q.loss);
}

namespace {
// The checkpoint's fp16 copy of the scales: round to nearest, ties to even, as a
// checkpoint writer's float32 -> float16 conversion (overflow to inf, underflow to
// subnormals or zero).  Four scales per thread.
__global__ void scales_fp16_kernel(const float* __restrict__ s, int64_t n, __half* __restrict__ h) {
  const int64_t i = 4 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i + 3 < n && (reinterpret_cast<uintptr_t>(s) % 16) == 0 &&
      (reinterpret_cast<uintptr_t>(h) % 8) == 0) {
    const float4 v = *reinterpret_cast<const float4*>(s + i);
    __align__(8) __half o[4] = {__float2half_rn(v.x), __float2half_rn(v.y),
                                __float2half_rn(v.z), __float2half_rn(v.w)};
    *reinterpret_cast<uint2*>(h + i) = *reinterpret_cast<const uint2*>(o);
  } else {
    for (int64_t k = i; k < n && k < i + 4; ++k) h[k] = __float2half_rn(s[k]);
  }
}
}  // namespace

void launch_scales_fp16(const float* scales, int64_t n, uint16_t* out, cudaStream_t s) {
  if (n <= 0) return;
  const unsigned grid = static_cast<unsigned>((n + 4 * 256 - 1) / (4 * 256));
  GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, scales_fp16_kernel, grid, 256, 0, scales, n,
              reinterpret_cast<__half*>(out));
}

}  // namespace gptq
