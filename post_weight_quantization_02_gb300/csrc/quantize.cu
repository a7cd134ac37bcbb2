// gptq_quantize_layer kernels: permuted working copy of W, group fit, the resident-block
// column loop, the lazy trailing update (float32 FMA path), packing and the loss sum.
//
// Method ("GPTQ Architecture, in depth", "The algorithm in code" and "Packing, tooling
// and serving"; "Same Ruler, Smarter Placement: GPTQ", sections 1.5 and 1.8):
//   for each block [i1, i2) of 128 columns in processing order:
//     for q in block: fit (s, z) at a group start on the current W[:, q:q+g];
//       code = clamp(round(w_q / s) + z, lowest, maxq); what = s (code - z);
//       e = (w_q - what) / U_qq; W[:, q+1:i2] -= e U[q, q+1:i2]; Err[:, q-i1] = e
//     W[:, i2:] -= Err U[i1:i2, i2:]          (the lazy update)
// Layouts in the workspace: Wp [m][d] float32 (processing order), codesT [d][m] uint8
// (column-major codes, so that a step's codes are one coalesced row), ErrT [128][m]
// float32, zeros [G][m] int32, loss_rows [m] float64, pos [d] int32 (inverse perm).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"

namespace gptq {

namespace {

constexpr int BLK = 128;   // columns per block of the loop
constexpr int CHUNK = 16;  // columns per register-shift chunk

// ---------------------------------------------------------------- permuted copy

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// Wp[r][k] = dead[perm[k]] ? 0 : W[r][perm[k]]; loss_rows[r] = 0.  One CTA per row,
// the source row staged in shared memory.
template <typename T>
__global__ void __launch_bounds__(256) gather_w_kernel(const T* __restrict__ W, int d,
                                                       const int32_t* __restrict__ perm,
                                                       const uint8_t* __restrict__ dead,
                                                       float* __restrict__ Wp,
                                                       double* __restrict__ loss_rows,
                                                       DevStatus* st) {
  extern __shared__ float srow[];
  const int r = blockIdx.x;
  const T* src = W + static_cast<size_t>(r) * d;
  bool bad = false;
  for (int j = threadIdx.x; j < d; j += 256) {
    float v = ldf(src + j);
    bad |= !isfinite(v);
    if (dead != nullptr && dead[j]) v = 0.0f;
    srow[j] = v;
  }
  if (bad) dev_fail(st, GPTQ_ERR_NONFINITE, r + 1);
  __syncthreads();
  float* dst = Wp + static_cast<size_t>(r) * d;
  for (int k = threadIdx.x; k < d; k += 256) dst[k] = srow[perm ? perm[k] : k];
  if (threadIdx.x == 0) loss_rows[r] = 0.0;
}

// pos[perm[k]] = k; g_idx[c] = pos[c] / group (0 for group == -1).
__global__ void gidx_kernel(const int32_t* __restrict__ perm, int d, int group,
                            int32_t* __restrict__ pos, int32_t* __restrict__ g_idx) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= d) return;
  const int c = perm ? perm[k] : k;
  pos[c] = k;
  g_idx[c] = (group == -1) ? 0 : k / group;
}

// ---------------------------------------------------------------- group fit

struct Grid {
  int bits;
  int sym;
  float maxq;
  float lowest;
  float zfix;
};

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

// ---------------------------------------------------------------- the column loop

// 4-byte asynchronous global -> shared copy; with valid == false it writes zero and
// reads nothing.
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}

struct LoopArgs {
  float* Wp;
  const float* U;
  int m, d;
  int i1, nb;          // block start and width (nb <= 128)
  int group;           // in-kernel fit width (16, 32, 64 or 128), or 0: fitted outside
  int gi_outer;        // group index of the outside fit (group 0 == -1 or wide groups)
  Grid g;
  float* scales;       // [G][m]
  int32_t* zeros;      // [G][m]
  uint8_t* codesT;     // [d][m]
  float* errT;         // [128][m]
  double* loss_rows;   // [m]
};

// Fit over the first `width` live columns of the rolling row (static width).
template <int WIDTH>
__device__ __forceinline__ void fit_regs(const float (&w)[BLK], int live, const Grid& g,
                                         float& s, float& z) {
  float mn = INFINITY, mx = -INFINITY, am = 0.0f;
#pragma unroll
  for (int j = 0; j < WIDTH; ++j) {
    if (j < live) {
      mn = fminf(mn, w[j]);
      mx = fmaxf(mx, w[j]);
      am = fmaxf(am, fabsf(w[j]));
    }
  }
  fit_from_range(g, mn, mx, am, s, z);
}

// One chunk of 16 columns.  On entry w[0] is column q0 = 16*C of the block and the row's
// live columns are w[0 .. nb-q0); each step quantises w[0], then writes the compensated
// later columns one slot down (w[j] <- w[j+1] - e u_{q, q+1+j}), so that w[0] is always
// the next column and every register index is static.
template <int C>
__device__ __forceinline__ void loop_chunk(float (&w)[BLK], const float (*ush)[BLK],
                                           const float* udiag, const LoopArgs& a, int r,
                                           bool active, float& s, float& z, double& loss) {
  constexpr int LEN = BLK - C * CHUNK;
  const int q0 = C * CHUNK;
  if (q0 >= a.nb) return;
  if (a.group > 0 && (q0 % a.group) == 0) {
    const int live = a.nb - q0;
    const int gi = (a.i1 + q0) / a.group;
    if (a.group == 16) fit_regs<(LEN < 16 ? LEN : 16)>(w, live, a.g, s, z);
    else if (a.group == 32) fit_regs<(LEN < 32 ? LEN : 32)>(w, live, a.g, s, z);
    else if (a.group == 64) fit_regs<(LEN < 64 ? LEN : 64)>(w, live, a.g, s, z);
    else fit_regs<LEN>(w, live, a.g, s, z);
    if (active) {
      a.scales[static_cast<size_t>(gi) * a.m + r] = s;
      a.zeros[static_cast<size_t>(gi) * a.m + r] = static_cast<int32_t>(z);
    }
  }
  const int steps = min(CHUNK, a.nb - q0);
#pragma unroll 1
  for (int t = 0; t < steps; ++t) {
    const int q = q0 + t;
    const float wq = w[0];
    const float v = __fdiv_rn(wq, s);
    const float code = fminf(fmaxf(rintf(v) + z, a.g.lowest), a.g.maxq);
    const float what = s * (code - z);
    const float e = __fdiv_rn(wq - what, udiag[q]);
    if (active) {
      a.codesT[static_cast<size_t>(a.i1 + q) * a.m + r] = static_cast<uint8_t>(code);
      a.errT[static_cast<size_t>(q) * a.m + r] = e;
      loss += 0.5 * static_cast<double>(e) * static_cast<double>(e);
    }
    const float* u = ush[q];
#pragma unroll
    for (int j = 0; j < LEN - 1; j += 4) {
      const float4 u4 = *reinterpret_cast<const float4*>(u + j);
      w[j] = fmaf(-e, u4.x, w[j + 1]);
      if (j + 1 < LEN - 1) w[j + 1] = fmaf(-e, u4.y, w[j + 2]);
      if (j + 2 < LEN - 1) w[j + 2] = fmaf(-e, u4.z, w[j + 3]);
      if (j + 3 < LEN - 1) w[j + 3] = fmaf(-e, u4.w, w[j + 4 < BLK ? j + 4 : BLK - 1]);
    }
  }
}

// One CTA per 128 rows; the block's U rows (shifted: ush[q][j] = U[i1+q][i1+q+1+j]) and
// diagonal sit in shared memory, each thread keeps its row's 128 columns in registers.
__global__ void __launch_bounds__(128) column_loop_kernel(const LoopArgs a) {
  extern __shared__ __align__(16) float smem_f[];
  float(*ush)[BLK] = reinterpret_cast<float(*)[BLK]>(smem_f);
  float* udiag = smem_f + BLK * BLK;
  const int i1 = a.i1, nb = a.nb;
  // The U block goes to shared memory through cp.async, so that all of its loads are in
  // flight at once; entries past the block's end are zero-filled.
  for (int q = 0; q < BLK; ++q) {
    const float* urow = a.U + static_cast<size_t>(i1 + (q < nb ? q : 0)) * a.d + i1 + q + 1;
    for (int j = threadIdx.x; j < BLK; j += blockDim.x) {
      const bool valid = (q + 1 + j < nb);
      cp_async4(&ush[q][j], valid ? urow + j : a.U, valid);
    }
  }
  for (int q = threadIdx.x; q < nb; q += blockDim.x)
    cp_async4(&udiag[q], a.U + static_cast<size_t>(i1 + q) * a.d + i1 + q, true);
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  __syncthreads();

  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = r < a.m;
  float w[BLK];
  const float* wrow = a.Wp + static_cast<size_t>(active ? r : 0) * a.d + i1;
#pragma unroll
  for (int j = 0; j < BLK; j += 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && j < nb) v = *reinterpret_cast<const float4*>(wrow + j);
    w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
  }
  float s = 1.0f, z = 0.0f;
  if (a.group == 0 && active) {
    s = a.scales[static_cast<size_t>(a.gi_outer) * a.m + r];
    z = static_cast<float>(a.zeros[static_cast<size_t>(a.gi_outer) * a.m + r]);
  }
  double loss = 0.0;
  loop_chunk<0>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<1>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<2>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<3>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<4>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<5>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<6>(w, ush, udiag, a, r, active, s, z, loss);
  loop_chunk<7>(w, ush, udiag, a, r, active, s, z, loss);
  if (active) a.loss_rows[r] += loss;
}

// ---------------------------------------------------------------- lazy update (FMA)

// Wp[r][c] -= sum_k ErrT[k][r] U[i1+k][c] for c >= i2 = i1 + nb.  64x64 output tiles,
// K in chunks of 32.
__global__ void __launch_bounds__(256) lazy_update_kernel(float* __restrict__ Wp,
                                                          const float* __restrict__ U,
                                                          const float* __restrict__ errT,
                                                          int m, int d, int i1, int nb) {
  __shared__ __align__(16) float se[32][64];
  __shared__ __align__(16) float su[32][64];
  const int i2 = i1 + nb;
  const int c0 = i2 + blockIdx.x * 64;
  const int r0 = blockIdx.y * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < nb; k0 += 32) {
    for (int e = threadIdx.x; e < 32 * 64; e += 256) {
      const int k = e / 64, x = e % 64;
      const bool kin = k0 + k < nb;
      se[k][x] = (kin && r0 + x < m) ? errT[static_cast<size_t>(k0 + k) * m + r0 + x] : 0.0f;
      su[k][x] = (kin && c0 + x < d) ? U[static_cast<size_t>(i1 + k0 + k) * d + c0 + x] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float4 a4 = *reinterpret_cast<const float4*>(&se[k][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&su[k][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = r0 + ty * 4 + u;
    if (r >= m) continue;
    float* wr = Wp + static_cast<size_t>(r) * d;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c = c0 + tx * 4 + v;
      if (c < d) wr[c] -= acc[u][v];
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

// qweight[wi][r]: codes of row r in original column order, packed along d.
__global__ void pack_qweight_kernel(const uint8_t* __restrict__ codesT,
                                    const int32_t* __restrict__ pos, int m, int d, int bits,
                                    int32_t* __restrict__ qweight) {
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

  GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gidx_kernel, (unsigned)ceil_div(d, 256), 256, 0, q.perm,
              d, q.group, q.pos, q.g_idx);
  if (m > 0) {
    const size_t row_smem = static_cast<size_t>(d) * sizeof(float);
    static size_t attr_f = 0, attr_b = 0;
    if (q.w_bf16) {
      if (row_smem > 48 * 1024 && row_smem > attr_b) {
        GPTQ_CUDA(cudaFuncSetAttribute(gather_w_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(row_smem)));
        attr_b = row_smem;
      }
      GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gather_w_kernel<__nv_bfloat16>, m, 256, row_smem,
                  static_cast<const __nv_bfloat16*>(q.W), d, q.perm, q.dead, q.Wp, q.loss_rows,
                  q.st);
    } else {
      if (row_smem > 48 * 1024 && row_smem > attr_f) {
        GPTQ_CUDA(cudaFuncSetAttribute(gather_w_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(row_smem)));
        attr_f = row_smem;
      }
      GPTQ_LAUNCH(GPTQ_K_QUANT_GATHER, s, gather_w_kernel<float>, m, 256, row_smem,
                  static_cast<const float*>(q.W), d, q.perm, q.dead, q.Wp, q.loss_rows, q.st);
    }

    const int loop_smem = (BLK * BLK + BLK) * static_cast<int>(sizeof(float));
    static bool loop_attr = false;
    if (!loop_attr) {
      GPTQ_CUDA(cudaFuncSetAttribute(column_loop_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, loop_smem));
      loop_attr = true;
    }
    const bool inblock_fit = (q.group > 0 && q.group <= BLK);
    for (int i1 = 0; i1 < d; i1 += BLK) {
      const int nb = (d - i1 < BLK) ? d - i1 : BLK;
      LoopArgs a;
      a.Wp = q.Wp;
      a.U = q.U;
      a.m = m;
      a.d = d;
      a.i1 = i1;
      a.nb = nb;
      a.group = inblock_fit ? q.group : 0;
      a.gi_outer = 0;
      a.g = g;
      a.scales = q.scales;
      a.zeros = q.zeros;
      a.codesT = q.codesT;
      a.errT = q.errT;
      a.loss_rows = q.loss_rows;
      if (!inblock_fit) {
        const bool start = (q.group == -1) ? (i1 == 0) : (i1 % q.group == 0);
        const int gi = (q.group == -1) ? 0 : i1 / q.group;
        if (start) {
          const int len = (q.group == -1) ? d : ((d - i1 < q.group) ? d - i1 : q.group);
          GPTQ_LAUNCH(GPTQ_K_QUANT_FIT, s, fit_kernel, (unsigned)ceil_div(m, 8), 256, 0, q.Wp, m,
                      d, i1, len, g, gi, q.scales, q.zeros);
        }
        a.gi_outer = gi;
      }
      GPTQ_LAUNCH(GPTQ_K_QUANT_LOOP, s, column_loop_kernel, (unsigned)ceil_div(m, 128), 128,
                  loop_smem, a);
      if (i1 + nb < d) {
        dim3 grid((unsigned)ceil_div(d - i1 - nb, 64), (unsigned)ceil_div(m, 64));
        GPTQ_LAUNCH(GPTQ_K_QUANT_LAZY, s, lazy_update_kernel, grid, 256, 0, q.Wp, q.U, q.errT, m,
                    d, i1, nb);
      }
    }
    dim3 gq((unsigned)ceil_div(m, 128), static_cast<unsigned>(q.bits * d / 32));
    GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, pack_qweight_kernel, gq, 128, 0, q.codesT, q.pos, m, d,
                q.bits, q.qweight);
    const int nz = q.G * (m * q.bits / 32);
    GPTQ_LAUNCH(GPTQ_K_QUANT_PACK, s, pack_qzeros_kernel, (unsigned)ceil_div(nz, 256), 256, 0,
                q.zeros, m, q.G, q.bits, q.qzeros);
  }
  GPTQ_LAUNCH(GPTQ_K_QUANT_LOSS, s, loss_sum_kernel, 1, 1024, 0, q.loss_rows, m, q.loss);
}

}  // namespace gptq
