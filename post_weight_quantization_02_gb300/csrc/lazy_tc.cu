// The lazy trailing update on the tensor cores: W[:, i2:] -= Err U[i1:i2, i2:].
//
// "Same Ruler, Smarter Placement: GPTQ", section 1.8, and "GPTQ Architecture, in
// depth", "The algorithm in code": after a block of 128 columns, its accumulated errors
// are pushed into every later column as one matrix product.  W is float32 and the update
// must keep float32 accuracy (the next blocks round these values), so each operand is
// split into two bf16 parts, x = hi + lo, and the product is accumulated in float32 TMEM
// as hi*hi + hi*lo + lo*hi (the lo*lo term, ~2^-16 relative, is dropped).
//
// Persistent kernel, one CTA per SM, one output tile (128 rows x 256 columns, K = 128)
// per unit:
//   warp 0      TMA: ErrT hi/lo [128 k x 128 rows] and U hi/lo [128 k x 256 columns],
//               both MN-major, 192 KB of operands per tile
//   warp 1      TMEM owner and MMA issuer: 8 k-steps x 3 tcgen05.mma 128x256x16
//   warps 2..9  epilogue: W[r, c] -= D[r, c], read-modify-write of the W tile
// Two 256-column TMEM accumulators let the epilogue (the HBM-bound part) of one tile
// overlap the MMAs of the next.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int BM = 128, BN = 256, BKT = 128;
constexpr int BOX = 64 * 64 * 2;                  // one TMA box: 64 x 64 bf16
constexpr int A_BYTES = BM * BKT * 2;            // per part (hi or lo): 32 KB
constexpr int B_BYTES = BN * BKT * 2;            // 64 KB
constexpr int OPS_BYTES = 2 * A_BYTES + 2 * B_BYTES;
constexpr int SMEM_BYTES = OPS_BYTES + 1024 + 256;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, true, true);

struct LazyArgs {
  float* W;       // Wp, [m][d]
  int m, d, i2;
  int n_mt, n_nt; // row tiles, column tiles
  DevStatus* st;
};

// smem offsets of part p (0 hi, 1 lo): A[p][kc][h], B[p][kc][h]
__device__ __forceinline__ uint32_t a_off(int p, int kc, int h) {
  return static_cast<uint32_t>(p * A_BYTES + (kc * 2 + h) * BOX);
}
__device__ __forceinline__ uint32_t b_off(int p, int kc, int h) {
  return static_cast<uint32_t>(2 * A_BYTES + p * B_BYTES + (kc * 4 + h) * BOX);
}

__global__ void __launch_bounds__(THREADS, 1)
    lazy_tc_kernel(const __grid_constant__ CUtensorMap tm_ehi, const __grid_constant__ CUtensorMap tm_elo,
                   const __grid_constant__ CUtensorMap tm_uhi, const __grid_constant__ CUtensorMap tm_ulo,
                   const LazyArgs a, int i1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OPS_BYTES);
  uint64_t* empty = full + 1;
  uint64_t* accfull = empty + 1;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_units = a.n_mt * a.n_nt;

  if (threadIdx.x == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(empty, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accfull[b], 1);
      tc::mbar_init(&accempty[b], EPI_WARPS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int mt = u % a.n_mt, nt = u / a.n_mt;
      if (!tc::mbar_wait(empty, phase ^ 1u, abort_flag)) { ok = false; break; }
      tc::mbar_arrive_expect_tx(full, OPS_BYTES);
      const int r0 = mt * BM, c0 = a.i2 + nt * BN;
      for (int kc = 0; kc < 2; ++kc) {
        const int k = i1 + kc * 64;  // U row / ErrT row coordinate
        for (int h = 0; h < 2; ++h) {
          tc::tma_load_2d(smem + a_off(0, kc, h), &tm_ehi, full, r0 + 64 * h, kc * 64);
          tc::tma_load_2d(smem + a_off(1, kc, h), &tm_elo, full, r0 + 64 * h, kc * 64);
        }
        for (int h = 0; h < 4; ++h) {
          tc::tma_load_2d(smem + b_off(0, kc, h), &tm_uhi, full, c0 + 64 * h, k);
          tc::tma_load_2d(smem + b_off(1, kc, h), &tm_ulo, full, c0 + 64 * h, k);
        }
      }
      phase ^= 1u;
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t phase = 0;
    int acc = 0;
    uint32_t accphase = 0;
    const uint32_t base = tc::smem_u32(smem);
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      if (!tc::mbar_wait(&accempty[acc], accphase ^ 1u, abort_flag)) { ok = false; break; }
      tc::fence_after();
      if (!tc::mbar_wait(full, phase, abort_flag)) { ok = false; break; }
      tc::fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
#pragma unroll
      for (int kk = 0; kk < BKT / 16; ++kk) {
        const int kc = kk / 4;
        const uint32_t ko = static_cast<uint32_t>((kk % 4) * 2048);
        const uint64_t ahi = tc::smem_desc(base + a_off(0, kc, 0) + ko, BOX, 1024, tc::kSwizzle128B);
        const uint64_t alo = tc::smem_desc(base + a_off(1, kc, 0) + ko, BOX, 1024, tc::kSwizzle128B);
        const uint64_t bhi = tc::smem_desc(base + b_off(0, kc, 0) + ko, BOX, 1024, tc::kSwizzle128B);
        const uint64_t blo = tc::smem_desc(base + b_off(1, kc, 0) + ko, BOX, 1024, tc::kSwizzle128B);
        tc::mma_f16(d_tmem, ahi, bhi, IDESC, kk != 0 ? 1u : 0u);
        tc::mma_f16(d_tmem, ahi, blo, IDESC, 1u);
        tc::mma_f16(d_tmem, alo, bhi, IDESC, 1u);
      }
      tc::mma_commit(empty);
      tc::mma_commit(&accfull[acc]);
      phase ^= 1u;
      acc ^= 1;
      if (acc == 0) accphase ^= 1u;
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp % 4;
    const int half = (warp - 2) / 4;
    int acc = 0;
    uint32_t accphase = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int mt = u % a.n_mt, nt = u / a.n_mt;
      if (!tc::mbar_wait(&accfull[acc], accphase, abort_flag)) { ok = false; break; }
      tc::fence_after();
      const int row = mt * BM + 32 * q + lane;
      const int col0 = a.i2 + nt * BN + half * 128;
      float* wrow = a.W + static_cast<size_t>(row < a.m ? row : 0) * a.d;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * BN + half * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
        tc::tmem_ld_wait();
        const int cc = col0 + c * 32;
        if (row < a.m) {
          float4 wv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (cc + 4 * k < a.d) wv[k] = *reinterpret_cast<const float4*>(wrow + cc + 4 * k);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (cc + 4 * k < a.d) {
              wv[k].x -= __uint_as_float(r[4 * k]);
              wv[k].y -= __uint_as_float(r[4 * k + 1]);
              wv[k].z -= __uint_as_float(r[4 * k + 2]);
              wv[k].w -= __uint_as_float(r[4 * k + 3]);
              *reinterpret_cast<float4*>(wrow + cc + 4 * k) = wv[k];
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&accempty[acc]);
      acc ^= 1;
      if (acc == 0) accphase ^= 1u;
    }
  }

  if (!ok) {
    *abort_flag = 1;
    if (lane == 0 || warp >= 2) {
      dev_fail(a.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&a.st->timeouts, 1);
    }
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

// hi = bf16(x), lo = bf16(x - hi) for the strict upper triangle of U (0 elsewhere).
__global__ void usplit_kernel(const float* __restrict__ U, int d, __nv_bfloat16* __restrict__ hi,
                              __nv_bfloat16* __restrict__ lo) {
  const int i = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= d) return;
  const size_t o = static_cast<size_t>(i) * d + j;
  const float x = (j > i) ? U[o] : 0.0f;
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi[o] = h;
  lo[o] = __float2bfloat16_rn(x - __bfloat162float(h));
}

}  // namespace

void launch_usplit(const float* U, int d, __nv_bfloat16* hi, __nv_bfloat16* lo, cudaStream_t s) {
  dim3 grid((unsigned)ceil_div(d, 256), d);
  GPTQ_LAUNCH(GPTQ_K_QUANT_SPLIT, s, usplit_kernel, grid, 256, 0, U, d, hi, lo);
}

LazyMaps make_lazy_maps(const __nv_bfloat16* ehi, const __nv_bfloat16* elo,
                        const __nv_bfloat16* uhi, const __nv_bfloat16* ulo, int m, int d) {
  LazyMaps mp;
  make_tmap_2d(&mp.ehi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ehi, m, 128, static_cast<uint64_t>(m) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.elo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, elo, m, 128, static_cast<uint64_t>(m) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.uhi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, uhi, d, d, static_cast<uint64_t>(d) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.ulo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ulo, d, d, static_cast<uint64_t>(d) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  return mp;
}

void launch_lazy_tc(const LazyMaps& mp, float* W, int m, int d, int i1, DevStatus* st,
                    cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    GPTQ_CUDA(cudaFuncSetAttribute(lazy_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM_BYTES));
    attr = true;
  }
  LazyArgs a;
  a.W = W;
  a.m = m;
  a.d = d;
  a.i2 = i1 + 128;
  a.n_mt = static_cast<int>(ceil_div(m, BM));
  a.n_nt = static_cast<int>(ceil_div(d - a.i2, BN));
  a.st = st;
  const int units = a.n_mt * a.n_nt;
  const int grid = units < sm_count() ? units : sm_count();
  GPTQ_LAUNCH(GPTQ_K_QUANT_LAZY, s, lazy_tc_kernel, grid, THREADS, SMEM_BYTES, mp.ehi, mp.elo,
              mp.uhi, mp.ulo, a, i1);
}

}  // namespace gptq
