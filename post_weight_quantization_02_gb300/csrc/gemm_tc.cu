// Float32-accurate tensor-core GEMM for the factorisation updates:
//   C[i][j] = beta C[i][j] + alpha sum_{k<128} A[i][k] B[j][k]
// with both operands K-major (rows of 128 consecutive k), read through tensor maps that
// cover whole matrices: the launch passes each operand's row and column offset.
//
// Each float32 operand x is split as x = hi + lo with hi = x truncated to tf32 (the
// tensor core reads the same bits as x) and lo = x - hi; the products hi*hi + hi*lo +
// lo*hi are accumulated in float32 TMEM with tcgen05.mma kind::tf32 (the dropped lo*lo is
// ~2^-21 relative).  TMA lands each K-quarter (32) of the fp32 tiles in shared memory
// with 128-byte swizzle; the CTA's threads then write the lo parts elementwise into twin
// buffers (same swizzled layout) before one thread issues the MMAs.  One CTA per
// 128 x 128 output tile, 64 KB of shared memory, so three CTAs share an SM and overlap
// their load / convert / MMA phases.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int TM = 128, TN = 128, TK = 128, KQ = 32;  // K-quarter per phase
constexpr int A_BYTES = TM * KQ * 4;                   // 16 KB
constexpr int B_BYTES = TN * KQ * 4;                   // 16 KB
constexpr int SMEM_BYTES = 2 * A_BYTES + 2 * B_BYTES + 1024 + 128;

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

struct TcGemmArgs {
  float* C;
  int ldc;
  int a_row0, a_k0;  // operand offsets inside the tensor maps
  int b_row0, b_k0;
  int M, N;
  float alpha, beta;
  int lower;     // only tiles with row tile >= column tile; only entries j <= i written
  int n_tiles;   // column tiles (non-lower enumeration)
  DevStatus* st;
};

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(128) gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tma,
                                                          const __grid_constant__ CUtensorMap tmb,
                                                          const TcGemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* a_hi = smem;
  uint8_t* a_lo = smem + A_BYTES;
  uint8_t* b_hi = smem + 2 * A_BYTES;
  uint8_t* b_lo = b_hi + B_BYTES;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + 2 * A_BYTES + 2 * B_BYTES);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int bi, bj;
  if (g.lower) {
    int rem = blockIdx.x;
    bi = 0;
    while (rem > bi) { rem -= bi + 1; ++bi; }
    bj = rem;
  } else {
    bi = blockIdx.x / g.n_tiles;
    bj = blockIdx.x % g.n_tiles;
  }
  const int i0 = bi * TM, j0 = bj * TN;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  if (tid == 0) {
    tc::mbar_init(bar_load, 1);
    tc::mbar_init(bar_mma, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t IDESC = idesc_tf32(TM, TN, false);
  bool ok = true;

  for (int ph = 0; ph < TK / KQ && ok; ++ph) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar_load, A_BYTES + B_BYTES);
      tc::tma_load_2d(a_hi, &tma, bar_load, g.a_k0 + ph * KQ, g.a_row0 + i0);
      tc::tma_load_2d(b_hi, &tmb, bar_load, g.b_k0 + ph * KQ, g.b_row0 + j0);
    }
    if (!tc::mbar_wait(bar_load, ph & 1, abort_flag)) { ok = false; break; }
    // lo = x - trunc_tf32(x), elementwise in the same swizzled layout
    {
      const float4* src_a = reinterpret_cast<const float4*>(a_hi);
      float4* dst_a = reinterpret_cast<float4*>(a_lo);
      const float4* src_b = reinterpret_cast<const float4*>(b_hi);
      float4* dst_b = reinterpret_cast<float4*>(b_lo);
#pragma unroll 4
      for (int e = tid; e < A_BYTES / 16; e += 128) {
        float4 x = src_a[e];
        x.x -= __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
        x.y -= __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
        x.z -= __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
        x.w -= __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
        dst_a[e] = x;
        float4 y = src_b[e];
        y.x -= __uint_as_float(__float_as_uint(y.x) & 0xFFFFE000u);
        y.y -= __uint_as_float(__float_as_uint(y.y) & 0xFFFFE000u);
        y.z -= __uint_as_float(__float_as_uint(y.z) & 0xFFFFE000u);
        y.w -= __uint_as_float(__float_as_uint(y.w) & 0xFFFFE000u);
        dst_b[e] = y;
      }
    }
    fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after();
      const uint32_t ah = tc::smem_u32(a_hi), al = tc::smem_u32(a_lo);
      const uint32_t bh = tc::smem_u32(b_hi), bl = tc::smem_u32(b_lo);
#pragma unroll
      for (int kk = 0; kk < KQ / 8; ++kk) {
        // A, K-major: 8 tf32 = 32 bytes along the 128-byte row; 8-row groups 1024 B apart
        const uint64_t dah = tc::smem_desc(ah + 32 * kk, 16, 1024, tc::kSwizzle128B);
        const uint64_t dal = tc::smem_desc(al + 32 * kk, 16, 1024, tc::kSwizzle128B);
        const uint64_t dbh = tc::smem_desc(bh + 32 * kk, 16, 1024, tc::kSwizzle128B);
        const uint64_t dbl = tc::smem_desc(bl + 32 * kk, 16, 1024, tc::kSwizzle128B);
        const uint32_t acc0 = (ph | kk) != 0 ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(dah), "l"(dbh), "r"(IDESC), "r"(acc0)
            : "memory");
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(dah), "l"(dbl), "r"(IDESC), "r"(1u)
            : "memory");
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(dal), "l"(dbh), "r"(IDESC), "r"(1u)
            : "memory");
      }
      tc::mma_commit(bar_mma);
    }
    if (!tc::mbar_wait(bar_mma, ph & 1, abort_flag)) { ok = false; break; }
    tc::fence_after();
  }

  if (ok) {
    // epilogue, in two 64-column halves staged through the (now free) operand buffers:
    // warp w moves TMEM lanes 32w..32w+31 (tile rows) into shared memory, then the CTA
    // reads and writes C as coalesced float4 rows
    float* stage = reinterpret_cast<float*>(smem);   // [128][68]
    constexpr int SROW = 68;
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + half * 64 + c * 32, r);
        tc::tmem_ld_wait();
        float* srow = stage + (32 * warp + lane) * SROW + c * 32;
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(srow + k) =
              make_float4(__uint_as_float(r[k]), __uint_as_float(r[k + 1]),
                          __uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]));
      }
      __syncthreads();
      for (int e = tid; e < TM * 16; e += 128) {
        const int rr = e / 16, c4 = (e % 16) * 4;
        const int row = i0 + rr, col = j0 + half * 64 + c4;
        if (row >= g.M || col >= g.N) continue;
        if (g.lower && col > row) continue;
        const float4 v = *reinterpret_cast<const float4*>(stage + rr * SROW + c4);
        float4* cp = reinterpret_cast<float4*>(g.C + static_cast<size_t>(row) * g.ldc + col);
        float4 o = (g.beta != 0.0f) ? *cp : make_float4(0.f, 0.f, 0.f, 0.f);
        // a lower tile's diagonal keeps the entries above it as they were
        const bool w1 = !g.lower || col + 1 <= row, w2 = !g.lower || col + 2 <= row,
                   w3 = !g.lower || col + 3 <= row;
        o.x = fmaf(g.alpha, v.x, o.x);
        if (w1) o.y = fmaf(g.alpha, v.y, o.y);
        if (w2) o.z = fmaf(g.alpha, v.z, o.z);
        if (w3) o.w = fmaf(g.alpha, v.w, o.w);
        if (g.beta == 0.0f) {
          if (!w1) o.y = cp->y;
          if (!w2) o.z = cp->z;
          if (!w3) o.w = cp->w;
        }
        *cp = o;
      }
      __syncthreads();
    }
  } else {
    *abort_flag = 1;
    if (lane == 0) {
      dev_fail(g.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&g.st->timeouts, 1);
    }
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
}

}  // namespace

void make_gemm_map(CUtensorMap* map, const float* base, int rows, int cols, int ld) {
  make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, static_cast<uint64_t>(cols),
               static_cast<uint64_t>(rows), static_cast<uint64_t>(ld) * 4, KQ, TM,
               CU_TENSOR_MAP_SWIZZLE_128B);
}

void launch_gemm_tf32x3(int kind, const CUtensorMap& ma, int a_row0, int a_k0,
                        const CUtensorMap& mb, int b_row0, int b_k0, float* C, int ldc, int M,
                        int N, float alpha, float beta, bool lower, DevStatus* st,
                        cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  static bool attr = false;
  if (!attr) {
    GPTQ_CUDA(cudaFuncSetAttribute(gemm_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM_BYTES));
    attr = true;
  }
  TcGemmArgs g;
  g.C = C;
  g.ldc = ldc;
  g.a_row0 = a_row0;
  g.a_k0 = a_k0;
  g.b_row0 = b_row0;
  g.b_k0 = b_k0;
  g.M = M;
  g.N = N;
  g.alpha = alpha;
  g.beta = beta;
  g.lower = lower ? 1 : 0;
  const int tm = static_cast<int>(ceil_div(M, TM)), tn = static_cast<int>(ceil_div(N, TN));
  g.n_tiles = tn;
  g.st = st;
  const unsigned grid = lower ? static_cast<unsigned>(tm * (tm + 1) / 2)
                              : static_cast<unsigned>(tm * tn);
  GPTQ_LAUNCH(kind, s, gemm_tf32x3_kernel, grid, 128, SMEM_BYTES, ma, mb, g);
}

}  // namespace gptq
