// dequant_matmul.cu: the product a W4A16-style serving kernel computes straight from the
// packed checkpoint ("GPTQ Architecture, in depth", "Packing, tooling and serving": the
// kernel unpacks each code and dequantises it with its group's scale and zero point just
// before the multiply):
//   y[t, r] = sum_c x[t, c] * s[g, r] * (code[r, c] - z[g, r]),  g = g_idx[c].
// It reads the checkpoint exactly as gptq_quantize_layer writes it, so it also checks
// the packing end to end.
//
// Design: one thread per output row; the row's packed words are read coalesced across
// the CTA's 128 rows (qweight is [bits*d/32, m]), 32 codes at a time from `bits` words
// with compile-time shifts; the scale and zero are reloaded only when the column's group
// changes (once per group with static groups, often with act-order groups).  d_in is
// split over the 8 CTAs of a cluster, and CTA 0 adds the 8 partial sums in rank order
// from the others' shared memory, so the result does not depend on timing.  The kernel
// is bound by the packed weight bytes (HBM) at decode batch sizes.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {
namespace {

constexpr int DQ_ROWS = 128;  // output rows per CTA, one per thread
constexpr int DQ_SPLIT = 8;   // CTAs of a cluster, each a slice of d_in
constexpr int DQ_KC = 128;    // columns staged per pass

struct DqArgs {
  const void* x;
  int x_bf16;
  int64_t n;
  int d, m, G;
  int kper;  // columns per CTA of the cluster (a multiple of 32)
  const int32_t* qweight;
  const float* scales;
  const int32_t* qzeros;
  const int32_t* g_idx;
  float* y;
  DevStatus* st;
};

__device__ __forceinline__ float ld_x(const DqArgs& a, int64_t t, int c) {
  const int64_t i = t * a.d + c;
  return a.x_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[i])
                  : static_cast<const float*>(a.x)[i];
}

// Bits [b, b + BITS) of a little-endian stream stored as 32-bit words.
template <int BITS>
__device__ __forceinline__ uint32_t stream_bits(const uint32_t* __restrict__ words, int b) {
  const int w = b >> 5, sh = b & 31;
  uint32_t v = words[w] >> sh;
  if (sh + BITS > 32) v |= words[w + 1] << (32 - sh);
  return v & ((1u << BITS) - 1u);
}

__device__ __forceinline__ float ld_dsmem(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

template <int BITS, int NT>
__global__ void __cluster_dims__(1, DQ_SPLIT, 1) __launch_bounds__(DQ_ROWS)
    dequant_matmul_kernel(const DqArgs a) {
  __shared__ __align__(16) float xs[NT][DQ_KC];
  __shared__ int gs[DQ_KC];
  __shared__ float part[NT][DQ_ROWS];
  const int tid = threadIdx.x;
  const int r = blockIdx.x * DQ_ROWS + tid;
  const bool row_ok = r < a.m;
  const int rank = static_cast<int>(tc::cluster_ctarank());  // the slice of d_in
  const int k0 = rank * a.kper, k1 = min(a.d, k0 + a.kper);
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.qweight);
  const uint32_t* qz = reinterpret_cast<const uint32_t*>(a.qzeros);
  const int zwords = BITS * a.m / 32;  // words of one group's zero stream
  for (int64_t t0 = 0; t0 < a.n; t0 += NT) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    for (int kc = k0; kc < k1; kc += DQ_KC) {
      const int kn = min(DQ_KC, k1 - kc);  // a multiple of 32
      for (int e = tid; e < NT * DQ_KC; e += DQ_ROWS) {
        const int t = e / DQ_KC, c = e % DQ_KC;
        xs[t][c] = (t0 + t < a.n && c < kn) ? ld_x(a, t0 + t, kc + c) : 0.0f;
      }
      for (int c = tid; c < DQ_KC; c += DQ_ROWS) {
        int g = (c < kn) ? a.g_idx[kc + c] : 0;
        if (g < 0 || g >= a.G) {  // a group index outside the scales: report, read group 0
          dev_fail(a.st, GPTQ_ERR_INVALID_ARG, kc + c + 1);
          g = 0;
        }
        gs[c] = g;
      }
      __syncthreads();
      if (row_ok) {
        int gprev = -1;
        float s = 0.0f, z = 0.0f;
        for (int c0 = 0; c0 < kn; c0 += 32) {
          uint32_t wds[BITS];  // the 32 codes of columns kc + c0 .. kc + c0 + 31
          const int w0 = BITS * (kc + c0) / 32;
#pragma unroll
          for (int i = 0; i < BITS; ++i) wds[i] = qw[static_cast<size_t>(w0 + i) * a.m + r];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float code = static_cast<float>(stream_bits<BITS>(wds, BITS * c));
            const int g = gs[c0 + c];
            if (g != gprev) {
              s = a.scales[static_cast<size_t>(g) * a.m + r];
              z = static_cast<float>(stream_bits<BITS>(qz + static_cast<size_t>(g) * zwords,
                                                       BITS * r));
              gprev = g;
            }
            const float w = s * (code - z);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t] = fmaf(xs[t][c0 + c], w, acc[t]);
          }
        }
      }
      __syncthreads();
    }
    // the cluster's slices, added by CTA 0 in rank order
#pragma unroll
    for (int t = 0; t < NT; ++t) part[t][tid] = acc[t];
    tc::cluster_sync();
    if (rank == 0 && row_ok) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t0 + t >= a.n) break;
        const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(&part[t][tid]));
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < DQ_SPLIT; ++j) sum += ld_dsmem(tc::mapa_shared(sa, j));
        a.y[(t0 + t) * a.m + r] = sum;
      }
    }
    tc::cluster_sync();  // the partial sums stay readable until CTA 0 is done
  }
}

template <int BITS>
void launch_bits(const DqArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(a.m, DQ_ROWS)), DQ_SPLIT);
  if (a.n == 1) {
    GPTQ_LAUNCH(GPTQ_K_DEQUANT_MATMUL, s, (dequant_matmul_kernel<BITS, 1>), grid, DQ_ROWS, 0, a);
  } else {
    GPTQ_LAUNCH(GPTQ_K_DEQUANT_MATMUL, s, (dequant_matmul_kernel<BITS, 8>), grid, DQ_ROWS, 0, a);
  }
}

}  // namespace

void launch_dequant_matmul(const void* x, bool x_bf16, int64_t n, int d, int m, int bits, int G,
                           const int32_t* qweight, const float* scales, const int32_t* qzeros,
                           const int32_t* g_idx, float* y, DevStatus* st, cudaStream_t s) {
  if (n <= 0 || m <= 0) return;
  DqArgs a;
  a.x = x;
  a.x_bf16 = x_bf16 ? 1 : 0;
  a.n = n;
  a.d = d;
  a.m = m;
  a.G = G;
  a.kper = static_cast<int>(ceil_div(ceil_div(d, DQ_SPLIT), 32)) * 32;
  a.qweight = qweight;
  a.scales = scales;
  a.qzeros = qzeros;
  a.g_idx = g_idx;
  a.y = y;
  a.st = st;
  switch (bits) {
    case 2: launch_bits<2>(a, s); break;
    case 3: launch_bits<3>(a, s); break;
    case 4: launch_bits<4>(a, s); break;
    default: launch_bits<8>(a, s); break;
  }
}

}  // namespace gptq
