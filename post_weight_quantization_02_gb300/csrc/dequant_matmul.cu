// dequant_matmul.cu: the product a W4A16-style serving kernel computes straight from the
// packed checkpoint ("GPTQ Architecture, in depth", "Packing, tooling and serving": the
// kernel unpacks each code and dequantises it with its group's scale and zero point just
// before the multiply):
//   y[t, r] = sum_c x[t, c] * s[g, r] * (code[r, c] - z[g, r]),  g = g_idx[c].
// It reads the checkpoint exactly as gptq_quantize_layer writes it, so it also checks
// the packing end to end.
//
// Design: two threads per output row, taking alternate 128-column chunks of the CTA's
// slice.  Each thread copies its own row's packed words of a chunk (read coalesced across
// the CTA's 128 rows: qweight is [bits*d/32, m]) into its own part of a shared-memory ring
// with cp.async, two chunks in flight; the first two are requested before anything else,
// so they land while the shared tables are filled.  Only the copying thread reads them, so
// waiting on its own copy groups is all the ordering needed.  Decoding loops over 32-column
// runs with the run's body unrolled: the whole kernel then fits the instruction cache,
// which a fully unrolled chunk (tens of KB of code) does not.  No integer-to-float
// conversion: the float whose exponent says 2^23 and whose low mantissa bits hold the code
// is exactly 2^23 + code, so one OR and one subtraction of (2^23 + z) give code - z
// exactly.  A run whose columns share one group (every run with static groups) sums
// x (code - z) and applies the scale once; other runs (act-order groups) look up the scale
// and zero per column, from a shared table of every group's (scale, 2^23 + zero) of the
// CTA's rows when it fits.  The CTA's slice of x sits in shared memory column-major.  d_in
// is split over the 8 CTAs of a cluster, and CTA 0 adds the 8 partial sums in rank order
// from the others' shared memory, so the result does not depend on timing.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {
namespace {

constexpr int DQ_ROWS = 128;  // output rows per CTA
constexpr int DQ_HALVES = 2;  // threads per row, taking alternate chunks of the slice
constexpr int DQ_THREADS = DQ_ROWS * DQ_HALVES;
constexpr int DQ_SPLIT = 8;   // CTAs of a cluster, each a slice of d_in
constexpr int DQ_KC = 128;    // columns per chunk of packed words

struct DqArgs {
  const void* x;
  int x_bf16;
  int64_t n;
  int d, m, G;
  int kper;  // columns per CTA of the cluster (a multiple of 32)
  int table; // the CTA keeps every group's scale and zero of its rows in shared memory
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

// The same from a register array (b known at compile time once the caller is unrolled).
template <int BITS, int N>
__device__ __forceinline__ uint32_t reg_bits(const uint32_t (&words)[N], int b) {
  const int w = b >> 5, sh = b & 31;
  uint32_t v = words[w] >> sh;
  if (sh + BITS > 32 && w + 1 < N) v |= words[w + 1] << (32 - sh);
  return v & ((1u << BITS) - 1u);
}

__device__ __forceinline__ float ld_dsmem(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Row r's zero point in group g (bits [BITS r, BITS r + BITS) of the group's stream).
template <int BITS>
__device__ __forceinline__ float zero_of(const uint32_t* __restrict__ qz, int zwords, int g,
                                         int zbit) {
  return static_cast<float>(stream_bits<BITS>(qz + static_cast<size_t>(g) * zwords, zbit));
}

constexpr uint32_t kTwo23Bits = 0x4B000000u;  // the float 2^23
constexpr float kTwo23 = 8388608.0f;

// code - z, exactly, for a code below 2^23 and zb = 2^23 + z.
__device__ __forceinline__ float code_minus(uint32_t code, float zb) {
  return __uint_as_float(code | kTwo23Bits) - zb;
}

__device__ __forceinline__ void cp_async4(uint32_t* dst, const uint32_t* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int DQ_STAGES = 2;  // a thread's chunks in flight

// Shared memory bytes of the ring of packed words: DQ_STAGES chunks of every thread.
template <int BITS>
constexpr int ring_bytes() {
  return DQ_STAGES * (BITS * DQ_KC / 32) * DQ_THREADS * static_cast<int>(sizeof(uint32_t));
}

template <int BITS, int NT>
__global__ void __cluster_dims__(1, DQ_SPLIT, 1) __launch_bounds__(DQ_THREADS, 2)
    dequant_matmul_kernel(const DqArgs a) {
  // dynamic shared memory: when a.table, (scale, 2^23 + zero) of every group of the
  // slice's range and row of the CTA; the ring of packed words, [stage][word][thread], each thread reading only
  // what it copied itself; x[t0 .. t0 + NT) over this CTA's slice of d_in, column-major
  // (the NT values of a column together); the slice's group indices; per 32-column run,
  // its group when every column of the run has the same one, else -1
  extern __shared__ __align__(16) float dsm[];
  constexpr int CW = BITS * DQ_KC / 32;                       // packed words per chunk
  constexpr int S = DQ_HALVES * DQ_KC;                        // a thread's chunk stride
  constexpr int WARPS = DQ_THREADS / 32;
  float2* tab = reinterpret_cast<float2*>(dsm);               // [G][DQ_ROWS] if a.table
  uint32_t* ring = reinterpret_cast<uint32_t*>(dsm + (a.table ? 2 * a.G * DQ_ROWS : 0));
  float* xs = reinterpret_cast<float*>(ring + DQ_STAGES * CW * DQ_THREADS);  // [kper][NT]
  int* gs = reinterpret_cast<int*>(xs + NT * a.kper);         // [kper]
  int* guni = gs + a.kper;                                    // [kper / 32]
  __shared__ float part[DQ_HALVES][NT][DQ_ROWS];
  __shared__ int grange[2];  // the smallest and largest group of the slice
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int rl = tid % DQ_ROWS, half = tid / DQ_ROWS;         // row within the CTA, chunk parity
  const int r = blockIdx.x * DQ_ROWS + rl;
  const bool row_ok = r < a.m;
  const int rank = static_cast<int>(tc::cluster_ctarank());   // the slice of d_in
  const int k0 = rank * a.kper, k1 = min(a.d, k0 + a.kper);
  const int kn_all = max(0, k1 - k0);                         // a multiple of 32
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.qweight);
  const uint32_t* qz = reinterpret_cast<const uint32_t*>(a.qzeros);
  const int zwords = BITS * a.m / 32;  // words of one group's zero stream
  const int zbit = BITS * (row_ok ? r : 0);
  const int kfirst = k0 + half * DQ_KC;  // this thread's chunks: every other one
  const int nch = (row_ok && kfirst < k1) ? (k1 - kfirst + S - 1) / S : 0;

  // chunk kc's words of this thread's row into ring stage `stage`, as one copy group
  auto issue = [&](int stage, int kc) {
    const int nw = BITS * min(DQ_KC, k1 - kc) / 32;
    const size_t w0 = static_cast<size_t>(BITS) * kc / 32;
    uint32_t* dst = ring + stage * CW * DQ_THREADS + tid;
#pragma unroll
    for (int u = 0; u < CW; ++u)
      if (u < nw) cp_async4(dst + u * DQ_THREADS, qw + (w0 + u) * a.m + r);
    cp_async_commit();
  };
  auto issue_first = [&]() {
    if (nch > 0) issue(0, kfirst);
    if (nch > 1) issue(1, kfirst + S);
  };
  issue_first();  // in flight while the shared tables are filled
  if (tid == 0) {
    grange[0] = a.G;
    grange[1] = -1;
  }
  __syncthreads();

  // the slice's group indices, a warp per 32-column run, four runs' loads at a time
  const int nruns = kn_all / 32;
  for (int run0 = warp; run0 < nruns; run0 += 4 * WARPS) {
    int gv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int run = run0 + u * WARPS;
      gv[u] = run < nruns ? a.g_idx[k0 + 32 * run + lane] : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int run = run0 + u * WARPS;  // the same for the whole warp
      if (run >= nruns) break;
      int g = gv[u];
      if (g < 0 || g >= a.G) {  // a group index outside the scales: report, read group 0
        dev_fail(a.st, GPTQ_ERR_INVALID_ARG, k0 + 32 * run + lane + 1);
        g = 0;
      }
      gs[32 * run + lane] = g;
      const int lo = __reduce_min_sync(0xffffffffu, g), hi = __reduce_max_sync(0xffffffffu, g);
      if (lane == 0) {
        guni[run] = lo == hi ? g : -1;
        atomicMin(&grange[0], lo);
        atomicMax(&grange[1], hi);
      }
    }
  }
  __syncthreads();
  const int glo = grange[0];  // the table holds groups glo .. grange[1]
  if (a.table) {
    // (with static groups a slice spans a few groups; with act-order groups, all)
    const int total = max(0, grange[1] - glo + 1) * DQ_ROWS;
    for (int e0 = tid; e0 < total; e0 += 16 * DQ_THREADS) {
      float sv[16], zv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int e = e0 + u * DQ_THREADS;
        const int g = glo + e / DQ_ROWS, row = blockIdx.x * DQ_ROWS + e % DQ_ROWS;
        const bool ok = e < total && row < a.m;
        sv[u] = ok ? a.scales[static_cast<size_t>(g) * a.m + row] : 0.0f;
        zv[u] = ok ? zero_of<BITS>(qz, zwords, g, BITS * row) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int e = e0 + u * DQ_THREADS;
        if (e < total) tab[e] = make_float2(sv[u], kTwo23 + zv[u]);
      }
    }
  }
  // (scale, 2^23 + zero) of this thread's row in group g, from global memory
  auto scale_zero_g = [&](int g) -> float2 {
    return make_float2(a.scales[static_cast<size_t>(g) * a.m + r],
                       kTwo23 + zero_of<BITS>(qz, zwords, g, zbit));
  };

  for (int64_t t0 = 0; t0 < a.n; t0 += NT) {
    for (int e0 = tid; e0 < NT * kn_all; e0 += 4 * DQ_THREADS) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * DQ_THREADS;
        const int c = e / NT, t = e % NT;
        v[u] = (e < NT * kn_all && t0 + t < a.n) ? ld_x(a, t0 + t, k0 + c) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * DQ_THREADS;
        if (e < NT * kn_all) xs[e] = v[u];
      }
    }
    __syncthreads();
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    // one chunk from ring stage `stage`: a loop over its 32-column runs, the run's body
    // unrolled (a small body: the whole kernel stays in the instruction cache)
    auto decode = [&](int stage, int kc) {
      const int nrun = min(DQ_KC, k1 - kc) / 32;
      const uint32_t* src = ring + stage * CW * DQ_THREADS + tid;
#pragma unroll 1
      for (int j = 0; j < nrun; ++j) {
        uint32_t w[BITS];  // the run's packed codes
#pragma unroll
        for (int i = 0; i < BITS; ++i) w[i] = src[(BITS * j + i) * DQ_THREADS];
        const int cb = kc - k0 + 32 * j;  // slice column of the run's first
        const float4* x4 = reinterpret_cast<const float4*>(xs + cb * NT);
        const int g0 = guni[cb / 32];
        if (g0 >= 0) {
          // one group for the whole run: sum x (code - z), then scale once
          const float2 sz = a.table ? tab[(g0 - glo) * DQ_ROWS + rl] : scale_zero_g(g0);
          float racc[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) racc[t] = 0.0f;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float xv[4 * NT];
#pragma unroll
            for (int q = 0; q < NT; ++q) *reinterpret_cast<float4*>(&xv[4 * q]) = x4[c4 * NT + q];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const float v = code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)), sz.y);
#pragma unroll
              for (int t = 0; t < NT; ++t) racc[t] = fmaf(xv[cc * NT + t], v, racc[t]);
            }
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[t] = fmaf(sz.x, racc[t], acc[t]);
        } else {
          // each column's own group (act-order)
          const int4* g4 = reinterpret_cast<const int4*>(gs + cb);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float xv[4 * NT];
#pragma unroll
            for (int q = 0; q < NT; ++q) *reinterpret_cast<float4*>(&xv[4 * q]) = x4[c4 * NT + q];
            const int4 gq = g4[c4];
            const int gg[4] = {gq.x, gq.y, gq.z, gq.w};
            float2 sz[4];
            if (a.table) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) sz[cc] = tab[(gg[cc] - glo) * DQ_ROWS + rl];
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) sz[cc] = scale_zero_g(gg[cc]);
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const float v = sz[cc].x *
                              code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)), sz[cc].y);
#pragma unroll
              for (int t = 0; t < NT; ++t) acc[t] = fmaf(xv[cc * NT + t], v, acc[t]);
            }
          }
        }
      }
    };
    // chunk i in stage i % 2; the stage is refilled with chunk i + 2 once decoded
    for (int i = 0; i < nch; ++i) {
      if (i + 1 < nch) cp_async_wait<1>();
      else cp_async_wait<0>();
      decode(i & 1, kfirst + i * S);
      if (i + 2 < nch) issue(i & 1, kfirst + (i + 2) * S);
    }
    if (t0 + NT < a.n) issue_first();  // the next tokens' pass, in flight during the sum
    // the cluster's slices and each slice's two halves, added by CTA 0 in a fixed order
#pragma unroll
    for (int t = 0; t < NT; ++t) part[half][t][rl] = acc[t];
    tc::cluster_sync();
    if (rank == 0 && row_ok && half == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t0 + t >= a.n) break;
        // every partial requested first, then added in rank order
        float v[DQ_SPLIT * DQ_HALVES];
#pragma unroll
        for (int j = 0; j < DQ_SPLIT; ++j) {
#pragma unroll
          for (int h = 0; h < DQ_HALVES; ++h) {
            const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(&part[h][t][rl]));
            v[DQ_HALVES * j + h] = ld_dsmem(tc::mapa_shared(sa, j));
          }
        }
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < DQ_SPLIT * DQ_HALVES; ++i) sum += v[i];
        a.y[(t0 + t) * a.m + r] = sum;
      }
    }
    tc::cluster_sync();  // the partial sums and x stay in place until CTA 0 is done
  }
}

template <int BITS, int NT>
void launch_nt(const DqArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(a.m, DQ_ROWS)), DQ_SPLIT);
  const int base = ring_bytes<BITS>() +
                   ((NT + 1) * a.kper + a.kper / 32) * static_cast<int>(sizeof(float));
  // the (scale, 2^23 + zero) table when it fits beside two CTAs' other shared memory on an SM
  const int tab = 2 * a.G * DQ_ROWS * static_cast<int>(sizeof(float));
  DqArgs b = a;
  b.table = (base + tab <= 100 * 1024) ? 1 : 0;
  const int smem = base + (b.table ? tab : 0);
  // the largest dynamic size allowed so far (the default allows 48 KB less the static
  // shared memory)
  static int attr = 0;
  if (smem > attr) {
    GPTQ_CUDA(cudaFuncSetAttribute(dequant_matmul_kernel<BITS, NT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    attr = smem;
  }
  GPTQ_LAUNCH(GPTQ_K_DEQUANT_MATMUL, s, (dequant_matmul_kernel<BITS, NT>), grid, DQ_THREADS, smem,
              b);
}

template <int BITS>
void launch_bits(const DqArgs& a, cudaStream_t s) {
  if (a.n == 1) launch_nt<BITS, 1>(a, s);
  else launch_nt<BITS, 8>(a, s);
}

// W_hat[r, c] = s[g, r] (code[r, c] - z[g, r]), g = g_idx[c], as bf16 or float32,
// row-major.  A CTA takes 32 rows x 128 columns: the packed words are read across its
// rows, decoded into a shared tile and written back along the rows.
template <int BITS, typename T>
__global__ void __launch_bounds__(256) dequantize_kernel(const int32_t* __restrict__ qweight,
                                                         const float* __restrict__ scales,
                                                         const int32_t* __restrict__ qzeros,
                                                         const int32_t* __restrict__ g_idx,
                                                         int m, int d, int G,
                                                         T* __restrict__ W, DevStatus* st) {
  __shared__ float tile[32][129];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 128;
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(qweight);
  const uint32_t* qz = reinterpret_cast<const uint32_t*>(qzeros);
  const int zwords = BITS * m / 32;
  {
    // thread: row r0 + (tid % 32) (a warp reads 32 rows' words together), columns
    // 16 run .. 16 run + 15 of the tile
    const int rl = threadIdx.x % 32, run = threadIdx.x / 32;
    const int r = r0 + rl;
    const int cb = c0 + 16 * run;
    if (r < m && cb < d) {
      const int zbit = BITS * r;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int col = cb + c;
        if (col >= d) break;
        int g = g_idx[col];
        if (g < 0 || g >= G) {
          dev_fail(st, GPTQ_ERR_INVALID_ARG, col + 1);
          g = 0;
        }
        const int bit = BITS * col;
        const int w = bit >> 5, sh = bit & 31;
        uint32_t v = qw[static_cast<size_t>(w) * m + r] >> sh;
        if (sh + BITS > 32) v |= qw[static_cast<size_t>(w + 1) * m + r] << (32 - sh);
        const float cv = static_cast<float>(v & ((1u << BITS) - 1u));
        const float sv = scales[static_cast<size_t>(g) * m + r];
        const float zv = zero_of<BITS>(qz, zwords, g, zbit);
        tile[rl][16 * run + c] = sv * (cv - zv);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 32 * 128; e += 256) {
    const int rl = e / 128, c = e % 128;
    const int r = r0 + rl, col = c0 + c;
    if (r < m && col < d) {
      if constexpr (sizeof(T) == 2) {
        W[static_cast<size_t>(r) * d + col] = __float2bfloat16_rn(tile[rl][c]);
      } else {
        W[static_cast<size_t>(r) * d + col] = tile[rl][c];
      }
    }
  }
}

template <int BITS>
void launch_dequantize_bits(const int32_t* qweight, const float* scales, const int32_t* qzeros,
                            const int32_t* g_idx, int m, int d, int G, void* W, bool w_bf16,
                            DevStatus* st, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(d, 128)), static_cast<unsigned>(ceil_div(m, 32)));
  if (w_bf16) {
    GPTQ_LAUNCH(GPTQ_K_DEQUANTIZE, s, (dequantize_kernel<BITS, __nv_bfloat16>), grid, 256, 0,
                qweight, scales, qzeros, g_idx, m, d, G, static_cast<__nv_bfloat16*>(W), st);
  } else {
    GPTQ_LAUNCH(GPTQ_K_DEQUANTIZE, s, (dequantize_kernel<BITS, float>), grid, 256, 0, qweight,
                scales, qzeros, g_idx, m, d, G, static_cast<float*>(W), st);
  }
}

}  // namespace

void launch_dequantize(const int32_t* qweight, const float* scales, const int32_t* qzeros,
                       const int32_t* g_idx, int m, int d, int bits, int G, void* W, bool w_bf16,
                       DevStatus* st, cudaStream_t s) {
  if (m <= 0 || d <= 0) return;
  switch (bits) {
    case 2: launch_dequantize_bits<2>(qweight, scales, qzeros, g_idx, m, d, G, W, w_bf16, st, s); break;
    case 3: launch_dequantize_bits<3>(qweight, scales, qzeros, g_idx, m, d, G, W, w_bf16, st, s); break;
    case 4: launch_dequantize_bits<4>(qweight, scales, qzeros, g_idx, m, d, G, W, w_bf16, st, s); break;
    default: launch_dequantize_bits<8>(qweight, scales, qzeros, g_idx, m, d, G, W, w_bf16, st, s); break;
  }
}

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
  a.table = 0;  // chosen per launch
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
