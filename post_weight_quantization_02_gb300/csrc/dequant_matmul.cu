// dequant_matmul.cu: the product a W4A16-style serving kernel computes straight from the
// packed checkpoint ("GPTQ Architecture, in depth", "Packing, tooling and serving": the
// kernel unpacks each code and dequantises it with its group's scale and zero point just
// before the multiply):
//   y[t, r] = sum_c x[t, c] * s[g, r] * (code[r, c] - z[g, r]),  g = g_idx[c].
// It reads the checkpoint exactly as gptq_quantize_layer writes it, so it also checks
// the packing end to end.
//
// Design: two threads per output row, taking alternate 128-column chunks of the CTA's
// slice.  The packed words go through a shared-memory ring of two stages (a stage: the
// CTA's 128 rows over 256 columns), copied with 16-byte cp.async (4 rows' words; a warp's
// copies read one word of the 128 rows, coalesced: qweight is [bits*d/32, m]).  The
// scales and packed zero words of every group of the CTA's rows are copied at the same
// time, and the first two stages are requested before anything else, so decoding can
// start as soon as stage 0 has landed while stage 1 streams in; after each stage a CTA
// barrier makes the next one visible and frees its buffer for the stage after it.
// Decoding loops over 32-column runs with the run's body unrolled: the whole kernel then
// fits the instruction cache, which a fully unrolled chunk (tens of KB of code) does not.
// No integer-to-float conversion: the float whose exponent says 2^23 and whose low
// mantissa bits hold the code is exactly 2^23 + code, so one OR and one subtraction of
// (2^23 + z) give code - z exactly.  A run whose columns share one group (every run with
// static groups) sums x (code - z) and applies the scale once; runs that mix groups
// (act-order) look up the scale and (2^23 + zero) per column from the shared table, built
// only when such a run exists, or from global memory when the table does not fit.  The
// CTA's slice of x sits in shared memory column-major.  d_in is split over the 8 CTAs of a
// cluster, and CTA 0 adds the 8 partial sums in rank order from the others' shared memory,
// so the result does not depend on timing.
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
constexpr int DQ_KC = 128;    // columns per thread's chunk of packed words
constexpr int DQ_RING = 2;    // stages in the shared-memory ring (a third one only costs
                              // occupancy: with x for eight tokens a wide layer's CTA no
                              // longer fits twice on an SM)

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

// Two floats in one 64-bit register pair, and the paired fused multiply-add of sm_100 and
// later (one instruction for both lanes, each lane rounded as the scalar fmaf).  With
// several tokens a pass pairs tokens 2p and 2p + 1 on the same weight.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Waits until at most `pending` (0 .. 2) of this thread's latest copy groups are in flight.
__device__ __forceinline__ void cp_async_wait_upto(int pending) {
  if (pending >= 2) cp_async_wait<2>();
  else if (pending == 1) cp_async_wait<1>();
  else cp_async_wait<0>();
}

// A stage is the CTA's 128 rows over DQ_HALVES * DQ_KC consecutive columns of its slice,
// half h taking columns [DQ_KC h, DQ_KC h + DQ_KC); the ring holds DQ_RING of them.
constexpr int DQ_STAGE_COLS = DQ_HALVES * DQ_KC;

template <int BITS>
constexpr int ring_bytes() {
  return DQ_RING * (BITS * DQ_KC / 32) * DQ_THREADS * static_cast<int>(sizeof(uint32_t));
}

// Shared memory bytes of the per-group table: the CTA's rows' scales and (2^23 + zero)
// as floats, and the packed zero words they come from.
template <int BITS>
constexpr int table_bytes_per_group() {
  return 2 * DQ_ROWS * static_cast<int>(sizeof(float)) +
         (BITS * DQ_ROWS / 32) * static_cast<int>(sizeof(uint32_t));
}

template <int BITS, int NT>
__global__ void __cluster_dims__(1, DQ_SPLIT, 1) __launch_bounds__(DQ_THREADS, 2)
    dequant_matmul_kernel(const DqArgs a) {
  // dynamic shared memory: when a.table, for every group the scales of the CTA's rows,
  // their (2^23 + zero) and the packed zero words; the ring of packed codes,
  // [stage][word][half][row]; x[t0 .. t0 + NT) over this CTA's slice of d_in, column-major
  // (the NT values of a column together); the slice's group indices; per 32-column run,
  // its group when every column of the run has the same one, else -1
  extern __shared__ __align__(16) float dsm[];
  constexpr int CW = BITS * DQ_KC / 32;                       // packed words per row and chunk
  constexpr int ZW = BITS * DQ_ROWS / 32;                     // zero words per group
  constexpr int WARPS = DQ_THREADS / 32;
  const int tg = a.table ? a.G : 0;
  float* stab = dsm;                                          // [tg][DQ_ROWS]
  float* ztab = stab + tg * DQ_ROWS;                          // [tg][DQ_ROWS]
  uint32_t* zraw = reinterpret_cast<uint32_t*>(ztab + tg * DQ_ROWS);  // [tg][ZW]
  uint32_t* ring = zraw + tg * ZW;                            // [DQ_RING][CW][DQ_THREADS]
  float* xs = reinterpret_cast<float*>(ring + DQ_RING * CW * DQ_THREADS);  // [kper][NT]
  int* gs = reinterpret_cast<int*>(xs + NT * a.kper);         // [kper]
  int* guni = gs + a.kper;                                    // [kper / 32]
  __shared__ float part[DQ_HALVES][NT][DQ_ROWS];
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int rl = tid % DQ_ROWS, half = tid / DQ_ROWS;         // row within the CTA, chunk parity
  const int r0 = blockIdx.x * DQ_ROWS, r = r0 + rl;
  const int rows = min(DQ_ROWS, a.m - r0);                    // a multiple of 32
  const bool row_ok = rl < rows;
  const int rank = static_cast<int>(tc::cluster_ctarank());   // the slice of d_in
  const int k0 = rank * a.kper, k1 = min(a.d, k0 + a.kper);
  const int kn_all = max(0, k1 - k0);                         // a multiple of 32
  const int nst = (kn_all + DQ_STAGE_COLS - 1) / DQ_STAGE_COLS;
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.qweight);
  const uint32_t* qz = reinterpret_cast<const uint32_t*>(a.qzeros);
  const int zwords = BITS * a.m / 32;  // words of one group's zero stream
  const int zbit = BITS * (row_ok ? r : 0);

  // stage i of the slice into ring buffer i % DQ_RING: 16 bytes (4 rows' words) per
  // copy, a warp's copies covering one word of 128 rows
  auto issue_stage = [&](int i) {
    constexpr int UNITS = DQ_HALVES * CW * (DQ_ROWS / 4);
    const int buf = i % DQ_RING;
#pragma unroll
    for (int e = tid; e < UNITS; e += DQ_THREADS) {
      const int h = e / (CW * (DQ_ROWS / 4)), u = (e / (DQ_ROWS / 4)) % CW, q = e % (DQ_ROWS / 4);
      const int kc = k0 + i * DQ_STAGE_COLS + h * DQ_KC;
      if (kc < k1 && u < BITS * min(DQ_KC, k1 - kc) / 32 && 4 * q < rows)
        cp_async16(ring + (buf * CW + u) * DQ_THREADS + h * DQ_ROWS + 4 * q,
                   qw + (static_cast<size_t>(BITS) * kc / 32 + u) * a.m + r0 + 4 * q);
    }
    cp_async_commit();
  };
  // the scales and packed zero words of every group for the CTA's rows
  auto issue_table = [&]() {
    for (int e = tid; e < tg * (DQ_ROWS / 4); e += DQ_THREADS) {
      const int g = e / (DQ_ROWS / 4), q = e % (DQ_ROWS / 4);
      if (4 * q < rows)
        cp_async16(stab + g * DQ_ROWS + 4 * q, a.scales + static_cast<size_t>(g) * a.m + r0 + 4 * q);
    }
    for (int e = tid; e < tg * ZW; e += DQ_THREADS) {
      const int g = e / ZW, i = e % ZW;
      if (i < BITS * rows / 32)
        cp_async4(zraw + e, qz + static_cast<size_t>(g) * zwords + BITS * r0 / 32 + i);
    }
    cp_async_commit();
  };
  // x of tokens t0 .. t0 + NT over the slice, four values per thread at a time
  auto x_load = [&](float (&v)[4], int e0, int64_t t0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * DQ_THREADS;
      const int c = e / NT, t = e % NT;
      v[u] = (e < NT * kn_all && t0 + t < a.n) ? ld_x(a, t0 + t, k0 + c) : 0.0f;
    }
  };
  auto x_store = [&](const float (&v)[4], int e0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * DQ_THREADS;
      if (e < NT * kn_all) xs[e] = v[u];
    }
  };
  // the slice's group indices, a warp per 32-column run, four runs at a time
  const int nruns = kn_all / 32;
  auto g_load = [&](int (&gv)[4], int run0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int run = run0 + u * WARPS;
      gv[u] = run < nruns ? a.g_idx[k0 + 32 * run + lane] : 0;
    }
  };
  bool mixed = false;  // a run of this warp's has columns of different groups
  auto g_store = [&](const int (&gv)[4], int run0) {
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
      const bool same = __all_sync(0xffffffffu, g == __shfl_sync(0xffffffffu, g, 0));
      if (lane == 0) guni[run] = same ? g : -1;
      mixed |= !same;
    }
  };

  // every copy the first pass needs is requested first; the loads of x and the group
  // indices overlap them
  issue_table();
  for (int i = 0; i < min(nst, DQ_RING); ++i) issue_stage(i);
  {
    float v[4];
    int gv[4];
    x_load(v, tid, 0);
    g_load(gv, warp);
    x_store(v, tid);
    g_store(gv, warp);
  }
  for (int e0 = tid + 4 * DQ_THREADS; e0 < NT * kn_all; e0 += 4 * DQ_THREADS) {
    float v[4];
    x_load(v, e0, 0);
    x_store(v, e0);
  }
  for (int run0 = warp + 4 * WARPS; run0 < nruns; run0 += 4 * WARPS) {
    int gv[4];
    g_load(gv, run0);
    g_store(gv, run0);
  }
  cp_async_wait_upto(min(nst, DQ_RING) - 1);  // the table and stage 0
  // (scale, 2^23 + zero) per group and row for runs that mix groups; a run of one
  // group reads its zero straight from the packed words
  if (__syncthreads_or(mixed) && tg > 0) {
    for (int e = tid; e < tg * DQ_ROWS; e += DQ_THREADS) {
      const int g = e / DQ_ROWS, row = e % DQ_ROWS;
      ztab[e] = kTwo23 + static_cast<float>(stream_bits<BITS>(zraw + g * ZW, BITS * row));
    }
    __syncthreads();
  }

  // (scale, 2^23 + zero) of this thread's row in group g, from global memory
  auto scale_zero_g = [&](int g) -> float2 {
    return make_float2(a.scales[static_cast<size_t>(g) * a.m + r],
                       kTwo23 + zero_of<BITS>(qz, zwords, g, zbit));
  };

  for (int64_t t0 = 0; t0 < a.n; t0 += NT) {
    if (t0 > 0) {
      // the next tokens: the first stages again (the ring is free: every thread has
      // passed the cluster barrier after its decoding) and x
      for (int i = 0; i < min(nst, DQ_RING); ++i) issue_stage(i);
      for (int e0 = tid; e0 < NT * kn_all; e0 += 4 * DQ_THREADS) {
        float v[4];
        x_load(v, e0, t0);
        x_store(v, e0);
      }
      cp_async_wait_upto(min(nst, DQ_RING) - 1);
      __syncthreads();
    }
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    // this thread's chunk of a stage in ring buffer `buf`: a loop over its 32-column
    // runs, the run's body unrolled (a small body: the whole kernel stays in the
    // instruction cache)
    auto decode = [&](int buf, int kc) {
      const int nrun = min(DQ_KC, k1 - kc) / 32;
      const uint32_t* src = ring + buf * CW * DQ_THREADS + tid;
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
          const float2 sz =
              a.table ? make_float2(stab[g0 * DQ_ROWS + rl],
                                    kTwo23 + static_cast<float>(stream_bits<BITS>(zraw + g0 * ZW, BITS * rl)))
                      : scale_zero_g(g0);
          if constexpr (NT == 1) {
            // one token: scalar (paired lanes over columns measured no faster here)
            float racc = 0.0f;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 xq = x4[c4];
              const float xv[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                racc = fmaf(xv[cc], code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)), sz.y), racc);
            }
            acc[0] = fmaf(sz.x, racc, acc[0]);
          } else {
            // lanes: tokens 2p and 2p + 1
            uint64_t r2[NT / 2];
#pragma unroll
            for (int p = 0; p < NT / 2; ++p) r2[p] = pack2(0.0f, 0.0f);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              float xv[4 * NT];
#pragma unroll
              for (int q = 0; q < NT; ++q) *reinterpret_cast<float4*>(&xv[4 * q]) = x4[c4 * NT + q];
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const float v = code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)), sz.y);
                const uint64_t v2 = pack2(v, v);
#pragma unroll
                for (int p = 0; p < NT / 2; ++p)
                  r2[p] = fma2(pack2(xv[cc * NT + 2 * p], xv[cc * NT + 2 * p + 1]), v2, r2[p]);
              }
            }
#pragma unroll
            for (int p = 0; p < NT / 2; ++p) {
              const float2 rr = unpack2(r2[p]);
              acc[2 * p] = fmaf(sz.x, rr.x, acc[2 * p]);
              acc[2 * p + 1] = fmaf(sz.x, rr.y, acc[2 * p + 1]);
            }
          }
        } else {
          // each column's own group (act-order)
          const int4* g4 = reinterpret_cast<const int4*>(gs + cb);
          uint64_t r2[NT == 1 ? 1 : NT / 2];
#pragma unroll
          for (int p = 0; p < (NT == 1 ? 1 : NT / 2); ++p) r2[p] = pack2(0.0f, 0.0f);
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
              for (int cc = 0; cc < 4; ++cc)
                sz[cc] = make_float2(stab[gg[cc] * DQ_ROWS + rl], ztab[gg[cc] * DQ_ROWS + rl]);
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) sz[cc] = scale_zero_g(gg[cc]);
            }
            if constexpr (NT == 1) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                acc[0] = fmaf(xv[cc], sz[cc].x * code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)),
                                                            sz[cc].y),
                              acc[0]);
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const float v = sz[cc].x *
                                code_minus(reg_bits<BITS>(w, BITS * (4 * c4 + cc)), sz[cc].y);
                const uint64_t v2 = pack2(v, v);
#pragma unroll
                for (int p = 0; p < NT / 2; ++p)
                  r2[p] = fma2(pack2(xv[cc * NT + 2 * p], xv[cc * NT + 2 * p + 1]), v2, r2[p]);
              }
            }
          }
          if constexpr (NT > 1) {
#pragma unroll
            for (int p = 0; p < NT / 2; ++p) {
              const float2 rr = unpack2(r2[p]);
              acc[2 * p] += rr.x;
              acc[2 * p + 1] += rr.y;
            }
          }
        }
      }
    };
    // stage i in buffer i % DQ_RING; once every thread is past stage i - 1 (the
    // barrier), its buffer takes stage i + DQ_RING - 1, in flight with the stages between
    for (int i = 0; i < nst; ++i) {
      if (i > 0) {
        cp_async_wait_upto(min(DQ_RING - 2, nst - 1 - i));
        __syncthreads();
        if (i + DQ_RING - 1 < nst) issue_stage(i + DQ_RING - 1);
      }
      const int kc = k0 + i * DQ_STAGE_COLS + half * DQ_KC;
      if (row_ok && kc < k1) decode(i % DQ_RING, kc);
    }
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

// Dynamic shared memory without the table, and the static partial sums, of one CTA.
template <int BITS, int NT>
int base_smem(int kper) {
  return ring_bytes<BITS>() + ((NT + 1) * kper + kper / 32) * static_cast<int>(sizeof(float));
}
template <int NT>
constexpr int static_smem() {
  return DQ_HALVES * NT * DQ_ROWS * static_cast<int>(sizeof(float));
}

template <int BITS, int NT>
void launch_nt(const DqArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(a.m, DQ_ROWS)), DQ_SPLIT);
  const int base = base_smem<BITS, NT>(a.kper);
  // the per-group table when two CTAs still fit on an SM (228 KB of shared memory, 1 KB
  // of it reserved per CTA, and the static partial sums)
  const int tab = a.G * table_bytes_per_group<BITS>();
  const int two_per_sm = 228 * 1024 / 2 - 1024 - static_smem<NT>();
  DqArgs b = a;
  b.table = (base + tab <= two_per_sm) ? 1 : 0;
  const int smem = base + (b.table ? tab : 0);
  // (the default limit is 48 KB less the static shared memory)
  ensure_dynamic_smem(dequant_matmul_kernel<BITS, NT>, smem);
  GPTQ_LAUNCH(GPTQ_K_DEQUANT_MATMUL, s, (dequant_matmul_kernel<BITS, NT>), grid, DQ_THREADS, smem,
              b);
}

template <int BITS>
void launch_bits(const DqArgs& a, cudaStream_t s) {
  // eight tokens per pass unless their slice of x does not fit beside the ring (a CTA may
  // have 227 KB of shared memory); then one token per pass
  if (a.n > 1 && base_smem<BITS, 8>(a.kper) + static_smem<8>() <= 227 * 1024)
    launch_nt<BITS, 8>(a, s);
  else
    launch_nt<BITS, 1>(a, s);
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
