// Float32-accurate tensor-core GEMM for the factorisation updates:
//   C[i][j] = beta C[i][j] + alpha sum_{k<K} A[i][k] B[j][k],   beta in {0, 1},
// with both operands K-major (rows of 128 consecutive k), read through tensor maps that
// cover whole matrices: the launch passes each operand's row and column offset.
//
// Each float32 operand x is split as x = hi + lo with hi = x truncated to tf32 (the
// tensor core reads the same bits as x) and lo = x - hi; the products hi*hi + hi*lo +
// lo*hi are accumulated in float32 TMEM with tcgen05.mma kind::tf32 (the dropped lo*lo is
// ~2^-21 relative).  TMA lands each K-quarter (32) of the fp32 tiles in shared memory
// with 128-byte swizzle, two quarters in flight (double-buffered), so the next quarter's
// load overlaps this quarter's split and MMAs; the CTA's threads write the lo parts
// elementwise into twin buffers (same swizzled layout) before one thread issues the MMAs.
//
// Epilogue: each warp moves 32-row x 32-column boxes of alpha D from TMEM through a
// swizzled shared buffer to C with one TMA bulk copy each: a store (beta = 0) or a
// reduce-add performed by the memory system (beta = 1), so the SM never reads C.  The C
// map spans exactly the M x N result, so partial tiles are clipped by the TMA unit; in
// `lower` mode the entries of a diagonal tile above its diagonal are sent as zeros (C
// unchanged).
//
// K is a multiple of 32 (128 for the panel steps, a superpanel's 1024 for the aggregated
// trailing updates); the K-quarters stream through the same two buffers, and every four
// quarters the TMEM sums are added into registers with round-to-nearest float32 adds.  In `lower` mode
// only the tiles on or below the diagonal of C (tile column <= tile row) are computed:
// with M > N that is a trapezoid, a triangle of N / 128 tile rows and whole rows below it.
//
// One CTA of 256 threads per 128 x 128 output tile, 96 KB of shared memory, two CTAs
// per SM.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int TM = 128, TN = 128, KQ = 32;  // K-quarter per phase
constexpr int THREADS = 256;
constexpr int A_BYTES = TM * KQ * 4;                   // 16 KB
constexpr int B_BYTES = TN * KQ * 4;                   // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// hi: two stages of (A, B) quarters; lo: one (A, B) quarter
constexpr int SMEM_BYTES = 3 * STAGE_BYTES + 1024 + 128;
constexpr int BOXB = 32 * 32 * 4;                      // one epilogue box: 32 x 32 float32
// K-quarters per TMEM accumulation chain.  The tensor core's float32 accumulation does not
// round to nearest, so its error grows with the chain; each chain covers K = 128 (as one
// panel step) and is then added into registers with round-to-nearest float32 adds.
constexpr int CHAIN_Q = 4;

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

struct TcGemmArgs {
  int a_row0, a_k0;  // operand offsets inside the tensor maps
  int b_row0, b_k0;
  int M, N;
  float alpha;
  int accumulate;  // beta = 1: reduce-add into C; beta = 0: store
  int lower;       // only tiles with row tile >= column tile; only entries j <= i change
  int n_tiles;     // column tiles
  int nq;          // K / 32
  DevStatus* st;
  uint64_t wait_ns;  // limit of each pipeline wait (the exit's drain waits use kWaitLimitNs)
};

// TMA of K-quarter ph of the A and B tiles into stage ph % 2
__device__ __forceinline__ void load_quarter(uint8_t* smem, uint64_t* bar_load,
                                             const CUtensorMap* tma, const CUtensorMap* tmb,
                                             const TcGemmArgs& g, int i0, int j0, int ph) {
  uint8_t* a_hi = smem + (ph & 1) * STAGE_BYTES;
  uint64_t* bar = bar_load + (ph & 1);
  tc::mbar_arrive_expect_tx(bar, A_BYTES + B_BYTES);
  tc::tma_load_2d(a_hi, tma, bar, g.a_k0 + ph * KQ, g.a_row0 + i0);
  tc::tma_load_2d(a_hi + A_BYTES, tmb, bar, g.b_k0 + ph * KQ, g.b_row0 + j0);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(tc::smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}

__global__ void __launch_bounds__(THREADS) gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tma,
                                                              const __grid_constant__ CUtensorMap tmb,
                                                              const __grid_constant__ CUtensorMap tmc,
                                                              const TcGemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // stage q: A hi at q * STAGE_BYTES, B hi right after it; the lo pair after both stages
  uint8_t* a_lo = smem + 2 * STAGE_BYTES;
  uint8_t* b_lo = a_lo + A_BYTES;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + 3 * STAGE_BYTES);  // [2]
  uint64_t* bar_mma = bar_load + 2;
  uint64_t* mma_drain = bar_mma + 1;  // the issuer's last commit at the exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int bi, bj;
  if (g.lower) {
    // the triangle of the first n_tiles tile rows, then whole tile rows
    const int tri = g.n_tiles * (g.n_tiles + 1) / 2;
    int rem = static_cast<int>(blockIdx.x);
    if (rem < tri) {
      bi = 0;
      while (rem > bi) { rem -= bi + 1; ++bi; }
      bj = rem;
    } else {
      rem -= tri;
      bi = g.n_tiles + rem / g.n_tiles;
      bj = rem % g.n_tiles;
    }
  } else {
    bi = blockIdx.x / g.n_tiles;
    bj = blockIdx.x % g.n_tiles;
  }
  const int i0 = bi * TM, j0 = bj * TN;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  griddep_launch_dependents();

  if (tid == 32) {
    // barriers first, then the first two K-quarters in flight while warp 0 allocates TMEM
    tc::mbar_init(bar_load, 1);
    tc::mbar_init(bar_load + 1, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    griddep_wait();
    load_quarter(smem, bar_load, &tma, &tmb, g, i0, j0, 0);
    if (g.nq > 1) load_quarter(smem, bar_load, &tma, &tmb, g, i0, j0, 1);
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  // no thread touches global memory before the previous kernel in the stream is done
  griddep_wait();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t IDESC = idesc_tf32(TM, TN, false);
  bool ok = true;
  // warp w owns TMEM lanes (tile rows) 32 (w % 4) .. and columns 64 (w / 4) .. + 64
  const int rq = warp % 4, ch = warp / 4;
  const uint32_t tmem_w = tmem + (static_cast<uint32_t>(32 * rq) << 16) + 64 * ch;
  float accr[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) accr[i] = 0.0f;

  // Every wait's outcome is made CTA-wide (__syncthreads_or) so that all threads leave the
  // loop at the same point; `landed` counts the quarters whose copies were seen to land and
  // `mmas_done` the quarters whose MMAs completed (quarters below mmas_done + 2 were loaded).
  int landed = 0, mmas_done = 0;
  for (int ph = 0; ph < g.nq && ok; ++ph) {
    uint8_t* a_hi = smem + (ph & 1) * STAGE_BYTES;
    uint8_t* b_hi = a_hi + A_BYTES;
    const bool bad_load = !tc::mbar_wait(bar_load + (ph & 1), (ph >> 1) & 1, abort_flag, g.wait_ns);
    // lo = x - trunc_tf32(x), elementwise in the same swizzled layout
    if (!bad_load) {
      const float4* src_a = reinterpret_cast<const float4*>(a_hi);
      float4* dst_a = reinterpret_cast<float4*>(a_lo);
      const float4* src_b = reinterpret_cast<const float4*>(b_hi);
      float4* dst_b = reinterpret_cast<float4*>(b_lo);
#pragma unroll
      for (int e = tid; e < A_BYTES / 16; e += THREADS) {
        float4 x = src_a[e];
        float4 y = src_b[e];
        x.x -= __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
        x.y -= __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
        x.z -= __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
        x.w -= __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
        y.x -= __uint_as_float(__float_as_uint(y.x) & 0xFFFFE000u);
        y.y -= __uint_as_float(__float_as_uint(y.y) & 0xFFFFE000u);
        y.z -= __uint_as_float(__float_as_uint(y.z) & 0xFFFFE000u);
        y.w -= __uint_as_float(__float_as_uint(y.w) & 0xFFFFE000u);
        dst_a[e] = x;
        dst_b[e] = y;
      }
    }
    tc::fence_proxy_async_shared();
    tc::fence_before();
    if (__syncthreads_or(bad_load)) { ok = false; break; }
    landed = ph + 1;
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
        const uint32_t acc0 = ((ph % CHAIN_Q) | kk) != 0 ? 1u : 0u;
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
    const bool bad_mma = !tc::mbar_wait(bar_mma, ph & 1, abort_flag, g.wait_ns);
    if (__syncthreads_or(bad_mma)) { ok = false; break; }
    mmas_done = ph + 1;
    tc::fence_after();
    // both buffers of this stage are free again: fetch the quarter after next into it
    if (tid == 32 && ph + 2 < g.nq) load_quarter(smem, bar_load, &tma, &tmb, g, i0, j0, ph + 2);
    if (ph % CHAIN_Q == CHAIN_Q - 1 || ph == g.nq - 1) {
      // end of a chain: its sums join the registers (the next chain's first MMAs
      // overwrite TMEM only after the next quarter's CTA-wide barrier)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem_w + 32 * c, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          accr[32 * c + j] = __fadd_rn(accr[32 * c + j], __uint_as_float(r[j]));
      }
      tc::fence_before();
    }
  }

  if (ok) {
    // warp w's rows and 64 columns as two 32 x 32 boxes, each staged in its own 4 KB
    // buffer (the operand buffers are free)
    const int row = i0 + 32 * rq + lane;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int colt = 64 * ch + 32 * c;  // column inside the tile
      uint8_t* box = smem + (warp * 2 + c) * BOXB;
      const float* r = accr + 32 * c;
      uint8_t* srow = box + lane * 128;  // 128-byte swizzle: chunk j at (j ^ (lane % 8))
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int col = j0 + colt + 4 * j;
        float4 v;
        v.x = (!g.lower || col <= row) ? g.alpha * r[4 * j] : 0.0f;
        v.y = (!g.lower || col + 1 <= row) ? g.alpha * r[4 * j + 1] : 0.0f;
        v.z = (!g.lower || col + 2 <= row) ? g.alpha * r[4 * j + 2] : 0.0f;
        v.w = (!g.lower || col + 3 <= row) ? g.alpha * r[4 * j + 3] : 0.0f;
        *reinterpret_cast<float4*>(srow + ((j ^ (lane & 7)) << 4)) = v;
      }
      tc::fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0 && i0 + 32 * rq < g.M && j0 + colt < g.N) {
        if (g.accumulate) tc::tma_reduce_add_2d(&tmc, box, j0 + colt, i0 + 32 * rq);
        else tma_store_2d(&tmc, box, j0 + colt, i0 + 32 * rq);
        tc::bulk_commit_group();
      }
    }
    // the boxes have been read out of shared memory; the memory system completes the
    // stores / reduce-adds before the grid is finished
    if (lane == 0) tc::bulk_wait_group_read0();
  } else {
    *abort_flag = 1;
    if (lane == 0) {
      dev_fail(g.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&g.st->timeouts, 1);
    }
  }
  // Drain, on every exit, so that nothing is in flight when the CTA's memory goes away:
  // the MMAs (one more commit, which arrives once every earlier MMA has completed) and the
  // copies of the quarters loaded but not seen to land (at most two, one per stage; the
  // slot's previous quarter was seen, so its current phase is this quarter's).
  bool drained = true;
  if (tid == 0) {
    tc::mma_commit(mma_drain);
    drained = tc::mbar_wait_for(mma_drain, 0, kWaitLimitNs);
  }
  if (tid == 32) {
    const int loaded = min(g.nq, mmas_done + 2);
    for (int q = landed; q < loaded; ++q)
      if (!tc::mbar_wait_for(bar_load + (q & 1), static_cast<uint32_t>(q >> 1) & 1u, kWaitLimitNs))
        drained = false;
  }
  if (!drained) {
    // a drain wait ran out (nothing should be left to land): record it, and give whatever
    // is still in flight time to land before the memory goes away
    dev_fail(g.st, GPTQ_ERR_TIMEOUT, 1);
    atomicAdd(&g.st->timeouts, 1);
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

// ---------------------------------------------------------------- long-K variant

// For K >= 256 (a superpanel's aggregated updates, K = 1024) the lo parts of both
// operands come precomputed from global memory (each operand element is split once, not
// once per tile that reads it), and a warp-specialised kernel on pairs of SMs keeps the
// tensor core fed.  What bounds the tf32x3 product is the operand bytes that must reach
// an SM per MMA cycle: a unit is one 256 x 256 tile of C computed by a cluster of two
// CTAs with paired-SM MMAs (tcgen05.mma.cta_group::2, M = 256): the even CTA's TMEM holds
// rows 0..127 of the tile and the odd CTA's rows 128..255, each CTA's shared memory holds
// its own 128 rows of A and one half (128 rows) of B, hi and lo, and the tensor cores of
// the pair read each other's half of B.  Per K-quarter an SM then receives 64 KB for
// 1536 MMA cycles, two thirds of what a one-SM 128 x 256 tile needs.
//   warp 0       TMA producer (both CTAs): A hi, A lo, B hi, B lo quarters into stage
//                q % NS, completion counted on the even CTA's barrier
//   warp 1       TMEM owner (both CTAs, paired allocation of two 256-column
//                accumulators); in the even CTA also the MMA issuer
//   warp 2       in the even CTA: waits for each quarter's copies (and, at a chain start,
//                for its accumulator to be drained by both CTAs) and releases warp 1
//                through a named barrier, so that the issuing warp never waits on an
//                mbarrier
//   warps 3..10  (both CTAs) drain each finished chain from TMEM into registers
//                (round-to-nearest adds) while the next chain accumulates in the other
//                accumulator; write the CTA's 128 x 256 part of the tile
struct PresplitPair {
  static constexpr int PART = TM * KQ * 4;   // 16 KB: 128 rows x one K-quarter
  static constexpr int STAGE = 4 * PART;     // A hi, A lo, B hi, B lo (this CTA's half)
  static constexpr int NS = 3;
  static constexpr int TNP = 256;            // columns of a unit
  static constexpr int WORKERS = 8;
  static constexpr int COLS = TNP / 2;       // columns per worker thread
  static constexpr int THREADS = 32 * (3 + WORKERS);
  static constexpr int SMEM = NS * STAGE + 1024 + 256;
  static_assert(SMEM <= 232448, "shared memory of one CTA");
  static_assert(WORKERS * (COLS / 32) * BOXB <= NS * STAGE, "epilogue boxes fit");
};
constexpr uint32_t kPsHandoff = 1;  // named barrier of warps 1 and 2

struct PresplitArgs {
  TcGemmArgs g;            // n_tiles: column tiles of 256
  int a_lo_row0, a_lo_k0;  // the lo parts' offsets in their own maps
  int b_lo_row0, b_lo_k0;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PresplitPair::THREADS, 1)
    gemm_tf32x3_presplit_kernel(const __grid_constant__ CUtensorMap tma,
                                const __grid_constant__ CUtensorMap tma_lo,
                                const __grid_constant__ CUtensorMap tmb,
                                const __grid_constant__ CUtensorMap tmb_lo,
                                const __grid_constant__ CUtensorMap tmc, const PresplitArgs pa) {
  using P = PresplitPair;
  const TcGemmArgs& g = pa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::NS * P::STAGE);  // [NS] copies
  uint64_t* empty = full + P::NS;                                         // [NS] MMAs done
  uint64_t* accfull = empty + P::NS;                                      // [2]
  uint64_t* accempty = accfull + 2;                                       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [0]: quarters this CTA's producer issued; [1] (even CTA): quarters the waiter saw land
  int* counts = const_cast<int*>(abort_flag) + 1;
  uint64_t* mma_drain = reinterpret_cast<uint64_t*>(counts + 2);  // the issuer's last commit

  // unit: row pair pi (256 rows), column tile bj (256 columns); in lower mode only the
  // units that reach the diagonal or below it (bj <= pi)
  const int unit = static_cast<int>(blockIdx.x / 2);
  int pi = 0, bj = 0;
  if (g.lower) {
    int rem = unit;
    for (;; ++pi) {
      const int cnt = min(pi + 1, g.n_tiles);
      if (rem < cnt) { bj = rem; break; }
      rem -= cnt;
    }
  } else {
    pi = unit / g.n_tiles;
    bj = unit % g.n_tiles;
  }
  const int crank = static_cast<int>(tc::cluster_ctarank());
  const int i0 = pi * 2 * TM + crank * TM;   // this CTA's rows of C
  const int j0 = bj * P::TNP;                // the unit's columns of C
  const int jb = j0 + crank * (P::TNP / 2);  // this CTA's half of B
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < P::NS; ++s) {
      tc::mbar_init(&full[s], 1);   // the even CTA's: both CTAs' bytes
      tc::mbar_init(&empty[s], 1);  // the pair's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accfull[b], 1);
      tc::mbar_init(&accempty[b], 2 * P::WORKERS);  // the even CTA's: both CTAs' workers
    }
    tc::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    counts[0] = counts[1] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, 2 * P::TNP);
    tc::tmem_relinquish_pair();
  }
  // no thread touches global memory before the previous kernel in the stream is done
  griddep_wait();
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // both CTAs' barriers exist before either copies into them
  tc::fence_after();
  const uint32_t tmem_base = *tmem_slot;
  constexpr uint32_t IDESC = idesc_tf32(2 * TM, P::TNP, false);  // paired: M = 256
  const int nq = g.nq;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int q = 0;
      for (; q < nq; ++q) {
        const int s = q % P::NS;
        const uint32_t ph = static_cast<uint32_t>(q / P::NS) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort_flag, g.wait_ns)) { ok = false; break; }
        uint8_t* base = smem + s * P::STAGE;
        const uint32_t bar = tc::mapa_shared(tc::smem_u32(&full[s]), 0);
        if (crank == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * P::STAGE);
        tc::tma_load_2d_pair(base, &tma, bar, g.a_k0 + q * KQ, g.a_row0 + i0);
        tc::tma_load_2d_pair(base + P::PART, &tma_lo, bar, pa.a_lo_k0 + q * KQ,
                             pa.a_lo_row0 + i0);
        tc::tma_load_2d_pair(base + 2 * P::PART, &tmb, bar, g.b_k0 + q * KQ, g.b_row0 + jb);
        tc::tma_load_2d_pair(base + 3 * P::PART, &tmb_lo, bar, pa.b_lo_k0 + q * KQ,
                             pa.b_lo_row0 + jb);
      }
      counts[0] = q;  // the quarters below q were issued
    }
  } else if (crank == 0 && (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------ MMA issuer and waiter
    const bool waiter = (warp == 2);
    int seen = 0;  // quarters whose copies the waiter saw land
    for (int q = 0; q < nq; ++q) {
      const int s = q % P::NS;
      const uint32_t ph = static_cast<uint32_t>(q / P::NS) & 1u;
      const int chain = q / CHAIN_Q, acc = chain & 1;
      bool bad = false;
      if (waiter && lane == 0) {
        if (q % CHAIN_Q == 0)
          bad = !tc::mbar_wait(&accempty[acc], (static_cast<uint32_t>(chain >> 1) & 1u) ^ 1u,
                               abort_flag, g.wait_ns);
        if (!bad) bad = !tc::mbar_wait(&full[s], ph, abort_flag, g.wait_ns);
        if (!bad) ++seen;
      }
      if (tc::handoff_or(kPsHandoff, 64, bad)) { ok = false; break; }
      if (!waiter && lane == 0) {
        tc::fence_after();
        const uint32_t ah = tc::smem_u32(smem + s * P::STAGE);
        const uint32_t al = ah + P::PART, bh = ah + 2 * P::PART, bl = ah + 3 * P::PART;
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * P::TNP);
#pragma unroll
        for (int kk = 0; kk < KQ / 8; ++kk) {
          const uint64_t dah = tc::smem_desc(ah + 32 * kk, 16, 1024, tc::kSwizzle128B);
          const uint64_t dal = tc::smem_desc(al + 32 * kk, 16, 1024, tc::kSwizzle128B);
          const uint64_t dbh = tc::smem_desc(bh + 32 * kk, 16, 1024, tc::kSwizzle128B);
          const uint64_t dbl = tc::smem_desc(bl + 32 * kk, 16, 1024, tc::kSwizzle128B);
          const uint32_t acc0 = ((q % CHAIN_Q) | kk) != 0 ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
              "l"(dah), "l"(dbh), "r"(IDESC), "r"(acc0)
              : "memory");
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
              "l"(dah), "l"(dbl), "r"(IDESC), "r"(1u)
              : "memory");
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
              "l"(dal), "l"(dbh), "r"(IDESC), "r"(1u)
              : "memory");
        }
        tc::mma_commit_pair(&empty[s], static_cast<uint16_t>(0x3));
        if (q % CHAIN_Q == CHAIN_Q - 1 || q == nq - 1)
          tc::mma_commit_pair(&accfull[acc], static_cast<uint16_t>(0x3));
      }
    }
    if (waiter && lane == 0) counts[1] = seen;
  } else if (warp >= 3) {
    // ------------------------------------------------------------ workers
    const int wk = warp - 3;                       // 0 .. WORKERS - 1
    const int rq = warp % 4, half = wk / 4;        // TMEM lane quarter, column half
    const uint32_t tmem_w =
        tmem_base + (static_cast<uint32_t>(32 * rq) << 16) + static_cast<uint32_t>(P::COLS * half);
    float accr[P::COLS];
#pragma unroll
    for (int i = 0; i < P::COLS; ++i) accr[i] = 0.0f;
    const int nchain = (nq + CHAIN_Q - 1) / CHAIN_Q;
    for (int chain = 0; chain < nchain; ++chain) {
      const int acc = chain & 1;
      if (!tc::mbar_wait(&accfull[acc], static_cast<uint32_t>(chain >> 1) & 1u, abort_flag,
                         g.wait_ns)) {
        ok = false;
        break;
      }
      tc::fence_after();
#pragma unroll
      for (int c = 0; c < P::COLS / 16; ++c) {
        uint32_t r[16];
        tc::tmem_ld_32x32b_x16(tmem_w + static_cast<uint32_t>(acc * P::TNP) + 16 * c, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          accr[16 * c + j] = __fadd_rn(accr[16 * c + j], __uint_as_float(r[j]));
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&accempty[acc]), 0));
    }
    if (ok) {
      // every MMA of the pair has completed (the last chain's commit) and every copy was
      // consumed: this CTA's stages hold the epilogue's boxes, COLS / 32 per worker warp
      const int row = i0 + 32 * rq + lane;
#pragma unroll
      for (int c = 0; c < P::COLS / 32; ++c) {
        const int colt = P::COLS * half + 32 * c;
        uint8_t* box = smem + (wk * (P::COLS / 32) + c) * BOXB;
        const float* r = accr + 32 * c;
        uint8_t* srow = box + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int col = j0 + colt + 4 * j;
          float4 v;
          v.x = (!g.lower || col <= row) ? g.alpha * r[4 * j] : 0.0f;
          v.y = (!g.lower || col + 1 <= row) ? g.alpha * r[4 * j + 1] : 0.0f;
          v.z = (!g.lower || col + 2 <= row) ? g.alpha * r[4 * j + 2] : 0.0f;
          v.w = (!g.lower || col + 3 <= row) ? g.alpha * r[4 * j + 3] : 0.0f;
          *reinterpret_cast<float4*>(srow + ((j ^ (lane & 7)) << 4)) = v;
        }
        tc::fence_proxy_async_shared();
        __syncwarp();
        // in lower mode a box wholly above the diagonal adds only zeros: skip it
        const bool live = !g.lower || j0 + colt <= i0 + 32 * rq + 31;
        if (lane == 0 && live && i0 + 32 * rq < g.M && j0 + colt < g.N) {
          if (g.accumulate) tc::tma_reduce_add_2d(&tmc, box, j0 + colt, i0 + 32 * rq);
          else tma_store_2d(&tmc, box, j0 + colt, i0 + 32 * rq);
          tc::bulk_commit_group();
        }
      }
      if (lane == 0) tc::bulk_wait_group_read0();
    }
  }

  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) {
      dev_fail(g.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&g.st->timeouts, 1);
    }
  }
  // Drain, on every exit, so that nothing is in flight when the CTAs' memory goes away:
  // the issuer's MMAs (one more commit, which arrives once every earlier MMA of the pair
  // has completed), then, once both producers have stopped, the pair's copies.
  bool drained = true;
  if (crank == 0 && warp == 1 && lane == 0) {
    tc::mma_commit_pair(mma_drain, static_cast<uint16_t>(1u));
    drained = tc::mbar_wait_for(mma_drain, 0, kWaitLimitNs);
  }
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // both producers have stopped; their counts are visible
  if (crank == 0 && threadIdx.x == 0) {
    const int odd = static_cast<int>(
        tc::ld_shared_cluster_u32(tc::mapa_shared(tc::smem_u32(counts), 1u)));
    drained = tc::drain_pair_stages(full, P::NS, counts[1], counts[0], odd, P::STAGE);
  }
  if (!drained) {
    // a drain wait ran out (nothing should be left to land): record it, and give whatever
    // is still in flight time to land before the memory goes away
    dev_fail(g.st, GPTQ_ERR_TIMEOUT, 1);
    atomicAdd(&g.st->timeouts, 1);
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // the pair's copies have landed; neither CTA signals the other any more
  if (warp == 1) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc_pair(tmem_base, 2 * P::TNP);
  }
}

// lo = x - trunc_tf32(x) for a rows x cols block (cols a multiple of 4, rows 16-byte
// aligned); one thread per 4 elements
__global__ void split_lo_kernel(const float* __restrict__ src, int ld, int rows, int cols,
                                float* __restrict__ lo, int ld_lo) {
  const int r = blockIdx.y;
  const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (r >= rows || c >= cols) return;
  float4 x = *reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * ld + c);
  x.x -= __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
  x.y -= __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
  x.z -= __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
  x.w -= __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
  *reinterpret_cast<float4*>(lo + static_cast<size_t>(r) * ld_lo + c) = x;
}

}  // namespace

void make_gemm_map(CUtensorMap* map, const float* base, int rows, int cols, int ld) {
  make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, static_cast<uint64_t>(cols),
               static_cast<uint64_t>(rows), static_cast<uint64_t>(ld) * 4, KQ, TM,
               CU_TENSOR_MAP_SWIZZLE_128B);
}

void launch_gemm_tf32x3(int kind, const CUtensorMap& ma, int a_row0, int a_k0,
                        const CUtensorMap& mb, int b_row0, int b_k0, int K, float* C, int ldc,
                        int M, int N, float alpha, float beta, bool lower, DevStatus* st,
                        cudaStream_t s, bool pdl) {
  if (M <= 0 || N <= 0) return;
  if ((beta != 0.0f && beta != 1.0f) || (lower && (beta != 1.0f || M < N)) || K <= 0 ||
      K % KQ != 0) {
    fail(GPTQ_ERR_INVALID_ARG,
         "launch_gemm_tf32x3: beta must be 0 or 1 (1 and M >= N in lower mode), K a positive "
         "multiple of 32");
  }
  // the M x N result, in boxes of 32 x 32 (128-byte rows, swizzled like the staging)
  CUtensorMap mc;
  make_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N),
               static_cast<uint64_t>(M), static_cast<uint64_t>(ldc) * 4, 32, 32,
               CU_TENSOR_MAP_SWIZZLE_128B);
  TcGemmArgs g;
  g.a_row0 = a_row0;
  g.a_k0 = a_k0;
  g.b_row0 = b_row0;
  g.b_k0 = b_k0;
  g.M = M;
  g.N = N;
  g.alpha = alpha;
  g.accumulate = (beta != 0.0f) ? 1 : 0;
  g.lower = lower ? 1 : 0;
  const int tm = static_cast<int>(ceil_div(M, TM)), tn = static_cast<int>(ceil_div(N, TN));
  g.n_tiles = tn;
  g.nq = K / KQ;
  g.st = st;
  g.wait_ns = wait_limit_ns();
  const unsigned grid = lower ? static_cast<unsigned>(tn * (tn + 1) / 2 + (tm - tn) * tn)
                              : static_cast<unsigned>(tm * tn);
  ensure_dynamic_smem(gemm_tf32x3_kernel, SMEM_BYTES);
  if (pdl) {
    GPTQ_LAUNCH_PDL(kind, s, gemm_tf32x3_kernel, grid, THREADS, SMEM_BYTES, ma, mb, mc, g);
  } else {
    GPTQ_LAUNCH(kind, s, gemm_tf32x3_kernel, grid, THREADS, SMEM_BYTES, ma, mb, mc, g);
  }
}

void launch_split_lo(const float* src, int ld, int rows, int cols, float* lo, int ld_lo,
                     cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return;
  dim3 grid(static_cast<unsigned>(ceil_div(cols / 4, 256)), static_cast<unsigned>(rows));
  GPTQ_LAUNCH(GPTQ_K_POTRF_UPDATE, s, split_lo_kernel, grid, 256, 0, src, ld, rows, cols, lo,
              ld_lo);
}

void launch_gemm_tf32x3_presplit(int kind, const CUtensorMap& ma, int a_row0, int a_k0,
                                 const CUtensorMap& ma_lo, int a_lo_row0, int a_lo_k0,
                                 const CUtensorMap& mb, int b_row0, int b_k0,
                                 const CUtensorMap& mb_lo, int b_lo_row0, int b_lo_k0, int K,
                                 float* C, int ldc, int M, int N, float alpha, float beta,
                                 bool lower, DevStatus* st, cudaStream_t s, bool pdl) {
  if (M <= 0 || N <= 0) return;
  if ((beta != 0.0f && beta != 1.0f) || (lower && (beta != 1.0f || M < N)) || K <= 0 ||
      K % KQ != 0) {
    fail(GPTQ_ERR_INVALID_ARG,
         "launch_gemm_tf32x3_presplit: beta must be 0 or 1 (1 and M >= N in lower mode), K a "
         "positive multiple of 32");
  }
  CUtensorMap mc;
  make_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N),
               static_cast<uint64_t>(M), static_cast<uint64_t>(ldc) * 4, 32, 32,
               CU_TENSOR_MAP_SWIZZLE_128B);
  PresplitArgs pa;
  pa.g.a_row0 = a_row0;
  pa.g.a_k0 = a_k0;
  pa.g.b_row0 = b_row0;
  pa.g.b_k0 = b_k0;
  pa.g.M = M;
  pa.g.N = N;
  pa.g.alpha = alpha;
  pa.g.accumulate = (beta != 0.0f) ? 1 : 0;
  pa.g.lower = lower ? 1 : 0;
  pa.g.nq = K / KQ;
  pa.g.st = st;
  pa.g.wait_ns = wait_limit_ns();
  pa.a_lo_row0 = a_lo_row0;
  pa.a_lo_k0 = a_lo_k0;
  pa.b_lo_row0 = b_lo_row0;
  pa.b_lo_k0 = b_lo_k0;
  using P = PresplitPair;
  const int tp = static_cast<int>(ceil_div(M, 2 * TM));  // row pairs
  const int tn = static_cast<int>(ceil_div(N, P::TNP));
  pa.g.n_tiles = tn;
  unsigned units = 0;
  if (lower) {
    for (int p = 0; p < tp; ++p) units += static_cast<unsigned>(std::min(p + 1, tn));
  } else {
    units = static_cast<unsigned>(tp * tn);
  }
  const unsigned grid = 2 * units;  // one cluster of two CTAs per unit
  ensure_dynamic_smem(gemm_tf32x3_presplit_kernel, P::SMEM);
  if (pdl) {
    GPTQ_LAUNCH_PDL(kind, s, gemm_tf32x3_presplit_kernel, grid, P::THREADS, P::SMEM, ma, ma_lo,
                    mb, mb_lo, mc, pa);
  } else {
    GPTQ_LAUNCH(kind, s, gemm_tf32x3_presplit_kernel, grid, P::THREADS, P::SMEM, ma, ma_lo, mb,
                mb_lo, mc, pa);
  }
}

}  // namespace gptq
