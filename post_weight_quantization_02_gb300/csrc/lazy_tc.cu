// The lazy trailing update on the tensor cores: W[:, c_begin:c_end] -= Err U[k-range, same].
//
// "Same Ruler, Smarter Placement: GPTQ", section 1.8, and "GPTQ Architecture, in
// depth", "The algorithm in code": after a block of columns is quantised, its
// accumulated errors are pushed into every later column as one matrix product.  The
// driver defers in two levels: after each 128-column block only the rest of its
// 1024-column superblock is updated (K = 128); after the superblock, every later column
// at once (K = 1024), so the far columns of W are rewritten an eighth as often.  W is
// float32 and the update must keep float32 accuracy (the next blocks round these
// values), so each operand is split into two bf16 parts, x = hi + lo, and the product is
// accumulated in float32 TMEM as hi*hi + hi*lo + lo*hi (the lo*lo term, ~2^-16
// relative, is dropped).
//
// Persistent kernel on pairs of SMs (clusters of two CTAs, one per SM) running paired
// MMAs: a unit is one 256 x 256 tile of W, the even CTA's TMEM holding rows 0..127 of it
// and the odd CTA's rows 128..255.  K goes in chunks of 64 through a three-stage operand
// pipeline; each CTA's stage holds its own 128 rows of ErrT and one half (128 columns) of
// U, hi and lo, 64 KB, and the tensor cores of the pair read each other's half of U.  Per
// chunk an SM so takes in 64 KB for 1536 MMA cycles, two thirds of what a one-SM
// 128 x 256 tile needs (the operand bytes that reach an SM per MMA cycle bound this
// product).
//   warp 0      TMA (both CTAs): ErrT hi/lo [64 k x 128 rows] and U hi/lo [64 k x 128
//               columns] per chunk, both MN-major; completion on the even CTA's barrier
//   warp 1      TMEM owner (both CTAs, paired allocation); in the even CTA also the MMA
//               issuer: 4 k-steps x 3 tcgen05.mma.cta_group::2 256x256x16 per chunk
//   warp 10     in the even CTA: waits for each chunk's data (and, per tile, for the
//               accumulator) and releases warp 1 through a named barrier, so that the
//               issuing warp never waits on an mbarrier (which would drain the tensor pipe
//               each chunk)
//   warps 2..9  epilogue (both CTAs): TMEM -> registers -> -D into a swizzled shared box
//               -> TMA reduce-add into W.  The memory system applies W += (-D) (one
//               rounding, as a float32 subtraction); the SM never reads W.
// Two 256-column TMEM accumulators let the epilogue of one tile overlap the MMAs of the
// next.
#include <cuda_bf16.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;      // BM rows per CTA, 2 BM per unit
constexpr int BOX = 64 * 64 * 2;                 // one TMA box: 64 x 64 bf16
constexpr int A_PART = BM * BK * 2;              // per part (hi or lo): 16 KB
constexpr int B_PART = (BN / 2) * BK * 2;        // this CTA's half of U: 16 KB
constexpr int STAGE = 2 * A_PART + 2 * B_PART;   // 64 KB
constexpr int NSTAGE = 3;
constexpr int EPI_WARPS = 8;
constexpr int STG_BYTES = 32 * 32 * 4;           // per epilogue warp: 32 rows x 32 columns
constexpr int SMEM_BYTES = NSTAGE * STAGE + EPI_WARPS * STG_BYTES + 1024 + 256;
constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;
constexpr int WAITER_WARP = 2 + EPI_WARPS;
constexpr uint32_t kHandoffBarrier = 1;  // named barrier of warps 1 and WAITER_WARP
constexpr uint32_t IDESC = tc::idesc_bf16_f32(2 * BM, BN, true, true);  // paired: M = 256
static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");

struct LazyArgs {
  int m, d;
  int e_row0;      // first ErrT row (k) of the product
  int u_row0;      // first U row (k)
  int nk;          // K / 64
  int c_begin;     // first W column updated
  int c_end;       // columns >= c_end are left alone
  int n_mt, n_nt;  // row-tile pairs (256 rows), column tiles
  DevStatus* st;
  uint64_t wait_ns;  // limit of each pipeline wait (the exit's drain waits use kWaitLimitNs)
};

// offsets inside a stage of part p (0 hi, 1 lo), box h
__device__ __forceinline__ uint32_t a_off(int p, int h) {
  return static_cast<uint32_t>(p * A_PART + h * BOX);
}
__device__ __forceinline__ uint32_t b_off(int p, int h) {
  return static_cast<uint32_t>(2 * A_PART + p * B_PART + h * BOX);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    lazy_tc_kernel(const __grid_constant__ CUtensorMap tm_ehi, const __grid_constant__ CUtensorMap tm_elo,
                   const __grid_constant__ CUtensorMap tm_uhi, const __grid_constant__ CUtensorMap tm_ulo,
                   const __grid_constant__ CUtensorMap tm_w, const LazyArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stg_base = smem + NSTAGE * STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_base + EPI_WARPS * STG_BYTES);  // [NSTAGE]
  uint64_t* empty = full + NSTAGE;                                                 // [NSTAGE]
  uint64_t* accfull = empty + NSTAGE;                                              // [2]
  uint64_t* accempty = accfull + 2;                                                // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [0]: stages this CTA's producer issued; [1] (even CTA): stages the waiter saw land
  int* counts = const_cast<int*>(abort_flag) + 1;
  uint64_t* mma_drain = reinterpret_cast<uint64_t*>(counts + 2);  // the issuer's last commit

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int crank = static_cast<int>(tc::cluster_ctarank());
  const int n_units = a.n_mt * a.n_nt;
  const int unit0 = static_cast<int>(blockIdx.x / 2), unit_step = static_cast<int>(gridDim.x / 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      tc::mbar_init(&full[s], 1);   // the even CTA's: both CTAs' bytes
      tc::mbar_init(&empty[s], 1);  // the pair's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accfull[b], 1);
      tc::mbar_init(&accempty[b], 2 * EPI_WARPS);  // the even CTA's: both CTAs' epilogues
    }
    tc::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    counts[0] = counts[1] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, 512);
    tc::tmem_relinquish_pair();
  }
  // launched as a programmatic dependent of the column loop before it: the set-up above
  // overlaps its tail, and no global memory is touched before it has completed
  griddep_launch_dependents();
  griddep_wait();
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // both CTAs' barriers exist before either copies into them
  tc::fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    for (int u = unit0; u < n_units && ok; u += unit_step) {
      const int mt = u % a.n_mt, nt = u / a.n_mt;
      const int r0 = mt * 2 * BM + crank * BM;                 // this CTA's rows of W
      const int c0 = a.c_begin + nt * BN + crank * (BN / 2);   // this CTA's half of U
      for (int kc = 0; kc < a.nk; ++kc, ++it) {
        const int s = static_cast<int>(it % NSTAGE);
        const uint32_t ph = (it / NSTAGE) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
        uint8_t* base = smem + s * STAGE;
        const uint32_t bar = tc::mapa_shared(tc::smem_u32(&full[s]), 0);
        if (crank == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * STAGE);
        const int ke = a.e_row0 + kc * BK, ku = a.u_row0 + kc * BK;
        for (int h = 0; h < 2; ++h) {
          tc::tma_load_2d_pair(base + a_off(0, h), &tm_ehi, bar, r0 + 64 * h, ke);
          tc::tma_load_2d_pair(base + a_off(1, h), &tm_elo, bar, r0 + 64 * h, ke);
          tc::tma_load_2d_pair(base + b_off(0, h), &tm_uhi, bar, c0 + 64 * h, ku);
          tc::tma_load_2d_pair(base + b_off(1, h), &tm_ulo, bar, c0 + 64 * h, ku);
        }
      }
    }
    counts[0] = static_cast<int>(it);  // the stage counter stops at the first one not issued
  } else if (crank == 0 && (warp == 1 || warp == WAITER_WARP)) {
    // ------------------------------------------------------------ MMA issuer and its
    // waiter: both walk the same chunks; the waiter's lane 0 waits, then both warps meet
    // at the named barrier, which also carries a failed wait
    const bool waiter = (warp == WAITER_WARP);
    uint32_t it = 0;
    int acc = 0;
    uint32_t accphase = 0;
    int seen = 0;  // stages whose copies the waiter saw land
    const uint32_t sbase = tc::smem_u32(smem);
    for (int u = unit0; u < n_units && ok; u += unit_step) {
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kc = 0; kc < a.nk; ++kc, ++it) {
        const int s = static_cast<int>(it % NSTAGE);
        const uint32_t ph = (it / NSTAGE) & 1u;
        bool bad = false;
        if (waiter && lane == 0) {
          if (kc == 0) bad = !tc::mbar_wait(&accempty[acc], accphase ^ 1u, abort_flag, a.wait_ns);
          if (!bad) bad = !tc::mbar_wait(&full[s], ph, abort_flag, a.wait_ns);
          if (!bad) ++seen;
        }
        if (tc::handoff_or(kHandoffBarrier, 64, bad)) { ok = false; break; }
        if (!waiter && lane == 0) {
          tc::fence_after();
          const uint32_t base = sbase + static_cast<uint32_t>(s * STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t ko = static_cast<uint32_t>(kk * 2048);  // 16 k-rows of 128 B
            const uint64_t ahi = tc::smem_desc(base + a_off(0, 0) + ko, BOX, 1024, tc::kSwizzle128B);
            const uint64_t alo = tc::smem_desc(base + a_off(1, 0) + ko, BOX, 1024, tc::kSwizzle128B);
            const uint64_t bhi = tc::smem_desc(base + b_off(0, 0) + ko, BOX, 1024, tc::kSwizzle128B);
            const uint64_t blo = tc::smem_desc(base + b_off(1, 0) + ko, BOX, 1024, tc::kSwizzle128B);
            tc::mma_f16_pair(d_tmem, ahi, bhi, IDESC, (kc | kk) != 0 ? 1u : 0u);
            tc::mma_f16_pair(d_tmem, ahi, blo, IDESC, 1u);
            tc::mma_f16_pair(d_tmem, alo, bhi, IDESC, 1u);
          }
          tc::mma_commit_pair(&empty[s], static_cast<uint16_t>(0x3));
          if (kc == a.nk - 1) tc::mma_commit_pair(&accfull[acc], static_cast<uint16_t>(0x3));
        }
      }
      if (!ok) break;
      acc ^= 1;
      if (acc == 0) accphase ^= 1u;
    }
    if (waiter && lane == 0) counts[1] = seen;
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int q = warp % 4;             // TMEM lane quarter = tile rows 32q..32q+31
    const int half = (warp - 2) / 4;    // tile columns half*128 ..
    uint8_t* stg = stg_base + (warp - 2) * STG_BYTES;
    int acc = 0;
    uint32_t accphase = 0;
    for (int u = unit0; u < n_units && ok; u += unit_step) {
      const int mt = u % a.n_mt, nt = u / a.n_mt;
      if (!tc::mbar_wait(&accfull[acc], accphase, abort_flag, a.wait_ns)) { ok = false; break; }
      tc::fence_after();
      const int row0 = mt * 2 * BM + crank * BM + 32 * q;
      const int col0 = a.c_begin + nt * BN + half * 128;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * BN + half * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
        tc::tmem_ld_wait();
        const int cc = col0 + c * 32;
        // the previous box's shared source has been read by the memory system
        if (lane == 0) tc::bulk_wait_group_read0();
        __syncwarp();
        // row `lane` of the box, 128-byte swizzle: 16-byte chunk j at (j ^ (lane % 8))
        uint8_t* srow = stg + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 v;
          v.x = (cc + 4 * j < a.c_end) ? -__uint_as_float(r[4 * j]) : 0.0f;
          v.y = (cc + 4 * j + 1 < a.c_end) ? -__uint_as_float(r[4 * j + 1]) : 0.0f;
          v.z = (cc + 4 * j + 2 < a.c_end) ? -__uint_as_float(r[4 * j + 2]) : 0.0f;
          v.w = (cc + 4 * j + 3 < a.c_end) ? -__uint_as_float(r[4 * j + 3]) : 0.0f;
          *reinterpret_cast<float4*>(srow + ((j ^ (lane & 7)) << 4)) = v;
        }
        tc::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && cc < a.c_end && row0 < a.m) {
          tc::tma_reduce_add_2d(&tm_w, stg, cc, row0);
          tc::bulk_commit_group();
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&accempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) accphase ^= 1u;
    }
    if (lane == 0) tc::bulk_wait_group0();
  }

  if (!ok) {
    *abort_flag = 1;
    if (lane == 0 || warp >= 2) {
      dev_fail(a.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&a.st->timeouts, 1);
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
    drained = tc::drain_pair_stages(full, NSTAGE, counts[1], counts[0], odd, STAGE);
  }
  if (!drained) {
    // a drain wait ran out (nothing should be left to land): record it, and give whatever
    // is still in flight time to land before the memory goes away
    dev_fail(a.st, GPTQ_ERR_TIMEOUT, 1);
    atomicAdd(&a.st->timeouts, 1);
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
    tc::tmem_dealloc_pair(tmem_base, 512);
  }
}

// hi = bf16(x), lo = bf16(x - hi) for the part of U that the lazy updates read: row i,
// columns from the first 128-column block past row i's block (an update takes U rows of
// its blocks and columns of later blocks only).  The rest of hi and lo is left unwritten.
// One CTA per row, 8 elements per thread and step: two 16-byte loads, two 16-byte stores
// (d a multiple of 8, rows 16-byte aligned).
__global__ void __launch_bounds__(256) usplit_kernel(const float* __restrict__ U, int d,
                                                     __nv_bfloat16* __restrict__ hi,
                                                     __nv_bfloat16* __restrict__ lo) {
  const int i = blockIdx.x;
  const size_t row = static_cast<size_t>(i) * d;
  for (int j = (i / 128 + 1) * 128 + 8 * static_cast<int>(threadIdx.x); j < d; j += 8 * 256) {
    const float4 x0 = *reinterpret_cast<const float4*>(U + row + j);
    const float4 x1 = *reinterpret_cast<const float4*>(U + row + j + 4);
    const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    __align__(16) __nv_bfloat16 h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      h[k] = __float2bfloat16_rn(x[k]);
      l[k] = __float2bfloat16_rn(x[k] - __bfloat162float(h[k]));
    }
    *reinterpret_cast<uint4*>(hi + row + j) = *reinterpret_cast<const uint4*>(h);
    *reinterpret_cast<uint4*>(lo + row + j) = *reinterpret_cast<const uint4*>(l);
  }
}

}  // namespace

void launch_usplit(const float* U, int d, __nv_bfloat16* hi, __nv_bfloat16* lo, cudaStream_t s) {
  if (d % 8 != 0) fail(GPTQ_ERR_INVALID_ARG, "launch_usplit: d must be a multiple of 8");
  GPTQ_LAUNCH(GPTQ_K_QUANT_SPLIT, s, usplit_kernel, static_cast<unsigned>(d), 256, 0, U, d, hi,
              lo);
}

LazyMaps make_lazy_maps(const __nv_bfloat16* ehi, const __nv_bfloat16* elo, int erows,
                        const __nv_bfloat16* uhi, const __nv_bfloat16* ulo, float* W, int m,
                        int d) {
  LazyMaps mp;
  make_tmap_2d(&mp.ehi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ehi, m, erows,
               static_cast<uint64_t>(m) * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.elo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, elo, m, erows,
               static_cast<uint64_t>(m) * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.uhi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, uhi, d, d, static_cast<uint64_t>(d) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  make_tmap_2d(&mp.ulo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ulo, d, d, static_cast<uint64_t>(d) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  // W boxes of 32 rows x 32 float32 columns (128 bytes, the swizzle span)
  make_tmap_2d(&mp.w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W, d, m, static_cast<uint64_t>(d) * 4, 32,
               32, CU_TENSOR_MAP_SWIZZLE_128B);
  mp.m = m;
  mp.d = d;
  return mp;
}

namespace {
// co-resident clusters of the kernel on the current device, looked up once per device
int resident_pairs() {
  static std::mutex mu;
  static std::map<int, int> per_dev;
  int dev = 0;
  GPTQ_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  int& r = per_dev[dev];
  const int most = sm_count() / 2;
  if (r <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * most));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lazy_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = most;
    }
    r = n < most ? n : most;
  }
  return r;
}
}  // namespace

void launch_lazy_tc(const LazyMaps& mp, int e_row0, int u_row0, int k, int c_begin, int c_end,
                    DevStatus* st, cudaStream_t s, int max_ctas) {
  if (k <= 0 || c_end <= c_begin || mp.m <= 0) return;
  ensure_dynamic_smem(lazy_tc_kernel, SMEM_BYTES);
  LazyArgs a;
  a.m = mp.m;
  a.d = mp.d;
  a.e_row0 = e_row0;
  a.u_row0 = u_row0;
  a.nk = static_cast<int>(ceil_div(k, BK));
  a.c_begin = c_begin;
  a.c_end = c_end;
  a.n_mt = static_cast<int>(ceil_div(mp.m, 2 * BM));
  a.n_nt = static_cast<int>(ceil_div(c_end - c_begin, BN));
  a.st = st;
  a.wait_ns = wait_limit_ns();
  const int units = a.n_mt * a.n_nt;
  // one cluster of two CTAs per pair of SMs that can hold one at once
  int clusters = resident_pairs();
  if (max_ctas > 0 && clusters > max_ctas / 2) clusters = max_ctas / 2 > 0 ? max_ctas / 2 : 1;
  const int grid = 2 * (units < clusters ? units : clusters);
  GPTQ_LAUNCH_PDL(GPTQ_K_QUANT_LAZY, s, lazy_tc_kernel, grid, THREADS, SMEM_BYTES, mp.ehi, mp.elo,
              mp.uhi, mp.ulo, mp.w, a);
}

}  // namespace gptq
