// Hessian accumulation on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes the token-split partials P[s] = X_s^T X_s of the streaming hook ("GPTQ
// Architecture, in depth", "The algorithm in code", HessianHook; "Same Ruler, Smarter
// Placement: GPTQ", section 1.4) for bf16 X, with float32 accumulation in TMEM.  Only
// tiles that touch the upper 128-tile triangle are computed.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: X tiles [64 tokens x 128 | 256 columns] into a 4-stage ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128x256x16, both operands
//               MN-major (the column index of X is contiguous in memory)
//   warps 2..9  epilogue: drain finished TMEM accumulators into float32 registers, then
//               store the unit's tile of P[s]
// A unit is (row tile I of 128, column tile J of 256, token split s).  The tensor core's
// float32 accumulation does not round to nearest, so its error grows with the length of
// an accumulation chain; each chain therefore covers only a few stages (512 tokens) and
// is then added, with round-to-nearest float32 adds in a fixed order, into the epilogue
// warps' registers.  Two 256-column TMEM accumulators alternate between chains, so the
// MMAs of one chain overlap the drain of the previous one.
#include <cuda_bf16.h>

#include <cstdlib>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // tokens per stage
constexpr int NSTAGE = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * BK * 2;  // one TMA box: 64 columns x 64 tokens
constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + 1024 + 256;
constexpr int CHAIN_DEFAULT = 8;    // stages per TMEM accumulation chain (512 tokens)
constexpr int EPI_WARPS = 8;        // two per TMEM lane quarter, 128 columns each
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, true, true);

struct SyrkArgs {
  int d;
  int64_t ntok;
  int64_t tok_per_split;
  int n_i;       // row tiles of 128
  int n_j;       // column tiles of 256
  int n_tiles;   // tiles intersecting the upper 128-tile triangle
  int splits;
  int chain;     // stages per accumulation chain
  float* P;      // [splits][d][d]
  DevStatus* st;
};

__device__ __forceinline__ void decode_tile(int tile, int n_i, int n_j, int& I, int& J) {
  int rem = tile;
  for (J = 0; J < n_j; ++J) {
    int cnt = min(2 * J + 2, n_i);
    if (rem < cnt) { I = rem; return; }
    rem -= cnt;
  }
  I = 0;
}

__global__ void __launch_bounds__(THREADS, 1)
    syrk_tc_kernel(const __grid_constant__ CUtensorMap tmap, const SyrkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * STAGE_BYTES);
  uint64_t* empty = full + NSTAGE;
  uint64_t* accfull = empty + NSTAGE;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t n_units = static_cast<int64_t>(a.n_tiles) * a.splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accfull[b], 1);
      tc::mbar_init(&accempty[b], EPI_WARPS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmap);
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
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int s = static_cast<int>(u / a.n_tiles);
      int I, J;
      decode_tile(static_cast<int>(u % a.n_tiles), a.n_i, a.n_j, I, J);
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      for (int kb = 0; kb < nk; ++kb) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        tc::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        const int tok = static_cast<int>(t0 + static_cast<int64_t>(kb) * BK);
        tc::tma_load_2d(sa, &tmap, &full[stage], I * BM, tok);
        tc::tma_load_2d(sa + BOX_BYTES, &tmap, &full[stage], I * BM + 64, tok);
#pragma unroll
        for (int h = 0; h < 4; ++h)
          tc::tma_load_2d(sb + h * BOX_BYTES, &tmap, &full[stage], J * BN + 64 * h, tok);
        if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t accphase = 0;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int s = static_cast<int>(u / a.n_tiles);
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      for (int kb = 0; kb < nk; ++kb) {
        const int kc = kb % a.chain;
        if (kc == 0) {
          if (!tc::mbar_wait(&accempty[acc], accphase ^ 1u, abort_flag)) { ok = false; break; }
          tc::fence_after();
        }
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        if (!tc::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
        tc::fence_after();
        const uint32_t abase = tc::smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t bbase = abase + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // 16 tokens = two 8-row core groups of 1024 B; 64-column atoms are one TMA box
          // (8192 B) apart.
          const uint64_t ad = tc::smem_desc(abase + kk * 2048, BOX_BYTES, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(bbase + kk * 2048, BOX_BYTES, 1024, tc::kSwizzle128B);
          tc::mma_f16(d_tmem, ad, bd, IDESC, (kc | kk) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[stage]);
        if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
        if (kc == a.chain - 1 || kb == nk - 1) {
          tc::mma_commit(&accfull[acc]);
          acc ^= 1;
          if (acc == 0) accphase ^= 1u;
        }
      }
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp % 4;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;   // which 128 of the 256 columns
    int acc = 0;
    uint32_t accphase = 0;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int s = static_cast<int>(u / a.n_tiles);
      int I, J;
      decode_tile(static_cast<int>(u % a.n_tiles), a.n_i, a.n_j, I, J);
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      const int nchain = (nk + a.chain - 1) / a.chain;
      float sum[128];
#pragma unroll
      for (int k = 0; k < 128; ++k) sum[k] = 0.0f;
      for (int ch = 0; ch < nchain; ++ch) {
        if (!tc::mbar_wait(&accfull[acc], accphase, abort_flag)) { ok = false; break; }
        tc::fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                               static_cast<uint32_t>(acc * BN + half * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t r[16];
          tc::tmem_ld_32x32b_x16(tbase + c * 16, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k)
            sum[c * 16 + k] = __fadd_rn(sum[c * 16 + k], __uint_as_float(r[k]));
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&accempty[acc]);
        acc ^= 1;
        if (acc == 0) accphase ^= 1u;
      }
      if (!ok) break;
      const int row = I * BM + 32 * q + lane;
      if (row < a.d) {
        float* prow = a.P + static_cast<size_t>(s) * a.d * a.d + static_cast<size_t>(row) * a.d;
        const int col0 = J * BN + half * 128;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (col0 + 4 * k < a.d) {
            *reinterpret_cast<float4*>(prow + col0 + 4 * k) =
                make_float4(sum[4 * k], sum[4 * k + 1], sum[4 * k + 2], sum[4 * k + 3]);
          }
        }
      }
    }
  }

  if (!ok) {
    *abort_flag = 1;
    if (lane == 0 || warp >= 2) {
      dev_fail(a.st, GPTQ_ERR_TIMEOUT, 0);
      atomicAdd(&a.st->timeouts, 1);
    }
    // let copies and MMAs already in flight land before the CTA's memory goes away
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

}  // namespace

int syrk_tc_tiles(int d) {
  const int n_i = (d + BM - 1) / BM, n_j = (d + BN - 1) / BN;
  int n = 0;
  for (int J = 0; J < n_j; ++J) n += (2 * J + 2 < n_i) ? 2 * J + 2 : n_i;
  return n;
}

int syrk_tc_token_granule() { return BK; }

void launch_syrk_tc(const void* X, int64_t ntok, int d, int splits, int64_t tok_per_split,
                    float* P, DevStatus* st, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    GPTQ_CUDA(cudaFuncSetAttribute(syrk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM_BYTES));
    attr_done = true;
  }
  CUtensorMap tmap;
  make_tmap_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(d),
               static_cast<uint64_t>(ntok), static_cast<uint64_t>(d) * 2, 64, BK,
               CU_TENSOR_MAP_SWIZZLE_128B);
  SyrkArgs a;
  a.d = d;
  a.ntok = ntok;
  a.tok_per_split = tok_per_split;
  a.n_i = (d + BM - 1) / BM;
  a.n_j = (d + BN - 1) / BN;
  a.n_tiles = syrk_tc_tiles(d);
  a.splits = splits;
  a.chain = CHAIN_DEFAULT;
  if (const char* e = std::getenv("GPTQ_SYRK_CHAIN")) {  // tuning knob: stages per chain
    const int c = std::atoi(e);
    if (c >= 1 && c <= 1024) a.chain = c;
  }
  a.P = P;
  a.st = st;
  const int64_t units = static_cast<int64_t>(a.n_tiles) * splits;
  const int grid = static_cast<int>(units < sm_count() ? units : sm_count());
  GPTQ_LAUNCH(GPTQ_K_SYRK_TC, s, syrk_tc_kernel, grid, THREADS, SMEM_BYTES, tmap, a);
}

}  // namespace gptq
