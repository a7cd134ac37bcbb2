// Hessian accumulation on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes the token-split partials P[s] = X_s^T X_s of the streaming hook ("GPTQ
// Architecture, in depth", "The algorithm in code", HessianHook; "Same Ruler, Smarter
// Placement: GPTQ", section 1.4) for bf16 X, with float32 accumulation in TMEM.  Only
// tiles that touch the upper 128-tile triangle are computed.
//
// Persistent, warp-specialised kernel, one CTA per SM, the CTAs in pairs that run
// paired-SM MMAs, NP pairs per cluster (NP = 2 on wide layers, else 1).  A unit is a
// 256 NP x 256 block of H (row tiles 2 NP Q .. 2 NP Q + 2 NP - 1 of 128, column tile J of
// 256) for one token split s: pair p of the cluster computes the 256 x 256 tile of row
// tiles 2 NP Q + 2p, + 1.  In a pair the even CTA's TMEM holds the first 128 rows and the
// odd CTA's the next 128; each CTA's shared memory holds its own 128 rows' operand and
// half of the 256-column operand, so an SM takes in 512 bytes of operands per token (768
// for a one-SM 128 x 256 tile).  With NP = 2 both pairs need the same column strip: CTAs 0
// and 2 hold its first half, CTAs 1 and 3 its second, and each half is read from L2 once,
// by two multicast copies of one 64-column box each (a quarter less L2 traffic than two
// separate pairs; under the power cap the clock rises with it).
//   warp 0      TMA producer (every CTA): its own X rows [BK tokens x 128 columns] and its
//               column half (NP = 2: one box of it, multicast to the same-parity CTA of
//               the other pair) into a 192 KB ring of BK-token stages (Stages below);
//               completion is counted on the even CTA of each pair
//   warp 1      TMEM owner (every CTA, paired allocation); in the even CTAs also the MMA
//               issuer: tcgen05.mma.cta_group::2 256x256x16, both operands MN-major (the
//               column index of X is contiguous in memory)
//   warps 2..9  epilogue (every CTA): drain finished TMEM accumulators into float32
//               registers, then store the CTA's 128 x 256 part of its pair's tile of P[s]
//   warp 10     in the even CTAs: waits for each stage's data (and, at a chain start, for
//               the accumulator) and releases warp 1 through a named barrier.  The issuing
//               warp never waits on an mbarrier: such a wait holds it until its
//               outstanding MMAs have read their operands, which empties the tensor pipe.
//               128 tokens (8 MMAs) per hand-off keep the pipe fed across it.
// A stage is refilled when every pair's MMAs have consumed it (each pair's commit arrives
// on every CTA's barrier of the cluster), since a multicast writes into the other pair's
// ring.  The tensor core's float32 accumulation does not round to nearest, so its error
// grows with the length of an accumulation chain; each chain therefore covers only a few
// stages (512 tokens) and is then added, with round-to-nearest float32 adds in a fixed
// order, into the epilogue warps' registers.  Two 256-column TMEM accumulators alternate
// between chains, so the MMAs of one chain overlap the drain of the previous one.
#include <cuda_bf16.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {

constexpr int BM = 128;  // rows of H per CTA
constexpr int BN = 256;  // columns of H per unit (128 in each CTA's shared memory)
// Stages by pairs per cluster: one pair (narrower layers, short Hessians at full clock,
// where moving operands into the SMs bounds the kernel) copies 128-token stages, 16 KB
// per TMA copy (q_proj: 2.55 against 2.81 ms with 64-token stages); two pairs (wide layers
// under the power cap) keep 64-token stages (128-token ones measured 1-3 % slower per
// clock there).  The ring holds the same 192 KB either way, and a TMEM accumulation chain
// covers 512 tokens.
template <int NP>
struct Stages {
  static constexpr int BK = NP == 1 ? 128 : 64;      // tokens per stage
  static constexpr int NSTAGE = NP == 1 ? 3 : 6;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / 2) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BOX_BYTES = 64 * BK * 2;      // one TMA box: 64 columns x BK tokens
  static constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + 1024 + 256;
  static constexpr int CHAIN = 512 / BK;             // stages per TMEM accumulation chain
};
constexpr int EPI_WARPS = 8;        // two per TMEM lane quarter, 128 columns each
constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;
constexpr int WAITER_WARP = 2 + EPI_WARPS;
constexpr uint32_t kHandoffBarrier = 1;  // named barrier of warps 1 and WAITER_WARP
constexpr uint32_t IDESC = tc::idesc_bf16_f32(2 * BM, BN, true, true);  // paired: M = 256

struct SyrkArgs {
  int d;
  int64_t ntok;
  int64_t tok_per_split;
  int n_i;       // row tiles of 128
  int n_j;       // column tiles of 256
  int n_units;   // units (NP pairs of row tiles) intersecting the upper 128-tile triangle
  int splits;
  float* P;      // [splits][d][d]
  DevStatus* st;
  uint64_t wait_ns;  // limit of each pipeline wait (the exit's drain waits use kWaitLimitNs)
};

// unit Q of column tile J: row tiles 2 NP Q .. 2 NP Q + 2 NP - 1.  Row tiles past 2J + 1
// (below the upper triangle, when NP = 2 and a column tile has an odd number of row-tile
// pairs) or past the last row tile are computed all the same, on the matrix or on zeros,
// so that every pair walks the same stages; the former land in the lower part of P[s],
// which nothing reads, the latter are not stored.  Units go column tile by column tile, so
// the units in flight at once share their column strip of X.  (A banded order of the
// one-pair kernel, 8 column tiles by row pair, which read fewer distinct strips per wave,
// measured 1.5-2 % slower at d_in = 28672.)
template <int NP>
__device__ __forceinline__ void decode_unit(int unit, int n_i, int n_j, int& Q, int& J) {
  int rem = unit;
  for (J = 0; J < n_j; ++J) {
    const int cnt = ((min(2 * J + 2, n_i) + 1) / 2 + NP - 1) / NP;
    if (rem < cnt) { Q = rem; return; }
    rem -= cnt;
  }
  Q = 0;
}

template <int NP>
__global__ void __cluster_dims__(2 * NP, 1, 1) __launch_bounds__(THREADS, 1)
    syrk_tc_kernel(const __grid_constant__ CUtensorMap tmap, const SyrkArgs a) {
  constexpr int BK = Stages<NP>::BK, NSTAGE = Stages<NP>::NSTAGE, CHAIN = Stages<NP>::CHAIN;
  constexpr int A_BYTES = Stages<NP>::A_BYTES, STAGE_BYTES = Stages<NP>::STAGE_BYTES;
  constexpr int BOX_BYTES = Stages<NP>::BOX_BYTES;
  constexpr int HS = 128 / BK;  // stages per hand-off
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * STAGE_BYTES);
  uint64_t* empty = full + NSTAGE;
  uint64_t* accfull = empty + NSTAGE;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [0]: stages this CTA's producer issued; [1] (even CTAs): stages the waiter saw land
  int* counts = const_cast<int*>(abort_flag) + 1;
  uint64_t* mma_drain = reinterpret_cast<uint64_t*>(counts + 2);  // the issuer's last commit

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int crank = static_cast<int>(tc::cluster_ctarank());
  const uint32_t lead = static_cast<uint32_t>(crank & ~1);  // the pair's even CTA
  const int64_t n_units = static_cast<int64_t>(a.n_units) * a.splits;
  const int64_t unit0 = blockIdx.x / (2 * NP), unit_step = gridDim.x / (2 * NP);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      tc::mbar_init(&full[s], 1);   // the even CTA's: both CTAs' bytes
      tc::mbar_init(&empty[s], NP);  // every pair's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accfull[b], 1);
      tc::mbar_init(&accempty[b], 2 * EPI_WARPS);  // the even CTA's: both CTAs' epilogues
    }
    tc::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    counts[0] = counts[1] = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmap);
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, 512);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // both CTAs' barriers exist before either multicasts into them
  tc::fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      const int s = static_cast<int>(u / a.n_units);
      int qq, J;
      decode_unit<NP>(static_cast<int>(u % a.n_units), a.n_i, a.n_j, qq, J);
      const int I = 2 * NP * qq + crank;
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      for (int kb = 0; kb < nk; ++kb) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        // both CTAs' 32 KB land on the even CTA's barrier
        const uint32_t bar = tc::mapa_shared(tc::smem_u32(&full[stage]), lead);
        if ((crank & 1) == 0) tc::mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
        const int tok = static_cast<int>(t0 + static_cast<int64_t>(kb) * BK);
        tc::tma_load_2d_pair(sa, &tmap, bar, I * BM, tok);
        tc::tma_load_2d_pair(sa + BOX_BYTES, &tmap, bar, I * BM + 64, tok);
        if constexpr (NP == 1) {
          tc::tma_load_2d_pair(sb, &tmap, bar, J * BN + 128 * crank, tok);
          tc::tma_load_2d_pair(sb + BOX_BYTES, &tmap, bar, J * BN + 128 * crank + 64, tok);
        } else {
          // the CTAs 0, 2 (1, 3) share their half of the column strip: each loads one box
          // of it into both
          const int hb = crank >> 1;
          tc::tma_load_2d_pair_mc(sb + hb * BOX_BYTES, &tmap, bar,
                                  J * BN + 128 * (crank & 1) + 64 * hb, tok,
                                  static_cast<uint16_t>(0x5u << (crank & 1)));
        }
        ++issued;
        if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
      }
    }
    counts[0] = issued;
  } else if ((crank & 1) == 0 && (warp == 1 || warp == WAITER_WARP)) {
    // ---------------------------------------------------------------- MMA issuer and its
    // waiter (even CTA): both walk the same stages, 128 tokens per hand-off; the waiter's lane 0
    // waits, then both warps meet at the named barrier, which also carries a failed wait
    const bool waiter = (warp == WAITER_WARP);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t accphase = 0;
    int seen = 0;  // stages whose copies the waiter saw land
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      const int s = static_cast<int>(u / a.n_units);
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      // HS stages (128 tokens, 8 MMAs) per hand-off; the loop keeps the two-stage form's
      // expressions, which measured faster than a general count
      for (int kb = 0; kb < nk; kb += HS) {
        const int nst = (HS == 2 && kb + 1 < nk) ? 2 : 1;
        bool bad = false;
        if (waiter && lane == 0) {
          if ((kb % CHAIN) == 0)
            bad = !tc::mbar_wait(&accempty[acc], accphase ^ 1u, abort_flag, a.wait_ns);
          if (!bad) bad = !tc::mbar_wait(&full[stage], phase, abort_flag, a.wait_ns);
          if (!bad) ++seen;
          if (!bad && nst == 2) {
            const int s2 = (stage + 1 == NSTAGE) ? 0 : stage + 1;
            bad = !tc::mbar_wait(&full[s2], (stage + 1 == NSTAGE) ? (phase ^ 1u) : phase,
                                 abort_flag, a.wait_ns);
            if (!bad) ++seen;
          }
        }
        if (tc::handoff_or(kHandoffBarrier, 64, bad)) { ok = false; break; }
        for (int q = 0; q < nst; ++q) {
          const int kq = kb + q;
          const int kc = kq % CHAIN;  // position in the accumulation chain
          if (!waiter && lane == 0) {
            tc::fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            const uint32_t abase = tc::smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t bbase = abase + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // 16 tokens = two 8-row core groups of 1024 B; 64-column atoms are one TMA
              // box (BOX_BYTES) apart.
              const uint64_t ad = tc::smem_desc(abase + kk * 2048, BOX_BYTES, 1024, tc::kSwizzle128B);
              const uint64_t bd = tc::smem_desc(bbase + kk * 2048, BOX_BYTES, 1024, tc::kSwizzle128B);
              tc::mma_f16_pair(d_tmem, ad, bd, IDESC, (kc | kk) != 0 ? 1u : 0u);
            }
            tc::mma_commit_pair(&empty[stage], static_cast<uint16_t>((1u << (2 * NP)) - 1));
            if (kc == CHAIN - 1 || kq == nk - 1)
              tc::mma_commit_pair(&accfull[acc], static_cast<uint16_t>(0x3u << lead));
          }
          if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
          if (kc == CHAIN - 1 || kq == nk - 1) {
            acc ^= 1;
            if (acc == 0) accphase ^= 1u;
          }
        }
      }
    }
    if (waiter && lane == 0) counts[1] = seen;
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp % 4;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;   // which 128 of the 256 columns
    int acc = 0;
    uint32_t accphase = 0;
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      const int s = static_cast<int>(u / a.n_units);
      int qq, J;
      decode_unit<NP>(static_cast<int>(u % a.n_units), a.n_i, a.n_j, qq, J);
      const int I = 2 * NP * qq + crank;
      const int64_t t0 = s * a.tok_per_split;
      const int64_t t1 = min(a.ntok, t0 + a.tok_per_split);
      const int nk = static_cast<int>((t1 - t0 + BK - 1) / BK);
      const int nchain = (nk + CHAIN - 1) / CHAIN;
      float sum[128];
#pragma unroll
      for (int k = 0; k < 128; ++k) sum[k] = 0.0f;
      for (int ch = 0; ch < nchain; ++ch) {
        if (!tc::mbar_wait(&accfull[acc], accphase, abort_flag, a.wait_ns)) { ok = false; break; }
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
        if (lane == 0) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&accempty[acc]), lead));
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
  }
  // Drain, on every exit, so that nothing is in flight when the CTAs' memory goes away.
  // First the issuer's MMAs: one more commit, which arrives once every earlier MMA of the
  // pair has completed (read its operands, written TMEM).
  bool drained = true;
  if ((crank & 1) == 0 && warp == 1 && lane == 0) {
    tc::mma_commit_pair(mma_drain, static_cast<uint16_t>(1u << crank));
    drained = tc::mbar_wait_for(mma_drain, 0, kWaitLimitNs);
  }
  tc::fence_before();
  __syncwarp();
  tc::cluster_sync();  // every producer has stopped; its count is visible cluster-wide
  if ((crank & 1) == 0 && threadIdx.x == 0) {
    // Then the copies: each pair's copies complete on its even CTA's barriers.  Stage k
    // (of every CTA's common sequence) sits in slot k % NSTAGE; the waiter saw stages
    // below counts[1] land, and no producer runs more than NSTAGE stages ahead of it, so
    // each later stage up to the largest count has a slot of its own, whose current phase
    // is that stage's.  A stage this CTA's producer did not arm is armed here, and the
    // bytes of every copy that was never issued are counted here, so the phase completes
    // exactly when the copies that were issued have landed.
    int cnt[2 * NP];
    int kmax = counts[1];
    for (int r = 0; r < 2 * NP; ++r) {
      cnt[r] = (r == crank) ? counts[0]
                            : static_cast<int>(tc::ld_shared_cluster_u32(
                                  tc::mapa_shared(tc::smem_u32(counts), static_cast<uint32_t>(r))));
      kmax = max(kmax, cnt[r]);
    }
    for (int k = counts[1]; k < kmax; ++k) {
      uint32_t missing = 0;  // bytes of this stage's copies that no producer issued
      for (int r = 0; r < 2 * NP; ++r) {
        if (k < cnt[r]) continue;
        // a CTA of this pair copies its rows and its box of the column half here; a CTA of
        // the other pair only its multicast box
        missing += ((r & ~1) == crank) ? static_cast<uint32_t>(NP == 1 ? STAGE_BYTES : A_BYTES + BOX_BYTES)
                                       : static_cast<uint32_t>(BOX_BYTES);
      }
      uint64_t* bar = &full[k % NSTAGE];
      if (k >= cnt[crank]) tc::mbar_arrive_expect_tx(bar, 2 * STAGE_BYTES);
      if (missing != 0) tc::mbar_complete_tx(bar, missing);
      if (!tc::mbar_wait_for(bar, static_cast<uint32_t>(k / NSTAGE) & 1u, kWaitLimitNs))
        drained = false;
    }
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
  tc::cluster_sync();  // every pair's copies have landed; no CTA signals another any more
  if (warp == 1) {
    __syncwarp();
    tc::fence_after();
    tc::tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace

// CTAs' tiles per token split (units of NP pairs of row tiles, a column's last unit
// padded).  Wide layers take clusters of two pairs (NP = 2): their Hessian streams run for
// seconds under the power cap, where the shared column strip's multicast (a quarter less
// L2 traffic) buys clock (70B-width down_proj: 337 against 350 ms per 524,288 tokens).  A
// cluster of four needs four SMs of one GPC, which leaves 8 of the 152 SMs idle, so the
// short Hessians of narrower layers, which run at full clock, keep one pair per cluster
// (q_proj, both with 64-token stages: 2.74 against 2.83 ms).
static int syrk_pairs_per_cluster(int d) { return d >= 8192 ? 2 : 1; }

int syrk_tc_tiles(int d) {
  const int np = syrk_pairs_per_cluster(d);
  const int n_i = (d + BM - 1) / BM, n_j = (d + BN - 1) / BN;
  int n = 0;
  for (int J = 0; J < n_j; ++J) {
    const int pairs = (((2 * J + 2 < n_i) ? 2 * J + 2 : n_i) + 1) / 2;
    n += 2 * np * ((pairs + np - 1) / np);
  }
  return n;
}

int syrk_tc_token_granule(int d) {
  return syrk_pairs_per_cluster(d) == 2 ? Stages<2>::BK : Stages<1>::BK;
}

namespace {
template <int NP>
int resident_clusters() {
  static std::mutex mu;
  static std::map<int, int> per_dev;  // device -> co-resident clusters of the kernel
  int dev = 0;
  GPTQ_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  int& r = per_dev[dev];
  const int most = sm_count() / (2 * NP);
  if (r <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * NP * most));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Stages<NP>::SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, syrk_tc_kernel<NP>, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = most;
    }
    r = n < most ? n : most;
  }
  return r;
}

template <int NP>
void launch_syrk_np(const CUtensorMap& tmap, SyrkArgs a, cudaStream_t s) {
  ensure_dynamic_smem(syrk_tc_kernel<NP>, Stages<NP>::SMEM_BYTES);
  a.n_units = syrk_tc_tiles(a.d) / (2 * NP);
  // one cluster of 2 NP CTAs per unit, no more clusters than can be resident at once (a
  // cluster needs 2 NP SMs of one GPC, so that may be fewer than the SMs allow); the
  // count is looked up once per device
  const int64_t units = static_cast<int64_t>(a.n_units) * a.splits;
  const int64_t clusters = resident_clusters<NP>();
  const int grid = 2 * NP * static_cast<int>(units < clusters ? units : clusters);
  GPTQ_LAUNCH(GPTQ_K_SYRK_TC, s, syrk_tc_kernel<NP>, grid, THREADS, Stages<NP>::SMEM_BYTES, tmap,
              a);
}
}  // namespace

void launch_syrk_tc(const void* X, int64_t ntok, int d, int splits, int64_t tok_per_split,
                    float* P, DevStatus* st, cudaStream_t s) {
  CUtensorMap tmap;
  make_tmap_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(d),
               static_cast<uint64_t>(ntok), static_cast<uint64_t>(d) * 2, 64,
               static_cast<uint32_t>(syrk_tc_token_granule(d)), CU_TENSOR_MAP_SWIZZLE_128B);
  SyrkArgs a;
  a.d = d;
  a.ntok = ntok;
  a.tok_per_split = tok_per_split;
  a.n_i = (d + BM - 1) / BM;
  a.n_j = (d + BN - 1) / BN;
  a.n_units = 0;
  a.splits = splits;
  a.P = P;
  a.st = st;
  a.wait_ns = wait_limit_ns();
  if (syrk_pairs_per_cluster(d) == 2) launch_syrk_np<2>(tmap, a, s);
  else launch_syrk_np<1>(tmap, a, s);
}

}  // namespace gptq
