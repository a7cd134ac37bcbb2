// Host-side launchers of the engine's kernels (one translation unit each).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gptq {

// hessian_simt.cu
int syrk_simt_tiles(int d);
void launch_syrk_simt(const void* X, bool bf16, int64_t ntok, int d, int splits,
                      int64_t tok_per_split, float* P, cudaStream_t s);
void launch_syrk_reduce(float* H, const float* P, int d, int splits, float alpha, float beta,
                        bool overwrite, cudaStream_t s);
// H <- factor * H on the upper 128-tile triangle (d a multiple of 4)
void launch_hessian_rescale(float* H, int d, float factor, cudaStream_t s);

// selfcheck.cu: one bounded wait on an mbarrier nothing arrives on
void launch_wait_timeout(DevStatus* st, uint64_t limit_ns, cudaStream_t s);

// hessian_tc.cu
int syrk_tc_tiles(int d);
int syrk_tc_token_granule(int d);  // tokens per pipeline stage at this width
void launch_syrk_tc(const void* X, int64_t ntok, int d, int splits, int64_t tok_per_split,
                    float* P, DevStatus* st, cudaStream_t s);

// lanes of the column loop per output row, and the floats of one 128-column block's
// layout of U for it (per row q of the block: kLoopLanesPerRow runs of 128 /
// kLoopLanesPerRow floats, each padded by 4; then 128 reciprocals)
constexpr int kLoopLanesPerRow = 4;
constexpr int kLoopUblkFloats = 128 * kLoopLanesPerRow * (128 / kLoopLanesPerRow + 4) + 128;

// prepare.cu
void launch_prepare(const float* H, int d, float damp, int actorder, int32_t* perm,
                    uint8_t* dead, float* U, float* S, float* Hr, float* diag_fixed,
                    float* lam, float* DI, float* Lo, DevStatus* st, cudaStream_t s);

// quantize.cu
struct QuantArgs {
  const void* W;
  bool w_bf16;
  const float* U;
  const int32_t* perm;  // may be null
  const uint8_t* dead;  // may be null
  int m, d, bits, group, sym, G;
  bool static_groups;   // groups fixed in the original column order before the loop
  // workspace
  float* Wp;
  uint8_t* codesT;
  __nv_bfloat16* ehi;   // [128][m] bf16 split of the block's errors
  __nv_bfloat16* elo;
  __nv_bfloat16* uhi;   // [d][d] bf16 split of U's strict upper triangle
  __nv_bfloat16* ulo;
  int32_t* zeros;
  double* loss_rows;
  int32_t* pos;
  float* Ublk;  // [ceil(d/128)][128*128 + 128]
  // outputs
  int32_t* qweight;
  float* scales;
  int32_t* qzeros;
  int32_t* g_idx;
  double* loss;
  DevStatus* st;
};
void launch_quantize(const QuantArgs& q, cudaStream_t s);

// dequant_matmul.cu: y[n, m] = x[n, d] W_hat^T from the packed checkpoint, and W_hat
void launch_dequantize(const int32_t* qweight, const float* scales, const int32_t* qzeros,
                       const int32_t* g_idx, int m, int d, int bits, int G, void* W, bool w_bf16,
                       DevStatus* st, cudaStream_t s);
void launch_dequant_matmul(const void* x, bool x_bf16, int64_t n, int d, int m, int bits, int G,
                           const int32_t* qweight, const float* scales, const int32_t* qzeros,
                           const int32_t* g_idx, float* y, DevStatus* st, cudaStream_t s);

// gemm_tc.cu: C[i][j] = beta C[i][j] + alpha sum_{k<K} A[a_row0+i][a_k0+k]
// B[b_row0+j][b_k0+k], float32-accurate (tf32 x3), K a multiple of 32; maps from
// make_gemm_map.  lower: only tiles with tile column <= tile row (M >= N), entries above the
// diagonal of C unchanged.  pdl: launched as a programmatic dependent of the kernel before
// it in the stream.
void make_gemm_map(CUtensorMap* map, const float* base, int rows, int cols, int ld);
void launch_gemm_tf32x3(int kind, const CUtensorMap& ma, int a_row0, int a_k0,
                        const CUtensorMap& mb, int b_row0, int b_k0, int K, float* C, int ldc,
                        int M, int N, float alpha, float beta, bool lower, DevStatus* st,
                        cudaStream_t s, bool pdl);

// gemm_tc.cu, long K: the same product with the lo parts of both operands precomputed
// (lo = x - tf32(x), read through their own maps at their own offsets); units of 256 x 256
// on pairs of SMs.  launch_split_lo writes those lo parts for a rows x cols block.
void launch_gemm_tf32x3_presplit(int kind, const CUtensorMap& ma, int a_row0, int a_k0,
                                 const CUtensorMap& ma_lo, int a_lo_row0, int a_lo_k0,
                                 const CUtensorMap& mb, int b_row0, int b_k0,
                                 const CUtensorMap& mb_lo, int b_lo_row0, int b_lo_k0, int K,
                                 float* C, int ldc, int M, int N, float alpha, float beta,
                                 bool lower, DevStatus* st, cudaStream_t s, bool pdl);
void launch_split_lo(const float* src, int ld, int rows, int cols, float* lo, int ld_lo,
                     cudaStream_t s);
// superpanel width of the prepare (panels whose update of later columns is grouped)
constexpr int kSuperpanel = 1024;

// lazy_tc.cu
// ErrT rows kept for the deferred update: one 1024-column superblock of the loop (the far
// update rewrites the later columns of W once per superblock; 1024 against 512 columns
// halved that traffic and took the update from 18.2 to 15.0 ms at d_in = 28672)
constexpr int kErrRows = 1024;

struct LazyMaps {
  CUtensorMap ehi, elo, uhi, ulo, w;
  int m, d;
};
// ErrT hi/lo [erows][m], U hi/lo [d][d] (bf16), W [m][d] (float32)
LazyMaps make_lazy_maps(const __nv_bfloat16* ehi, const __nv_bfloat16* elo, int erows,
                        const __nv_bfloat16* uhi, const __nv_bfloat16* ulo, float* W, int m,
                        int d);
// bf16 halves of U (x = hi + lo) on the blocks the lazy updates read: row i, columns from
// the 128-column block after row i's block on (d a multiple of 8)
void launch_usplit(const float* U, int d, __nv_bfloat16* hi, __nv_bfloat16* lo, cudaStream_t s);
// quantize.cu: the checkpoint's fp16 copy of n float32 scales (round to nearest even)
void launch_scales_fp16(const float* scales, int64_t n, uint16_t* out, cudaStream_t s);
// W[:, c_begin:c_end] -= ErrT[e_row0 : e_row0 + k]^T U[u_row0 : u_row0 + k, c_begin:c_end];
// max_ctas > 0 caps the persistent grid (to leave SMs to concurrent work)
void launch_lazy_tc(const LazyMaps& mp, int e_row0, int u_row0, int k, int c_begin, int c_end,
                    DevStatus* st, cudaStream_t s, int max_ctas);

}  // namespace gptq
