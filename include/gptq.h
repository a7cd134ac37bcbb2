/*
 * gptq.h -- C ABI of the GB300 GPTQ layer-quantization engine (libgptq_gb300.so).
 *
 * The engine quantises one linear layer with GPTQ.  Three calls follow the method's
 * statement of the problem:
 *
 *   gptq_hessian_accumulate  H = 2/n * sum x x^T over calibration tokens, streamed
 *   gptq_prepare             dead-column fix, act-order permutation, damping and the
 *                            upper Cholesky factor U of H_damp^-1
 *   gptq_quantize_layer      the fixed-order column loop in 128-column blocks with the
 *                            lazy trailing update, group scales / zeros, g_idx and
 *                            bit packing
 *
 * and two calls consume the packed checkpoint: gptq_dequant_matmul (y = x W_hat^T) and
 * gptq_dequantize (the dense W_hat).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Device pointers are CUDA device memory on the current device, allocated and owned by
 *   the caller.  The library allocates no device memory at run time: scratch comes from
 *   the caller's workspace `ws` of `ws_bytes` bytes (size it with gptq_workspace_size; the
 *   base must be 256-byte aligned).  The one exception is the fixed static array behind
 *   gptq_hessian_accumulate_noalloc (16 MiB + 256 B per GPU that loads the library).
 *   Host pointers are named as such below.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *   call enqueues its kernels on `stream`, then synchronises `stream` and returns the
 *   status of the work it enqueued (device-side failures such as a non-positive-definite
 *   matrix are reported this way); gptq_hessian_accumulate_async is the one call that
 *   returns without synchronising (gptq_hessian_status reports its device-side status).
 * - Matrices are row-major.  Indices and sizes are 32-bit unless stated.
 * - On any status other than GPTQ_OK, gptq_last_error() (thread-local) describes it.
 *   Invalid arguments are detected before anything is enqueued; outputs are then
 *   untouched.
 * - Calls may come from several host threads and for several devices in one process;
 *   the library's own state (kernel attributes, internal streams) is kept per device.
 *   gptq_prepare and gptq_quantize_layer(_ex) (also inside gptq_quantize_layer_host)
 *   share internal streams, so concurrent calls of those run one after the other.
 */
#ifndef GPTQ_GB300_H
#define GPTQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned buffer       */
  GPTQ_ERR_UNSUPPORTED = 2,   /* a valid value this engine does not implement          */
  GPTQ_ERR_NOT_PD = 3,        /* H_damp is not positive definite (Cholesky pivot <= 0) */
  GPTQ_ERR_NONFINITE = 4,     /* NaN or Inf in an input                                */
  GPTQ_ERR_CUDA = 5,          /* a CUDA runtime call failed                            */
  GPTQ_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out                    */
  GPTQ_ERR_WORKSPACE = 7      /* ws too small (see gptq_workspace_size)                */
} gptq_status;

typedef enum { GPTQ_F32 = 0, GPTQ_BF16 = 1 } gptq_dtype;

typedef enum {
  GPTQ_OP_HESSIAN = 0, GPTQ_OP_PREPARE = 1, GPTQ_OP_QUANTIZE = 2, GPTQ_OP_DEQUANT_MATMUL = 3
} gptq_op;

/*
 * gptq_workspace_size -- bytes of workspace the call `op` wants for these sizes on the
 * current device.  Arguments that do not apply to `op` are ignored.  For GPTQ_OP_HESSIAN
 * the value is the size that lets the call split the token axis as it prefers; any ws of
 * at least d_in*d_in*4 + 256 bytes is accepted (fewer splits).  Returns 0 for invalid
 * sizes.
 */
size_t gptq_workspace_size(int op, int64_t ntok, int32_t d_out, int32_t d_in, int bits,
                           int group);

/*
 * gptq_hessian_accumulate -- one step of the streaming Hessian hook.
 *
 * Defined by "GPTQ Architecture, in depth", "The algorithm in code" (HessianHook) and
 * "Same Ruler, Smarter Placement: GPTQ" section 1.4 (H = 2 X X^T): for a chunk of t =
 * ntok tokens and n = *nseen tokens seen so far,
 *     H <- H * n/(n+t) + 2/(n+t) * X^T X ,   *nseen <- n + t .
 * When *nseen == 0 the previous contents of H are ignored (H may be uninitialised).
 *
 * H      device float32 [d_in, d_in], in/out.  Only the upper triangle, at the
 *        granularity of 128x128 tiles (every element (i, j) with i/128 <= j/128), is
 *        written and is authoritative; the rest is left as it was.
 * nseen  host int64, in/out: the running token count n.
 * X      device [ntok, d_in] row-major (token-major: a Linear's input flattened to
 *        [tokens, cols]), element type `xdtype` (GPTQ_BF16: bfloat16, computed on the
 *        tensor cores with float32 accumulation; GPTQ_F32: float32, computed in float32
 *        FMA).  Row stride d_in elements; d_in must be a multiple of 8.
 * ntok   >= 0; ntok == 0 is a no-op.
 * Errors: INVALID_ARG, UNSUPPORTED (d_in % 8 != 0), WORKSPACE, CUDA, TIMEOUT.
 */
gptq_status gptq_hessian_accumulate(float* H, int64_t* nseen, const void* X, int xdtype,
                                    int64_t ntok, int32_t d_in, void* ws, size_t ws_bytes,
                                    void* stream);

/*
 * gptq_hessian_accumulate_noalloc -- gptq_hessian_accumulate for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an interface addition.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator while it feeds
 * calibration batches -- a host framework that owns the device pool and forbids
 * allocations after start-up, a plug-in living inside another program's memory manager,
 * or a loop that must not take an allocation's implicit device synchronisation.  The
 * caller still owns and passes H, nseen and X; the scratch (status word and token-split
 * partials) comes from a fixed 16 MiB (+256 B) array in device memory that the library
 * holds on every GPU that loads it, until the process exits.
 *
 * Same arguments, semantics and errors as gptq_hessian_accumulate, without ws/ws_bytes.
 * Limit: d_in * d_in * 4 <= 16 MiB, i.e. d_in <= 2048; larger d_in returns
 * GPTQ_ERR_UNSUPPORTED without touching anything.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture.  All calls share the one array and it keeps the
 * last call's contents (each call clears its status word and rewrites the partials it
 * reads), so calls whose work overlaps on the GPU -- from two streams or two threads --
 * race and must be serialised by the caller.
 */
gptq_status gptq_hessian_accumulate_noalloc(float* H, int64_t* nseen, const void* X,
                                            int xdtype, int64_t ntok, int32_t d_in,
                                            void* stream);

/*
 * gptq_hessian_accumulate_async -- gptq_hessian_accumulate without the synchronisation.
 * An interface addition (the pages' hook is a synchronous PyTorch call): it lets a
 * caller overlap the host-to-device copy of the next batch with this batch's kernels.
 *
 * Same arguments, arithmetic and argument checks as gptq_hessian_accumulate ("GPTQ
 * Architecture, in depth", HessianHook; "Same Ruler, Smarter Placement: GPTQ" section
 * 1.4).  It enqueues the batch's kernels on `stream` and returns without waiting: *nseen
 * is updated at once, H when the work completes.  X must stay valid and unmodified until
 * then (order its reuse after the work with an event on `stream`).  Device-side failures
 * (TIMEOUT, CUDA faults of the kernels) are not returned here: they collect in the status
 * word at the start of `ws`, which a call with *nseen == 0 clears, and
 * gptq_hessian_status reports and clears them.  All calls on one `ws` must be issued on
 * one stream (they share its token-split partials).
 * Errors returned directly: INVALID_ARG, UNSUPPORTED, WORKSPACE (nothing enqueued), CUDA
 * (a launch failed).
 */
gptq_status gptq_hessian_accumulate_async(float* H, int64_t* nseen, const void* X,
                                          int xdtype, int64_t ntok, int32_t d_in, void* ws,
                                          size_t ws_bytes, void* stream);

/*
 * gptq_hessian_rescale -- H <- H * n_from / n_to on the upper 128-tile triangle.
 *
 * gptq_hessian_accumulate leaves H normalised by the tokens it has seen (2/n sum x x^T,
 * "GPTQ Architecture, in depth", "The algorithm in code", HessianHook; "Same Ruler,
 * Smarter Placement: GPTQ" section 1.4).  Rescaled from its n_from tokens to n_to, it
 * becomes those tokens' share of the Hessian of an n_to-token stream: when a calibration
 * stream is split across GPUs, each rank rescales its partial from its own token count
 * to the total, and the sum of the partials (one all-reduce) is the Hessian of the whole
 * stream.  The interface is an addition for that split; the pages run one GPU.
 *
 * H       device float32 [d_in, d_in], in/out (upper 128-tile triangle, as written by
 *         gptq_hessian_accumulate; the rest is left as it was).  With n_from == 0 the
 *         upper triangle is set to zero whatever it held (a rank that saw no tokens).
 * d_in    > 0, multiple of 8.   n_from >= 0, n_to > 0.
 * Synchronous on `stream`.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
gptq_status gptq_hessian_rescale(float* H, int32_t d_in, int64_t n_from, int64_t n_to,
                                 void* stream);

/*
 * gptq_hessian_status -- synchronise `stream` and return the status collected by the
 * gptq_hessian_accumulate_async calls on `ws` since the last call with *nseen == 0 (the
 * first failure, as GPTQ_OK or the error code with gptq_last_error() describing it); the
 * status word is cleared afterwards.
 *
 * ws, ws_bytes  the same workspace the async calls used (device, 256-byte aligned).
 * Errors: INVALID_ARG (null, unaligned or too small ws), CUDA, TIMEOUT, and whatever the
 *         kernels recorded.
 */
gptq_status gptq_hessian_status(void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_prepare -- everything GPTQ does to H before the column loop.
 *
 * Defined by "GPTQ Architecture, in depth", "The algorithm in code" and "Groups,
 * act-order and other knobs", "Same Ruler, Smarter Placement: GPTQ" sections 1.6, 1.7
 * and 1.9, "GPTQ > ActOrder: Activation-Based Column Ordering":
 *   dead[j]   = (H_jj == 0); such channels get H_jj = 1 (their weights are zeroed later)
 *   perm      = columns by descending diagonal (after the dead fix), ties by ascending
 *               index; identity when actorder == 0
 *   H_damp    = H[perm][:, perm] + lambda I, lambda = damp * mean(diag H)
 *   Hinv_chol = U, upper triangular, H_damp^-1 = U^T U (the upper Cholesky factor of the
 *               inverse), in permuted order.
 *
 * H          device float32 [d_in, d_in], read only; the upper 128-tile triangle (as
 *            written by gptq_hessian_accumulate) is read, the rest ignored.
 * damp       relative damping, >= 0 (0.01 on the pages).
 * perm       device int32 [d_in], out: perm[k] = original column processed k-th.
 * dead       device uint8 [d_in], out: 1 for dead channels (original order).
 * Hinv_chol  device float32 [d_in, d_in], out: U (strict lower triangle written as 0).
 * info       host int32, out, may be NULL: 0, or for GPTQ_ERR_NOT_PD the 1-based
 *            position in processing order of the first column whose pivot failed.
 * Errors: INVALID_ARG, WORKSPACE, NOT_PD (raise damp; the pages suggest up to 0.1),
 *         NONFINITE, CUDA, TIMEOUT.
 */
gptq_status gptq_prepare(const float* H, int32_t d_in, float damp, int actorder,
                         int32_t* perm, uint8_t* dead, float* Hinv_chol, int32_t* info,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_quantize_layer -- the GPTQ column loop and the packed checkpoint tensors.
 *
 * Defined by "GPTQ Architecture, in depth", "The algorithm in code" (gptq, fit_group)
 * and "Packing, tooling and serving", "Same Ruler, Smarter Placement: GPTQ" sections
 * 1.5 and 1.8, "04 - GPTQ" section 8.  With W' = W with dead columns zeroed, in
 * processing order, for each column q in order: at a group start fit (s, z) per row on
 * the current W'[:, q:q+g] (asymmetric: lo = min(w,0), hi = max(w,0),
 * s = max((hi-lo)/maxq, 1e-8), z = round(-lo/s); symmetric: s = max(max|w| /
 * (2^(bits-1)-1), 1e-8), z = 2^(bits-1)); code = clamp(round(w/s) + z, lowest, maxq)
 * (lowest = 0 asymmetric, 1 symmetric; round half to even; w/s in float32);
 * e = (w - s(code - z)) / U_qq; every later column j: w_j -= e U_qj.  Results equal the
 * unblocked loop up to float32 rounding; the engine applies updates inside 128-column
 * blocks at once and pushes each block's errors to later columns as one matrix product.
 *
 * W          device [d_out, d_in] row-major, `wdtype` (float32 or bfloat16); read only.
 * Hinv_chol  device float32 [d_in, d_in], U from gptq_prepare (upper triangle read).
 * perm       device int32 [d_in], or NULL for natural order.
 * dead       device uint8 [d_in], or NULL for no dead channels.
 * d_out      >= 0 (0: only g_idx and *loss = 0 are written); multiple of 32.
 * d_in       >= 1, multiple of 32.
 * bits       2, 3, 4 or 8.   group: -1 (one group per row), 16, 32, 64, or a multiple
 *            of 128.   sym: 0 asymmetric, 1 symmetric.
 * blocksize  1..128.  Results do not depend on it (beyond rounding); it is accepted for
 *            the pages' interface.  With group != -1, group and blocksize must divide
 *            one another, else GPTQ_ERR_UNSUPPORTED.
 * qweight    device int32 [bits*d_in/32, d_out], out: codes in original column order
 *            packed along d_in as a little-endian bit stream (code k of output row r at
 *            bits [bits*k, bits*k+bits) of column r's stream).
 * scales     device float32 [G, d_out], out; G = ceil(d_in/group) (1 when group=-1),
 *            groups in processing order (original order with static groups, below).
 * qzeros     device int32 [G, bits*d_out/32], out: zero points packed along d_out.
 * g_idx      device int32 [d_in], out: g_idx[c] = (position of c in perm) / group.
 * loss       device float64 scalar, out: sum over rows and columns of e^2 / 2, the OBS
 *            loss (w - what)^2 / (2 [H_cond^-1]_qq) ("04 - GPTQ", section 2).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, NONFINITE (W), CUDA, TIMEOUT.
 */
gptq_status gptq_quantize_layer(const void* W, int wdtype, const float* Hinv_chol,
                                const int32_t* perm, const uint8_t* dead, int32_t d_out,
                                int32_t d_in, int bits, int group, int sym, int blocksize,
                                int32_t* qweight, float* scales, int32_t* qzeros,
                                int32_t* g_idx, double* loss, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * gptq_quantize_layer_ex -- gptq_quantize_layer with option flags (the same arguments,
 * plus `flags` after `blocksize`; flags = 0 is gptq_quantize_layer).
 *
 * GPTQ_QUANT_STATIC_GROUPS: static groups ("GPTQ Architecture, in depth", "Groups,
 * act-order and other knobs": groups fixed in the original order before permuting, so
 * that a serving kernel reads its scales contiguously).  Group G is the original columns
 * [G*group, (G+1)*group); its (s, z) per row are fitted once, before the column loop, on
 * W after the dead fix (no permutation, no compensation yet), with the same formulas as
 * above; processed column q then rounds on the grid of group perm[q] / group.  scales
 * and qzeros come in original group order and g_idx[c] = c / group.  With group = -1 it
 * is the same as flags = 0.
 * Errors: as gptq_quantize_layer; INVALID_ARG for an unknown flag.
 */
#define GPTQ_QUANT_STATIC_GROUPS 1
gptq_status gptq_quantize_layer_ex(const void* W, int wdtype, const float* Hinv_chol,
                                   const int32_t* perm, const uint8_t* dead, int32_t d_out,
                                   int32_t d_in, int bits, int group, int sym, int blocksize,
                                   int flags, int32_t* qweight, float* scales, int32_t* qzeros,
                                   int32_t* g_idx, double* loss, void* ws, size_t ws_bytes,
                                   void* stream);

/*
 * gptq_layer_host_size -- bytes of device memory gptq_quantize_layer_host needs for these
 * sizes and element types on the current device; 0 for invalid or unsupported values.
 */
size_t gptq_layer_host_size(int64_t chunk_tokens, int32_t d_out, int32_t d_in, int bits,
                            int group, int xdtype, int wdtype);

/*
 * gptq_quantize_layer_host -- one linear layer end to end from host memory: the Hessian
 * hook over every calibration token, gptq_prepare and gptq_quantize_layer_ex, with the
 * inputs read from and the packed checkpoint written to host buffers.
 *
 * The method is the one the three device calls define ("GPTQ Architecture, in depth",
 * "The algorithm in code": the hook over the calibration batches, then gptq; "Same
 * Ruler, Smarter Placement: GPTQ", sections 1.4-1.9); the outputs equal those of the
 * device calls run one after the other on the same inputs with the same chunking.  The
 * interface itself is an addition: the pages run the method from PyTorch on device
 * tensors.
 *
 * X      host [ntok, d_in] row-major, `xdtype`; ntok > 0.  It is copied to the device in
 *        chunks of chunk_tokens tokens through two staging buffers, each copy overlapping
 *        the Hessian kernels of the chunk before it.  Page-locked host memory (for example
 *        from cudaHostAlloc) lets the copies run asynchronously; pageable memory works but
 *        serialises them.
 * W      host [d_out, d_in] row-major, `wdtype`; copied once, after the tokens.
 * damp, actorder: as gptq_prepare.  bits, group, sym, blocksize, flags: as
 *        gptq_quantize_layer_ex (d_out and d_in multiples of 32, d_out > 0).
 * qweight, scales, qzeros, g_idx: host outputs with the layouts of gptq_quantize_layer.
 * perm   host int32 [d_in], out: the processing order gptq_prepare chose.
 * loss   host double, out: the OBS loss as in gptq_quantize_layer.
 * info   host int32, out, may be NULL: as gptq_prepare.
 * dev    device buffer of at least gptq_layer_host_size(chunk_tokens, d_out, d_in, bits,
 *        group, xdtype, wdtype) bytes, 256-byte aligned, owned by the caller: it holds H,
 *        U, the staging buffers, device copies of W and of the outputs, and the scratch
 *        the three device calls use in turn.  Its contents afterwards are unspecified.
 * stream as elsewhere; the host-to-device copies run on a library-internal copy stream of
 *        the device, ordered after the work already queued on `stream`.  The call returns
 *        after the outputs have arrived in host memory.  On every return no copy of this
 *        call is still in flight.
 * Errors: INVALID_ARG (also ntok == 0: nothing to prepare), UNSUPPORTED, WORKSPACE, and
 *         those of the three device calls (NOT_PD, NONFINITE, CUDA, TIMEOUT).
 */
gptq_status gptq_quantize_layer_host(const void* X, int xdtype, int64_t ntok,
                                     int64_t chunk_tokens, const void* W, int wdtype,
                                     int32_t d_out, int32_t d_in, float damp, int actorder,
                                     int bits, int group, int sym, int blocksize, int flags,
                                     int32_t* qweight, float* scales, int32_t* qzeros,
                                     int32_t* g_idx, int32_t* perm, double* loss, int32_t* info,
                                     void* dev, size_t dev_bytes, void* stream);

/*
 * gptq_dequant_matmul -- y = x W_hat^T from the packed checkpoint, the product a W4A16-
 * style serving kernel computes ("GPTQ Architecture, in depth", "Packing, tooling and
 * serving": codes are unpacked and dequantised with their group's scale and zero point
 * just before the multiply):
 *   y[t, r] = sum_c x[t, c] * scales[g, r] * (code[r, c] - zero[g, r]),  g = g_idx[c].
 * It reads exactly what gptq_quantize_layer(_ex) writes.
 *
 * x        device [n, d_in] row-major, `xdtype` (bfloat16 or float32).
 * n        tokens, >= 0 (0: nothing is written).
 * d_in     >= 32, multiple of 32;  d_out >= 0, multiple of 32.
 * bits     2, 3, 4 or 8.
 * qweight  device int32 [bits*d_in/32, d_out], scales device float32 [G, d_out], qzeros
 *          device int32 [G, bits*d_out/32], g_idx device int32 [d_in] with values in
 *          [0, G): the layout gptq_quantize_layer documents.  qweight and scales are
 *          16-byte aligned (they are copied to shared memory 16 bytes at a time).
 * G        number of groups (rows of scales).
 * y        device float32 [n, d_out], out.
 * ws       device workspace of gptq_workspace_size(GPTQ_OP_DEQUANT_MATMUL, ...) bytes
 *          (256-byte aligned; holds the status word).
 * Accumulation is float32; the result does not depend on timing (the d_in slices are
 * added in a fixed order).
 * Errors: INVALID_ARG (arguments; a g_idx value outside [0, G), reported after the
 *         kernel, which then read group 0 for it), UNSUPPORTED (bits, sizes), CUDA.
 */
gptq_status gptq_dequant_matmul(const void* x, int xdtype, int64_t n, int32_t d_in,
                                int32_t d_out, int bits, const int32_t* qweight,
                                const float* scales, const int32_t* qzeros,
                                const int32_t* g_idx, int32_t G, float* y, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * gptq_dequantize -- the dense weights the packed checkpoint stands for,
 *   W_hat[r, c] = scales[g, r] * (code[r, c] - zero[g, r]),  g = g_idx[c]
 * ("GPTQ Architecture, in depth", "Packing, tooling and serving"), e.g. to re-run a
 * quantised block on many tokens with a dense matrix product.
 *
 * qweight, scales, qzeros, g_idx, G, bits, d_in, d_out: as gptq_dequant_matmul.
 * W      device [d_out, d_in] row-major, out, `wdtype` (bfloat16 or float32).
 * ws     device workspace of gptq_workspace_size(GPTQ_OP_DEQUANT_MATMUL, ...) bytes.
 * Errors: as gptq_dequant_matmul.
 */
gptq_status gptq_dequantize(const int32_t* qweight, const float* scales, const int32_t* qzeros,
                            const int32_t* g_idx, int32_t d_out, int32_t d_in, int bits,
                            int32_t G, void* W, int wdtype, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * gptq_scales_fp16 -- the checkpoint's fp16 copy of the group scales.
 *
 * The checkpoint format stores the scales as fp16 ("GPTQ Architecture, in depth",
 * "Packing, tooling and serving"; the bytes of "04 - GPTQ" section 8 count 2 bytes per
 * scale).  The column loop fits and uses them in float32; this call converts the scales
 * of gptq_quantize_layer to fp16 with round to nearest, ties to even (overflow to
 * infinity, underflow to subnormals or zero; a scale of an all-zero group, 1e-8, becomes
 * 0, which dequantizes that group to zeros as before).
 *
 * scales  device float32 [n], in.
 * out     device binary16 [n] (uint16 bit patterns), out; may not overlap scales.
 * n       number of scales (G * d_out), >= 0.
 * Errors: INVALID_ARG (null pointer with n > 0, n < 0), CUDA.
 */
gptq_status gptq_scales_fp16(const float* scales, int64_t n, uint16_t* out, void* stream);

/*
 * gptq_check_wait_timeout -- self-check of the library's failure path for device waits.
 *
 * Every wait of the tensor-core kernels on an mbarrier (a copy or a matrix operation that
 * has not landed yet) is bounded: after a time limit it gives up, the kernel records
 * GPTQ_ERR_TIMEOUT in the call's status word and returns, and the call reports it, so a
 * wait that can never end does not hang the device.  This call runs that same bounded
 * wait, for limit_ns nanoseconds, on an mbarrier nothing ever arrives on, in a kernel with
 * nothing else in flight.  Not part of the method (the pages have no counterpart).
 *
 * limit_ns  1 .. 1e9 (at most one second).
 * ws        device workspace of at least 256 bytes (the status word), 256-byte aligned.
 * Returns GPTQ_ERR_TIMEOUT when the wait gave up as designed (gptq_last_error() says how
 * many waits ran out); GPTQ_OK would mean the wait ended by itself, which it cannot.
 * Errors: INVALID_ARG, CUDA.
 */
gptq_status gptq_check_wait_timeout(uint64_t limit_ns, void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_set_wait_limit -- the time limit of the tensor-core kernels' device waits (the
 * Hessian SYRK, the prepare's tf32x3 GEMMs, the lazy update), for every later call in
 * this process (all threads, all devices).  Not part of the method: a diagnostic that lets
 * a test make the kernels' pipeline waits run out on purpose.
 *
 * A pipeline wait (for a copy, a matrix operation or an accumulator) gives up after
 * limit_ns nanoseconds (2 s by default); the kernel then records GPTQ_ERR_TIMEOUT in the
 * call's status word and drains before it returns: it waits for every matrix operation
 * and every copy it issued to complete (the drain does not use this limit), so the device
 * memory and the context stay usable, and the call reports GPTQ_ERR_TIMEOUT; its outputs
 * are then unset.
 *
 * limit_ns  0 restores the default; else 1 .. 1e10.
 * Errors: INVALID_ARG.
 */
gptq_status gptq_set_wait_limit(uint64_t limit_ns);

/* Thread-local description of the last failure on this thread ("" if none). */
const char* gptq_last_error(void);

/* Name of a gptq_status value. */
const char* gptq_status_string(int status);

/* ABI version of this header: 1. */
int gptq_abi_version(void);

/*
 * Tracing.  gptq_profile_enable(1) makes every later call bracket each of its kernel
 * launches with CUDA events on the call's stream and accumulate the device time per
 * kernel kind; gptq_profile_read(kind, &ms, &launches) returns the totals and
 * gptq_profile_reset() clears them.  Kinds are the gptq_kernel_kind values; the name of
 * a kind is gptq_kernel_name(kind).  gptq_profile_select(kinds) limits the tracing to the
 * kinds whose bit (1 << kind) is set (all of them after load): the events between
 * consecutive kernels cost time and keep dependent launches apart, so a caller that
 * times whole calls traces only the kinds it needs.  gptq_launch_count() counts every
 * kernel launched by the library since load (profiling or not).
 */
typedef enum {
  GPTQ_K_SYRK_TC = 0, GPTQ_K_SYRK_SIMT, GPTQ_K_SYRK_REDUCE,
  GPTQ_K_PREP_DIAG, GPTQ_K_PREP_RANK, GPTQ_K_PREP_MIRROR, GPTQ_K_PREP_GATHER,
  GPTQ_K_POTRF_PANEL, GPTQ_K_POTRF_TRSM, GPTQ_K_POTRF_UPDATE,
  GPTQ_K_TRTRI_DIAG, GPTQ_K_TRTRI_UPDATE, GPTQ_K_PREP_REVERSE,
  GPTQ_K_QUANT_GATHER, GPTQ_K_QUANT_FIT, GPTQ_K_QUANT_LOOP, GPTQ_K_QUANT_LAZY,
  GPTQ_K_QUANT_PACK, GPTQ_K_QUANT_LOSS, GPTQ_K_QUANT_SPLIT, GPTQ_K_DEQUANT_MATMUL,
  GPTQ_K_DEQUANTIZE, GPTQ_K_HESSIAN_RESCALE, GPTQ_K_SELFCHECK,
  GPTQ_K_COUNT
} gptq_kernel_kind;

void gptq_profile_enable(int on);
void gptq_profile_select(uint32_t kinds);
int gptq_profile_read(int kind, double* ms_total, int64_t* launches);
void gptq_profile_reset(void);
const char* gptq_kernel_name(int kind);
int64_t gptq_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_GB300_H */
