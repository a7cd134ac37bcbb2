// The C ABI: argument checks, workspace layout, split choice and call orchestration.
// Every entry point enqueues its kernels on the caller's stream, synchronises that
// stream and returns the status of the work (see include/gptq.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>

#include "common.cuh"
#include "kernels.cuh"

namespace gptq {
namespace {

template <typename F>
gptq_status guarded(F&& f) {
  try {
    f();
    set_last_error("");
    return GPTQ_OK;
  } catch (const Error& e) {
    trace_discard();
    set_last_error(e.msg);
    return e.status;
  } catch (const std::exception& e) {
    trace_discard();
    set_last_error(std::string("internal error: ") + e.what());
    return GPTQ_ERR_CUDA;
  } catch (...) {
    trace_discard();
    set_last_error("internal error");
    return GPTQ_ERR_CUDA;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

void require(bool ok, gptq_status s, const char* msg) {
  if (!ok) fail(s, "%s", msg);
}

void begin_call(DevStatus* st, cudaStream_t s) {
  GPTQ_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
}

// Synchronise, read the device status word, fold in the tracing events.
DevStatus finish_call(DevStatus* st, cudaStream_t s) {
  DevStatus h;
  std::memset(&h, 0, sizeof(h));
  GPTQ_CUDA(cudaMemcpyAsync(&h, st, 3 * sizeof(int), cudaMemcpyDeviceToHost, s));
  GPTQ_CUDA(cudaStreamSynchronize(s));
  trace_flush();
  return h;
}

void raise_device_status(const DevStatus& h, const char* call) {
  switch (h.code) {
    case 0:
      return;
    case GPTQ_ERR_NOT_PD:
      fail(GPTQ_ERR_NOT_PD, "%s: H_damp is not positive definite (pivot at processing position %d);"
           " raise damp", call, h.info);
    case GPTQ_ERR_NONFINITE:
      fail(GPTQ_ERR_NONFINITE, "%s: NaN or Inf in the input (detail %d)", call, h.info);
    case GPTQ_ERR_TIMEOUT:
      fail(GPTQ_ERR_TIMEOUT, "%s: %d device-side wait(s) ran out", call, h.timeouts);
    default:
      fail(static_cast<gptq_status>(h.code), "%s: device reported status %d", call, h.code);
  }
}

// ------------------------------------------------------------------ Hessian

// bf16 tokens run on the tensor-core SYRK, float32 tokens on the float32 FMA kernel
bool use_tensor_cores(int xdtype) { return xdtype == GPTQ_BF16; }

int planning_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) {
    return n;
  }
  cudaGetLastError();
  return 152;  // sizing only: GB300
}

struct SplitPlan {
  int splits;
  int64_t tok_per_split;
};

// Splits of the token axis: enough units to fill the SMs evenly, at least 8 token
// stages per unit, and no more partials than the workspace holds.
SplitPlan plan_splits(int64_t ntok, int d, bool tc, int64_t max_splits, int nsm) {
  const int granule = tc ? syrk_tc_token_granule(d) : 16;
  const int64_t tiles = tc ? syrk_tc_tiles(d) : syrk_simt_tiles(d);
  const int64_t slots = tc ? nsm : 4LL * nsm;  // the SIMT kernel keeps ~4 CTAs per SM
  int64_t smax = ntok / (8LL * granule);
  if (smax < 1) smax = 1;
  if (smax > 16) smax = 16;
  if (smax > max_splits) smax = max_splits;
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= smax; ++s) {
    const int64_t units = tiles * s;
    const int64_t waves = (units + slots - 1) / slots;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * slots);
    if (eff > best_eff + 0.03) {
      best_eff = eff;
      best = s;
    }
    if (eff >= 0.9) break;
  }
  int64_t tps = (ntok + best - 1) / best;
  tps = (tps + granule - 1) / granule * granule;
  SplitPlan p;
  p.tok_per_split = tps;
  p.splits = static_cast<int>((ntok + tps - 1) / tps);
  return p;
}

size_t hessian_ws_bytes(int d, int splits) {
  WsPlan w;
  w.add<DevStatus>(1);
  w.add<float>(static_cast<size_t>(splits) * d * d);
  return w.bytes;
}

size_t prepare_ws_bytes(int d) {
  WsPlan w;
  w.add<DevStatus>(1);
  w.add<float>(static_cast<size_t>(d) * d);  // symmetric copy, then the inverse
  w.add<float>(static_cast<size_t>(d) * d);  // reversed, permuted, damped H -> factor
  w.add<float>(d);                           // fixed diagonal
  w.add<float>(1);                           // lambda
  w.add<float>(static_cast<size_t>(ceil_div(d, 128)) * 128 * 128);  // diagonal-block inverses
  w.add<float>(static_cast<size_t>(2) * d * kSuperpanel);  // lo parts of two superpanels
  return w.bytes;
}

size_t quantize_ws_bytes(int m, int d, int G) {
  WsPlan w;
  w.add<DevStatus>(1);
  w.add<float>(static_cast<size_t>(m) * d);    // Wp
  w.add<uint8_t>(static_cast<size_t>(m) * d);  // codesT
  w.add<uint16_t>(static_cast<size_t>(kErrRows) * m);  // errors, bf16 hi
  w.add<uint16_t>(static_cast<size_t>(kErrRows) * m);  // errors, bf16 lo
  w.add<uint16_t>(static_cast<size_t>(d) * d);    // U, bf16 hi
  w.add<uint16_t>(static_cast<size_t>(d) * d);    // U, bf16 lo
  w.add<int32_t>(static_cast<size_t>(G) * m);  // zeros
  w.add<double>(m);                            // loss_rows
  w.add<int32_t>(d);                           // pos
  w.add<float>(static_cast<size_t>(ceil_div(d, 128)) * kLoopUblkFloats);  // loop layout of U
  return w.bytes;
}

int groups_of(int d, int group) { return group == -1 ? 1 : static_cast<int>(ceil_div(d, group)); }

bool group_supported(int group) {
  return group == -1 || group == 16 || group == 32 || group == 64 || (group > 0 && group % 128 == 0);
}

// Device layout of gptq_quantize_layer_host: the layer's persistent buffers, two staging
// buffers for token chunks, the device copies of W and of the outputs, and one scratch
// region shared in turn by the Hessian, prepare and quantize workspaces.
struct HostLayout {
  size_t hess, prep, quant, scratch, total;
};

size_t hessian_ws_for(int64_t ntok, int d);

HostLayout host_layout(int64_t chunk, int m, int d, int bits, int group, int xdtype,
                       int wdtype) {
  HostLayout L;
  const int G = groups_of(d, group);
  const size_t xe = (xdtype == GPTQ_BF16) ? 2 : 4, we = (wdtype == GPTQ_BF16) ? 2 : 4;
  L.hess = hessian_ws_for(chunk, d);
  L.prep = prepare_ws_bytes(d);
  L.quant = quantize_ws_bytes(m, d, G);
  L.scratch = std::max(L.hess, std::max(L.prep, L.quant));
  WsPlan w;
  w.add<float>(static_cast<size_t>(d) * d);                    // H
  w.add<float>(static_cast<size_t>(d) * d);                    // U
  w.add<int32_t>(d);                                           // perm
  w.add<uint8_t>(d);                                           // dead
  w.add<uint8_t>(static_cast<size_t>(m) * d * we);             // W
  w.add<uint8_t>(static_cast<size_t>(chunk) * d * xe);         // token chunk, buffer 0
  w.add<uint8_t>(static_cast<size_t>(chunk) * d * xe);         // token chunk, buffer 1
  w.add<int32_t>(static_cast<size_t>(bits) * d / 32 * m);      // qweight
  w.add<float>(static_cast<size_t>(G) * m);                    // scales
  w.add<int32_t>(static_cast<size_t>(G) * bits * m / 32);      // qzeros
  w.add<int32_t>(d);                                           // g_idx
  w.add<double>(1);                                            // loss
  w.add<uint8_t>(L.scratch);
  L.total = w.bytes;
  return L;
}

// The Hessian step behind gptq_hessian_accumulate (sync) and its enqueue-only form.
void hessian_step(float* H, int64_t* nseen, const void* X, int xdtype, int64_t ntok,
                  int32_t d_in, void* ws, size_t ws_bytes, void* stream, bool sync) {
  require(H != nullptr && nseen != nullptr && ws != nullptr, GPTQ_ERR_INVALID_ARG,
          "gptq_hessian_accumulate: null H, nseen or ws");
  require(d_in > 0 && ntok >= 0 && *nseen >= 0, GPTQ_ERR_INVALID_ARG,
          "gptq_hessian_accumulate: need d_in > 0, ntok >= 0, *nseen >= 0");
  require(xdtype == GPTQ_F32 || xdtype == GPTQ_BF16, GPTQ_ERR_INVALID_ARG,
          "gptq_hessian_accumulate: xdtype must be GPTQ_F32 or GPTQ_BF16");
  require(d_in % 8 == 0, GPTQ_ERR_UNSUPPORTED, "gptq_hessian_accumulate: d_in must be a multiple of 8");
  require(ntok == 0 || X != nullptr, GPTQ_ERR_INVALID_ARG, "gptq_hessian_accumulate: null X");
  require(aligned(H, 16) && aligned(X, 16) && aligned(ws, 256), GPTQ_ERR_INVALID_ARG,
          "gptq_hessian_accumulate: H and X must be 16-byte aligned, ws 256-byte aligned");
  require(ntok < (int64_t(1) << 31), GPTQ_ERR_UNSUPPORTED,
          "gptq_hessian_accumulate: at most 2^31 - 1 tokens per call");
  const int64_t one = hessian_ws_bytes(d_in, 1);
  require(ws_bytes >= static_cast<size_t>(one), GPTQ_ERR_WORKSPACE,
          "gptq_hessian_accumulate: workspace smaller than d_in*d_in*4 + 256 bytes");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsCarver wc(ws, ws_bytes);
  DevStatus* st = wc.take<DevStatus>(1);
  // the enqueue-only form clears the status word at a layer's first batch and lets it
  // collect failures until gptq_hessian_status reads it
  if (!sync && *nseen == 0) begin_call(st, s);
  if (ntok == 0) return;
  const bool tc = use_tensor_cores(xdtype);
  const size_t per = static_cast<size_t>(d_in) * d_in * sizeof(float);
  const int64_t cap = static_cast<int64_t>((ws_bytes - 256) / per);
  SplitPlan p = plan_splits(ntok, d_in, tc, cap, sm_count());
  float* P = wc.take<float>(static_cast<size_t>(p.splits) * d_in * d_in);

  const int64_t n_old = *nseen;
  const double n_new = static_cast<double>(n_old) + static_cast<double>(ntok);
  const float alpha = static_cast<float>(2.0 / n_new);
  const float beta = static_cast<float>(static_cast<double>(n_old) / n_new);

  if (sync) begin_call(st, s);
  if (tc) launch_syrk_tc(X, ntok, d_in, p.splits, p.tok_per_split, P, st, s);
  else launch_syrk_simt(X, xdtype == GPTQ_BF16, ntok, d_in, p.splits, p.tok_per_split, P, s);
  launch_syrk_reduce(H, P, d_in, p.splits, alpha, beta, n_old == 0, s);
  if (sync) raise_device_status(finish_call(st, s), "gptq_hessian_accumulate");
  *nseen = n_old + ntok;
}

// The Hessian workspace gptq_workspace_size reports for a call of ntok tokens.
size_t hessian_ws_for(int64_t ntok, int d) {
  const int64_t t = ntok > 0 ? ntok : 1;
  SplitPlan p = plan_splits(t, d, true, 16, planning_sm_count());
  SplitPlan q = plan_splits(t, d, false, 16, planning_sm_count());
  return hessian_ws_bytes(d, p.splits > q.splits ? p.splits : q.splits);
}

// Events of one gptq_quantize_layer_host call.  On every exit the copy stream is drained
// first, so that no copy still reads the caller's host buffers or writes the device
// buffer after the call returns.
struct HostCallEvents {
  cudaStream_t copy = nullptr;
  cudaEvent_t ev[6] = {};
  int n = 0;
  ~HostCallEvents() {
    if (copy != nullptr) cudaStreamSynchronize(copy);
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
};

}  // namespace
}  // namespace gptq

using namespace gptq;

extern "C" {

size_t gptq_workspace_size(int op, int64_t ntok, int32_t d_out, int32_t d_in, int bits,
                           int group) {
  (void)bits;
  if (d_in <= 0) return 0;
  switch (op) {
    case GPTQ_OP_HESSIAN:
      if (ntok < 0) return 0;
      return hessian_ws_for(ntok, d_in);
    case GPTQ_OP_PREPARE:
      return prepare_ws_bytes(d_in);
    case GPTQ_OP_QUANTIZE:
      if (d_out < 0 || !group_supported(group)) return 0;
      return quantize_ws_bytes(d_out, d_in, groups_of(d_in, group));
    case GPTQ_OP_DEQUANT_MATMUL:
      return 256;  // the status word
    default:
      return 0;
  }
}

gptq_status gptq_hessian_accumulate(float* H, int64_t* nseen, const void* X, int xdtype,
                                    int64_t ntok, int32_t d_in, void* ws, size_t ws_bytes,
                                    void* stream) {
  return guarded([&] { hessian_step(H, nseen, X, xdtype, ntok, d_in, ws, ws_bytes, stream, true); });
}

gptq_status gptq_hessian_accumulate_async(float* H, int64_t* nseen, const void* X, int xdtype,
                                          int64_t ntok, int32_t d_in, void* ws,
                                          size_t ws_bytes, void* stream) {
  return guarded([&] { hessian_step(H, nseen, X, xdtype, ntok, d_in, ws, ws_bytes, stream, false); });
}

gptq_status gptq_hessian_status(void* ws, size_t ws_bytes, void* stream) {
  return guarded([&] {
    require(ws != nullptr && aligned(ws, 256) && ws_bytes >= sizeof(DevStatus),
            GPTQ_ERR_INVALID_ARG, "gptq_hessian_status: null, unaligned or too small ws");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    DevStatus* st = wc.take<DevStatus>(1);
    const DevStatus h = finish_call(st, s);
    GPTQ_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
    GPTQ_CUDA(cudaStreamSynchronize(s));
    raise_device_status(h, "gptq_hessian_accumulate_async");
  });
}

gptq_status gptq_hessian_rescale(float* H, int32_t d_in, int64_t n_from, int64_t n_to,
                                 void* stream) {
  return guarded([&] {
    require(H != nullptr, GPTQ_ERR_INVALID_ARG, "gptq_hessian_rescale: null H");
    require(d_in > 0 && n_from >= 0 && n_to > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_hessian_rescale: need d_in > 0, n_from >= 0, n_to > 0");
    require(d_in % 8 == 0, GPTQ_ERR_UNSUPPORTED, "gptq_hessian_rescale: d_in must be a multiple of 8");
    require(aligned(H, 16), GPTQ_ERR_INVALID_ARG, "gptq_hessian_rescale: H must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float factor = static_cast<float>(static_cast<double>(n_from) / static_cast<double>(n_to));
    launch_hessian_rescale(H, d_in, factor, s);
    GPTQ_CUDA(cudaStreamSynchronize(s));
    trace_flush();
  });
}

gptq_status gptq_prepare(const float* H, int32_t d_in, float damp, int actorder,
                         int32_t* perm, uint8_t* dead, float* Hinv_chol, int32_t* info,
                         void* ws, size_t ws_bytes, void* stream) {
  if (info != nullptr) *info = 0;
  int32_t pivot = 0;
  gptq_status st_code = guarded([&] {
    require(H != nullptr && perm != nullptr && dead != nullptr && Hinv_chol != nullptr &&
                ws != nullptr,
            GPTQ_ERR_INVALID_ARG, "gptq_prepare: null pointer argument");
    require(d_in > 0, GPTQ_ERR_INVALID_ARG, "gptq_prepare: d_in must be positive");
    require(std::isfinite(damp) && damp >= 0.0f, GPTQ_ERR_INVALID_ARG,
            "gptq_prepare: damp must be finite and >= 0");
    require(d_in % 8 == 0, GPTQ_ERR_UNSUPPORTED, "gptq_prepare: d_in must be a multiple of 8");
    require(aligned(H, 16) && aligned(Hinv_chol, 16) && aligned(ws, 256), GPTQ_ERR_INVALID_ARG,
            "gptq_prepare: H and Hinv_chol must be 16-byte aligned, ws 256-byte aligned");
    require(ws_bytes >= prepare_ws_bytes(d_in), GPTQ_ERR_WORKSPACE,
            "gptq_prepare: workspace too small (see gptq_workspace_size)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    DevStatus* st = wc.take<DevStatus>(1);
    float* S = wc.take<float>(static_cast<size_t>(d_in) * d_in);
    float* Hr = wc.take<float>(static_cast<size_t>(d_in) * d_in);
    float* diag = wc.take<float>(d_in);
    float* lam = wc.take<float>(1);
    float* DI = wc.take<float>(static_cast<size_t>(ceil_div(d_in, 128)) * 128 * 128);
    float* Lo = wc.take<float>(static_cast<size_t>(2) * d_in * kSuperpanel);
    std::lock_guard<std::mutex> lk(aux_mutex());  // the internal streams are shared
    begin_call(st, s);
    launch_prepare(H, d_in, damp, actorder ? 1 : 0, perm, dead, Hinv_chol, S, Hr, diag, lam, DI,
                   Lo, st, s);
    DevStatus h = finish_call(st, s);
    if (h.code == GPTQ_ERR_NOT_PD) pivot = h.info;
    raise_device_status(h, "gptq_prepare");
  });
  if (info != nullptr) *info = pivot;
  return st_code;
}

gptq_status gptq_quantize_layer_ex(const void* W, int wdtype, const float* Hinv_chol,
                                   const int32_t* perm, const uint8_t* dead, int32_t d_out,
                                   int32_t d_in, int bits, int group, int sym, int blocksize,
                                   int flags, int32_t* qweight, float* scales, int32_t* qzeros,
                                   int32_t* g_idx, double* loss, void* ws, size_t ws_bytes,
                                   void* stream) {
  return guarded([&] {
    require((flags & ~GPTQ_QUANT_STATIC_GROUPS) == 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: unknown flags");
    require(d_in > 0 && d_out >= 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: need d_in > 0 and d_out >= 0");
    require(Hinv_chol != nullptr && g_idx != nullptr && loss != nullptr && ws != nullptr,
            GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer: null Hinv_chol, g_idx, loss or ws");
    require(d_out == 0 || (W != nullptr && qweight != nullptr && scales != nullptr &&
                           qzeros != nullptr),
            GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer: null W or output");
    require(wdtype == GPTQ_F32 || wdtype == GPTQ_BF16, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: wdtype must be GPTQ_F32 or GPTQ_BF16");
    require(sym == 0 || sym == 1, GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer: sym must be 0 or 1");
    require(blocksize >= 1 && blocksize <= 128, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: blocksize must be in 1..128");
    require(group == -1 || group > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: group must be -1 or positive");
    require(bits == 2 || bits == 3 || bits == 4 || bits == 8, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer: bits must be 2, 3, 4 or 8");
    require(group_supported(group), GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer: group must be -1, 16, 32, 64 or a multiple of 128");
    require(group == -1 || group % blocksize == 0 || blocksize % group == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer: group and blocksize must divide one another");
    require(d_in % 32 == 0 && d_out % 32 == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer: d_in and d_out must be multiples of 32");
    require(aligned(W, 16) && aligned(Hinv_chol, 16) && aligned(ws, 256), GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer: W and Hinv_chol must be 16-byte aligned, ws 256-byte aligned");
    const int G = groups_of(d_in, group);
    require(ws_bytes >= quantize_ws_bytes(d_out, d_in, G), GPTQ_ERR_WORKSPACE,
            "gptq_quantize_layer: workspace too small (see gptq_workspace_size)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    QuantArgs q;
    q.st = wc.take<DevStatus>(1);
    q.Wp = wc.take<float>(static_cast<size_t>(d_out) * d_in);
    q.codesT = wc.take<uint8_t>(static_cast<size_t>(d_out) * d_in);
    q.ehi = wc.take<__nv_bfloat16>(static_cast<size_t>(kErrRows) * d_out);
    q.elo = wc.take<__nv_bfloat16>(static_cast<size_t>(kErrRows) * d_out);
    q.uhi = wc.take<__nv_bfloat16>(static_cast<size_t>(d_in) * d_in);
    q.ulo = wc.take<__nv_bfloat16>(static_cast<size_t>(d_in) * d_in);
    q.zeros = wc.take<int32_t>(static_cast<size_t>(G) * d_out);
    q.loss_rows = wc.take<double>(d_out);
    q.pos = wc.take<int32_t>(d_in);
    q.Ublk = wc.take<float>(static_cast<size_t>(ceil_div(d_in, 128)) * kLoopUblkFloats);
    q.W = W;
    q.w_bf16 = (wdtype == GPTQ_BF16);
    q.U = Hinv_chol;
    q.perm = perm;
    q.dead = dead;
    q.m = d_out;
    q.d = d_in;
    q.bits = bits;
    q.group = group;
    q.static_groups = (flags & GPTQ_QUANT_STATIC_GROUPS) != 0;
    q.sym = sym;
    q.G = G;
    q.qweight = qweight;
    q.scales = scales;
    q.qzeros = qzeros;
    q.g_idx = g_idx;
    q.loss = loss;
    begin_call(q.st, s);
    launch_quantize(q, s);
    raise_device_status(finish_call(q.st, s), "gptq_quantize_layer");
  });
}

gptq_status gptq_quantize_layer(const void* W, int wdtype, const float* Hinv_chol,
                                const int32_t* perm, const uint8_t* dead, int32_t d_out,
                                int32_t d_in, int bits, int group, int sym, int blocksize,
                                int32_t* qweight, float* scales, int32_t* qzeros,
                                int32_t* g_idx, double* loss, void* ws, size_t ws_bytes,
                                void* stream) {
  return gptq_quantize_layer_ex(W, wdtype, Hinv_chol, perm, dead, d_out, d_in, bits, group, sym,
                                blocksize, 0, qweight, scales, qzeros, g_idx, loss, ws,
                                ws_bytes, stream);
}

size_t gptq_layer_host_size(int64_t chunk_tokens, int32_t d_out, int32_t d_in, int bits,
                            int group, int xdtype, int wdtype) {
  if (chunk_tokens <= 0 || d_out <= 0 || d_in <= 0 || d_in % 32 != 0 || d_out % 32 != 0 ||
      !(bits == 2 || bits == 3 || bits == 4 || bits == 8) || !group_supported(group) ||
      !(xdtype == GPTQ_F32 || xdtype == GPTQ_BF16) || !(wdtype == GPTQ_F32 || wdtype == GPTQ_BF16)) {
    return 0;
  }
  return host_layout(chunk_tokens, d_out, d_in, bits, group, xdtype, wdtype).total;
}

gptq_status gptq_quantize_layer_host(const void* X, int xdtype, int64_t ntok, int64_t chunk_tokens,
                                     const void* W, int wdtype, int32_t d_out, int32_t d_in,
                                     float damp, int actorder, int bits, int group, int sym,
                                     int blocksize, int flags, int32_t* qweight, float* scales,
                                     int32_t* qzeros, int32_t* g_idx, int32_t* perm, double* loss,
                                     int32_t* info, void* dev, size_t dev_bytes, void* stream) {
  if (info != nullptr) *info = 0;
  int32_t pivot = 0;
  gptq_status rc = guarded([&] {
    const char* fn = "gptq_quantize_layer_host";
    require(ntok > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: no calibration tokens (ntok must be positive)");
    require(X != nullptr && W != nullptr && qweight != nullptr && scales != nullptr &&
                qzeros != nullptr && g_idx != nullptr && perm != nullptr && loss != nullptr &&
                dev != nullptr,
            GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer_host: null pointer argument");
    require(chunk_tokens > 0 && chunk_tokens < (int64_t(1) << 31), GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: chunk_tokens must be in 1 .. 2^31 - 1");
    require(d_out > 0 && d_in > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: need d_out > 0 and d_in > 0");
    require((xdtype == GPTQ_F32 || xdtype == GPTQ_BF16) && (wdtype == GPTQ_F32 || wdtype == GPTQ_BF16),
            GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer_host: dtypes must be GPTQ_F32 or GPTQ_BF16");
    require(std::isfinite(damp) && damp >= 0.0f, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: damp must be finite and >= 0");
    require((flags & ~GPTQ_QUANT_STATIC_GROUPS) == 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: unknown flags");
    require(sym == 0 || sym == 1, GPTQ_ERR_INVALID_ARG, "gptq_quantize_layer_host: sym must be 0 or 1");
    require(blocksize >= 1 && blocksize <= 128, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: blocksize must be in 1..128");
    require(group == -1 || group > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: group must be -1 or positive");
    require(bits == 2 || bits == 3 || bits == 4 || bits == 8, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer_host: bits must be 2, 3, 4 or 8");
    require(group_supported(group), GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer_host: group must be -1, 16, 32, 64 or a multiple of 128");
    require(group == -1 || group % blocksize == 0 || blocksize % group == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer_host: group and blocksize must divide one another");
    require(d_in % 32 == 0 && d_out % 32 == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_quantize_layer_host: d_in and d_out must be multiples of 32");
    require(aligned(dev, 256), GPTQ_ERR_INVALID_ARG,
            "gptq_quantize_layer_host: the device buffer must be 256-byte aligned");
    const HostLayout lay = host_layout(chunk_tokens, d_out, d_in, bits, group, xdtype, wdtype);
    require(dev_bytes >= lay.total, GPTQ_ERR_WORKSPACE,
            "gptq_quantize_layer_host: device buffer too small (see gptq_layer_host_size)");
    const int m = d_out, d = d_in, G = groups_of(d, group);
    const size_t xe = (xdtype == GPTQ_BF16) ? 2 : 4, we = (wdtype == GPTQ_BF16) ? 2 : 4;
    WsCarver wc(dev, dev_bytes);
    float* H = wc.take<float>(static_cast<size_t>(d) * d);
    float* U = wc.take<float>(static_cast<size_t>(d) * d);
    int32_t* perm_d = wc.take<int32_t>(d);
    uint8_t* dead_d = wc.take<uint8_t>(d);
    uint8_t* W_d = wc.take<uint8_t>(static_cast<size_t>(m) * d * we);
    uint8_t* xs[2];
    xs[0] = wc.take<uint8_t>(static_cast<size_t>(chunk_tokens) * d * xe);
    xs[1] = wc.take<uint8_t>(static_cast<size_t>(chunk_tokens) * d * xe);
    const size_t qw_words = static_cast<size_t>(bits) * d / 32 * m;
    const size_t qz_words = static_cast<size_t>(G) * bits * m / 32;
    int32_t* qw_d = wc.take<int32_t>(qw_words);
    float* sc_d = wc.take<float>(static_cast<size_t>(G) * m);
    int32_t* qz_d = wc.take<int32_t>(qz_words);
    int32_t* gi_d = wc.take<int32_t>(d);
    double* loss_d = wc.take<double>(1);
    void* scratch = wc.take<uint8_t>(lay.scratch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    HostCallEvents he;
    {
      std::lock_guard<std::mutex> lk(aux_mutex());
      he.copy = copy_stream();
    }
    for (; he.n < 6; ++he.n) {
      GPTQ_CUDA(cudaEventCreateWithFlags(&he.ev[he.n], cudaEventDisableTiming));
    }
    cudaEvent_t* done = he.ev;       // [2] the Hessian step that read staging buffer b
    cudaEvent_t* ready = he.ev + 2;  // [2] the copy into staging buffer b
    cudaEvent_t fork = he.ev[4], wready = he.ev[5];
    // the copies follow whatever the caller queued on `stream` before this call
    GPTQ_CUDA(cudaEventRecord(fork, s));
    GPTQ_CUDA(cudaStreamWaitEvent(he.copy, fork, 0));
    // the Hessian hook over the token stream: chunk c is copied into staging buffer c % 2
    // while the Hessian kernels of chunk c - 1 run
    int64_t nseen = 0;
    const int64_t nchunks = (ntok + chunk_tokens - 1) / chunk_tokens;
    for (int64_t c = 0; c < nchunks; ++c) {
      const int b = static_cast<int>(c & 1);
      const int64_t t = std::min(chunk_tokens, ntok - c * chunk_tokens);
      if (c >= 2) GPTQ_CUDA(cudaStreamWaitEvent(he.copy, done[b], 0));
      GPTQ_CUDA(cudaMemcpyAsync(xs[b], static_cast<const char*>(X) + c * chunk_tokens * d * xe,
                                static_cast<size_t>(t) * d * xe, cudaMemcpyHostToDevice, he.copy));
      GPTQ_CUDA(cudaEventRecord(ready[b], he.copy));
      GPTQ_CUDA(cudaStreamWaitEvent(s, ready[b], 0));
      hessian_step(H, &nseen, xs[b], xdtype, t, d, scratch, lay.hess, stream, false);
      GPTQ_CUDA(cudaEventRecord(done[b], s));
    }
    // the weights follow the tokens on the copy stream
    GPTQ_CUDA(cudaMemcpyAsync(W_d, W, static_cast<size_t>(m) * d * we, cudaMemcpyHostToDevice,
                              he.copy));
    GPTQ_CUDA(cudaEventRecord(wready, he.copy));
    {
      WsCarver hw(scratch, lay.hess);
      raise_device_status(finish_call(hw.take<DevStatus>(1), s), fn);
    }
    gptq_status st = gptq_prepare(H, d, damp, actorder, perm_d, dead_d, U, &pivot, scratch,
                                  lay.scratch, stream);
    if (st != GPTQ_OK) fail(st, "%s", last_error().c_str());
    GPTQ_CUDA(cudaStreamWaitEvent(s, wready, 0));
    st = gptq_quantize_layer_ex(W_d, wdtype, U, perm_d, dead_d, m, d, bits, group, sym, blocksize,
                                flags, qw_d, sc_d, qz_d, gi_d, loss_d, scratch, lay.scratch, stream);
    if (st != GPTQ_OK) fail(st, "%s", last_error().c_str());
    double loss_h = 0.0;
    GPTQ_CUDA(cudaMemcpyAsync(qweight, qw_d, qw_words * 4, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaMemcpyAsync(scales, sc_d, static_cast<size_t>(G) * m * 4, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaMemcpyAsync(qzeros, qz_d, qz_words * 4, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaMemcpyAsync(g_idx, gi_d, static_cast<size_t>(d) * 4, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaMemcpyAsync(perm, perm_d, static_cast<size_t>(d) * 4, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaMemcpyAsync(&loss_h, loss_d, sizeof(double), cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA(cudaStreamSynchronize(s));
    *loss = loss_h;
  });
  if (info != nullptr) *info = pivot;
  return rc;
}

gptq_status gptq_dequant_matmul(const void* x, int xdtype, int64_t n, int32_t d_in,
                                int32_t d_out, int bits, const int32_t* qweight,
                                const float* scales, const int32_t* qzeros,
                                const int32_t* g_idx, int32_t G, float* y, void* ws,
                                size_t ws_bytes, void* stream) {
  return guarded([&] {
    require(n >= 0 && d_in > 0 && d_out >= 0 && G > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_dequant_matmul: need n >= 0, d_in > 0, d_out >= 0, G > 0");
    require(xdtype == GPTQ_F32 || xdtype == GPTQ_BF16, GPTQ_ERR_INVALID_ARG,
            "gptq_dequant_matmul: xdtype must be GPTQ_F32 or GPTQ_BF16");
    require(bits == 2 || bits == 3 || bits == 4 || bits == 8, GPTQ_ERR_UNSUPPORTED,
            "gptq_dequant_matmul: bits must be 2, 3, 4 or 8");
    require(d_in % 32 == 0 && d_out % 32 == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_dequant_matmul: d_in and d_out must be multiples of 32");
    require(ws != nullptr && aligned(ws, 256) && ws_bytes >= sizeof(DevStatus),
            GPTQ_ERR_INVALID_ARG, "gptq_dequant_matmul: null, unaligned or too small ws");
    require(n == 0 || d_out == 0 ||
                (x != nullptr && qweight != nullptr && scales != nullptr && qzeros != nullptr &&
                 g_idx != nullptr && y != nullptr),
            GPTQ_ERR_INVALID_ARG, "gptq_dequant_matmul: null input or output");
    require(aligned(qweight, 16) && aligned(scales, 16), GPTQ_ERR_INVALID_ARG,
            "gptq_dequant_matmul: qweight and scales must be 16-byte aligned");
    if (n == 0 || d_out == 0) return;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    DevStatus* st = wc.take<DevStatus>(1);
    begin_call(st, s);
    launch_dequant_matmul(x, xdtype == GPTQ_BF16, n, d_in, d_out, bits, G, qweight, scales,
                          qzeros, g_idx, y, st, s);
    raise_device_status(finish_call(st, s), "gptq_dequant_matmul");
  });
}

gptq_status gptq_dequantize(const int32_t* qweight, const float* scales, const int32_t* qzeros,
                            const int32_t* g_idx, int32_t d_out, int32_t d_in, int bits,
                            int32_t G, void* W, int wdtype, void* ws, size_t ws_bytes,
                            void* stream) {
  return guarded([&] {
    require(d_in > 0 && d_out >= 0 && G > 0, GPTQ_ERR_INVALID_ARG,
            "gptq_dequantize: need d_in > 0, d_out >= 0, G > 0");
    require(wdtype == GPTQ_F32 || wdtype == GPTQ_BF16, GPTQ_ERR_INVALID_ARG,
            "gptq_dequantize: wdtype must be GPTQ_F32 or GPTQ_BF16");
    require(bits == 2 || bits == 3 || bits == 4 || bits == 8, GPTQ_ERR_UNSUPPORTED,
            "gptq_dequantize: bits must be 2, 3, 4 or 8");
    require(d_in % 32 == 0 && d_out % 32 == 0, GPTQ_ERR_UNSUPPORTED,
            "gptq_dequantize: d_in and d_out must be multiples of 32");
    require(ws != nullptr && aligned(ws, 256) && ws_bytes >= sizeof(DevStatus),
            GPTQ_ERR_INVALID_ARG, "gptq_dequantize: null, unaligned or too small ws");
    require(d_out == 0 || (qweight != nullptr && scales != nullptr && qzeros != nullptr &&
                           g_idx != nullptr && W != nullptr),
            GPTQ_ERR_INVALID_ARG, "gptq_dequantize: null input or output");
    if (d_out == 0) return;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    DevStatus* st = wc.take<DevStatus>(1);
    begin_call(st, s);
    launch_dequantize(qweight, scales, qzeros, g_idx, d_out, d_in, bits, G, W,
                      wdtype == GPTQ_BF16, st, s);
    raise_device_status(finish_call(st, s), "gptq_dequantize");
  });
}

gptq_status gptq_scales_fp16(const float* scales, int64_t n, uint16_t* out, void* stream) {
  return guarded([&] {
    require(n >= 0, GPTQ_ERR_INVALID_ARG, "gptq_scales_fp16: n must be >= 0");
    require(n == 0 || (scales != nullptr && out != nullptr), GPTQ_ERR_INVALID_ARG,
            "gptq_scales_fp16: null pointer");
    launch_scales_fp16(scales, n, out, static_cast<cudaStream_t>(stream));
  });
}

gptq_status gptq_set_wait_limit(uint64_t limit_ns) {
  return guarded([&] {
    require(limit_ns <= 10000000000ull, GPTQ_ERR_INVALID_ARG,
            "gptq_set_wait_limit: limit_ns must be 0 (the default) or 1 .. 1e10");
    set_wait_limit_ns(limit_ns);
  });
}

gptq_status gptq_check_wait_timeout(uint64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  return guarded([&] {
    require(limit_ns >= 1 && limit_ns <= 1000000000ull, GPTQ_ERR_INVALID_ARG,
            "gptq_check_wait_timeout: limit_ns must be in 1 .. 1e9");
    require(ws != nullptr && aligned(ws, 256) && ws_bytes >= sizeof(DevStatus),
            GPTQ_ERR_INVALID_ARG, "gptq_check_wait_timeout: null, unaligned or too small ws");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsCarver wc(ws, ws_bytes);
    DevStatus* st = wc.take<DevStatus>(1);
    begin_call(st, s);
    launch_wait_timeout(st, limit_ns, s);
    raise_device_status(finish_call(st, s), "gptq_check_wait_timeout");
  });
}

const char* gptq_last_error(void) { return last_error().c_str(); }

const char* gptq_status_string(int status) {
  switch (status) {
    case GPTQ_OK: return "GPTQ_OK";
    case GPTQ_ERR_INVALID_ARG: return "GPTQ_ERR_INVALID_ARG";
    case GPTQ_ERR_UNSUPPORTED: return "GPTQ_ERR_UNSUPPORTED";
    case GPTQ_ERR_NOT_PD: return "GPTQ_ERR_NOT_PD";
    case GPTQ_ERR_NONFINITE: return "GPTQ_ERR_NONFINITE";
    case GPTQ_ERR_CUDA: return "GPTQ_ERR_CUDA";
    case GPTQ_ERR_TIMEOUT: return "GPTQ_ERR_TIMEOUT";
    case GPTQ_ERR_WORKSPACE: return "GPTQ_ERR_WORKSPACE";
    default: return "GPTQ_ERR_UNKNOWN";
  }
}

int gptq_abi_version(void) { return 1; }

void gptq_profile_enable(int on) { profile_enable(on != 0); }
void gptq_profile_select(uint32_t kinds) { profile_select(kinds); }
int gptq_profile_read(int kind, double* ms_total, int64_t* launches) {
  return profile_read(kind, ms_total, launches) ? 0 : -1;
}
void gptq_profile_reset(void) { profile_reset(); }

const char* gptq_kernel_name(int kind) {
  static const char* names[GPTQ_K_COUNT] = {
      "syrk_tc", "syrk_simt", "syrk_reduce", "prep_diag", "prep_rank", "prep_mirror",
      "prep_gather", "potrf_panel", "potrf_trsm", "potrf_update", "trtri_diag", "trtri_update",
      "prep_reverse", "quant_gather", "quant_fit", "quant_loop", "quant_lazy", "quant_pack",
      "quant_loss", "quant_split", "dequant_matmul", "dequantize", "hessian_rescale",
      "selfcheck"};
  if (kind < 0 || kind >= GPTQ_K_COUNT) return "";
  return names[kind];
}

int64_t gptq_launch_count(void) { return launch_count(); }

}  // extern "C"
