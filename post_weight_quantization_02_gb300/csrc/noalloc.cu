// gptq_hessian_accumulate_noalloc: the Hessian hook for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they feed
// calibration batches: a host framework that owns the whole device pool and forbids
// allocations after start-up, a plug-in running inside someone else's memory manager, or
// a latency-sensitive loop that must not hit an allocation's implicit device
// synchronisation.  They still own H and X; this entry point takes its scratch (the
// token-split partials and the status word) from a fixed array that the library itself
// places in device memory, so it needs no workspace argument and allocates nothing.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <string>

#include "common.cuh"

namespace gptq {
namespace {

// 256 bytes of status word plus 16 MiB of float32 partials: room for one d_in x d_in
// partial at d_in <= 2048 (more token splits at smaller d_in).  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoallocPartialBytes = static_cast<size_t>(16) << 20;
constexpr size_t kNoallocScratchBytes = kNoallocPartialBytes + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_ptr;  // device ordinal -> device address of the array

// Device address of the array on the current device.  In host code the array's name is
// only a host-side stand-in, so its address is asked from the runtime once per device,
// with that device current.
void* noalloc_scratch_ptr() {
  int dev = 0;
  cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_ptr.find(dev);
  if (it != g_noalloc_ptr.end()) return it->second;
  void* p = nullptr;
  cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress");
  g_noalloc_ptr[dev] = p;
  return p;
}

}  // namespace
}  // namespace gptq

extern "C" gptq_status gptq_hessian_accumulate_noalloc(float* H, int64_t* nseen, const void* X,
                                                       int xdtype, int64_t ntok, int32_t d_in,
                                                       void* stream) {
  using namespace gptq;
  if (d_in > 0 && static_cast<uint64_t>(d_in) * static_cast<uint64_t>(d_in) * sizeof(float) >
                      kNoallocPartialBytes) {
    set_last_error("gptq_hessian_accumulate_noalloc: d_in = " + std::to_string(d_in) +
                   " exceeds the built-in scratch (16 MiB: d_in <= 2048); use "
                   "gptq_hessian_accumulate with a caller workspace");
    return GPTQ_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  try {
    scratch = noalloc_scratch_ptr();
  } catch (const Error& e) {
    set_last_error(e.msg);
    return e.status;
  }
  // The status word at the start of the array is cleared by every call; the partials are
  // rewritten in full before the reduction reads them.
  return gptq_hessian_accumulate(H, nseen, X, xdtype, ntok, d_in, scratch, kNoallocScratchBytes,
                                 stream);
}
