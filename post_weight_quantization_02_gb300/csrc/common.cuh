// Shared host and device helpers of the GPTQ engine: errors, workspace carving, the
// device status word, bounded waits and launch tracing.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/gptq.h"

namespace gptq {

// ------------------------------------------------------------------ host-side errors

struct Error {
  gptq_status status;
  std::string msg;
};

[[noreturn]] void fail(gptq_status s, const char* fmt, ...);
void cuda_check(cudaError_t e, const char* what);
void set_last_error(const std::string& msg);

#define GPTQ_CUDA(call) ::gptq::cuda_check((call), #call)

// Lets kernel `func` take at least `bytes` of dynamic shared memory on the current device
// (raised once per device and size; safe to call from several host threads).
void ensure_dynamic_smem(const void* func, int bytes);
template <typename F>
void ensure_dynamic_smem(F* func, int bytes) {
  ensure_dynamic_smem(reinterpret_cast<const void*>(func), bytes);
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carves 256-byte aligned sub-buffers out of the caller's workspace.
class WsCarver {
 public:
  WsCarver(void* base, size_t bytes) : base_(static_cast<char*>(base)), size_(bytes) {}
  template <typename T>
  T* take(size_t count) {
    size_t need = align_up(count * sizeof(T), 256);
    if (off_ + need > size_) {
      fail(GPTQ_ERR_WORKSPACE, "workspace too small: need more than %zu bytes", size_);
    }
    T* p = reinterpret_cast<T*>(base_ + off_);
    off_ += need;
    return p;
  }
  size_t used() const { return off_; }

 private:
  char* base_;
  size_t size_;
  size_t off_ = 0;
};

// Counts bytes the way WsCarver lays them out.
struct WsPlan {
  size_t bytes = 0;
  template <typename T>
  void add(size_t count) { bytes += align_up(count * sizeof(T), 256); }
};

// ------------------------------------------------------------------ device status

// The first 256 bytes of every workspace: written by kernels, read after the call's
// stream synchronisation.
struct DevStatus {
  int code;      // gptq_status of the first device-side failure (0 = none)
  int info;      // failing pivot (1-based) or other detail
  int timeouts;  // number of bounded waits that ran out
  int pad[61];
};

__device__ __forceinline__ void dev_fail(DevStatus* st, int code, int info) {
  if (atomicCAS(&st->code, 0, code) == 0) st->info = info;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every spin-wait in the library gives up after this long and records a timeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------------ launch tracing

void trace_begin(int kind, cudaStream_t s);
void trace_end(int kind, cudaStream_t s);
void trace_flush();    // after the call's stream is synchronised
void trace_discard();  // on failure: drop this thread's pending events
void profile_enable(bool on);
void profile_select(uint32_t mask);
void profile_reset();
bool profile_read(int kind, double* ms, int64_t* n);
int64_t launch_count();
const std::string& last_error();

#define GPTQ_LAUNCH(kind, stream, kernel, grid, block, smem, ...)                 \
  do {                                                                            \
    ::gptq::trace_begin((kind), (stream));                                        \
    kernel<<<(grid), (block), (smem), (stream)>>>(__VA_ARGS__);                   \
    ::gptq::cuda_check(cudaGetLastError(), #kernel);                              \
    ::gptq::trace_end((kind), (stream));                                          \
  } while (0)

// Programmatic dependent launch.  A kernel launched with GPTQ_LAUNCH_PDL may start while
// the kernel before it in the stream is still running: it must call griddep_wait() before
// it reads or writes global memory that earlier work in the stream touches (the wait
// returns once the earlier grid has completed and its writes are visible; for a kernel
// launched without the attribute it returns at once).  griddep_launch_dependents() lets
// the next such kernel start as soon as every CTA of this one has issued it.
#ifdef __CUDACC__
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

template <typename... P, typename... A>
void launch_pdl(const char* name, void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                cudaStream_t s, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cuda_check(cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...), name);
}

#define GPTQ_LAUNCH_PDL(kind, stream, kernel, grid, block, smem, ...)                    \
  do {                                                                                  \
    ::gptq::trace_begin((kind), (stream));                                              \
    ::gptq::launch_pdl(#kernel, kernel, dim3(grid), dim3(block), (smem), (stream),      \
                       __VA_ARGS__);                                                    \
    ::gptq::trace_end((kind), (stream));                                                \
  } while (0)

// Number of SMs of the current device.
int sm_count();

// Limit of the tensor-core kernels' pipeline waits for the launches that follow
// (process-wide; kWaitLimitNs unless gptq_set_wait_limit changed it).
uint64_t wait_limit_ns();
void set_wait_limit_ns(uint64_t ns);

// Three library-internal streams of the current device (a: highest priority, c: middle,
// b: lowest) and at least `nevents` timing-free events, created on first use and kept for the life
// of the process.  Calls that use them hold aux_mutex() until their work has finished.
struct AuxStreams {
  cudaStream_t a = nullptr;
  cudaStream_t b = nullptr;
  cudaStream_t c = nullptr;
  std::vector<cudaEvent_t> ev;
  cudaStream_t copy = nullptr;  // host <-> device copies of gptq_quantize_layer_host
};
AuxStreams& aux_streams(int nevents);
std::mutex& aux_mutex();
// The current device's copy stream (created on first use); call with aux_mutex() held.
cudaStream_t copy_stream();

}  // namespace gptq
