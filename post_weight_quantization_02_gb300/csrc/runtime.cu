// Host runtime of the engine: thread-local errors, launch tracing with CUDA events, the
// device's SM count and tensor-map encoding.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <map>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "tc_common.cuh"

namespace gptq {

namespace {
thread_local std::string g_last_error;
}

void set_last_error(const std::string& msg) { g_last_error = msg; }
const std::string& last_error() { return g_last_error; }

void fail(gptq_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  throw Error{s, std::string(buf)};
}

void cuda_check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fail(GPTQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  }
}

// ------------------------------------------------------------------ tracing

namespace {

struct Pending {
  int kind;
  cudaEvent_t start;
  cudaEvent_t stop;
};

std::mutex g_mu;
std::atomic<bool> g_enabled{false};
std::atomic<uint32_t> g_mask{0xffffffffu};  // kinds that are traced while enabled
std::atomic<int64_t> g_launches{0};
double g_ms[GPTQ_K_COUNT] = {};
int64_t g_count[GPTQ_K_COUNT] = {};
thread_local std::vector<Pending> t_pending;
thread_local std::vector<cudaEvent_t> t_pool;

cudaEvent_t pool_get() {
  if (!t_pool.empty()) {
    cudaEvent_t e = t_pool.back();
    t_pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  cuda_check(cudaEventCreate(&e), "cudaEventCreate");
  return e;
}

}  // namespace

static bool traced(int kind) {
  return g_enabled.load(std::memory_order_relaxed) && kind >= 0 && kind < 32 &&
         ((g_mask.load(std::memory_order_relaxed) >> kind) & 1u) != 0;
}

void trace_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!traced(kind)) return;
  Pending p{kind, pool_get(), nullptr};
  cuda_check(cudaEventRecord(p.start, s), "cudaEventRecord");
  t_pending.push_back(p);
}

void trace_end(int kind, cudaStream_t s) {
  if (!traced(kind) || t_pending.empty()) return;
  Pending& p = t_pending.back();
  if (p.stop != nullptr) return;
  p.stop = pool_get();
  cuda_check(cudaEventRecord(p.stop, s), "cudaEventRecord");
}

void trace_flush() {
  if (t_pending.empty()) return;
  std::vector<Pending> done;
  done.swap(t_pending);
  std::lock_guard<std::mutex> lk(g_mu);
  for (const Pending& p : done) {
    float ms = 0.f;
    if (p.stop != nullptr && cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess &&
        p.kind >= 0 && p.kind < GPTQ_K_COUNT) {
      g_ms[p.kind] += ms;
      g_count[p.kind] += 1;
    }
    t_pool.push_back(p.start);
    if (p.stop != nullptr) t_pool.push_back(p.stop);
  }
}

void trace_discard() {
  for (const Pending& p : t_pending) {
    t_pool.push_back(p.start);
    if (p.stop != nullptr) t_pool.push_back(p.stop);
  }
  t_pending.clear();
}

void profile_enable(bool on) { g_enabled.store(on); }
void profile_select(uint32_t mask) { g_mask.store(mask); }

void ensure_dynamic_smem(const void* func, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> limit;  // (device, kernel) -> bytes
  int dev = 0;
  GPTQ_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  int& cur = limit[{dev, func}];
  if (bytes > cur) {
    GPTQ_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    cur = bytes;
  }
}
void profile_reset() {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int k = 0; k < GPTQ_K_COUNT; ++k) {
    g_ms[k] = 0.0;
    g_count[k] = 0;
  }
}
bool profile_read(int kind, double* ms, int64_t* n) {
  if (kind < 0 || kind >= GPTQ_K_COUNT) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (ms) *ms = g_ms[kind];
  if (n) *n = g_count[kind];
  return true;
}
int64_t launch_count() { return g_launches.load(); }

// ------------------------------------------------------------------ device facts

namespace {
std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};
}

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
void set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kWaitLimitNs : ns, std::memory_order_relaxed);
}

int sm_count() {
  int dev = 0;
  cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  thread_local int cached_dev = -1, cached = 0;  // per host thread: no shared state
  if (dev != cached_dev) {
    cuda_check(cudaDeviceGetAttribute(&cached, cudaDevAttrMultiProcessorCount, dev),
               "cudaDeviceGetAttribute");
    cached_dev = dev;
  }
  return cached;
}

AuxStreams& aux_streams(int nevents) {
  static std::map<int, AuxStreams> per_dev;
  int dev = 0;
  cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  AuxStreams& a = per_dev[dev];
  if (a.a == nullptr) {
    int least = 0, greatest = 0;
    cuda_check(cudaDeviceGetStreamPriorityRange(&least, &greatest),
               "cudaDeviceGetStreamPriorityRange");
    cuda_check(cudaStreamCreateWithPriority(&a.a, cudaStreamNonBlocking, greatest),
               "cudaStreamCreateWithPriority");
    cuda_check(cudaStreamCreateWithPriority(&a.b, cudaStreamNonBlocking, least),
               "cudaStreamCreateWithPriority");
    cuda_check(cudaStreamCreateWithPriority(&a.c, cudaStreamNonBlocking, (least + greatest) / 2),
               "cudaStreamCreateWithPriority");
    cuda_check(cudaStreamCreateWithFlags(&a.copy, cudaStreamNonBlocking), "cudaStreamCreateWithFlags");
  }
  while (static_cast<int>(a.ev.size()) < nevents) {
    cudaEvent_t e;
    cuda_check(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreateWithFlags");
    a.ev.push_back(e);
  }
  return a;
}

cudaStream_t copy_stream() { return aux_streams(0).copy; }

std::mutex& aux_mutex() {
  static std::mutex m;
  return m;
}

void make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                  uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  // looked up once (a function-local static's initialisation is thread-safe)
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cuda_check(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                cudaEnableDefault, &q),
               "cudaGetDriverEntryPointByVersion");
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) {
      fail(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) fail(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
}

}  // namespace gptq
