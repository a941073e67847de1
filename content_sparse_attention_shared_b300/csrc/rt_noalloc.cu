// rt_route_assign_noalloc: routing for callers that cannot allocate device
// memory.
//
// rt_route_assign needs a scratch buffer for the fp32 score matrix
// [B*H, k, n]; normally the caller allocates it as the workspace.  Some
// callers cannot call cudaMalloc (or any allocating routine) at the point
// where they route -- for example code that runs inside a host framework
// whose device allocator it does not own, or a program that fixes its device
// memory footprint at start-up.  This entry point uses a fixed array in
// device memory that belongs to the library instead: RT_NOALLOC_MAX_SCORES
// fp32 elements (32 MiB) per context that uses it, held until the process
// exits.  With lazy module loading (the CUDA default) the array is reserved
// when the first call in a context looks up its address, so that first call
// can fail with RT_ERR_CUDA when device memory is short; callers with a fixed
// memory budget should make it at start-up.
//
// The array is a file-scope __device__ symbol, so host code cannot use its
// name as a device address.  The first call in each context (with that
// context's device current) looks the address up with cudaGetSymbolAddress
// and caches it under the context's unique id; make that first call before
// any stream capture.  All calls share the one array: the score kernel
// overwrites every element the select kernel reads, so nothing needs clearing
// between calls, but calls that overlap on the GPU (different streams, or
// different host threads) race on it.
//
// A bounded wait that runs out inside the score kernel sets a status word
// that also lives in the library (one per context, zero at load);
// rt_check_device_status(NULL, 0, stream) reads and clears it.
#include <cstdio>
#include <mutex>

#include "noalloc_cache.h"
#include "rt_internal.cuh"

static __device__ __align__(256) float g_noalloc_scores[RT_NOALLOC_MAX_SCORES];
static __device__ __align__(16) unsigned int g_noalloc_status;

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_setup_mu;
rt::ContextAddressCache<64> g_cache;

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}

// Unique id of the current context, making the device's primary context
// current first if the calling thread has none.
rt_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id)
    return rt::record_error(RT_ERR_CUDA, "the driver lacks cuCtxGetCurrent/cuCtxGetId");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    // cudaSetDevice initialises the device's primary context and makes it
    // current (CUDA 12 and later)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
      return rt::record_error(RT_ERR_CUDA, "no current CUDA context");
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return rt::record_error(RT_ERR_CUDA, "no current CUDA context");
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) return rt::record_error(RT_ERR_CUDA, "cuCtxGetId failed");
  return RT_OK;
}

// Device addresses of the scratch array and the status word in the current
// context (looked up on the first call in each context).
rt_status scratch_addresses(rt::NoallocAddrs* out) {
  unsigned long long id = 0;
  rt_status st = current_context_id(&id);
  if (st != RT_OK) return st;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (const rt::NoallocAddrs* hit = g_cache.find(id)) {
    *out = *hit;
    return RT_OK;
  }
  rt::NoallocAddrs a;
  cudaError_t e = cudaGetSymbolAddress(&a.scores, g_noalloc_scores);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&a.status, g_noalloc_status);
  if (e != cudaSuccess || a.scores == nullptr || a.status == nullptr) {
    char msg[160];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress for the routing scratch failed: %s",
             cudaGetErrorString(e));
    return rt::record_error(RT_ERR_CUDA, msg);
  }
  g_cache.put(id, a);
  *out = a;
  return RT_OK;
}

}  // namespace

namespace rt {

// Reads and clears the no-alloc status word of the current context after
// synchronising `s`.  A context in which the entry point never ran has no
// status to report.
rt_status noalloc_check_status(cudaStream_t s) {
  unsigned long long id = 0;
  rt_status st = current_context_id(&id);
  if (st != RT_OK) return st;
  void* addr = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    const NoallocAddrs* hit = g_cache.find(id);
    if (hit == nullptr) return record_error(RT_OK, "");
    addr = hit->status;
  }
  unsigned int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, addr, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return record_error(RT_ERR_CUDA, cudaGetErrorString(e));
  if (word == DEV_OK) return record_error(RT_OK, "");
  e = cudaMemsetAsync(addr, 0, sizeof(word), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (word == DEV_TIMEOUT)
    return record_error(RT_ERR_TIMEOUT, "a device-side wait of rt_route_assign_noalloc ran out");
  return record_error(RT_ERR_CUDA, "rt_route_assign_noalloc device status word set");
}

}  // namespace rt

extern "C" rt_status rt_route_assign_noalloc(const void* qk, rt_dtype dt, int B, int H, int n,
                                             int d, const float* centroids, int k, int w,
                                             int32_t* idx, int32_t* assign, void* stream) {
  rt_status st = rt::validate_shape(dt, B, H, n, d, k, w);
  if (st != RT_OK) return st;
  if (!qk || !centroids || !idx) return rt::record_error(RT_ERR_INVALID_ARG, "null qk/centroids/idx");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(qk) | reinterpret_cast<uintptr_t>(centroids) |
                        reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(assign);
  if (mis & 15u) return rt::record_error(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const unsigned long long elems = (unsigned long long)B * H * k * n;
  if (elems > RT_NOALLOC_MAX_SCORES) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "B*H*k*n = %llu scores exceed the fixed scratch of %u (use rt_route_assign with a "
             "caller workspace)", elems, (unsigned)RT_NOALLOC_MAX_SCORES);
    return rt::record_error(RT_ERR_UNSUPPORTED, msg);
  }
  rt::NoallocAddrs addrs;
  st = scratch_addresses(&addrs);
  if (st != RT_OK) return st;
  float* S = static_cast<float*>(addrs.scores);
  unsigned int* err = static_cast<unsigned int*>(addrs.status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  cudaError_t e =
      rt::launch_score(qk, dt, B, H, n, d, centroids, k, S, assign, nullptr, nullptr, nullptr, err, s);
  if (e != cudaSuccess) return rt::record_error(RT_ERR_CUDA, cudaGetErrorString(e));
  e = rt::launch_select(S, nullptr, BH, n, k, w, idx, nullptr, nullptr, s);
  if (e != cudaSuccess) return rt::record_error(RT_ERR_CUDA, cudaGetErrorString(e));
  return rt::record_error(RT_OK, "");
}
