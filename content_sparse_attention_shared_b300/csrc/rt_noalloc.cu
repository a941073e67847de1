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
// fp32 elements (32 MiB), held on every GPU that loads the library until the
// process exits.
//
// The array is a file-scope __device__ symbol, so host code cannot use its
// name as a device address.  The first call on each device (with that device
// current) looks the address up with cudaGetSymbolAddress and caches it;
// make that first call before any stream capture.  All calls share the one
// array: the score kernel overwrites every element the select kernel reads,
// so nothing needs clearing between calls, but calls that overlap on the GPU
// (different streams, or different host threads) race on it.
#include <cstdio>
#include <mutex>

#include "rt_internal.cuh"

static __device__ __align__(256) float g_noalloc_scores[RT_NOALLOC_MAX_SCORES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
float* g_scores_addr[kMaxDevices] = {};

// Device address of the scratch array for the current device (set-up on the
// first call per device).
rt_status scratch_address(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return rt::record_error(RT_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return rt::record_error(RT_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scores_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scores);
    if (e != cudaSuccess || p == nullptr) {
      char msg[160];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress for the routing scratch failed: %s",
               cudaGetErrorString(e));
      return rt::record_error(RT_ERR_CUDA, msg);
    }
    g_scores_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scores_addr[dev];
  return RT_OK;
}

}  // namespace

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
  float* S = nullptr;
  st = scratch_address(&S);
  if (st != RT_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  cudaError_t e = rt::launch_score(qk, dt, B, H, n, d, centroids, k, S, assign, nullptr, nullptr, nullptr, s);
  if (e != cudaSuccess) return rt::record_error(RT_ERR_CUDA, cudaGetErrorString(e));
  e = rt::launch_select(S, BH, n, k, w, idx, nullptr, nullptr, s);
  if (e != cudaSuccess) return rt::record_error(RT_ERR_CUDA, cudaGetErrorString(e));
  return rt::record_error(RT_OK, "");
}
