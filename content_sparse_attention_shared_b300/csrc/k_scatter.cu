// Scatter-average of the per-cluster outputs back to positions.
//
// The combination of a position's outputs is left open by the pages
// ("Efficient Content-Based Sparse Attention with Routing Transformers", §4
// only restricts attention to same-cluster pairs); this library takes the
// arithmetic mean over the clusters that chose the position, and a zero row
// for a position no cluster chose.
//
// Positions chosen by exactly one cluster were written by the attention
// epilogue already.  One warp per remaining position: a zero row, or the
// clusters holding the position are found by binary search in each
// cluster's ascending member list (lanes split the clusters), and the slot
// rows are summed in ascending cluster order -- a fixed order, so the result
// is deterministic.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS = 256;

template <typename T, int D>
__global__ void __launch_bounds__(THREADS)
scatter_kernel(int BHn, int n, int k, int w, const int32_t* __restrict__ idx,
               const int32_t* __restrict__ mcount, const float* __restrict__ yslot,
               T* __restrict__ out) {
  const int warp_global = (blockIdx.x * THREADS + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= BHn) return;
  const int bh = warp_global / n;
  const int t = warp_global % n;
  const int m = mcount[warp_global];
  if (m == 1) return;
  T* orow = out + (size_t)warp_global * D;
  if (m == 0) {
#pragma unroll
    for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = from_f32<T>(0.0f);
    return;
  }
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.0f;
  const int32_t* base = idx + (size_t)bh * k * w;
  for (int c0 = 0; c0 < k; c0 += 32) {
    const int c = c0 + lane;
    int slot = -1;
    if (c < k) {
      const int32_t* list = base + (size_t)c * w;
      int lo = 0, hi = w - 1;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int v = list[mid];
        if (v == t) { slot = mid; break; }
        if (v < t) lo = mid + 1; else hi = mid - 1;
      }
    }
    unsigned found = __ballot_sync(0xffffffffu, slot >= 0);
    while (found) {
      const int src = __ffs(found) - 1;
      found &= found - 1;
      const int s = __shfl_sync(0xffffffffu, slot, src);
      const float* yrow = yslot + (((size_t)bh * k + c0 + src) * w + s) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[i] += yrow[lane + 32 * i];
    }
  }
  const float fm = (float)m;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = from_f32<T>(acc[i] / fm);
}

template <typename T, int D>
cudaError_t launch_t(int BH, int n, int k, int w, const int32_t* idx, const int32_t* mcount,
                     const float* yslot, void* out, cudaStream_t s) {
  const long long warps = (long long)BH * n;
  const int blocks = (int)((warps * 32 + THREADS - 1) / THREADS);
  launch_begin(K_SCATTER, s);
  scatter_kernel<T, D><<<blocks, THREADS, 0, s>>>((int)warps, n, k, w, idx, mcount, yslot,
                                                  static_cast<T*>(out));
  cudaError_t e = cudaGetLastError();
  launch_end(K_SCATTER, s);
  return e;
}

}  // namespace

cudaError_t launch_scatter(rt_dtype dt, int BH, int n, int d, int k, int w,
                           const int32_t* idx, const int32_t* mcount, const float* yslot,
                           void* out, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_t<float, 64>(BH, n, k, w, idx, mcount, yslot, out, s)
                   : launch_t<float, 128>(BH, n, k, w, idx, mcount, yslot, out, s);
  }
  return d == 64 ? launch_t<__nv_bfloat16, 64>(BH, n, k, w, idx, mcount, yslot, out, s)
                 : launch_t<__nv_bfloat16, 128>(BH, n, k, w, idx, mcount, yslot, out, s);
}

}  // namespace rt
