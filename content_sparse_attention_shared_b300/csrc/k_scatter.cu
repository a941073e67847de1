// Scatter-average of the per-cluster outputs back to positions.
//
// The combination of a position's outputs is left open by the pages
// ("Efficient Content-Based Sparse Attention with Routing Transformers", §4
// only restricts attention to same-cluster pairs); this library takes the
// arithmetic mean over the clusters that chose the position, and a zero row
// for a position no cluster chose.
//
// Positions chosen by exactly one cluster were written by the attention
// epilogue already.  A warp takes 32 consecutive positions, reads their
// membership counts with one coalesced load, and then serves the positions
// that need work one after the other: a zero row, or the mean of the slot
// rows.  The slots of a position come from the (cluster, slot) list the
// select kernel recorded (up to SLOTS_PER_ROW entries), put in ascending
// order; a position in more clusters than that finds its slots by binary
// search in every cluster's ascending member list.  Either way the rows are
// summed in ascending cluster order, so the result is deterministic.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS = 256;

template <typename T, int PER>
__device__ __forceinline__ void store_row(T* dst, const float (&v)[PER]) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (PER == 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(dst) = u;
    } else {
      *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(v[0], v[1]);
    }
  } else {
    if constexpr (PER == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
    }
  }
}

template <int PER>
__device__ __forceinline__ void add_row(float (&acc)[PER], const float* src) {
  if constexpr (PER == 4) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
  } else {
    const float2 x = *reinterpret_cast<const float2*>(src);
    acc[0] += x.x; acc[1] += x.y;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(THREADS)
scatter_kernel(long long BHn, int n, int k, int w, const int32_t* __restrict__ idx,
               const int32_t* __restrict__ mcount, const int32_t* __restrict__ slots,
               const float* __restrict__ yslot, T* __restrict__ out) {
  constexpr int PER = D / 32;  // contiguous features per lane
  const long long warp_global = ((long long)blockIdx.x * THREADS + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long g0 = warp_global * 32;
  if (g0 >= BHn) return;
  const long long g = g0 + lane;
  const int m = (g < BHn) ? mcount[g] : 1;
  unsigned todo = __ballot_sync(0xffffffffu, m != 1);
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const long long gt = g0 + src;  // row index bh * n + t
    const int mm = __shfl_sync(0xffffffffu, m, src);
    T* orow = out + gt * D + lane * PER;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.0f;
    if (mm == 0) {
      store_row<T, PER>(orow, acc);
      continue;
    }
    const long long bh = gt / n;
    const int t = (int)(gt - bh * n);
    const float* ybase = yslot + (size_t)bh * k * w * D;
    if (slots != nullptr && mm <= SLOTS_PER_ROW) {
      const int sid = lane < mm ? slots[gt * SLOTS_PER_ROW + lane] : 0x7fffffff;
      // rank of this lane's slot id among the first mm lanes (ids are distinct)
      int rank = 0;
#pragma unroll
      for (int j = 0; j < SLOTS_PER_ROW; ++j) {
        const int other = __shfl_sync(0xffffffffu, sid, j);
        if (j < mm && other < sid) ++rank;
      }
      for (int r = 0; r < mm; ++r) {
        const unsigned who = __ballot_sync(0xffffffffu, lane < mm && rank == r);
        const int sl = __shfl_sync(0xffffffffu, sid, __ffs(who) - 1);
        add_row<PER>(acc, ybase + (size_t)sl * D + lane * PER);
      }
    } else {
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
          const int fl = __ffs(found) - 1;
          found &= found - 1;
          const int s = __shfl_sync(0xffffffffu, slot, fl);
          add_row<PER>(acc, ybase + ((size_t)(c0 + fl) * w + s) * D + lane * PER);
        }
      }
    }
    const float fm = (float)mm;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = acc[i] / fm;
    store_row<T, PER>(orow, acc);
  }
}

template <typename T, int D>
cudaError_t launch_t(int BH, int n, int k, int w, const int32_t* idx, const int32_t* mcount,
                     const int32_t* slots, const float* yslot, void* out, cudaStream_t s) {
  const long long rows = (long long)BH * n;
  const long long warps = (rows + 31) / 32;
  const long long blocks = (warps * 32 + THREADS - 1) / THREADS;
  launch_begin(K_SCATTER, s);
  scatter_kernel<T, D><<<(unsigned)blocks, THREADS, 0, s>>>(rows, n, k, w, idx, mcount, slots,
                                                            yslot, static_cast<T*>(out));
  cudaError_t e = cudaGetLastError();
  launch_end(K_SCATTER, s);
  return e;
}

}  // namespace

cudaError_t launch_scatter(rt_dtype dt, int BH, int n, int d, int k, int w,
                           const int32_t* idx, const int32_t* mcount, const int32_t* slots,
                           const float* yslot, void* out, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_t<float, 64>(BH, n, k, w, idx, mcount, slots, yslot, out, s)
                   : launch_t<float, 128>(BH, n, k, w, idx, mcount, slots, yslot, out, s);
  }
  return d == 64 ? launch_t<__nv_bfloat16, 64>(BH, n, k, w, idx, mcount, slots, yslot, out, s)
                 : launch_t<__nv_bfloat16, 128>(BH, n, k, w, idx, mcount, slots, yslot, out, s);
}

}  // namespace rt
