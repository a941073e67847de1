// Scatter-average of the per-cluster outputs back to positions.
//
// The combination of a position's outputs is left open by the pages
// ("Efficient Content-Based Sparse Attention with Routing Transformers", §4
// only restricts attention to same-cluster pairs); this library takes the
// arithmetic mean over the clusters that chose the position, and a zero row
// for a position no cluster chose.
//
// Positions chosen by exactly one cluster were written by the attention
// epilogue already.  One thread per (position, 8-feature chunk): it reads the
// position's membership count and, for a position in m = 0 clusters, writes
// zeros; for 2 <= m <= SLOTS_PER_ROW it reads the (cluster, slot) ids the
// select kernel recorded, sorts them (a fixed 8-input network), and sums its
// chunk of the m slot rows in ascending cluster order -- the m row loads are
// independent, so they are all in flight at once.  A position in more
// clusters than that (only with many near-identical centroids) is served by
// the whole warp: every lane binary-searches a different cluster's ascending
// member list, and the rows found are summed in ascending cluster order.
// Either way the result is deterministic.  With separate queries and keys a
// position's divisor is its count of visible memberships (`mdiv`; the rows of
// memberships without a visible key are zero), and 0 gives a zero row.
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

__device__ __forceinline__ void cswap(int& a, int& b) {
  const int lo = min(a, b), hi = max(a, b);
  a = lo;
  b = hi;
}

// ascending sort of 8 ints (Batcher odd-even merge network, 19 exchanges)
__device__ __forceinline__ void sort8(int (&v)[8]) {
  cswap(v[0], v[1]); cswap(v[2], v[3]); cswap(v[4], v[5]); cswap(v[6], v[7]);
  cswap(v[0], v[2]); cswap(v[1], v[3]); cswap(v[4], v[6]); cswap(v[5], v[7]);
  cswap(v[1], v[2]); cswap(v[5], v[6]);
  cswap(v[0], v[4]); cswap(v[1], v[5]); cswap(v[2], v[6]); cswap(v[3], v[7]);
  cswap(v[2], v[4]); cswap(v[3], v[5]);
  cswap(v[1], v[2]); cswap(v[3], v[4]); cswap(v[5], v[6]);
}
static_assert(SLOTS_PER_ROW == 8, "sort8 covers the recorded slot list");

template <typename T>
__device__ __forceinline__ void store8(T* dst, const float (&v)[8]) {
  if constexpr (sizeof(T) == 2) {
    uint4 u;
    __nv_bfloat162 p;
    p = __floats2bfloat162_rn(v[0], v[1]); u.x = *reinterpret_cast<uint32_t*>(&p);
    p = __floats2bfloat162_rn(v[2], v[3]); u.y = *reinterpret_cast<uint32_t*>(&p);
    p = __floats2bfloat162_rn(v[4], v[5]); u.z = *reinterpret_cast<uint32_t*>(&p);
    p = __floats2bfloat162_rn(v[6], v[7]); u.w = *reinterpret_cast<uint32_t*>(&p);
    *reinterpret_cast<uint4*>(dst) = u;
  } else {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// SUM = false: the forward's averaging scatter (single-membership rows were
// written by the attention kernel).  SUM = true: the backward's gather of
// per-slot gradient rows -- every position with m >= 1 gets the plain sum of
// its slot rows (fp32), m = 0 a zero row.
template <typename T, int D, bool SUM>
__global__ void __launch_bounds__(THREADS, 6)
scatter_kernel(long long BHn, int n, int k, int w, const int32_t* __restrict__ idx,
               const int32_t* __restrict__ mcount, const int32_t* __restrict__ mdiv,
               const int32_t* __restrict__ slots, const float* __restrict__ yslot,
               T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  constexpr int CH = D / 8;    // 8-feature chunks per row
  constexpr int PER = D / 32;  // contiguous features per lane on the warp-wide path
  const long long g = (long long)blockIdx.x * THREADS + threadIdx.x;
  const long long r = g / CH;  // row index bh * n + t
  const int ch = (int)(g - r * CH);
  const int lane = threadIdx.x & 31;
  const bool active = r < BHn;
  const int m = active ? __ldcg(mcount + r) : 1;
  // divisor of the mean (m itself unless the visible count is given)
  const int dv = (active && mdiv != nullptr && m >= 2) ? __ldcg(mdiv + r) : m;
  // the recorded slot ids are loaded together with the count (one round trip
  // instead of two); only rows with 2 <= m <= SLOTS_PER_ROW use them
  int4 sa = make_int4(0, 0, 0, 0), sb = sa;
  if (active) {
    const int4* sp = reinterpret_cast<const int4*>(slots + r * SLOTS_PER_ROW);
    sa = __ldcg(sp);
    sb = __ldcg(sp + 1);
  }

  // rare: positions in more than SLOTS_PER_ROW clusters, one warp pass each
  unsigned slow = __ballot_sync(0xffffffffu, active && ch == 0 && m > SLOTS_PER_ROW);
  while (slow) {
    const int src = __ffs(slow) - 1;
    slow &= slow - 1;
    const long long gt = __shfl_sync(0xffffffffu, r, src);
    const int mm = __shfl_sync(0xffffffffu, dv, src);
    const long long bh = gt / n;
    const int t = (int)(gt - bh * n);
    const float* ybase = yslot + (size_t)bh * k * w * D;
    const int32_t* base = idx + (size_t)bh * k * w;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.0f;
    for (int c0 = 0; c0 < k; c0 += 32) {
      const int c = c0 + lane;
      int slot = -1;
      if (c < k) {
        const int32_t* list = base + (size_t)c * w;
        int lo = 0, hi = w - 1;
        while (lo <= hi) {
          const int mid = (lo + hi) >> 1;
          const int v = __ldcg(list + mid);
          if (v == t) { slot = mid; break; }
          if (v < t) lo = mid + 1; else hi = mid - 1;
        }
      }
      unsigned found = __ballot_sync(0xffffffffu, slot >= 0);
      while (found) {
        const int fl = __ffs(found) - 1;
        found &= found - 1;
        const int sl = __shfl_sync(0xffffffffu, slot, fl);
        add_row<PER>(acc, ybase + ((size_t)(c0 + fl) * w + sl) * D + lane * PER);
      }
    }
    const float fm = (float)mm;
    float o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = SUM ? acc[i] : (mm > 0 ? acc[i] / fm : 0.0f);
    store_row<T, PER>(out + gt * D + lane * PER, o);
  }

  if (!active || (!SUM && m == 1) || m > SLOTS_PER_ROW) return;
  T* dst = out + r * D + ch * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if (m == 0) {
    store8<T>(dst, acc);
    return;
  }
  int ids[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
  const int kw = k * w;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i >= m || (unsigned)ids[i] >= (unsigned)kw) ids[i] = 0x7fffffff;  // (defensive)
  sort8(ids);
  const long long bh = r / n;
  const float* ybase = yslot + (size_t)bh * k * w * D + ch * 8;
  // slot rows summed in ascending cluster order, two rows in flight at a time
  // (four would not fit the 40 registers that six CTAs an SM leave, and
  // spilling them, or fewer CTAs, measured slower)
#pragma unroll
  for (int i0 = 0; i0 < 8; i0 += 2) {
    if (i0 >= m) break;
    float4 y[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (i0 + u < m && ids[i0 + u] != 0x7fffffff) {
        const float4* p = reinterpret_cast<const float4*>(ybase + (size_t)ids[i0 + u] * D);
        y[u][0] = __ldcg(p);
        y[u][1] = __ldcg(p + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (i0 + u < m && ids[i0 + u] != 0x7fffffff) {
        acc[0] += y[u][0].x; acc[1] += y[u][0].y; acc[2] += y[u][0].z; acc[3] += y[u][0].w;
        acc[4] += y[u][1].x; acc[5] += y[u][1].y; acc[6] += y[u][1].z; acc[7] += y[u][1].w;
      }
    }
  }
  const float fm = (float)dv;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = SUM ? acc[i] : (dv > 0 ? acc[i] / fm : 0.0f);
  store8<T>(dst, acc);
}

template <typename T, int D>
cudaError_t launch_t(int BH, int n, int k, int w, const int32_t* idx, const int32_t* mcount,
                     const int32_t* mdiv, const int32_t* slots, const float* yslot, void* out,
                     cudaStream_t s) {
  const long long rows = (long long)BH * n;
  const long long threads = rows * (D / 8);
  const long long blocks = (threads + THREADS - 1) / THREADS;
  launch_begin(K_SCATTER, s);
  cudaError_t e = launch_pdl(scatter_kernel<T, D, false>, dim3((unsigned)blocks), dim3(THREADS), 0, s,
                             rows, n, k, w, idx, mcount, mdiv, slots, yslot, static_cast<T*>(out));
  launch_end(K_SCATTER, s);
  return e;
}

template <int D>
cudaError_t launch_sum_t(int BH, int n, int k, int w, const int32_t* idx, const int32_t* mcount,
                         const int32_t* slots, const float* yslot, float* out, cudaStream_t s) {
  const long long rows = (long long)BH * n;
  const long long blocks = (rows * (D / 8) + THREADS - 1) / THREADS;
  launch_begin(K_SCATTER, s);
  cudaError_t e = launch_pdl(scatter_kernel<float, D, true>, dim3((unsigned)blocks), dim3(THREADS),
                             0, s, rows, n, k, w, idx, mcount,
                             static_cast<const int32_t*>(nullptr), slots, yslot, out);
  launch_end(K_SCATTER, s);
  return e;
}

}  // namespace

cudaError_t launch_gather_sum(int BH, int n, int d, int k, int w, const int32_t* idx,
                              const int32_t* mcount, const int32_t* slots, const float* yslot,
                              float* out, cudaStream_t s) {
  return d == 64 ? launch_sum_t<64>(BH, n, k, w, idx, mcount, slots, yslot, out, s)
                 : launch_sum_t<128>(BH, n, k, w, idx, mcount, slots, yslot, out, s);
}

cudaError_t launch_scatter(rt_dtype dt, int BH, int n, int d, int k, int w,
                           const int32_t* idx, const int32_t* mcount, const int32_t* mdiv,
                           const int32_t* slots, const float* yslot, void* out, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_t<float, 64>(BH, n, k, w, idx, mcount, mdiv, slots, yslot, out, s)
                   : launch_t<float, 128>(BH, n, k, w, idx, mcount, mdiv, slots, yslot, out, s);
  }
  return d == 64 ? launch_t<__nv_bfloat16, 64>(BH, n, k, w, idx, mcount, mdiv, slots, yslot, out, s)
                 : launch_t<__nv_bfloat16, 128>(BH, n, k, w, idx, mcount, mdiv, slots, yslot, out, s);
}

}  // namespace rt
