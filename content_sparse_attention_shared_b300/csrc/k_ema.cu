// Online spherical k-means step on the shared centroids.
//
// "Efficient Content-Based Sparse Attention with Routing Transformers":
// the routing centroids are learned online with mini-batch spherical k-means
// (§2 "Attention with Content-Based Sparsity"), shared across sequences
// (§4).  The update rule itself is left open by the pages; this library reads
// it as: for every head and centroid c with N > 0 assigned rows (argmax
// assignment, all sequences of the batch),
//     mu_c <- normalise(decay * mu_c + (1 - decay) * mean of the assigned r_t),
// and leaves a centroid without rows untouched.
//
// No floating-point atomics and one kernel: each (centroid, head) CTA scans
// the head's assignments itself (coalesced 16-byte loads, 8192 rows per pass),
// lists its rows in a fixed order with one block-wide scan, re-normalises
// each row on the fly, sums them in that order, blends and renormalises.  The
// result is deterministic.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS2 = 256;
constexpr int WARPS2 = THREADS2 / 32;
constexpr int SCAN_PER_THREAD = 32;                    // assignments per thread per pass
constexpr int SCAN_ROWS = THREADS2 * SCAN_PER_THREAD;  // rows per pass
constexpr int LIST = 1024;                             // rows listed per summation round
constexpr int STAGE_BYTES = 24 * 1024;                 // rows staged in shared memory per round

// 8 consecutive features of a row, kept in their storage format and read as
// fp32 on use.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    u = __ldcg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ void load_shared(const uint8_t* p) {
    u = *reinterpret_cast<const uint4*>(p);
  }
  __device__ __forceinline__ void zero() { u = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float at(int j) const {
    const uint32_t w = j < 2 ? u.x : j < 4 ? u.y : j < 6 ? u.z : u.w;
    return (j & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldcg(reinterpret_cast<const float4*>(p));
    b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void load_shared(const uint8_t* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 16);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float at(int j) const {
    const float4& q = j < 4 ? a : b;
    const int e = j & 3;
    return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
  }
};

// Sum over the CH consecutive lanes that hold one row (CH a power of two).
template <int CH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = CH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (unsigned)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

// Adds the normalised rows rowlist[0 .. nl) of head h into acc (this
// thread's 8 features).  Round by round, the rows are first copied into the
// shared stage with 16-byte cp.async copies (every row of the round in flight
// at once), then CH threads share each staged row: its mean and centred norm
// come from shuffles inside the group, and the thread adds its 8 normalised
// features into registers.  The trip counts are uniform: the shuffles involve
// every lane of the warp.  Ends with a block barrier (the stage is free).
template <typename T, int D>
__device__ __forceinline__ void add_rows(const T* __restrict__ qk, int H, int n, int h,
                                         const int* rowlist, int nl, float (&acc)[8],
                                         uint8_t* stage) {
  constexpr int CH = D / 8;
  constexpr int RS = THREADS2 / CH;
  constexpr int RB = D * (int)sizeof(T);  // bytes per row
  constexpr int CPR = RB / 16;            // 16-byte chunks per row
  constexpr int SR = STAGE_BYTES / RB;    // rows per round
  const int tid = threadIdx.x;
  const int ch = tid % CH, rs = tid / CH;
  for (int r0 = 0; r0 < nl; r0 += SR) {
    const int nr = min(SR, nl - r0);
    for (int i = tid; i < nr * CPR; i += THREADS2) {
      const int r = i / CPR, cc = i - r * CPR;
      const int g = rowlist[r0 + r];
      const int b = g / n, t = g - b * n;
      cp_async16(stage + r * RB + cc * 16,
                 reinterpret_cast<const uint8_t*>(qk + (((size_t)b * H + h) * n + t) * D) +
                     cc * 16);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    for (int base = 0; base < nr; base += RS) {
      const int i = base + rs;
      Raw8<T> x;
      if (i < nr) x.load_shared(stage + i * RB + ch * 8 * (int)sizeof(T));
      else x.zero();
      float sx = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) sx += x.at(j);
      const float mean = group_sum<CH>(sx) / (float)D;
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float a = x.at(j) - mean;
        ss = fmaf(a, a, ss);
      }
      ss = group_sum<CH>(ss);
      const float inv = (i < nr && ss > 0.0f) ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(x.at(j) - mean, inv, acc[j]);
    }
    __syncthreads();  // the stage may be refilled
  }
}

// Sums the row slots' partial sums in a fixed order, blends the mean into
// the centroid (`old` = its previous value, loaded by threads < D) and
// renormalises it.  Every thread of the block calls it.
template <int D>
__device__ __forceinline__ void finish_centroid(const float (&acc)[8], int N, float old,
                                                float decay, float* __restrict__ mu_c,
                                                float (*red)[D] /* [RS][D], shared */) {
  constexpr int CH = D / 8;
  constexpr int RS = THREADS2 / CH;
  __shared__ float nrm_part[WARPS2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = tid % CH, rs = tid / CH;
#pragma unroll
  for (int j = 0; j < 8; ++j) red[rs][ch * 8 + j] = acc[j];
  __syncthreads();
  float vj = 0.0f;
  if (tid < D) {
    float sum = 0.0f;
    for (int r = 0; r < RS; ++r) sum += red[r][tid];
    const float mean_j = sum / (float)N;
    vj = decay * old + (1.0f - decay) * mean_j;
  }
  float sq = warp_sum(vj * vj);
  if (lane == 0) nrm_part[warp] = sq;
  __syncthreads();
  if (tid < D) {
    float tot = 0.0f;
    for (int wv = 0; wv < WARPS2; ++wv) tot += nrm_part[wv];
    mu_c[tid] = tot > 0.0f ? vj / sqrtf(tot) : vj;
  }
}

// One CTA per (centroid, head).  Pass by pass over each sequence's n
// positions, thread i examines positions base + 1024 j + 4 i + e (j < 8,
// e < 4; one coalesced 16-byte load per j), keeps a 32-bit mask of the rows
// assigned to this centroid, and a block-wide exclusive scan of the mask
// counts places them in a shared list in (thread, j, e) order.  The listed
// rows are then staged in shared memory and summed (add_rows); the row slots'
// partial sums are combined in a fixed order at the end, so the result is
// deterministic.
template <typename T, int D>
__global__ void __launch_bounds__(THREADS2, 7)
ema_update_kernel(const T* __restrict__ qk, const int32_t* __restrict__ assign, int B, int H,
                  int n, int k, float* __restrict__ mu, float decay) {
  pdl_trigger();
  __shared__ int rowlist[LIST];
  __shared__ int wsum[WARPS2];
  __shared__ __align__(16) uint8_t stage[STAGE_BYTES];  // staged rows, then the partial sums
  static_assert(STAGE_BYTES >= THREADS2 / (D / 8) * D * 4, "the stage holds the partial sums");
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(assign) & 15u) == 0;
  pdl_wait();
  const float old = (tid < D) ? __ldcg(mu + ((size_t)h * k + c) * D + tid) : 0.0f;

  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  int N = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t* arow = assign + ((size_t)b * H + h) * n;
    for (int t0 = 0; t0 < n; t0 += SCAN_ROWS) {
      // this thread's rows of the pass: bit 4 j + e <-> position t0 + 1024 j + 4 tid + e
      uint32_t mask = 0u;
#pragma unroll 4
      for (int j = 0; j < SCAN_PER_THREAD / 4; ++j) {
        const int t = t0 + j * (4 * THREADS2) + 4 * tid;
        if (vec && t + 3 < n) {
          const int4 a4 = __ldcg(reinterpret_cast<const int4*>(arow + t));
          mask |= (uint32_t)(a4.x == c) << (4 * j + 0);
          mask |= (uint32_t)(a4.y == c) << (4 * j + 1);
          mask |= (uint32_t)(a4.z == c) << (4 * j + 2);
          mask |= (uint32_t)(a4.w == c) << (4 * j + 3);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (t + e < n) mask |= (uint32_t)(__ldcg(arow + t + e) == c) << (4 * j + e);
        }
      }
      int total;
      const int ex = block_exclusive_scan<THREADS2>(__popc(mask), wsum, total);
      // (out-of-range assignments never equal c, so they are never listed)
      for (int sub = 0; sub < total; sub += LIST) {
        int r = ex;
        for (uint32_t mm = mask; mm != 0u; mm &= mm - 1u, ++r) {
          const int bit = __ffs(mm) - 1;
          if (r >= sub && r < sub + LIST)
            rowlist[r - sub] = b * n + t0 + (bit >> 2) * (4 * THREADS2) + 4 * tid + (bit & 3);
        }
        __syncthreads();
        add_rows<T, D>(qk, H, n, h, rowlist, min(LIST, total - sub), acc, stage);
      }
      N += total;
    }
  }
  if (N == 0) return;  // no assigned row: centroid unchanged (uniform)
  finish_centroid<D>(acc, N, old, decay, mu + ((size_t)h * k + c) * D,
                     reinterpret_cast<float (*)[D]>(stage));
}

// The variant driven by the top-w membership.  One CTA per (centroid, head)
// lists the positions of its own lists idx[b, h, c, :] for every sequence b
// (four consecutive entries per thread, one block scan keeps the list order,
// entries outside [0, n) are skipped), then stages and sums the rows exactly
// as above and blends with N = the number of listed rows.
template <typename T, int D>
__global__ void __launch_bounds__(THREADS2, 7)
ema_topw_kernel(const T* __restrict__ qk, const int32_t* __restrict__ idx, int B, int H, int n,
                int k, int w, float* __restrict__ mu, float decay) {
  pdl_trigger();
  __shared__ int rowlist[LIST];
  __shared__ int wsum[WARPS2];
  __shared__ __align__(16) uint8_t stage[STAGE_BYTES];  // staged rows, then the partial sums
  static_assert(LIST == 4 * THREADS2, "four list entries per thread");
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  pdl_wait();
  const float old = (tid < D) ? __ldcg(mu + ((size_t)h * k + c) * D + tid) : 0.0f;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  int N = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t* list = idx + (((size_t)b * H + h) * k + c) * w;
    for (int i0 = 0; i0 < w; i0 += LIST) {
      const int here = min(LIST, w - i0);
      int ent[4];
      uint32_t vm = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * tid + e;
        ent[e] = i < here ? __ldcg(list + i0 + i) : -1;
        vm |= (ent[e] >= 0 && ent[e] < n ? 1u : 0u) << e;
      }
      int total;
      int o = block_exclusive_scan<THREADS2>(__popc(vm), wsum, total);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((vm >> e) & 1u) rowlist[o++] = b * n + ent[e];
      __syncthreads();
      add_rows<T, D>(qk, H, n, h, rowlist, total, acc, stage);
      N += total;
    }
  }
  if (N == 0) return;  // no valid entry: centroid unchanged (uniform)
  finish_centroid<D>(acc, N, old, decay, mu + ((size_t)h * k + c) * D,
                     reinterpret_cast<float (*)[D]>(stage));
}

template <typename T, int D>
cudaError_t launch_topw(const void* qk, const int32_t* idx, int B, int H, int n, int k, int w,
                        float* mu, float decay, cudaStream_t s) {
  auto kern = ema_topw_kernel<T, D>;
  launch_begin(K_EMA_TOPW, s);
  cudaError_t e = launch_pdl(kern, dim3(k, H), dim3(THREADS2), 0, s, static_cast<const T*>(qk),
                             idx, B, H, n, k, w, mu, decay);
  launch_end(K_EMA_TOPW, s);
  return e;
}

template <typename T, int D>
cudaError_t launch_update(const void* qk, const int32_t* assign, int B, int H, int n, int k,
                          float* mu, float decay, cudaStream_t s) {
  auto kern = ema_update_kernel<T, D>;
  launch_begin(K_EMA_UPDATE, s);
  cudaError_t e = launch_pdl(kern, dim3(k, H), dim3(THREADS2), 0, s, static_cast<const T*>(qk),
                             assign, B, H, n, k, mu, decay);
  launch_end(K_EMA_UPDATE, s);
  return e;
}

}  // namespace

size_t ema_workspace_bytes(int, int, int, int) { return 0; }

cudaError_t launch_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                       const int32_t* assign, float* mu, int k, float decay,
                       void* /*ws*/, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_update<float, 64>(qk, assign, B, H, n, k, mu, decay, s)
                   : launch_update<float, 128>(qk, assign, B, H, n, k, mu, decay, s);
  }
  return d == 64 ? launch_update<__nv_bfloat16, 64>(qk, assign, B, H, n, k, mu, decay, s)
                 : launch_update<__nv_bfloat16, 128>(qk, assign, B, H, n, k, mu, decay, s);
}

cudaError_t launch_ema_topw(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                            const int32_t* idx, int w, float* mu, int k, float decay,
                            cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_topw<float, 64>(qk, idx, B, H, n, k, w, mu, decay, s)
                   : launch_topw<float, 128>(qk, idx, B, H, n, k, w, mu, decay, s);
  }
  return d == 64 ? launch_topw<__nv_bfloat16, 64>(qk, idx, B, H, n, k, w, mu, decay, s)
                 : launch_topw<__nv_bfloat16, 128>(qk, idx, B, H, n, k, w, mu, decay, s);
}

}  // namespace rt
