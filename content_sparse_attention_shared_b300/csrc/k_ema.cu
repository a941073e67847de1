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
// No floating-point atomics: kernel 1 counting-sorts the rows of every tile
// of 256 rows by centroid (a stable, position-ordered bucket per centroid),
// kernel 2 gives each (centroid, head) one CTA that lists its rows from the
// buckets, re-normalises each row on the fly, sums them in a fixed order,
// blends and renormalises.  The result is deterministic.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int TE = 256;  // rows per tile = threads of kernel 1
constexpr int WARPS1 = TE / 32;
constexpr int THREADS2 = 256;
constexpr int WARPS2 = THREADS2 / 32;

struct EmaLayout {
  int T;  // tiles per head
  int32_t* counts;  // [H][k][T]
  int32_t* starts;  // [H][k][T]
  int32_t* perm;    // [H][T*TE]
};

EmaLayout ema_layout(void* ws, int B, int H, int n, int k) {
  EmaLayout L;
  const long long rows = (long long)B * n;
  L.T = (int)((rows + TE - 1) / TE);
  char* p = static_cast<char*>(ws);
  L.counts = reinterpret_cast<int32_t*>(p);
  p += ((size_t)H * k * L.T * 4 + 255) / 256 * 256;
  L.starts = reinterpret_cast<int32_t*>(p);
  p += ((size_t)H * k * L.T * 4 + 255) / 256 * 256;
  L.perm = reinterpret_cast<int32_t*>(p);
  return L;
}

__global__ void __launch_bounds__(TE)
ema_bucket_kernel(const int32_t* __restrict__ assign, int B, int H, int n, int k, int T,
                  int32_t* __restrict__ counts, int32_t* __restrict__ starts,
                  int32_t* __restrict__ perm) {
  pdl_trigger();
  extern __shared__ int32_t sm[];
  int32_t* warp_cnt = sm;                 // [WARPS1][k]
  int32_t* tot = sm + WARPS1 * k;         // [k]
  int32_t* start = tot + k;               // [k]
  const int tile = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (WARPS1 + 2) * k; i += TE) sm[i] = 0;
  pdl_wait();
  __syncthreads();

  const long long g = (long long)tile * TE + tid;
  const long long rows = (long long)B * n;
  int a = -1;
  if (g < rows) {
    const int b = (int)(g / n), t = (int)(g % n);
    a = __ldcg(assign + ((size_t)b * H + h) * n + t);
    if (a < 0 || a >= k) a = -1;  // out-of-range assignment: ignored
  }
  const unsigned peers = __match_any_sync(0xffffffffu, a);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (a >= 0 && rank == 0) warp_cnt[warp * k + a] = __popc(peers);
  __syncthreads();
  // per centroid: exclusive prefix over warps (in place) and the tile total
  for (int c = tid; c < k; c += TE) {
    int run = 0;
    for (int wv = 0; wv < WARPS1; ++wv) {
      const int x = warp_cnt[wv * k + c];
      warp_cnt[wv * k + c] = run;
      run += x;
    }
    tot[c] = run;
  }
  __syncthreads();
  {
    // exclusive prefix of the tile totals over centroids (bucket starts)
    __shared__ int wsum[WARPS1];
    int carry = 0;
    for (int c0 = 0; c0 < k; c0 += TE) {
      const int c = c0 + tid;
      int total;
      const int ex = block_exclusive_scan<TE>(c < k ? tot[c] : 0, wsum, total);
      if (c < k) start[c] = carry + ex;
      carry += total;
    }
  }
  __syncthreads();
  for (int c = tid; c < k; c += TE) {
    counts[((size_t)h * k + c) * T + tile] = tot[c];
    starts[((size_t)h * k + c) * T + tile] = start[c];
  }
  if (a >= 0) {
    const int p = start[a] + warp_cnt[warp * k + a] + rank;
    perm[(size_t)h * T * TE + (size_t)tile * TE + p] = (int32_t)g;
  }
}

// 8 consecutive features of a row, kept in their storage format and read as
// fp32 on use.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    u = __ldcg(reinterpret_cast<const uint4*>(p));
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

// Adds the normalised rows rowlist[0 .. nl) of head h into acc (this
// thread's 8 features; CH threads share a row, RS rows in flight).  The trip
// count is uniform: the shuffles involve every lane of the warp.  Two rows in
// flight per thread, each kept as its raw 16 bytes (8 bf16 or 2 x 4 fp32) and
// converted when used, which keeps the register count low.
template <typename T, int D>
__device__ __forceinline__ void add_rows(const T* __restrict__ qk, int H, int n, int h,
                                         const int* rowlist, int nl, float (&acc)[8]) {
  constexpr int CH = D / 8;
  constexpr int RS = THREADS2 / CH;
  const int ch = threadIdx.x % CH, rs = threadIdx.x / CH;
  for (int base = 0; base < nl; base += 2 * RS) {
    Raw8<T> x[2];
    int gg[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = base + rs + u * RS;
      gg[u] = (i < nl) ? rowlist[i] : -1;
      if (gg[u] >= 0) {
        const int b = gg[u] / n, t = gg[u] - b * n;
        x[u].load(qk + (((size_t)b * H + h) * n + t) * D + ch * 8);
      } else {
        x[u].zero();
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float sx = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) sx += x[u].at(j);
      const float mean = group_sum<CH>(sx) / (float)D;
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float a = x[u].at(j) - mean;
        ss = fmaf(a, a, ss);
      }
      ss = group_sum<CH>(ss);
      const float inv = (gg[u] >= 0 && ss > 0.0f) ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(x[u].at(j) - mean, inv, acc[j]);
    }
  }
}

// Sums the row slots' partial sums in a fixed order, blends the mean into
// the centroid (`old` = its previous value, loaded by threads < D) and
// renormalises it.  Every thread of the block calls it.
template <int D>
__device__ __forceinline__ void finish_centroid(const float (&acc)[8], int N, float old,
                                                float decay, float* __restrict__ mu_c) {
  constexpr int CH = D / 8;
  constexpr int RS = THREADS2 / CH;
  __shared__ float red[RS][D];
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

// One CTA per (centroid, head).  The centroid's rows (bucket entries of every
// tile, in tile order, so in position order) are first listed in shared
// memory, one lookup per row by one thread; then CH threads share each row,
// every thread reading one 16-byte chunk of 8 features: the row's mean and
// centred norm come from shuffles inside the group and the thread adds its
// 8 normalised features into registers.  Row slots are summed in a fixed
// order at the end, so the result is deterministic.
template <typename T, int D>
__global__ void __launch_bounds__(THREADS2, 8)
ema_update_kernel(const T* __restrict__ qk, int B, int H, int n, int k, int Tn,
                  const int32_t* __restrict__ counts, const int32_t* __restrict__ starts,
                  const int32_t* __restrict__ perm, float* __restrict__ mu, float decay) {
  pdl_trigger();
  pdl_wait();
  constexpr int LIST = 1024;         // rows listed per round
  extern __shared__ int32_t offs[];  // [Tn + 1] offsets, then [Tn] bucket starts
  int32_t* sts = offs + Tn + 1;
  __shared__ int rowlist[LIST];
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  const int32_t* cnt = counts + ((size_t)h * k + c) * Tn;
  const int32_t* st = starts + ((size_t)h * k + c) * Tn;
  const long long rows_total = (long long)B * n;
  const float old = (tid < D) ? __ldcg(mu + ((size_t)h * k + c) * D + tid) : 0.0f;  // early

  // exclusive prefix of the per-tile counts over the tiles
  {
    __shared__ int wsum[WARPS2];
    int carry = 0;
    for (int i0 = 0; i0 < Tn; i0 += THREADS2) {
      const int i = i0 + tid;
      int total;
      const int ex = block_exclusive_scan<THREADS2>(i < Tn ? __ldcg(cnt + i) : 0, wsum, total);
      if (i < Tn) {
        offs[i] = carry + ex;
        sts[i] = __ldcg(st + i);
      }
      carry += total;
    }
    if (tid == 0) offs[Tn] = carry;
  }
  __syncthreads();
  const int N = offs[Tn];
  if (N == 0) return;  // no assigned row: centroid unchanged

  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

  for (int f0 = 0; f0 < N; f0 += LIST) {
    const int nl = min(LIST, N - f0);
    __syncthreads();  // the previous round's list is consumed
    for (int i = tid; i < nl; i += THREADS2) {
      const int f = f0 + i;
      // tile holding flattened entry f: last tl with offs[tl] <= f
      int a0 = 0, a1 = Tn - 1;
      while (a0 < a1) {
        const int mid = (a0 + a1 + 1) >> 1;
        if (offs[mid] <= f) a0 = mid; else a1 = mid - 1;
      }
      const int p = sts[a0] + (f - offs[a0]);
      int g = -1;
      if (p >= 0 && p < TE) g = __ldcg(perm + (size_t)h * Tn * TE + (size_t)a0 * TE + p);
      if (g < 0 || (long long)g >= rows_total) g = -1;  // defensive
      rowlist[i] = g;
    }
    __syncthreads();
    add_rows<T, D>(qk, H, n, h, rowlist, nl, acc);
  }
  finish_centroid<D>(acc, N, old, decay, mu + ((size_t)h * k + c) * D);
}

template <typename T, int D>
cudaError_t launch_update(const void* qk, int B, int H, int n, int k, const EmaLayout& L,
                          float* mu, float decay, cudaStream_t s) {
  const size_t smem = (size_t)(2 * L.T + 1) * sizeof(int32_t);
  auto kern = ema_update_kernel<T, D>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)(smem < 48 * 1024 ? 48 * 1024 : smem));
  if (e != cudaSuccess) return e;
  launch_begin(K_EMA_UPDATE, s);
  e = launch_pdl(kern, dim3(k, H), dim3(THREADS2), smem, s, static_cast<const T*>(qk), B, H, n, k,
                 L.T, (const int32_t*)L.counts, (const int32_t*)L.starts, (const int32_t*)L.perm,
                 mu, decay);
  launch_end(K_EMA_UPDATE, s);
  return e;
}

}  // namespace

size_t ema_workspace_bytes(int B, int H, int n, int k) {
  const long long rows = (long long)B * n;
  const long long T = (rows + TE - 1) / TE;
  size_t a = ((size_t)H * k * T * 4 + 255) / 256 * 256;
  size_t p = ((size_t)H * T * TE * 4 + 255) / 256 * 256;
  return 2 * a + p;
}

cudaError_t launch_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                       const int32_t* assign, float* mu, int k, float decay,
                       void* ws, cudaStream_t s) {
  EmaLayout L = ema_layout(ws, B, H, n, k);
  const size_t smem1 = (size_t)(WARPS1 + 2) * k * sizeof(int32_t);
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(ema_bucket_kernel), (int)(smem1 < 48 * 1024 ? 48 * 1024 : smem1));
  if (e != cudaSuccess) return e;
  launch_begin(K_EMA_BUCKET, s);
  e = launch_pdl(ema_bucket_kernel, dim3(L.T, H), dim3(TE), smem1, s, assign, B, H, n, k, L.T,
                 L.counts, L.starts, L.perm);
  launch_end(K_EMA_BUCKET, s);
  if (e != cudaSuccess) return e;
  if (dt == RT_F32) {
    return d == 64 ? launch_update<float, 64>(qk, B, H, n, k, L, mu, decay, s)
                   : launch_update<float, 128>(qk, B, H, n, k, L, mu, decay, s);
  }
  return d == 64 ? launch_update<__nv_bfloat16, 64>(qk, B, H, n, k, L, mu, decay, s)
                 : launch_update<__nv_bfloat16, 128>(qk, B, H, n, k, L, mu, decay, s);
}

}  // namespace rt
