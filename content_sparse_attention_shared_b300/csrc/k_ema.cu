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
// kernel 2 gives each (head, centroid) one CTA that walks its buckets tile by
// tile, re-normalises each row on the fly, sums in a fixed order (warp
// round-robin, then warps in order), blends and renormalises.  The result is
// deterministic.
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
  extern __shared__ int32_t sm[];
  int32_t* warp_cnt = sm;                 // [WARPS1][k]
  int32_t* tot = sm + WARPS1 * k;         // [k]
  int32_t* start = tot + k;               // [k]
  const int tile = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (WARPS1 + 2) * k; i += TE) sm[i] = 0;
  __syncthreads();

  const long long g = (long long)tile * TE + tid;
  const long long rows = (long long)B * n;
  int a = -1;
  if (g < rows) {
    const int b = (int)(g / n), t = (int)(g % n);
    a = assign[((size_t)b * H + h) * n + t];
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
  if (tid == 0) {
    int run = 0;
    for (int c = 0; c < k; ++c) {
      start[c] = run;
      run += tot[c];
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

template <typename T, int D>
__global__ void __launch_bounds__(THREADS2)
ema_update_kernel(const T* __restrict__ qk, int B, int H, int n, int k, int Tn,
                  const int32_t* __restrict__ counts, const int32_t* __restrict__ starts,
                  const int32_t* __restrict__ perm, float* __restrict__ mu, float decay) {
  extern __shared__ int32_t offs[];  // [Tn + 1]
  __shared__ int part[THREADS2];
  __shared__ float red[WARPS2][D];
  __shared__ float nrm_part[WARPS2];
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t* cnt = counts + ((size_t)h * k + c) * Tn;
  const int32_t* st = starts + ((size_t)h * k + c) * Tn;

  // exclusive prefix of the per-tile counts: contiguous chunk per thread
  const int per = (Tn + THREADS2 - 1) / THREADS2;
  const int lo = tid * per, hi = min(Tn, lo + per);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += cnt[i];
  part[tid] = local;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < THREADS2; ++i) {
      const int x = part[i];
      part[i] = run;
      run += x;
    }
    offs[Tn] = run;
  }
  __syncthreads();
  {
    int run = part[tid];
    for (int i = lo; i < hi; ++i) {
      offs[i] = run;
      run += cnt[i];
    }
  }
  __syncthreads();
  const int N = offs[Tn];
  if (N == 0) return;  // no assigned row: centroid unchanged

  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.0f;
  for (int f = warp; f < N; f += WARPS2) {
    // tile holding flattened entry f: last tl with offs[tl] <= f
    int a0 = 0, a1 = Tn - 1;
    while (a0 < a1) {
      const int mid = (a0 + a1 + 1) >> 1;
      if (offs[mid] <= f) a0 = mid; else a1 = mid - 1;
    }
    const int tl = a0;
    const int p = st[tl] + (f - offs[tl]);
    const int g = perm[(size_t)h * Tn * TE + (size_t)tl * TE + p];
    if (g < 0 || (long long)g >= (long long)B * n) continue;  // defensive
    const int b = g / n, t = g % n;
    const T* row = qk + (((size_t)b * H + h) * n + t) * D;
    float x[D / 32];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) { x[i] = to_f32(row[lane + 32 * i]); s += x[i]; }
    const float mean = warp_sum(s) / (float)D;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) { x[i] -= mean; ss = fmaf(x[i], x[i], ss); }
    ss = warp_sum(ss);
    const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] += x[i] * inv;
  }
#pragma unroll
  for (int i = 0; i < D / 32; ++i) red[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  float vj = 0.0f;
  if (tid < D) {
    float sum = 0.0f;
    for (int wv = 0; wv < WARPS2; ++wv) sum += red[wv][tid];
    const float mean_j = sum / (float)N;
    const float old = mu[((size_t)h * k + c) * D + tid];
    vj = decay * old + (1.0f - decay) * mean_j;
  }
  float sq = warp_sum(vj * vj);
  if (lane == 0) nrm_part[warp] = sq;
  __syncthreads();
  if (tid < D) {
    float tot = 0.0f;
    for (int wv = 0; wv < WARPS2; ++wv) tot += nrm_part[wv];
    const float out = tot > 0.0f ? vj / sqrtf(tot) : vj;
    mu[((size_t)h * k + c) * D + tid] = out;
  }
}

template <typename T, int D>
cudaError_t launch_update(const void* qk, int B, int H, int n, int k, const EmaLayout& L,
                          float* mu, float decay, cudaStream_t s) {
  const size_t smem = (size_t)(L.T + 1) * sizeof(int32_t);
  auto kern = ema_update_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(smem < 48 * 1024 ? 48 * 1024 : smem));
  if (e != cudaSuccess) return e;
  launch_begin(K_EMA_UPDATE, s);
  kern<<<dim3(k, H), THREADS2, smem, s>>>(static_cast<const T*>(qk), B, H, n, k, L.T, L.counts,
                                           L.starts, L.perm, mu, decay);
  e = cudaGetLastError();
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
  cudaError_t e = cudaFuncSetAttribute(ema_bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(smem1 < 48 * 1024 ? 48 * 1024 : smem1));
  if (e != cudaSuccess) return e;
  launch_begin(K_EMA_BUCKET, s);
  ema_bucket_kernel<<<dim3(L.T, H), TE, smem1, s>>>(assign, B, H, n, k, L.T, L.counts, L.starts,
                                                     L.perm);
  e = cudaGetLastError();
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
