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
// A segmented reduction with no floating-point atomics that reads every
// assignment and every row once: a bucketing kernel sorts every chunk's rows
// by centroid with integer counts, then one CTA per (centroid, head)
// concatenates its own rows chunk by chunk and sums them, normalised, in that
// order -- an order fixed by the assignments alone, so the result is
// deterministic.  The second kernel can stop before the blend and write each
// centroid's raw sum and count instead, so that shards of a batch can be
// combined with one all-reduce.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS2 = 256;
constexpr int WARPS2 = THREADS2 / 32;
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

// Blends the mean sum/N into the centroid (`old` = its previous value) and
// renormalises it; threads tid < D hold feature tid.  Every thread of the
// block calls it (it contains a barrier); N > 0.
template <int D>
__device__ __forceinline__ void blend_store(float sum, int N, float old, float decay,
                                            float* __restrict__ mu_c) {
  __shared__ float nrm_part[WARPS2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float vj = 0.0f;
  if (tid < D) vj = decay * old + (1.0f - decay) * (sum / (float)N);
  const float sq = warp_sum(vj * vj);
  if (lane == 0) nrm_part[warp] = sq;
  __syncthreads();
  if (tid < D) {
    float tot = 0.0f;
    for (int wv = 0; wv < WARPS2; ++wv) tot += nrm_part[wv];
    mu_c[tid] = tot > 0.0f ? vj / sqrtf(tot) : vj;
  }
}

// Sums the row slots' partial sums in a fixed order.  FINAL: blends the mean
// into the centroid (`old` = its previous value, loaded by threads < D; a
// centroid with N = 0 is left untouched).  Otherwise writes the raw sum and
// the count N (as a float) to part_c[0 .. D].  Every thread of the block calls
// it.
template <int D, bool FINAL>
__device__ __forceinline__ void finish_centroid(const float (&acc)[8], int N, float old,
                                                float decay, float* __restrict__ mu_c,
                                                float* __restrict__ part_c,
                                                float (*red)[D] /* [RS][D], shared */) {
  constexpr int CH = D / 8;
  constexpr int RS = THREADS2 / CH;
  const int tid = threadIdx.x;
  const int ch = tid % CH, rs = tid / CH;
#pragma unroll
  for (int j = 0; j < 8; ++j) red[rs][ch * 8 + j] = acc[j];
  __syncthreads();
  float sum = 0.0f;
  if (tid < D)
    for (int r = 0; r < RS; ++r) sum += red[r][tid];
  if (!FINAL) {
    if (tid < D) part_c[tid] = sum;
    if (tid == 0) part_c[D] = (float)N;
    return;
  }
  if (N == 0) return;  // uniform
  blend_store<D>(sum, N, old, decay, mu_c);
}

// ---------------------------------------------------------------------------
// Argmax-driven step as a segmented reduction in two kernels, with no
// floating-point atomics and no per-centroid re-scan of the assignments:
//
// ema_bucket_kernel: one CTA per (chunk of R = 1024*M consecutive positions of
//   one sequence, head).  It reads the chunk's assignments once and sorts the
//   chunk's rows by centroid, stably, with integer counts only: warp w owns a
//   stripe of 128*M consecutive positions, handled 32 at a time in position
//   order; __match_any_sync gives each row its rank among the earlier rows of
//   the stripe with the same centroid (per-warp counters in shared memory),
//   and one block-wide exclusive scan over the (centroid, warp) counts turns
//   ranks into places.  Writes, per chunk and centroid, (first place, count)
//   and, per place, the row id b*n + t (`perm`, the chunk's own range of the
//   head's B*n entries).  Rows with an assignment outside [0, k) are skipped.
// ema_segment_kernel: one CTA per (centroid, head) concatenates its rows
//   chunk by chunk in chunk order (a block scan over the chunks' counts), so
//   it reads B*n/R pairs and its own rows only; the rows are then staged,
//   normalised and summed in that fixed order (add_rows), the mean blended
//   into the centroid and renormalised (finish_centroid).
// The order of every sum is a function of the assignments alone, so the
// result is deterministic.
// ---------------------------------------------------------------------------
constexpr int BUCKET_THREADS = 256;
constexpr int BUCKET_WARPS = BUCKET_THREADS / 32;
constexpr int BUCKET_ROWS = 1024;  // positions per chunk for M = 1

template <int M>
__global__ void __launch_bounds__(BUCKET_THREADS)
ema_bucket_kernel(const int32_t* __restrict__ assign, int H, int n, int k, int cps,
                  int nchunks, int2* __restrict__ offcnt, int32_t* __restrict__ perm, int Bn) {
  pdl_trigger();
  constexpr int G = 4 * M;  // groups of 32 positions per warp stripe
  constexpr int R = BUCKET_ROWS * M;
  extern __shared__ int whist[];  // [BUCKET_WARPS][k]: counts, then places
  __shared__ int wsum[BUCKET_WARPS];
  const int j = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = j / cps;
  const int t0 = (j - b * cps) * R;
  for (int i = tid; i < BUCKET_WARPS * k; i += BUCKET_THREADS) whist[i] = 0;
  pdl_wait();
  const int32_t* arow = assign + ((size_t)b * H + h) * n;
  int a[G];
#pragma unroll
  for (int e = 0; e < G; ++e) {
    const int t = t0 + warp * (32 * G) + 32 * e + lane;
    int c = t < n ? __ldcg(arow + t) : -1;
    a[e] = (c >= 0 && c < k) ? c : -1;
  }
  __syncthreads();  // counters cleared
  // rank of each row among the earlier rows of this warp's stripe with the
  // same centroid (groups in position order, lanes in position order)
  int rank[G];
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int e = 0; e < G; ++e) {
    const int c = a[e];
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    rank[e] = c >= 0 ? whist[warp * k + c] + __popc(peers & lt) : 0;
    __syncwarp();
    if (c >= 0 && lane == __ffs(peers) - 1) whist[warp * k + c] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // exclusive scan of the counts in (centroid, warp) order: thread tid takes
  // the consecutive items [tid*P, tid*P + P) of item c*BUCKET_WARPS + w
  const int items = BUCKET_WARPS * k;
  const int P = (items + BUCKET_THREADS - 1) / BUCKET_THREADS;
  const int i0 = tid * P;
  int local = 0;
  for (int i = i0; i < i0 + P && i < items; ++i)
    local += whist[(i % BUCKET_WARPS) * k + i / BUCKET_WARPS];
  int total;
  int run = block_exclusive_scan<BUCKET_THREADS>(local, wsum, total);
  for (int i = i0; i < i0 + P && i < items; ++i) {
    int& x = whist[(i % BUCKET_WARPS) * k + i / BUCKET_WARPS];
    const int cnt = x;
    x = run;
    run += cnt;
  }
  __syncthreads();
  // (first place, count) of every centroid in this chunk
  int2* oc = offcnt + ((size_t)h * nchunks + j) * k;
  for (int c = tid; c < k; c += BUCKET_THREADS) {
    const int first = whist[c];
    const int next = c + 1 < k ? whist[c + 1] : total;
    oc[c] = make_int2(first, next - first);
  }
  int32_t* pp = perm + (size_t)h * Bn + (size_t)b * n + t0;
#pragma unroll
  for (int e = 0; e < G; ++e) {
    const int c = a[e];
    if (c >= 0) {
      const int t = t0 + warp * (32 * G) + 32 * e + lane;
      pp[whist[warp * k + c] + rank[e]] = b * n + t;
    }
  }
}

template <typename T, int D, bool FINAL>
__global__ void __launch_bounds__(THREADS2, 7)
ema_segment_kernel(const T* __restrict__ qk, const int2* __restrict__ offcnt,
                   const int32_t* __restrict__ perm, int H, int n, int k, int cps, int R,
                   int nchunks, int Bn, float* __restrict__ mu, float decay,
                   float* __restrict__ out) {
  pdl_trigger();
  __shared__ int rowlist[LIST];
  __shared__ int wsum[WARPS2];
  __shared__ __align__(16) uint8_t stage[STAGE_BYTES];  // staged rows, then the partial sums
  static_assert(STAGE_BYTES >= THREADS2 / (D / 8) * D * 4, "the stage holds the partial sums");
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  pdl_wait();
  const float old = (FINAL && tid < D) ? __ldcg(mu + ((size_t)h * k + c) * D + tid) : 0.0f;

  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  int N = 0;
  const int32_t* perm_h = perm + (size_t)h * Bn;
  __shared__ int ex_s[THREADS2];        // first list place of each chunk of the block
  __shared__ long long base_s[THREADS2];  // perm index of its first entry
  for (int j0 = 0; j0 < nchunks; j0 += THREADS2) {
    // chunk j0 + tid: its rows of centroid c, perm_h[base + first .. + cnt)
    const int j = j0 + tid;
    const int nthis = min(THREADS2, nchunks - j0);
    int2 fc = make_int2(0, 0);
    long long base = 0;
    if (j < nchunks) {
      fc = __ldcg(offcnt + ((size_t)h * nchunks + j) * k + c);
      const int b = j / cps;
      base = (long long)b * n + (long long)(j - b * cps) * R + fc.x;
    }
    int total;
    const int ex = block_exclusive_scan<THREADS2>(fc.y, wsum, total);
    ex_s[tid] = ex;
    base_s[tid] = base;
    __syncthreads();
    for (int sub = 0; sub < total; sub += LIST) {
      // one entry per thread: the chunk holding list place p is the last one
      // whose first place is <= p (ex_s is non-decreasing)
      const int nl = min(LIST, total - sub);
      for (int i = tid; i < nl; i += THREADS2) {
        const int p = sub + i;
        int lo = 0, hi = nthis - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (ex_s[mid] <= p) lo = mid; else hi = mid - 1;
        }
        rowlist[i] = __ldcg(perm_h + base_s[lo] + (p - ex_s[lo]));
      }
      __syncthreads();
      add_rows<T, D>(qk, H, n, h, rowlist, nl, acc, stage);
    }
    N += total;
    __syncthreads();  // ex_s / base_s may be rewritten
  }
  finish_centroid<D, FINAL>(acc, N, old, decay, mu + ((size_t)h * k + c) * D,
                            out + ((size_t)h * k + c) * (D + 1),
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
  finish_centroid<D, true>(acc, N, old, decay, mu + ((size_t)h * k + c) * D, nullptr,
                           reinterpret_cast<float (*)[D]>(stage));
}

// The step from combined sums: red [H][k][D+1] holds every centroid's sum of
// normalised rows and its count (as produced above, summed over shards).
template <int D>
__global__ void __launch_bounds__(THREADS2)
ema_apply_kernel(const float* __restrict__ red, int k, float* __restrict__ mu, float decay) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const float* r = red + ((size_t)h * k + c) * (D + 1);
  const float Nf = __ldcg(r + D);
  const float sum = tid < D ? __ldcg(r + tid) : 0.0f;
  const float old = tid < D ? __ldcg(mu + ((size_t)h * k + c) * D + tid) : 0.0f;
  const int N = (int)Nf;
  if (N <= 0) return;  // uniform
  blend_store<D>(sum, N, old, decay, mu + ((size_t)h * k + c) * D);
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

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// ---- plan of the bucket-and-segment path ----------------------------------
// rows per bucketing chunk: 1024 * M, with M the smallest of 1, 2, 4 whose
// chunk covers at least k positions (so the per-chunk counts never outgrow the
// row list)
inline int bucket_m(int k) { return k <= 1024 ? 1 : k <= 2048 ? 2 : 4; }

struct BucketPlan {
  int M, R, cps, nchunks;
  size_t perm_bytes, offcnt_bytes;
};

inline BucketPlan bucket_plan(int B, int H, int n, int k) {
  BucketPlan p;
  p.M = bucket_m(k);
  p.R = BUCKET_ROWS * p.M;
  p.cps = (n + p.R - 1) / p.R;
  p.nchunks = B * p.cps;
  p.perm_bytes = align256((size_t)H * B * n * sizeof(int32_t));
  p.offcnt_bytes = align256((size_t)H * p.nchunks * k * sizeof(int2));
  return p;
}

// FINAL: update mu in place.  Otherwise write every centroid's raw sum and
// count to out [H][k][D+1] and leave mu alone.
template <typename T, int D, bool FINAL>
cudaError_t launch_update(const void* qk, const int32_t* assign, int B, int H, int n, int k,
                          float* mu, float decay, float* out, void* ws, cudaStream_t s) {
  cudaError_t e;
  const BucketPlan p = bucket_plan(B, H, n, k);
  int32_t* perm = static_cast<int32_t*>(ws);
  int2* offcnt = reinterpret_cast<int2*>(static_cast<uint8_t*>(ws) + p.perm_bytes);
  const int Bn = B * n;
  const size_t smem = (size_t)BUCKET_WARPS * k * sizeof(int);
  auto bucket = p.M == 1 ? ema_bucket_kernel<1> : p.M == 2 ? ema_bucket_kernel<2> : ema_bucket_kernel<4>;
  e = set_smem_limit(reinterpret_cast<const void*>(bucket), (int)smem);
  if (e != cudaSuccess) return e;
  launch_begin(K_EMA_BUCKET, s);
  e = launch_pdl(bucket, dim3(p.nchunks, H), dim3(BUCKET_THREADS), smem, s, assign, H, n, k,
                 p.cps, p.nchunks, offcnt, perm, Bn);
  launch_end(K_EMA_BUCKET, s);
  if (e != cudaSuccess) return e;
  auto kern = ema_segment_kernel<T, D, FINAL>;
  launch_begin(K_EMA_UPDATE, s);
  e = launch_pdl(kern, dim3(k, H), dim3(THREADS2), 0, s, static_cast<const T*>(qk),
                 static_cast<const int2*>(offcnt), static_cast<const int32_t*>(perm), H, n, k,
                 p.cps, p.R, p.nchunks, Bn, mu, decay, out);
  launch_end(K_EMA_UPDATE, s);
  return e;
}

template <bool FINAL>
cudaError_t launch_update_any(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                              const int32_t* assign, float* mu, int k, float decay, float* out,
                              void* ws, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_update<float, 64, FINAL>(qk, assign, B, H, n, k, mu, decay, out, ws, s)
                   : launch_update<float, 128, FINAL>(qk, assign, B, H, n, k, mu, decay, out, ws, s);
  }
  return d == 64
             ? launch_update<__nv_bfloat16, 64, FINAL>(qk, assign, B, H, n, k, mu, decay, out, ws, s)
             : launch_update<__nv_bfloat16, 128, FINAL>(qk, assign, B, H, n, k, mu, decay, out, ws, s);
}

}  // namespace

size_t ema_workspace_bytes(int B, int H, int n, int /*d*/, int k, rt_dtype /*dt*/) {
  const BucketPlan p = bucket_plan(B, H, n, k);
  return p.perm_bytes + p.offcnt_bytes;
}

cudaError_t launch_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                       const int32_t* assign, float* mu, int k, float decay, void* ws,
                       cudaStream_t s) {
  return launch_update_any<true>(qk, dt, B, H, n, d, assign, mu, k, decay, nullptr, ws, s);
}

cudaError_t launch_ema_sums(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                            const int32_t* assign, int k, float* sums, void* ws,
                            cudaStream_t s) {
  return launch_update_any<false>(qk, dt, B, H, n, d, assign, nullptr, k, 0.0f, sums, ws, s);
}

cudaError_t launch_ema_apply(const float* sums, int H, int d, float* mu, int k, float decay,
                             cudaStream_t s) {
  launch_begin(K_EMA_UPDATE, s);
  cudaError_t e = d == 64 ? launch_pdl(ema_apply_kernel<64>, dim3(k, H), dim3(THREADS2), 0, s, sums, k, mu, decay)
                          : launch_pdl(ema_apply_kernel<128>, dim3(k, H), dim3(THREADS2), 0, s, sums, k, mu, decay);
  launch_end(K_EMA_UPDATE, s);
  return e;
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
