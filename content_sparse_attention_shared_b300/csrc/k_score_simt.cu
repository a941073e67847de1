// Normalise + score + argmax on CUDA cores (fp32 FMA).
//
// Routing step of "Efficient Content-Based Sparse Attention with Routing
// Transformers" (§4, "Routing attention with clustering"): every shared
// query/key row is put on the unit sphere (mean removed, divided by its
// norm) and compared with every centroid by inner product; the nearest
// centroid is the one with the largest score (ties to the lower index).
//
// One CTA scores a tile of 64 rows of one (batch, head) against all k
// centroids in chunks of 64.  The normalised tile and the centroid chunk are
// staged transposed in shared memory; each thread accumulates a 4x4 block of
// scores over the head dimension in a fixed order, so a score is the same
// fp32 value in every call.  Scores are written centroid-major [BH,k,n] so
// that a warp stores 16 consecutive positions per centroid, optionally with
// the group bins of the select kernel (the 8 positions of a group are 8 lanes
// of a warp, reduced by shuffles).
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int TOK = 64;      // rows per CTA
constexpr int CCH = 64;      // centroids per chunk
constexpr int THREADS = 256;
constexpr int PAD = TOK + 1;

template <typename T, int D>
__global__ void __launch_bounds__(THREADS)
score_simt_kernel(const T* __restrict__ qk, int H, int n, const float* __restrict__ mu,
                  int k, float* __restrict__ S, int32_t* __restrict__ assign,
                  int32_t* __restrict__ mcount, uint16_t* __restrict__ gbins, int gstride) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float smem[];
  float* rT = smem;             // [D][PAD]
  float* muT = smem + D * PAD;  // [D][PAD]
  __shared__ float best_v[16][TOK];
  __shared__ int best_c[16][TOK];

  const int bh = blockIdx.y;
  const int h = bh % H;
  const int t0 = blockIdx.x * TOK;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // --- normalise 64 rows: warp per row ---------------------------------
  for (int tl = warp; tl < TOK; tl += THREADS / 32) {
    const int t = t0 + tl;
    float x[D / 32];
    if (t < n) {
      const T* row = qk + ((size_t)bh * n + t) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) x[i] = to_f32(__ldcg(row + lane + 32 * i));
    } else {
#pragma unroll
      for (int i = 0; i < D / 32; ++i) x[i] = 0.0f;
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) s += x[i];
    const float mean = warp_sum(s) / (float)D;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      x[i] -= mean;
      ss = fmaf(x[i], x[i], ss);
    }
    ss = warp_sum(ss);
    const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) rT[(lane + 32 * i) * PAD + tl] = x[i] * inv;
    if (mcount != nullptr && t < n && lane == 0) mcount[(size_t)bh * n + t] = 0;
  }

  const int tx = tid & 15, ty = tid >> 4;
  float bv[4];
  int bc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) { bv[i] = -INFINITY; bc[i] = 0x7fffffff; }

  for (int c0 = 0; c0 < k; c0 += CCH) {
    __syncthreads();  // rT ready / previous chunk consumed
    for (int e = tid; e < CCH * D; e += THREADS) {
      const int cl = e / D, j = e % D;
      const int c = c0 + cl;
      muT[j * PAD + cl] = (c < k) ? __ldcg(mu + ((size_t)h * k + c) * D + j) : 0.0f;
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) acc[i][jj] = 0.0f;
#pragma unroll 8
    for (int j = 0; j < D; ++j) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = rT[j * PAD + tx + 16 * i];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) b[jj] = muT[j * PAD + ty + 16 * jj];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int c = c0 + ty + 16 * jj;
      if (c >= k) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = t0 + tx + 16 * i;
        if (t < n) {
          if (S != nullptr) S[((size_t)bh * k + c) * n + t] = acc[i][jj];
          if (acc[i][jj] > bv[i]) { bv[i] = acc[i][jj]; bc[i] = c; }
        }
      }
    }
    if (gbins != nullptr) {
      // group bins: the lanes tx = 8m .. 8m+7 of a half-warp hold one group of
      // 8 positions; its 16 (i, jj) columns are reduced in two rounds of 8
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float m[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = 2 * r + (q >> 2), jj = q & 3;
          m[q] = (t0 + tx + 16 * i < n) ? acc[i][jj] : -INFINITY;
        }
        const float gm = octet_column_max(m, lane);
        const int q = lane & 7, i = 2 * r + (q >> 2), jj = q & 3;
        const int c = c0 + ty + 16 * jj;
        const int g = (t0 + 16 * i) / GROUP_SIZE + (tx >> 3);
        if (c < k && g * GROUP_SIZE < n)
          gbins[((size_t)bh * k + c) * gstride + g] = (uint16_t)score_bin(gm);
      }
    }
  }

  if (assign != nullptr) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      best_v[ty][tx + 16 * i] = bv[i];
      best_c[ty][tx + 16 * i] = bc[i];
    }
    __syncthreads();
    if (tid < TOK) {
      const int t = t0 + tid;
      float v = best_v[0][tid];
      int c = best_c[0][tid];
      for (int y = 1; y < 16; ++y) {
        const float v2 = best_v[y][tid];
        const int c2 = best_c[y][tid];
        if (v2 > v || (v2 == v && c2 < c)) { v = v2; c = c2; }
      }
      if (t < n) assign[(size_t)bh * n + t] = c;
    }
  }
}

template <typename T, int D>
cudaError_t launch_t(const void* qk, int BH, int H, int n, const float* mu, int k, float* S,
                     int32_t* a, int32_t* mcount, uint16_t* gbins, cudaStream_t s) {
  const size_t smem = 2 * (size_t)D * PAD * sizeof(float);
  auto kern = score_simt_kernel<T, D>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((n + TOK - 1) / TOK, BH);
  launch_begin(K_SCORE_SIMT, s);
  e = launch_pdl(kern, grid, dim3(THREADS), smem, s, static_cast<const T*>(qk), H, n, mu, k, S, a,
                 mcount, S != nullptr ? gbins : nullptr, gbin_stride(n));
  launch_end(K_SCORE_SIMT, s);
  return e;
}

}  // namespace

cudaError_t launch_score_simt(const void* qk, rt_dtype dt, int BH, int H, int n, int d,
                              const float* mu, int k, float* S, int32_t* a,
                              int32_t* mcount, uint16_t* gbins, cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_t<float, 64>(qk, BH, H, n, mu, k, S, a, mcount, gbins, s)
                   : launch_t<float, 128>(qk, BH, H, n, mu, k, S, a, mcount, gbins, s);
  }
  return d == 64 ? launch_t<__nv_bfloat16, 64>(qk, BH, H, n, mu, k, S, a, mcount, gbins, s)
                 : launch_t<__nv_bfloat16, 128>(qk, BH, H, n, mu, k, S, a, mcount, gbins, s);
}

}  // namespace rt
