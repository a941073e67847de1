// In-cluster softmax attention on CUDA cores (fp32).  Serves fp32 inputs and
// is the generic path for shapes the tensor-core kernel does not take.
//
// "Efficient Content-Based Sparse Attention with Routing Transformers":
// §3 (attention weights from query/key dot products, rows normalised by
// softmax, autoregressive queries only see earlier positions, output =
// weights times values) restricted by §4 to query/key pairs of one cluster.
// A cluster's members are listed in ascending position order, so the causal
// mask on original positions is the lower triangle in slot order, diagonal
// included.
//
// One CTA takes 64 query slots of one cluster (16 when the problem has too
// few clusters to fill the GPU that way) and walks the cluster's key slots in
// blocks of 64 with an online (running max / running sum) softmax.
// With SEP (separate queries and keys) the key and value rows come from the
// keys' own lists (idx_k) and the causal mask compares original positions; a
// query with no visible key gets a zero row and is not counted in mvis.
// Gathered K and V rows are staged in shared memory as fp32; each warp owns
// 8 (or 2) query rows.  The epilogue writes a row straight to the output when the
// position belongs to exactly one cluster, else to the per-slot buffer that
// the scatter kernel averages.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int KB = 64;
constexpr int THREADS = 256;

template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* __restrict__ src,
                                          const int32_t* __restrict__ pos, int first, int count,
                                          int limit, int n_rows_total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < count; r += THREADS / 32) {
    const int slot = first + r;
    const int t = (slot < limit) ? __ldcg(pos + slot) : -1;
    if ((unsigned)t < (unsigned)n_rows_total) {  // defensive: never read outside the head
      const T* row = src + (size_t)t * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) dst[r * ld + lane + 32 * i] = to_f32(__ldcg(row + lane + 32 * i));
    } else {
#pragma unroll
      for (int i = 0; i < D / 32; ++i) dst[r * ld + lane + 32 * i] = 0.0f;
    }
  }
}

template <typename T, int D, bool SEP, int QB>
__global__ void __launch_bounds__(THREADS)
attention_simt_kernel(const T* __restrict__ q, const T* __restrict__ kk, const T* __restrict__ v,
                      int n, int k, int w, int causal, float scale,
                      const int32_t* __restrict__ idx, const int32_t* __restrict__ idx_k,
                      const int32_t* __restrict__ mcount, int32_t* __restrict__ mvis,
                      T* __restrict__ out, float* __restrict__ yslot) {
  pdl_trigger();
  pdl_wait();
  constexpr int ROWS_PER_WARP = QB / (THREADS / 32);
  extern __shared__ float smem[];
  constexpr int LDQ = D + 1;
  float* Qs = smem;              // [QB][D+1]
  float* Ks = Qs + QB * LDQ;     // [KB][D+1]
  float* Vs = Ks + KB * LDQ;     // [KB][D]

  const int q0 = blockIdx.x * QB;
  const int c = blockIdx.y;
  const int bh = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* pos = idx + ((size_t)bh * k + c) * w;
  const int32_t* kpos = SEP ? idx_k + ((size_t)bh * k + c) * w : pos;
  const size_t head_off = (size_t)bh * n * D;
  __shared__ int qp_s[QB], kp_s[KB];  // positions (SEP's causal mask)

  load_rows<T, D>(Qs, LDQ, q + head_off, pos, q0, QB, w, n);
  if (SEP)
    for (int i = threadIdx.x; i < QB; i += THREADS) qp_s[i] = q0 + i < w ? __ldcg(pos + q0 + i) : -1;

  float m[ROWS_PER_WARP], l[ROWS_PER_WARP], acc[ROWS_PER_WARP][D / 32];
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[r][i] = 0.0f;
  }

  const int kend = (causal && !SEP) ? min(w, q0 + QB) : w;
  for (int kb0 = 0; kb0 < kend; kb0 += KB) {
    __syncthreads();
    load_rows<T, D>(Ks, LDQ, kk + head_off, kpos, kb0, KB, w, n);
    load_rows<T, D>(Vs, D, v + head_off, kpos, kb0, KB, w, n);
    if (SEP)
      for (int i = threadIdx.x; i < KB; i += THREADS) kp_s[i] = kb0 + i < w ? __ldcg(kpos + kb0 + i) : -1;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
      const int rl = warp * ROWS_PER_WARP + r;
      const int qi = q0 + rl;
      if (qi >= w) continue;
      const float* qrow = Qs + rl * LDQ;
      const float* k0 = Ks + lane * LDQ;
      const float* k1 = Ks + (lane + 32) * LDQ;
      float d0 = 0.0f, d1 = 0.0f;
#pragma unroll 16
      for (int j = 0; j < D; ++j) {
        const float qv = qrow[j];
        d0 = fmaf(qv, k0[j], d0);
        d1 = fmaf(qv, k1[j], d1);
      }
      const int j0 = kb0 + lane, j1 = kb0 + lane + 32;
      bool v0, v1;
      if (SEP) {
        const int qp = qp_s[rl];
        v0 = j0 < w && (!causal || kp_s[lane] <= qp);
        v1 = j1 < w && (!causal || kp_s[lane + 32] <= qp);
      } else {
        v0 = j0 < w && (!causal || j0 <= qi);
        v1 = j1 < w && (!causal || j1 <= qi);
      }
      const float s0 = v0 ? d0 * scale : -INFINITY;
      const float s1 = v1 ? d1 * scale : -INFINITY;
      const float mb = warp_max(fmaxf(s0, s1));
      if (mb == -INFINITY) continue;
      const float mnew = fmaxf(m[r], mb);
      const float alpha = (m[r] == -INFINITY) ? 0.0f : expf(m[r] - mnew);
      const float p0 = v0 ? expf(s0 - mnew) : 0.0f;
      const float p1 = v1 ? expf(s1 - mnew) : 0.0f;
      l[r] = l[r] * alpha + warp_sum(p0 + p1);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[r][i] *= alpha;
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const float pa = __shfl_sync(0xffffffffu, p0, jj);
        const float pb = __shfl_sync(0xffffffffu, p1, jj);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          acc[r][i] = fmaf(pa, Vs[jj * D + lane + 32 * i], acc[r][i]);
          acc[r][i] = fmaf(pb, Vs[(jj + 32) * D + lane + 32 * i], acc[r][i]);
        }
      }
      m[r] = mnew;
    }
  }

#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    const int qi = q0 + warp * ROWS_PER_WARP + r;
    if (qi >= w) continue;
    const int t = pos[qi];
    if ((unsigned)t >= (unsigned)n) continue;
    const float inv_l = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;  // no visible key: zero row
    const int m_all = __ldcg(mcount + (size_t)bh * n + t);
    if (SEP && m_all != 1 && l[r] > 0.0f && lane == 0) atomicAdd(mvis + (size_t)bh * n + t, 1);
    if (m_all == 1) {
      T* orow = out + head_off + (size_t)t * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = from_f32<T>(acc[r][i] * inv_l);
    } else {
      float* yrow = yslot + (((size_t)bh * k + c) * w + qi) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) yrow[lane + 32 * i] = acc[r][i] * inv_l;
    }
  }
}

template <typename T, int D>
cudaError_t launch_t(const void* q, const void* kk, const void* v, int BH, int n, int k, int w,
                     int causal, float scale, const int32_t* idx, const int32_t* idx_k,
                     const int32_t* mcount, int32_t* mvis, void* out, float* yslot,
                     cudaStream_t s) {
  // 64 query rows a CTA, or 16 when that would leave most SMs idle
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool small = (long long)((w + 63) / 64) * k * BH < 2LL * sms;
  const int QB = small ? 16 : 64;
  const size_t smem = ((size_t)(QB + KB) * (D + 1) + (size_t)KB * D) * sizeof(float);
  auto kern = idx_k != nullptr
                  ? (small ? attention_simt_kernel<T, D, true, 16> : attention_simt_kernel<T, D, true, 64>)
                  : (small ? attention_simt_kernel<T, D, false, 16> : attention_simt_kernel<T, D, false, 64>);
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((w + QB - 1) / QB, k, BH);
  launch_begin(K_ATTN_SIMT, s);
  e = launch_pdl(kern, grid, dim3(THREADS), smem, s, static_cast<const T*>(q),
                 static_cast<const T*>(kk), static_cast<const T*>(v), n, k, w, causal, scale, idx,
                 idx_k, mcount, mvis, static_cast<T*>(out), yslot);
  launch_end(K_ATTN_SIMT, s);
  return e;
}

}  // namespace

cudaError_t launch_attention_simt(const void* q, const void* kk, const void* v, rt_dtype dt,
                                  int BH, int n, int d, int k, int w, int causal,
                                  float scale, const int32_t* idx, const int32_t* idx_k,
                                  const int32_t* mcount, int32_t* mvis, void* out, float* yslot,
                                  cudaStream_t s) {
  if (dt == RT_F32) {
    return d == 64 ? launch_t<float, 64>(q, kk, v, BH, n, k, w, causal, scale, idx, idx_k, mcount, mvis, out, yslot, s)
                   : launch_t<float, 128>(q, kk, v, BH, n, k, w, causal, scale, idx, idx_k, mcount, mvis, out, yslot, s);
  }
  return d == 64
             ? launch_t<__nv_bfloat16, 64>(q, kk, v, BH, n, k, w, causal, scale, idx, idx_k, mcount, mvis, out, yslot, s)
             : launch_t<__nv_bfloat16, 128>(q, kk, v, BH, n, k, w, causal, scale, idx, idx_k, mcount, mvis, out, yslot, s);
}

}  // namespace rt
