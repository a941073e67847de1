// Backward pass of the in-cluster attention and the averaging scatter, with
// the routing held fixed.
//
// "Efficient Content-Based Sparse Attention with Routing Transformers": the
// centroids are learned by the online k-means step, not by gradients (§2,
// §4), and the routing is piecewise constant in the rows, so the gradient of
// the layer flows through the softmax attention of each cluster (§3) and the
// averaging of a position's cluster outputs.  With shared QK a row is both a
// query and a key of its cluster, so dq collects both roles.  Per cluster c
// with members p_0 < ... < p_{w-1}:
//   P  = softmax(scale Q_c Q_c^T + causal mask)      (recomputed here)
//   dY = dO[p_i] / m(p_i)                             (m = membership count)
//   dV_c = P^T dY;  dP = dY V_c^T;  D_i = sum_j P_ij dP_ij
//   dS = P * (dP - D);  dQ_c = scale (dS Q_c + dS^T Q_c)
// and a position's gradient is the sum of its rows over its clusters.
//
// backward_cluster_kernel: one CTA per (cluster, batch*head), fp32 on CUDA
// cores, blocks of 64 slots.  For each query block i it makes three passes
// over the key blocks j <= i (all j when not causal): the row maxima and
// sums of exp, then D, then dS -- adding dS Q_j into the block's query-role
// rows (shared memory) and dS^T Q_i and P^T dY_i into key block j's slot rows
// in global memory.  Only this CTA touches its cluster's slot rows, in a
// fixed order, so the result is deterministic.  A gather kernel then adds each
// position's slot rows in ascending cluster order (membership lists rebuilt
// from idx).
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int BTHREADS = 256;
constexpr int BB = 64;        // slots per block
constexpr int LDT = BB + 1;   // padded row of a 64 x 64 tile

template <int D>
struct BwdSmem {
  static constexpr int LDR = D + 1;  // padded row of a 64 x D block
  // Qi, dYi, Qj, Vj (64 x (D+1)), P and dP/dS tiles (64 x 65), dQi (64 x D)
  static constexpr size_t FLOATS = 4 * (size_t)BB * LDR + 2 * (size_t)BB * LDT + (size_t)BB * D;
  static constexpr size_t BYTES = FLOATS * 4;
};

template <typename T, int D>
__device__ __forceinline__ void load_block(float* dst, const T* __restrict__ src, const int* pos,
                                           const float* mult) {
  // rows pos[r] (-1: zero row) of src [n, D] into dst [64][D+1], times mult[r]
  constexpr int LDR = D + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < BB; r += BTHREADS / 32) {
    const int p = pos[r];
    const float f = mult ? mult[r] : 1.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i)
      dst[r * LDR + lane + 32 * i] = p >= 0 ? to_f32(__ldcg(src + (size_t)p * D + lane + 32 * i)) * f : 0.0f;
  }
}

// out[r][c] = sum_kk A[r][kk] * B[c][kk] for a 64 x 64 tile (A, B: 64 x K,
// row strides lda, ldb); thread (ty, tx) computes rows 4ty.., cols 4tx..
template <int K>
__device__ __forceinline__ void tile_abt(const float* A, int lda, const float* B, int ldb,
                                         float (&acc)[4][4]) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
#pragma unroll 4
  for (int kk = 0; kk < K; ++kk) {
    float x[4], y[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) x[a] = A[(4 * ty + a) * lda + kk];
#pragma unroll
    for (int b = 0; b < 4; ++b) y[b] = B[(4 * tx + b) * ldb + kk];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(x[a], y[b], acc[a][b]);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(BTHREADS, 1)
backward_cluster_kernel(const T* __restrict__ q, const T* __restrict__ v, int n, int k, int w,
                        int causal, float scale, const int32_t* __restrict__ idx,
                        const int32_t* __restrict__ mcount, const float* __restrict__ dout,
                        float* __restrict__ dq_slot, float* __restrict__ dv_slot) {
  pdl_trigger();
  pdl_wait();
  constexpr int LDR = D + 1;
  extern __shared__ float bsm[];
  float* Qi = bsm;
  float* dYi = Qi + BB * LDR;
  float* Qj = dYi + BB * LDR;
  float* Vj = Qj + BB * LDR;
  float* Pt = Vj + BB * LDR;   // [64][65]
  float* Gt = Pt + BB * LDT;   // dP, then dS [64][65]
  float* dQi = Gt + BB * LDT;  // [64][D]
  __shared__ int pi[BB], pj[BB];
  __shared__ float minv[BB], mrow[BB], lrow[BB], drow[BB];

  const int c = blockIdx.x, bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tx = tid & 15, ty = tid >> 4;
  const int32_t* list = idx + ((size_t)bh * k + c) * w;
  const T* q_bh = q + (size_t)bh * n * D;
  const T* v_bh = v + (size_t)bh * n * D;
  const float* do_bh = dout + (size_t)bh * n * D;
  float* dqs = dq_slot + ((size_t)bh * k + c) * w * D;
  float* dvs = dv_slot + ((size_t)bh * k + c) * w * D;
  const int nb = (w + BB - 1) / BB;

  // the cluster's slot rows start at zero (only this CTA writes them)
  for (int i = tid; i < w * D; i += BTHREADS) { dqs[i] = 0.0f; dvs[i] = 0.0f; }

  // valid key columns of row r (slot si) in key block jb: [0, jmax)
  auto col_limit = [&](int si, int jb) {
    int jm = min(BB, w - jb * BB);
    if (causal) jm = min(jm, si - jb * BB + 1);
    return jm;
  };
  // S tile of (ib, jb) scaled, into acc (thread tile)
  for (int ib = 0; ib < nb; ++ib) {
    __syncthreads();
    for (int r = tid; r < BB; r += BTHREADS) {
      const int s = ib * BB + r;
      int p = s < w ? __ldcg(list + s) : -1;
      if ((unsigned)p >= (unsigned)n) p = -1;
      pi[r] = p;
      const int m = p >= 0 ? __ldcg(mcount + (size_t)bh * n + p) : 0;
      minv[r] = m > 0 ? 1.0f / (float)m : 0.0f;
      mrow[r] = -INFINITY;
      lrow[r] = 0.0f;
      drow[r] = 0.0f;
    }
    __syncthreads();
    load_block<T, D>(Qi, q_bh, pi, nullptr);
    load_block<float, D>(dYi, do_bh, pi, minv);
    for (int i = tid; i < BB * D; i += BTHREADS) dQi[i] = 0.0f;
    const int jb_end = causal ? ib + 1 : nb;

    for (int pass = 0; pass < 3; ++pass) {
      for (int jb = 0; jb < jb_end; ++jb) {
        __syncthreads();  // Qj / Vj / tiles free
        for (int r = tid; r < BB; r += BTHREADS) {
          const int s = jb * BB + r;
          int p = s < w ? __ldcg(list + s) : -1;
          if ((unsigned)p >= (unsigned)n) p = -1;
          pj[r] = p;
        }
        __syncthreads();
        load_block<T, D>(Qj, q_bh, pj, nullptr);
        if (pass > 0) load_block<T, D>(Vj, v_bh, pj, nullptr);
        __syncthreads();
        // S tile (scaled logits) into Pt
        {
          float acc[4][4];
          tile_abt<D>(Qi, LDR, Qj, LDR, acc);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) Pt[(4 * ty + a) * LDT + 4 * tx + b] = acc[a][b] * scale;
        }
        if (pass > 0) {  // dP = dY_i V_j^T into Gt
          float acc[4][4];
          tile_abt<D>(dYi, LDR, Vj, LDR, acc);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) Gt[(4 * ty + a) * LDT + 4 * tx + b] = acc[a][b];
        }
        __syncthreads();
        // row-wise work: warp per 8 rows, lane per 2 columns
        for (int rr = 0; rr < BB / 8; ++rr) {
          const int r = warp * (BB / 8) + rr;
          const int si = ib * BB + r;
          const bool rv = pi[r] >= 0;
          const int jm = rv ? col_limit(si, jb) : 0;
          const bool v0 = lane < jm, v1 = lane + 32 < jm;
          const float s0 = v0 ? Pt[r * LDT + lane] : -INFINITY;
          const float s1 = v1 ? Pt[r * LDT + lane + 32] : -INFINITY;
          if (pass == 0) {
            // online row maximum and sum of exp
            const float mb = warp_max(fmaxf(s0, s1));
            if (mb != -INFINITY) {
              const float mo = mrow[r];
              const float mn = fmaxf(mo, mb);
              const float e = (v0 ? expf(s0 - mn) : 0.0f) + (v1 ? expf(s1 - mn) : 0.0f);
              const float es = warp_sum(e);
              if (lane == 0) {
                lrow[r] = lrow[r] * (mo == -INFINITY ? 0.0f : expf(mo - mn)) + es;
                mrow[r] = mn;
              }
            }
          } else {
            const float inv_l = lrow[r] > 0.0f ? 1.0f / lrow[r] : 0.0f;
            const float p0 = v0 ? expf(s0 - mrow[r]) * inv_l : 0.0f;
            const float p1 = v1 ? expf(s1 - mrow[r]) * inv_l : 0.0f;
            if (pass == 1) {
              const float dd = warp_sum(p0 * Gt[r * LDT + lane] + p1 * Gt[r * LDT + lane + 32]);
              if (lane == 0) drow[r] += dd;
            } else {
              // P into Pt, dS into Gt
              const float dr = drow[r];
              Gt[r * LDT + lane] = p0 * (Gt[r * LDT + lane] - dr);
              Gt[r * LDT + lane + 32] = p1 * (Gt[r * LDT + lane + 32] - dr);
              Pt[r * LDT + lane] = p0;
              Pt[r * LDT + lane + 32] = p1;
            }
          }
          __syncwarp();
        }
        if (pass < 2) continue;
        __syncthreads();
        // dQ_i += scale dS Q_j (query role); key block rows: dQ_j += scale dS^T Q_i,
        // dV_j += P^T dY_i.  Thread (ty, tx): rows 4ty..4ty+3, features tx + 16 e.
        constexpr int FE = D / 16;
        {
          float a1[4][FE];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int e = 0; e < FE; ++e) a1[a][e] = 0.0f;
          for (int jj = 0; jj < BB; ++jj) {
            float g[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) g[a] = Gt[(4 * ty + a) * LDT + jj];
#pragma unroll
            for (int e = 0; e < FE; ++e) {
              const float y = Qj[jj * LDR + tx + 16 * e];
#pragma unroll
              for (int a = 0; a < 4; ++a) a1[a][e] = fmaf(g[a], y, a1[a][e]);
            }
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int e = 0; e < FE; ++e) dQi[(4 * ty + a) * D + tx + 16 * e] += scale * a1[a][e];
        }
        {
          float a2[4][FE], a3[4][FE];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int e = 0; e < FE; ++e) { a2[a][e] = 0.0f; a3[a][e] = 0.0f; }
          for (int ii = 0; ii < BB; ++ii) {
            float g[4], pp[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              g[a] = Gt[ii * LDT + 4 * ty + a];
              pp[a] = Pt[ii * LDT + 4 * ty + a];
            }
#pragma unroll
            for (int e = 0; e < FE; ++e) {
              const float x = Qi[ii * LDR + tx + 16 * e];
              const float y = dYi[ii * LDR + tx + 16 * e];
#pragma unroll
              for (int a = 0; a < 4; ++a) {
                a2[a][e] = fmaf(g[a], x, a2[a][e]);
                a3[a][e] = fmaf(pp[a], y, a3[a][e]);
              }
            }
          }
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int sj = jb * BB + 4 * ty + a;
            if (sj >= w) continue;
#pragma unroll
            for (int e = 0; e < FE; ++e) {
              dqs[(size_t)sj * D + tx + 16 * e] += scale * a2[a][e];
              dvs[(size_t)sj * D + tx + 16 * e] += a3[a][e];
            }
          }
        }
      }
    }
    __syncthreads();
    // the query role of block ib
    for (int i = tid; i < BB * D; i += BTHREADS) {
      const int r = i / D, f = i - r * D;
      const int si = ib * BB + r;
      if (si < w) dqs[(size_t)si * D + f] += dQi[i];
    }
  }
}

// Membership lists from the index lists: mcount[t] = the number of clusters
// listing t, slots[t][0..7] the first (cluster*w + slot) ids (any order).
__global__ void __launch_bounds__(256)
membership_kernel(const int32_t* __restrict__ idx, int n, int k, int w, long long total,
                  int32_t* __restrict__ mcount, int32_t* __restrict__ slots) {
  pdl_trigger();
  pdl_wait();
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= total) return;
  const long long bh = g / ((long long)k * w);
  const int cs = (int)(g - bh * k * w);
  const int t = __ldcg(idx + g);
  if ((unsigned)t >= (unsigned)n) return;
  const int prev = atomicAdd(&mcount[bh * n + t], 1);
  if (prev < SLOTS_PER_ROW) slots[(bh * n + t) * SLOTS_PER_ROW + prev] = cs;
}

template <typename T, int D>
cudaError_t launch_bwd_t(const void* q, const void* v, int BH, int n, int k, int w, int causal,
                         float scale, const int32_t* idx, const int32_t* mcount,
                         const float* dout, float* dq_slot, float* dv_slot, cudaStream_t s) {
  const size_t smem = BwdSmem<D>::BYTES;
  auto kern = backward_cluster_kernel<T, D>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  launch_begin(K_BACKWARD, s);
  e = launch_pdl(kern, dim3(k, BH), dim3(BTHREADS), smem, s, static_cast<const T*>(q),
                 static_cast<const T*>(v), n, k, w, causal, scale, idx, mcount, dout, dq_slot,
                 dv_slot);
  launch_end(K_BACKWARD, s);
  return e;
}

}  // namespace

cudaError_t launch_membership(const int32_t* idx, int BH, int n, int k, int w, int32_t* mcount,
                              int32_t* slots, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(mcount, 0, (size_t)BH * n * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const long long total = (long long)BH * k * w;
  launch_begin(K_MEMBERSHIP, s);
  e = launch_pdl(membership_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, s, idx, n,
                 k, w, total, mcount, slots);
  launch_end(K_MEMBERSHIP, s);
  return e;
}

cudaError_t launch_backward_clusters(const void* q, const void* v, rt_dtype dt, int BH, int n,
                                     int d, int k, int w, int causal, float scale,
                                     const int32_t* idx, const int32_t* mcount, const float* dout,
                                     float* dq_slot, float* dv_slot, cudaStream_t s) {
  if (dt == RT_F32)
    return d == 64 ? launch_bwd_t<float, 64>(q, v, BH, n, k, w, causal, scale, idx, mcount, dout, dq_slot, dv_slot, s)
                   : launch_bwd_t<float, 128>(q, v, BH, n, k, w, causal, scale, idx, mcount, dout, dq_slot, dv_slot, s);
  return d == 64 ? launch_bwd_t<__nv_bfloat16, 64>(q, v, BH, n, k, w, causal, scale, idx, mcount, dout, dq_slot, dv_slot, s)
                 : launch_bwd_t<__nv_bfloat16, 128>(q, v, BH, n, k, w, causal, scale, idx, mcount, dout, dq_slot, dv_slot, s);
}

}  // namespace rt
