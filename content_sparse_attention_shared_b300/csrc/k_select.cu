// Top-w per centroid, emitted in ascending position order.
//
// Balanced clusters of "Efficient Content-Based Sparse Attention with
// Routing Transformers" (§4, "Routing attention with clustering": each query
// compares with about n/k keys through a top-k assignment).  Each centroid
// keeps the w positions with the largest score; equal scores go to the lower
// position; the kept positions are listed in ascending order.
//
// One CTA per (batch*head, centroid).  Scores are mapped to order-preserving
// 32-bit keys.  A most-significant-digit radix select (4 passes of 8 bits,
// over shared memory when the row fits, else over the L2-resident row) finds
// the key K* of the w-th largest score and how many keys equal to K* are
// needed.  A final ordered compaction walks the row in position order and
// keeps keys > K* plus the first `need` keys == K*; a block-wide prefix sum
// gives each kept position its output slot, so the list comes out sorted
// without a sort.  Membership counts are incremented here with integer
// atomics (the totals are order independent).
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_STAGED = 48 * 1024;  // keys staged in shared memory (192 KiB)

template <bool STAGED>
__device__ __forceinline__ uint32_t key_at(const uint32_t* keys, const float* row, int t) {
  return STAGED ? keys[t] : score_key(__ldg(row + t));
}

// exclusive block prefix of two predicates at once; returns block totals
__device__ __forceinline__ void block_scan2(bool p0, bool p1, int& ex0, int& ex1, int& tot0,
                                            int& tot1, int* sm /* [2*WARPS] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const unsigned b0 = __ballot_sync(0xffffffffu, p0);
  const unsigned b1 = __ballot_sync(0xffffffffu, p1);
  if (lane == 0) { sm[warp] = __popc(b0); sm[WARPS + warp] = __popc(b1); }
  __syncthreads();
  int pre0 = 0, pre1 = 0, t0 = 0, t1 = 0;
  for (int i = 0; i < WARPS; ++i) {
    const int c0 = sm[i], c1 = sm[WARPS + i];
    if (i < warp) { pre0 += c0; pre1 += c1; }
    t0 += c0; t1 += c1;
  }
  ex0 = pre0 + __popc(b0 & lt);
  ex1 = pre1 + __popc(b1 & lt);
  tot0 = t0; tot1 = t1;
  __syncthreads();
}

template <bool STAGED>
__global__ void __launch_bounds__(THREADS)
select_topw_kernel(const float* __restrict__ S, int n, int k, int w, int32_t* __restrict__ idx,
                   int32_t* __restrict__ mcount) {
  extern __shared__ uint32_t keys[];  // n keys when STAGED
  __shared__ unsigned hist[256];
  __shared__ int scan_sm[2 * WARPS];
  __shared__ unsigned s_digit;
  __shared__ int s_remaining;

  const int c = blockIdx.x;
  const int bh = blockIdx.y;
  const float* row = S + ((size_t)bh * k + c) * n;
  int32_t* out = idx + ((size_t)bh * k + c) * w;
  const int tid = threadIdx.x;

  if (STAGED) {
    for (int t = tid; t < n; t += THREADS) keys[t] = score_key(__ldg(row + t));
  }

  uint32_t prefix = 0, mask = 0;
  int remaining = w;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += THREADS) hist[b] = 0u;
    __syncthreads();
    for (int t = tid; t < n; t += THREADS) {
      const uint32_t key = key_at<STAGED>(keys, row, t);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns bins 255-8L ... 248-8L (descending)
      const int lane = tid;
      unsigned lsum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) lsum += hist[255 - 8 * lane - q];
      unsigned incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned excl = incl - lsum;
      if (excl < (unsigned)remaining && (unsigned)remaining <= incl) {
        unsigned cum = excl;
        for (int q = 0; q < 8; ++q) {
          const int b = 255 - 8 * lane - q;
          const unsigned hb = hist[b];
          if (cum + hb >= (unsigned)remaining) {
            s_digit = (unsigned)b;
            s_remaining = remaining - (int)cum;
            break;
          }
          cum += hb;
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    remaining = s_remaining;
    __syncthreads();
  }
  const uint32_t kstar = prefix;
  const int need_eq = remaining;

  // ordered compaction in position order
  int out_base = 0, eq_base = 0;
  for (int t0 = 0; t0 < n && out_base < w; t0 += THREADS) {
    const int t = t0 + tid;
    uint32_t key = 0;
    if (t < n) key = key_at<STAGED>(keys, row, t);
    const bool gt = (t < n) && key > kstar;
    const bool eq = (t < n) && key == kstar;
    int eq_rank, dummy, eq_tot, dummy_tot;
    block_scan2(eq, false, eq_rank, dummy, eq_tot, dummy_tot, scan_sm);
    const bool sel = gt || (eq && (eq_base + eq_rank) < need_eq);
    int pos, pos2, sel_tot, tot2;
    block_scan2(sel, false, pos, pos2, sel_tot, tot2, scan_sm);
    if (sel) {
      const int o = out_base + pos;
      if (o < w) {
        out[o] = t;
        if (mcount != nullptr) atomicAdd(&mcount[(size_t)bh * n + t], 1);
      }
    }
    out_base += sel_tot;
    eq_base += eq_tot;
  }
}

}  // namespace

cudaError_t launch_select(const float* S, int BH, int n, int k, int w, int32_t* idx,
                          int32_t* mcount, cudaStream_t s) {
  dim3 grid(k, BH);
  cudaError_t e;
  launch_begin(K_SELECT, s);
  if (n <= MAX_STAGED) {
    const size_t smem = (size_t)n * sizeof(uint32_t);
    e = cudaFuncSetAttribute(select_topw_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_STAGED * 4);
    if (e == cudaSuccess) {
      select_topw_kernel<true><<<grid, THREADS, smem, s>>>(S, n, k, w, idx, mcount);
      e = cudaGetLastError();
    }
  } else {
    select_topw_kernel<false><<<grid, THREADS, 0, s>>>(S, n, k, w, idx, mcount);
    e = cudaGetLastError();
  }
  launch_end(K_SELECT, s);
  return e;
}

}  // namespace rt
