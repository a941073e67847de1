// Top-w per centroid, emitted in ascending position order.
//
// Balanced clusters of "Efficient Content-Based Sparse Attention with
// Routing Transformers" (§4, "Routing attention with clustering": each query
// compares with about n/k keys through a top-k assignment).  Each centroid
// keeps the w positions with the largest score; equal scores go to the lower
// position; the kept positions are listed in ascending order.
//
// One CTA per (batch*head, centroid), in three steps over the row of n
// scores:
//   1. one read of the row: every score gets a bin of a 2048-bin linear
//      partition of [-1, 1] (a non-decreasing function of the score, so all
//      scores of a higher bin are strictly larger); the bin index is staged in
//      shared memory (u16) and counted in a shared histogram;
//   2. the bin b* holding the w-th largest score is found by a descending scan
//      of the histogram; its members (the candidates, typically a handful) are
//      collected and ranked exactly by (score desc, position asc) -- a
//      candidate is kept iff its rank is below the number still needed;
//   3. an ordered compaction walks the positions in order and keeps bin > b*
//      plus the kept candidates; a block prefix sum gives each kept position
//      its output slot, so the list comes out sorted without a sort.
// Membership counts are incremented here with integer atomics (the totals are
// order independent), and the first SLOTS_PER_ROW (cluster, slot) entries of
// every position are recorded for the scatter.
// Rows whose boundary bin holds too many candidates (many equal scores), or
// that do not fit in shared memory, use an exact 32-bit most-significant-digit
// radix select over order-preserving keys instead.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int NBINS = 2048;
constexpr int CAND_CAP = 2048;
constexpr int MAX_STAGED_BINS = 80 * 1024;  // u16 bins staged in shared memory

__device__ __forceinline__ int score_bin(float s) {
  // non-decreasing in s; [-1, 1] -> [0, 2047]
  float f = (s + 1.0f) * 1024.0f;
  f = fminf(fmaxf(f, 0.0f), (float)(NBINS - 1));
  return (int)f;
}

struct SelectOut {
  int32_t* out;
  int32_t* mcount;
  int32_t* slots;
  int bh, c, n, w;
  __device__ __forceinline__ void emit(int o, int t) const {
    out[o] = t;
    if (mcount != nullptr) {
      const int prev = atomicAdd(&mcount[(size_t)bh * n + t], 1);
      if (slots != nullptr && prev < SLOTS_PER_ROW)
        slots[((size_t)bh * n + t) * SLOTS_PER_ROW + prev] = c * w + o;
    }
  }
};

// Ordered compaction: keep(t) is evaluated for t = 0, 1, ... in chunks of
// THREADS; one barrier per chunk (double-buffered warp totals).
template <typename Keep>
__device__ __forceinline__ void ordered_compact(int n, int w, int* wsum /* [2][WARPS] */,
                                                const SelectOut& so, Keep keep) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int out_base = 0, buf = 0;
  for (int t0 = 0; t0 < n && out_base < w; t0 += THREADS, buf ^= 1) {
    const int t = t0 + threadIdx.x;
    const bool sel = (t < n) && keep(t);
    const unsigned b = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) wsum[buf * WARPS + warp] = __popc(b);
    __syncthreads();
    int pre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < WARPS; ++i) {
      const int x = wsum[buf * WARPS + i];
      pre += (i < warp) ? x : 0;
      tot += x;
    }
    if (sel) {
      const int o = out_base + pre + __popc(b & ((1u << lane) - 1u));
      if (o < w) so.emit(o, t);
    }
    out_base += tot;
  }
}

// Exact fallback: 32-bit MSD radix select on order-preserving keys.
__device__ void radix_select_row(const float* __restrict__ row, int n, int w, const SelectOut& so,
                                 unsigned* hist /* >= 256 */, int* wsum /* [4][WARPS] */) {
  __shared__ unsigned s_digit;
  __shared__ int s_remaining;
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
  int remaining = w;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += THREADS) hist[b] = 0u;
    __syncthreads();
    for (int t = tid; t < n; t += THREADS) {
      const uint32_t key = score_key(__ldg(row + t));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
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
  // keys > K* plus the first need_eq keys == K*, in position order
  const int lane = tid & 31, warp = tid >> 5;
  int out_base = 0, eq_base = 0, buf = 0;
  for (int t0 = 0; t0 < n && out_base < w; t0 += THREADS, buf ^= 1) {
    const int t = t0 + tid;
    const uint32_t key = (t < n) ? score_key(__ldg(row + t)) : 0u;
    const bool gt = (t < n) && key > kstar;
    const bool eq = (t < n) && key == kstar;
    const unsigned be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) wsum[buf * 2 * WARPS + warp] = __popc(be);
    __syncthreads();
    int epre = 0, etot = 0;
    for (int i = 0; i < WARPS; ++i) {
      const int x = wsum[buf * 2 * WARPS + i];
      epre += (i < warp) ? x : 0;
      etot += x;
    }
    const int erank = eq_base + epre + __popc(be & ((1u << lane) - 1u));
    const bool sel = gt || (eq && erank < need_eq);
    const unsigned bs = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) wsum[buf * 2 * WARPS + WARPS + warp] = __popc(bs);
    __syncthreads();
    int spre = 0, stot = 0;
    for (int i = 0; i < WARPS; ++i) {
      const int x = wsum[buf * 2 * WARPS + WARPS + i];
      spre += (i < warp) ? x : 0;
      stot += x;
    }
    if (sel) {
      const int o = out_base + spre + __popc(bs & ((1u << lane) - 1u));
      if (o < w) so.emit(o, t);
    }
    out_base += stot;
    eq_base += etot;
  }
}

__global__ void __launch_bounds__(THREADS)
select_topw_kernel(const float* __restrict__ S, int n, int k, int w, int32_t* __restrict__ idx,
                   int32_t* __restrict__ mcount, int32_t* __restrict__ slots, int staged) {
  extern __shared__ uint16_t sbin[];  // [n] when staged
  __shared__ unsigned hist[NBINS];
  __shared__ int cand_t[CAND_CAP];
  __shared__ float cand_s[CAND_CAP];
  __shared__ int wsum[4 * WARPS];
  __shared__ int s_bstar, s_need, s_ncand;
  __shared__ unsigned keep_bits[CAND_CAP / 32];

  const int c = blockIdx.x;
  const int bh = blockIdx.y;
  const float* row = S + ((size_t)bh * k + c) * n;
  const SelectOut so{idx + ((size_t)bh * k + c) * w, mcount, slots, bh, c, n, w};
  const int tid = threadIdx.x, lane = tid & 31;

  if (!staged) {
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }

  for (int b = tid; b < NBINS; b += THREADS) hist[b] = 0u;
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  // 1. bins + histogram (one read of the row)
  for (int t = tid; t < n; t += THREADS) {
    const int b = score_bin(__ldg(row + t));
    sbin[t] = (uint16_t)b;
    atomicAdd(&hist[b], 1u);
  }
  __syncthreads();
  // 2a. boundary bin: the descending cumulative count reaches w inside b*
  if (tid < 32) {
    constexpr int PER = NBINS / 32;  // bins per lane, lane 0 = highest bins
    unsigned lsum = 0;
    for (int q = 0; q < PER; ++q) lsum += hist[NBINS - 1 - PER * lane - q];
    unsigned incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned excl = incl - lsum;
    if (excl < (unsigned)w && (unsigned)w <= incl) {
      unsigned cum = excl;
      for (int q = 0; q < PER; ++q) {
        const int b = NBINS - 1 - PER * lane - q;
        const unsigned hb = hist[b];
        if (cum + hb >= (unsigned)w) {
          s_bstar = b;
          s_need = w - (int)cum;
          break;
        }
        cum += hb;
      }
    }
  }
  __syncthreads();
  const int bstar = s_bstar, need = s_need;
  const int ncand_total = (int)hist[bstar];
  if (ncand_total > CAND_CAP) {  // many equal or near-equal scores: exact radix path
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }
  // 2b. collect the candidates (order irrelevant) and rank them exactly
  for (int t0 = 0; t0 < n; t0 += THREADS) {
    const int t = t0 + tid;
    const bool is_c = (t < n) && sbin[t] == bstar;
    const unsigned bm = __ballot_sync(0xffffffffu, is_c);
    int base = 0;
    if (lane == 0 && bm) base = atomicAdd(&s_ncand, __popc(bm));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (is_c) {
      const int slot = base + __popc(bm & ((1u << lane) - 1u));
      cand_t[slot] = t;
      cand_s[slot] = __ldg(row + t);
    }
  }
  for (int i = tid; i < CAND_CAP / 32; i += THREADS) keep_bits[i] = 0u;
  __syncthreads();
  const int nc = s_ncand;
  for (int i = tid; i < nc; i += THREADS) {
    const float si = cand_s[i];
    const int ti = cand_t[i];
    int rank = 0;
    for (int j = 0; j < nc; ++j) {
      const float sj = cand_s[j];
      rank += (sj > si) || (sj == si && cand_t[j] < ti);
    }
    if (rank < need) atomicOr(&keep_bits[i >> 5], 1u << (i & 31));
  }
  __syncthreads();
  // kept candidates get bin value NBINS (> every b*)
  for (int i = tid; i < nc; i += THREADS)
    if (keep_bits[i >> 5] & (1u << (i & 31))) sbin[cand_t[i]] = (uint16_t)NBINS;
  __syncthreads();
  // 3. ordered compaction: bin > b*
  ordered_compact(n, w, wsum, so, [&](int t) { return (int)sbin[t] > bstar; });
}

}  // namespace

cudaError_t launch_select(const float* S, int BH, int n, int k, int w, int32_t* idx,
                          int32_t* mcount, int32_t* slots, cudaStream_t s) {
  dim3 grid(k, BH);
  const int staged = n <= MAX_STAGED_BINS ? 1 : 0;
  const size_t smem = staged ? (size_t)n * sizeof(uint16_t) : 0;
  cudaError_t e = cudaFuncSetAttribute(select_topw_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       MAX_STAGED_BINS * (int)sizeof(uint16_t));
  if (e != cudaSuccess) return e;
  launch_begin(K_SELECT, s);
  select_topw_kernel<<<grid, THREADS, smem, s>>>(S, n, k, w, idx, mcount, slots, staged);
  e = cudaGetLastError();
  launch_end(K_SELECT, s);
  return e;
}

}  // namespace rt
