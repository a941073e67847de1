// Top-w per centroid, emitted in ascending position order.
//
// Balanced clusters of "Efficient Content-Based Sparse Attention with
// Routing Transformers" (§4, "Routing attention with clustering": each query
// compares with about n/k keys through a top-k assignment).  Each centroid
// keeps the w positions with the largest score; equal scores go to the lower
// position; the kept positions are listed in ascending order.
//
// One CTA of 256 threads per (batch*head, centroid) row of n scores, with a
// handful of block barriers in total (the cost of this kernel is latency, not
// bytes: the row is read once, usually from L2 right after the score kernel
// wrote it):
//   1. one vectorised read of the row: every score gets a bin of a 2048-bin
//      linear partition of [-1, 1] (non-decreasing in the score, so every
//      score of a higher bin is strictly larger); bins are staged in shared
//      memory (u16) and counted in a shared histogram;
//   2. a block-wide scan of the histogram from the top bin down finds the bin
//      b* holding the w-th largest score and how many of its members are
//      still needed;
//   3. one pass over the staged bins records, per 32-position chunk, the
//      mask of positions above b* and the mask of members of b* (the
//      candidates, typically a few); the candidates are ranked exactly by
//      (score desc, position asc) and the first `need` join the kept mask;
//   4. ordered emission: a block-wide scan over the chunks' kept counts gives
//      every chunk its first output slot, so the list comes out sorted by
//      position without a sort.
// Membership counts are incremented here with integer atomics (the totals are
// order independent), and the first SLOTS_PER_ROW (cluster, slot) entries of
// every position are recorded for the scatter.
// Rows whose boundary bin holds more than CAND_CAP candidates (many equal
// scores), or too long to stage in shared memory, use an exact 32-bit
// most-significant-digit radix select over order-preserving keys instead.
// Rows of n <= 8192 scores (n a multiple of 4, w <= 256) take the per-thread
// maximum bound kernel, longer rows with n a multiple of 4 the group-maximum
// kernel; this histogram kernel serves the rest.
#include "rt_internal.cuh"

namespace rt {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int NBINS = SCORE_BINS;  // score_bin: [-1, 1] -> [0, 2047], non-decreasing
constexpr int BINS_PER_THREAD = NBINS / THREADS;
constexpr int CAND_CAP = 1024;
constexpr int MAX_STAGED_BINS = 80 * 1024;  // u16 bins staged in shared memory

struct SelectOut {
  int32_t* out;
  int32_t* mcount;
  int32_t* slots;
  int bh, c, n, w;
  __device__ __forceinline__ void emit(int o, int t) const {
    out[o] = t;
    if (mcount != nullptr) {
      const int prev = atomicAdd(&mcount[(size_t)bh * n + t], 1);
      if (slots != nullptr && (unsigned)prev < (unsigned)SLOTS_PER_ROW)
        slots[((size_t)bh * n + t) * SLOTS_PER_ROW + prev] = c * w + o;
    }
  }
  // Emits the positions of the set bits of `word` (bit b = position base + b,
  // ascending) to output slots o, o + 1, ...; returns the next slot.  The
  // membership atomics of up to NB positions are issued together, so a
  // thread with several kept positions waits for one round trip, not one
  // per position.
  template <int NB = 8>
  __device__ __forceinline__ int emit_word(int o, unsigned word, int base) const {
    while (word != 0u) {
      int p[NB], prev[NB];
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        p[i] = 0;
        prev[i] = SLOTS_PER_ROW;
        if (word != 0u) {
          p[i] = base + __ffs(word) - 1;
          word &= word - 1u;
          cnt = i + 1;
        }
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i < cnt && o + i < w) {
          out[o + i] = p[i];
          if (mcount != nullptr) prev[i] = atomicAdd(&mcount[(size_t)bh * n + p[i]], 1);
        }
      }
      if (slots != nullptr) {
#pragma unroll
        for (int i = 0; i < NB; ++i)
          if (i < cnt && o + i < w && (unsigned)prev[i] < (unsigned)SLOTS_PER_ROW)
            slots[((size_t)bh * n + p[i]) * SLOTS_PER_ROW + prev[i]] = c * w + o + i;
      }
      o += cnt;
    }
    return o;
  }
  // The same over the words [q0, q1) of a position bitmap (word q: positions
  // 32q..32q+31): the kept positions of all the words are batched together,
  // so a thread owning several words waits for one round trip, not one per
  // non-empty word.
  template <int NB = 8>
  __device__ __forceinline__ int emit_words(int o, const unsigned* words, int q0, int q1) const {
    int q = q0;
    unsigned word = q < q1 ? words[q] : 0u;
    while (true) {
      int p[NB], prev[NB];
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        p[i] = 0;
        prev[i] = SLOTS_PER_ROW;
        while (word == 0u && q + 1 < q1) word = words[++q];
        if (word != 0u) {
          p[i] = q * 32 + __ffs(word) - 1;
          word &= word - 1u;
          cnt = i + 1;
        }
      }
      if (cnt == 0) break;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i < cnt && o + i < w) {
          out[o + i] = p[i];
          if (mcount != nullptr) prev[i] = atomicAdd(&mcount[(size_t)bh * n + p[i]], 1);
        }
      }
      if (slots != nullptr) {
#pragma unroll
        for (int i = 0; i < NB; ++i)
          if (i < cnt && o + i < w && (unsigned)prev[i] < (unsigned)SLOTS_PER_ROW)
            slots[((size_t)bh * n + p[i]) * SLOTS_PER_ROW + prev[i]] = c * w + o + i;
      }
      o += cnt;
    }
    return o;
  }
};

// Exact fallback: 32-bit MSD radix select on order-preserving keys, reading
// the row from global memory (L2).  Slow but general.
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
      const uint32_t key = score_key(__ldcg(row + t));
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
    const uint32_t key = (t < n) ? score_key(__ldcg(row + t)) : 0u;
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
  pdl_trigger();
  extern __shared__ __align__(16) uint16_t sbin[];  // [n] when staged
  __shared__ unsigned hist[NBINS];
  __shared__ int cand_t[CAND_CAP];
  __shared__ float cand_s[CAND_CAP];
  __shared__ int wsum[4 * WARPS];
  __shared__ int s_bstar, s_need, s_ncand;

  const int c = blockIdx.x;
  const int bh = blockIdx.y;
  const float* row = S + ((size_t)bh * k + c) * n;
  const SelectOut so{idx + ((size_t)bh * k + c) * w, mcount, slots, bh, c, n, w};
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (!staged) {
    pdl_wait();
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }

  for (int b = tid; b < NBINS; b += THREADS) hist[b] = 0u;
  if (tid == 0) s_ncand = 0;
  pdl_wait();
  __syncthreads();

  // 1. bins + histogram: one vectorised read of the row
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
  const int n4 = vec ? (n >> 2) : 0;
  {
    const float4* row4 = reinterpret_cast<const float4*>(row);
    int i = tid;
    for (; i + 3 * THREADS < n4; i += 4 * THREADS) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(row4 + i + u * THREADS);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b0 = score_bin(v[u].x), b1 = score_bin(v[u].y);
        const int b2 = score_bin(v[u].z), b3 = score_bin(v[u].w);
        uint2 packed;
        packed.x = (uint32_t)b0 | ((uint32_t)b1 << 16);
        packed.y = (uint32_t)b2 | ((uint32_t)b3 << 16);
        *reinterpret_cast<uint2*>(sbin + 4 * (i + u * THREADS)) = packed;
        atomicAdd(&hist[b0], 1u);
        atomicAdd(&hist[b1], 1u);
        atomicAdd(&hist[b2], 1u);
        atomicAdd(&hist[b3], 1u);
      }
    }
    for (; i < n4; i += THREADS) {
      const float4 v = __ldcg(row4 + i);
      const int b0 = score_bin(v.x), b1 = score_bin(v.y);
      const int b2 = score_bin(v.z), b3 = score_bin(v.w);
      uint2 packed;
      packed.x = (uint32_t)b0 | ((uint32_t)b1 << 16);
      packed.y = (uint32_t)b2 | ((uint32_t)b3 << 16);
      *reinterpret_cast<uint2*>(sbin + 4 * i) = packed;
      atomicAdd(&hist[b0], 1u);
      atomicAdd(&hist[b1], 1u);
      atomicAdd(&hist[b2], 1u);
      atomicAdd(&hist[b3], 1u);
    }
    for (int t = 4 * n4 + tid; t < n; t += THREADS) {
      const int b = score_bin(__ldcg(row + t));
      sbin[t] = (uint16_t)b;
      atomicAdd(&hist[b], 1u);
    }
  }
  __syncthreads();

  // 2. boundary bin: thread i owns bins [top - 8i - 7, top - 8i] (descending)
  {
    const int hi_bin = NBINS - 1 - BINS_PER_THREAD * tid;
    unsigned hb[BINS_PER_THREAD];
    int lsum = 0;
#pragma unroll
    for (int q = 0; q < BINS_PER_THREAD; ++q) {
      hb[q] = hist[hi_bin - q];
      lsum += (int)hb[q];
    }
    int total;
    const int excl = block_exclusive_scan<THREADS>(lsum, wsum, total);
    if (excl < w && w <= excl + lsum) {
      int cum = excl;
#pragma unroll
      for (int q = 0; q < BINS_PER_THREAD; ++q) {
        if (cum < w && cum + (int)hb[q] >= w) {
          s_bstar = hi_bin - q;
          s_need = w - cum;
        }
        cum += (int)hb[q];
      }
    }
  }
  __syncthreads();
  const int bstar = s_bstar, need = s_need;
  const int ncand_total = (int)hist[bstar];
  if (ncand_total > CAND_CAP) {  // many equal or near-equal scores: exact radix path
    __syncthreads();             // every thread has read hist[b*] before it is reused
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }

  // 3. one pass over the staged bins: per 32-position chunk q, the mask of
  //    positions in a bin above b* (kept) and of members of b* (candidates)
  const int nq = (n + 31) >> 5;
  uint32_t* hmask = reinterpret_cast<uint32_t*>(sbin + ((n + 7) & ~7));  // [nq]
  uint32_t* emask = hmask + nq;                                          // [nq]
  for (int q = warp; q < nq; q += WARPS) {
    const int t = q * 32 + lane;
    const int bv = (t < n) ? (int)sbin[t] : -1;
    const unsigned hi = __ballot_sync(0xffffffffu, bv > bstar);
    const unsigned eq = __ballot_sync(0xffffffffu, bv == bstar);
    if (lane == 0) {
      hmask[q] = hi;
      emask[q] = eq;
    }
  }
  __syncthreads();
  if (need == ncand_total) {
    // every member of b* is kept
    for (int q = tid; q < nq; q += THREADS) hmask[q] |= emask[q];
  } else {
    // rank the members of b* exactly by (score desc, position asc)
    for (int q = tid; q < nq; q += THREADS) {
      unsigned em = emask[q];
      while (em) {
        const int b = __ffs(em) - 1;
        em &= em - 1;
        const int slot = atomicAdd(&s_ncand, 1);
        const int t = q * 32 + b;
        cand_t[slot] = t;
        cand_s[slot] = __ldcg(row + t);
      }
    }
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
      if (rank < need) atomicOr(&hmask[ti >> 5], 1u << (ti & 31));
    }
  }
  __syncthreads();

  // 4. ordered emission: chunk q's kept positions go to the output slots after
  //    those of chunks 0..q-1 (a block-wide scan over the chunk counts)
  int carry = 0;
  for (int q0 = 0; q0 < nq; q0 += THREADS) {
    const int q = q0 + tid;
    const unsigned km = (q < nq) ? hmask[q] : 0u;
    int total;
    const int ex = block_exclusive_scan<THREADS>(__popc(km), wsum, total);
    so.emit_word(carry + ex, km, q * 32);
    carry += total;
  }
}

// ---------------------------------------------------------------------------
// Rows of n <= THREADS * 32 scores, n a multiple of 4.  Warp j owns the
// contiguous segment [j*seg, (j+1)*seg) (seg a multiple of 128), in chunks of
// 128 positions; lane l owns positions 4l..4l+3 of every chunk, so every load
// is a coalesced float4 (512 bytes per warp), four in flight per thread.
// The w-th largest of the per-thread maxima is a lower bound on the w-th
// largest score (the w threads holding the largest maxima own w distinct
// scores at least that large), so every kept score lies in a bin at or above
// the bin b_L of that maximum; b_L is found by bisection over the bins with
// block-wide counts (no histogram).  Only threads whose maximum reaches b_L
// read their scores again; the scores of bin >= b_L (typically a few more than
// w) become candidates, each taking a slot with a shared-memory atomic, packed
// as 64-bit keys (score key, complemented position) so that one integer
// compare orders them by (score desc, position asc).  A candidate is kept when
// fewer than w keys exceed its own; when fewer than w candidates lie above the
// boundary bin (the usual case) those are all kept and only the boundary bin's
// few candidates are ranked.  Kept positions are set in a position bitmap, and
// a block-wide scan over the bitmap words puts them out in ascending order.
// Rows where the bound leaves more than RCAP candidates (many equal scores), or
// with fewer than w non-empty threads, use the exact radix select.
// ---------------------------------------------------------------------------
constexpr int CHUNKS_MAX = 8;  // 128-position chunks per warp
constexpr int BOUND_N_MAX = THREADS * 4 * CHUNKS_MAX;
constexpr int RCAP = 1024;
static_assert(BOUND_N_MAX / 32 == THREADS, "one position-bitmap word per thread");

__device__ __forceinline__ unsigned long long cand_key(float x, int p) {
  return ((unsigned long long)score_key(x) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)p);
}

__global__ void __launch_bounds__(THREADS, 7)
select_topw_bound_kernel(const float* __restrict__ S, int n, int k, int w,
                         int32_t* __restrict__ idx, int32_t* __restrict__ mcount,
                         int32_t* __restrict__ slots) {
  pdl_trigger();
  __shared__ unsigned hist[256];  // radix fallback
  __shared__ __align__(16) unsigned long long ckey[RCAP];
  __shared__ unsigned kept[THREADS];  // position bitmap, 32 positions per word
  __shared__ int wsum[4 * WARPS];
  __shared__ int s_ncand, s_nedge;

  const int c = blockIdx.x;
  const int bh = blockIdx.y;
  const float* row = S + ((size_t)bh * k + c) * n;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  const SelectOut so{idx + ((size_t)bh * k + c) * w, mcount, slots, bh, c, n, w};
  const int tid = threadIdx.x, warp = tid >> 5;
  const int seg = ((n + WARPS * 128 - 1) / (WARPS * 128)) * 128;  // <= 128 * CHUNKS_MAX
  const int w0 = warp * seg + 4 * (tid & 31);                     // first position of this thread

  kept[tid] = 0u;
  if (tid == 0) { s_ncand = 0; s_nedge = 0; }
  pdl_wait();

  auto load_chunks = [&](int i0, float4 (&v)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u;
      const int p = w0 + 128 * i;
      v[u] = (128 * i < seg && p < n) ? __ldcg(row4 + (p >> 2))
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
  };

  // 1. per-thread maximum
  float m = -INFINITY;
#pragma unroll
  for (int i0 = 0; i0 < CHUNKS_MAX; i0 += 4) {
    float4 v[4];
    load_chunks(i0, v);
#pragma unroll
    for (int u = 0; u < 4; ++u) m = fmaxf(m, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
  }
  const int mbin = w0 < n ? score_bin(m) : -1;

  // 2. b_L = the largest bin b with at least w thread maxima in bins >= b,
  //    by bisection over the bins with block-wide counts (no histogram, no
  //    shared-memory atomics); -1 when fewer than w threads hold scores
  int bl;
  {
    int lo = 0, hi = NBINS - 1;  // invariant: count(>= lo) >= w, count(>= hi + 1) < w
    if (__syncthreads_count(mbin >= 0) < w) {
      bl = -1;
    } else {
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__syncthreads_count(mbin >= mid) >= w) lo = mid;
        else hi = mid - 1;
      }
      bl = lo;
    }
  }

  // 3. candidates: scores of bin >= b_L, read again only by the threads whose
  //    maximum qualifies.  A float compare against a value a little below the
  //    bin's lower edge filters first; the bin itself is only computed for
  //    the few scores that pass.  A candidate above the boundary bin takes a
  //    slot from the front of ckey, one in it a slot from the back (shared
  //    atomics; the ranking below does not depend on the slot order).
  {
    const bool mine = bl >= 0 && mbin >= bl;
    // (finite for bin 0, so that the -inf padding past n never qualifies)
    const float pre = bl > 0 ? (float)bl * (1.0f / 1024.0f) - 1.0f - 1.0e-5f : -3.0e38f;
    if (mine) {
#pragma unroll
      for (int i0 = 0; i0 < CHUNKS_MAX; i0 += 4) {
        float4 v[4];
        load_chunks(i0, v);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (e4[e] >= pre) {
              const int sb = score_bin(e4[e]);
              if (sb >= bl) {
                const int p = w0 + 128 * (i0 + u) + e;
                if (sb > bl) {
                  const int slot = atomicAdd(&s_ncand, 1);
                  if (slot < RCAP) ckey[slot] = cand_key(e4[e], p);
                } else {
                  const int slot = atomicAdd(&s_nedge, 1);
                  if (slot < RCAP) ckey[RCAP - 1 - slot] = cand_key(e4[e], p);
                }
              }
            }
          }
        }
      }
    }
  }
  __syncthreads();
  const int nA = s_ncand, nE = s_nedge;
  if (bl < 0 || nA + nE > RCAP) {
    radix_select_row(row, n, w, so, hist, wsum);  // uniform branch
    return;
  }

  // 4. kept: fewer than w candidate keys above its own.  Usually fewer than w
  //    scores lie above the boundary bin: those are all kept, and only the
  //    boundary bin's candidates are ranked, among themselves, for the
  //    remaining w - nA places.  Otherwise every candidate is ranked.
  {
    const unsigned long long* cE = ckey + (RCAP - nE);
    const bool above_all = nA < w;
    if (above_all) {
      for (int i = tid; i < nA; i += THREADS) {
        const int p = (int)(0xFFFFFFFFu - (uint32_t)ckey[i]);
        atomicOr(&kept[p >> 5], 1u << (p & 31));
      }
    }
    const int need = above_all ? w - nA : w;
    const int total = above_all ? nE : nA + nE;
    for (int i = tid; i < total; i += THREADS) {
      const unsigned long long ki = (above_all || i >= nA) ? cE[above_all ? i : i - nA] : ckey[i];
      int rank = 0;
      for (int j = 0; j < nE; ++j) rank += cE[j] > ki;
      if (!above_all)
        for (int j = 0; j < nA; ++j) rank += ckey[j] > ki;
      if (rank < need) {
        const int p = (int)(0xFFFFFFFFu - (uint32_t)ki);
        atomicOr(&kept[p >> 5], 1u << (p & 31));
      }
    }
  }
  __syncthreads();

  // 5. ordered emission: word q's kept positions go to the output slots after
  //    those of words 0..q-1
  {
    const unsigned km = kept[tid];
    int total;
    const int o = block_exclusive_scan<THREADS>(__popc(km), wsum, total);
    so.emit_word<4>(o, km, tid * 32);
  }
}

// ---------------------------------------------------------------------------
// Long rows (n a multiple of 4, up to GROUP_N_MAX): group maxima.  The bound
// of the kernel above, with groups of GSIZE consecutive scores in place of a
// thread's scores, so that it stays tight for any n:
//   1. one streaming read of the row (two float4 per group, four groups in
//      flight per thread): the bin of every group's maximum goes to shared
//      memory (u16); the bins at or above the smallest thread maximum (a
//      lower bound on the w-th largest group maximum when w <= 256) are
//      counted in a 2048-bin histogram, one shared atomic per distinct bin of
//      a warp;
//   2. b_L = the largest bin with at least w group maxima in bins >= b_L: the
//      w groups holding the largest maxima own w distinct scores at least
//      that large, so every kept score lies in a bin >= b_L (a block scan of
//      the histogram from the top bin down);
//   3. only the groups whose maximum reaches b_L are read again (from L2,
//      right after the first pass): they are listed first, then read one per
//      thread with every load in flight; their scores of bin >= b_L become the
//      candidates (typically a few more than w), packed as 64-bit keys (score
//      key, complemented position), appended with one shared atomic per warp;
//   4. a candidate is kept when fewer than w candidate keys exceed its own;
//      when fewer than w scores lie above the boundary bin (the usual case)
//      those are all kept and only the boundary bin's few candidates are
//      ranked, among themselves; kept positions go into a position bitmap;
//   5. a block scan over the bitmap words (consecutive words per thread) puts
//      them out in ascending order.
// Rows where fewer than w groups exist or the bound leaves more than GCAP
// candidates (many equal scores) use the exact radix select.
// Shared memory: about n/4 + n/8 bytes + 16 KB, so several CTAs share an SM
// and the first pass keeps enough loads in flight to stream at HBM speed.
// ---------------------------------------------------------------------------
constexpr int GSIZE = GROUP_SIZE;
constexpr int GCAP = 1024;
constexpr int GROUP_N_MAX = 262144;

// Shared memory: the group bins [NG] (u16), whose space the position bitmap
// [NW] takes over once the qualifying groups are listed, then the candidate
// keys and the qualifying-group list.
inline size_t group_region0_bytes(int n) {
  const size_t ng = (size_t)(n + GSIZE - 1) / GSIZE, nw = (size_t)(n + 31) / 32;
  return std::max((ng * 2 + 15) & ~(size_t)15, (nw * 4 + 15) & ~(size_t)15);
}
inline size_t group_smem_bytes(int n) {
  return group_region0_bytes(n) + (size_t)(GCAP + 1) * 8 + (size_t)GCAP * 4;
}

// (5 CTAs an SM: about 37 KB of shared memory each at n = 65536)
template <bool FROM_GBINS>
__global__ void __launch_bounds__(THREADS, 5)
select_topw_group_kernel(const float* __restrict__ S, const uint16_t* __restrict__ gbins, int n,
                         int k, int w, int32_t* __restrict__ idx, int32_t* __restrict__ mcount,
                         int32_t* __restrict__ slots) {
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t gsm[];
  __shared__ unsigned hist[NBINS];
  __shared__ int wsum[4 * WARPS];
  __shared__ int s_bl, s_ncand, s_nq, s_nq2;
  const int NG = (n + GSIZE - 1) / GSIZE;
  const int NW = (n + 31) / 32;
  const int R0 = max((NG * 2 + 15) & ~15, (NW * 4 + 15) & ~15);
  uint16_t* gbin = reinterpret_cast<uint16_t*>(gsm);  // [NG], until the groups are listed
  unsigned* kept = reinterpret_cast<unsigned*>(gsm);  // [NW], after that
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(gsm + R0);
  int* qlist = reinterpret_cast<int*>(ckey + GCAP + 1);  // [GCAP] qualifying groups

  const int c = blockIdx.x;
  const int bh = blockIdx.y;
  const float* row = S + ((size_t)bh * k + c) * n;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  const SelectOut so{idx + ((size_t)bh * k + c) * w, mcount, slots, bh, c, n, w};
  const int tid = threadIdx.x, lane = tid & 31;

  for (int i = tid; i < NBINS; i += THREADS) hist[i] = 0u;
  if (tid == 0) { s_ncand = 0; s_nq = 0; s_nq2 = 0; s_bl = -1; }
  pdl_wait();
  __syncthreads();

  const int n4 = n >> 2;
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  int b0 = 0;
  if constexpr (FROM_GBINS) {
    // 1. the group bins the score kernel wrote: 8 groups per 16-byte load,
    //    copied to shared memory (the padding past NG comes along, unused);
    //    a thread's largest bin feeds the prefilter below
    const uint4* src = reinterpret_cast<const uint4*>(gbins + ((size_t)bh * k + c) * gbin_stride(n));
    uint4* dst = reinterpret_cast<uint4*>(gbin);
    const int NV = (NG + 7) / 8;
    int tb = -1;
    for (int v0 = tid; v0 < NV; v0 += 4 * THREADS) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = v0 + u * THREADS;
        v[u] = i < NV ? __ldcg(src + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = v0 + u * THREADS;
        if (i < NV) {
          dst[i] = v[u];
          const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (8 * i + e < NG) tb = max(tb, (int)((wv[e >> 1] >> (16 * (e & 1))) & 0xffffu));
        }
      }
    }
    // Prefilter: the min(THREADS, NV) threads that own groups own distinct
    // groups, each one of bin >= the smallest thread maximum b0; with w no
    // more than them, b_L >= b0, and only bins >= b0 need counting.
    __shared__ int wmin_b[WARPS];
    {
      int tm = tb >= 0 ? tb : NBINS;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tm = min(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      if (lane == 0) wmin_b[tid >> 5] = tm;
    }
    __syncthreads();
    if (w <= min(THREADS, NV)) {
      int t0 = wmin_b[0];
      for (int i = 1; i < WARPS; ++i) t0 = min(t0, wmin_b[i]);
      b0 = t0;
    }
  } else {
    // 1. bins of the group maxima (and this thread's largest group maximum)
    float tmax = -INFINITY;
    for (int g0 = tid; g0 < NG; g0 += 4 * THREADS) {
      float4 v[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * THREADS;
        v[u][0] = (g < NG && 2 * g < n4) ? __ldcg(row4 + 2 * g) : ninf;
        v[u][1] = (g < NG && 2 * g + 1 < n4) ? __ldcg(row4 + 2 * g + 1) : ninf;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * THREADS;
        if (g < NG) {
          const float m = fmaxf(fmaxf(fmaxf(v[u][0].x, v[u][0].y), fmaxf(v[u][0].z, v[u][0].w)),
                                fmaxf(fmaxf(v[u][1].x, v[u][1].y), fmaxf(v[u][1].z, v[u][1].w)));
          gbin[g] = (uint16_t)score_bin(m);
          tmax = fmaxf(tmax, m);
        }
      }
    }
    // Prefilter: when every thread owns a group and w <= THREADS, the smallest
    // thread maximum T0 is at most the w-th largest group maximum (the THREADS
    // threads own THREADS distinct groups with maxima >= T0), so b_L >= bin(T0)
    // and only group maxima in bins >= bin(T0) need counting.  This keeps the
    // histogram small and its atomics spread over few, uncontended bins.
    __shared__ float wmin[WARPS];
    {
      float tm = tmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tm = fminf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      if (lane == 0) wmin[tid >> 5] = tm;
    }
    __syncthreads();
    if (w <= THREADS && NG >= THREADS) {
      float t0 = wmin[0];
      for (int i = 1; i < WARPS; ++i) t0 = fminf(t0, wmin[i]);
      b0 = score_bin(t0);
    }
  }
  // counts of the bins >= b0: two bins per 32-bit shared load, a shared
  // atomic for each bin at or above b0 (few of them, spread over many bins;
  // a bin outside the histogram, which only an unfinished score kernel
  // could leave, is not counted)
  {
    const uint32_t* gb2 = reinterpret_cast<const uint32_t*>(gbin);
    for (int v = tid; 2 * v < NG; v += THREADS) {
      const uint32_t pr = gb2[v];
      const int lo = (int)(pr & 0xffffu), hi = (int)(pr >> 16);
      if (lo >= b0 && lo < NBINS) atomicAdd(&hist[lo], 1u);
      if (2 * v + 1 < NG && hi >= b0 && hi < NBINS) atomicAdd(&hist[hi], 1u);
    }
  }
  __syncthreads();

  // 2. b_L: thread i owns bins [top - 8i - 7, top - 8i] (descending)
  {
    const int hi_bin = NBINS - 1 - BINS_PER_THREAD * tid;
    unsigned hb[BINS_PER_THREAD];
    int lsum = 0;
#pragma unroll
    for (int q = 0; q < BINS_PER_THREAD; ++q) {
      hb[q] = hist[hi_bin - q];
      lsum += (int)hb[q];
    }
    int total;
    const int excl = block_exclusive_scan<THREADS>(lsum, wsum, total);
    if (excl < w && w <= excl + lsum) {
      int cum = excl;
#pragma unroll
      for (int q = 0; q < BINS_PER_THREAD; ++q) {
        if (cum < w && cum + (int)hb[q] >= w) s_bl = hi_bin - q;
        cum += (int)hb[q];
      }
    }
  }
  __syncthreads();
  const int bl = s_bl;
  if (bl < 0) {  // fewer than w groups: exact radix path (uniform)
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }

  // 3. candidates from the groups whose maximum reaches b_L: first the list of
  //    those groups (shared memory only: each warp counts its groups with
  //    ballots, reserves its range with one atomic, then writes them), then
  //    two groups per thread, every load in flight at once
  {
    const unsigned lt = (1u << lane) - 1u;
    int wcount = 0;
    for (int g0 = 0; g0 < NG; g0 += THREADS) {
      const int g = g0 + tid;
      wcount += __popc(__ballot_sync(0xffffffffu, g < NG && (int)gbin[g] >= bl));
    }
    int base = 0;
    if (lane == 0 && wcount != 0) base = atomicAdd(&s_nq, wcount);
    base = __shfl_sync(0xffffffffu, base, 0);
    for (int g0 = 0; g0 < NG; g0 += THREADS) {
      const int g = g0 + tid;
      const bool ok = g < NG && (int)gbin[g] >= bl;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      const int slot = base + __popc(bal & lt);
      if (ok && slot < GCAP) qlist[slot] = g;
      base += __popc(bal);
    }
  }
  __syncthreads();
  const int nq = s_nq;
  if (nq > GCAP) {  // many groups in the boundary bin: exact radix path (uniform)
    radix_select_row(row, n, w, so, hist, wsum);
    return;
  }
  // the group bins are read no more: their space becomes the position bitmap
  // (cleared here, first written after the barrier that ends the candidates)
  for (int i = tid; i < NW; i += THREADS) kept[i] = 0u;
  // candidates above the boundary bin fill ckey from the front (nA), those in
  // it from the back (nE)
  {
    // groups a thread loads at once: two on the long rows that come with
    // precomputed group bins, one on the shorter rows below them
    constexpr int GPT = FROM_GBINS ? 2 : 1;
    const float pre = bl > 0 ? (float)bl * (1.0f / 1024.0f) - 1.0f - 1.0e-5f : -3.0e38f;
    for (int i0 = 0; i0 < nq; i0 += GPT * THREADS) {
      uint32_t ca[GPT], ce[GPT];  // above the boundary bin / in it
      float x[GPT][GSIZE];
      int g[GPT];
#pragma unroll
      for (int u = 0; u < GPT; ++u) {
        ca[u] = 0u;
        ce[u] = 0u;
        g[u] = 0;
        const int i = i0 + u * THREADS + tid;
        float4 a = ninf, b = ninf;
        if (i < nq) {
          g[u] = qlist[i];
          if (2 * g[u] < n4) a = __ldcg(row4 + 2 * g[u]);
          if (2 * g[u] + 1 < n4) b = __ldcg(row4 + 2 * g[u] + 1);
        }
        x[u][0] = a.x; x[u][1] = a.y; x[u][2] = a.z; x[u][3] = a.w;
        x[u][4] = b.x; x[u][5] = b.y; x[u][6] = b.z; x[u][7] = b.w;
      }
#pragma unroll
      for (int u = 0; u < GPT; ++u) {
#pragma unroll
        for (int e = 0; e < GSIZE; ++e) {
          if (x[u][e] >= pre) {
            const int sb = score_bin(x[u][e]);
            if (sb > bl) ca[u] |= 1u << e;
            else if (sb == bl) ce[u] |= 1u << e;
          }
        }
      }
      int sa, se;
      {
        int cnt = 0;  // both counts in one scan
#pragma unroll
        for (int u = 0; u < GPT; ++u) cnt += __popc(ca[u]) | (__popc(ce[u]) << 16);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int wtot = __shfl_sync(0xffffffffu, incl, 31);
        int baseA = 0, baseE = 0;
        if (lane == 31) {
          if (wtot & 0xffff) baseA = atomicAdd(&s_ncand, wtot & 0xffff);
          if (wtot >> 16) baseE = atomicAdd(&s_nq2, wtot >> 16);
        }
        baseA = __shfl_sync(0xffffffffu, baseA, 31);
        baseE = __shfl_sync(0xffffffffu, baseE, 31);
        const int ex = incl - cnt;
        sa = baseA + (ex & 0xffff);
        se = baseE + (ex >> 16);
      }
#pragma unroll
      for (int u = 0; u < GPT; ++u) {
#pragma unroll
        for (int e = 0; e < GSIZE; ++e) {
          if ((ca[u] >> e) & 1u) {
            if (sa < GCAP) ckey[sa] = cand_key(x[u][e], g[u] * GSIZE + e);
            ++sa;
          } else if ((ce[u] >> e) & 1u) {
            if (se < GCAP) ckey[GCAP - 1 - se] = cand_key(x[u][e], g[u] * GSIZE + e);
            ++se;
          }
        }
      }
    }
  }
  __syncthreads();
  const int nA = s_ncand, nE = s_nq2;
  if (nA + nE > GCAP) {
    radix_select_row(row, n, w, so, hist, wsum);  // uniform branch
    return;
  }

  // 4. kept: fewer than w candidate keys above its own.  Usually fewer than w
  //    scores lie above the boundary bin: those are all kept, and only the
  //    boundary bin's candidates are ranked, among themselves, for the
  //    remaining w - nA places.  Otherwise every candidate is ranked.
  {
    const unsigned long long* cE = ckey + (GCAP - nE);
    const bool above_all = nA < w;
    if (above_all) {
      for (int i = tid; i < nA; i += THREADS) {
        const int p = (int)(0xFFFFFFFFu - (uint32_t)ckey[i]);
        atomicOr(&kept[p >> 5], 1u << (p & 31));
      }
    }
    const int need = above_all ? w - nA : w;
    const int total = above_all ? nE : nA + nE;
    for (int i = tid; i < total; i += THREADS) {
      const unsigned long long ki = (above_all || i >= nA) ? cE[above_all ? i : i - nA] : ckey[i];
      int rank = 0;
      for (int j = 0; j < nE; ++j) rank += cE[j] > ki;
      if (!above_all)
        for (int j = 0; j < nA; ++j) rank += ckey[j] > ki;
      if (rank < need) {
        const int p = (int)(0xFFFFFFFFu - (uint32_t)ki);
        atomicOr(&kept[p >> 5], 1u << (p & 31));
      }
    }
  }
  __syncthreads();

  // 5. ordered emission: thread tid takes words [tid*WPT, tid*WPT + WPT)
  {
    const int WPT = (NW + THREADS - 1) / THREADS;
    const int q0 = tid * WPT;
    int cnt = 0;
    for (int q = q0; q < q0 + WPT && q < NW; ++q) cnt += __popc(kept[q]);
    int total;
    const int o = block_exclusive_scan<THREADS>(cnt, wsum, total);
    so.emit_words(o, kept, q0, min(q0 + WPT, NW));
  }
}

}  // namespace

// Group bins from the score epilogue cost that kernel a shuffle reduction per
// 8 columns; they pay only where the select would otherwise stream long rows:
// measured on B300, n = 65536 (256 KiB rows) gains about 75 us a forward at
// H = 8, k = 256, while n = 8192 and n = 12288 lose 8 and 15 us.
constexpr int GROUP_BINS_MIN_N = 32768;

bool select_wants_group_bins(int n) {
  return n >= GROUP_BINS_MIN_N && n <= GROUP_N_MAX && (n & 3) == 0;
}

cudaError_t launch_select(const float* S, const uint16_t* gbins, int BH, int n, int k, int w,
                          int32_t* idx, int32_t* mcount, int32_t* slots, cudaStream_t s) {
  dim3 grid(k, BH);
  const int staged = n <= MAX_STAGED_BINS ? 1 : 0;
  // staged bins (u16, padded to 16 bytes) + two chunk masks per 32 positions
  auto stage_bytes = [](int nn) {
    return (size_t)((nn + 7) & ~7) * sizeof(uint16_t) + 2 * (size_t)((nn + 31) / 32) * 4;
  };
  const size_t smem = staged ? stage_bytes(n) : 0;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(select_topw_kernel), (int)stage_bytes(MAX_STAGED_BINS));
  if (e != cudaSuccess) return e;
  if (gbins != nullptr && n <= GROUP_N_MAX && (n & 3) == 0) {
    const size_t gsmem = group_smem_bytes(n);
    e = set_smem_limit(reinterpret_cast<const void*>(select_topw_group_kernel<true>), (int)gsmem);
    if (e != cudaSuccess) return e;
    launch_begin(K_SELECT, s);
    e = launch_pdl(select_topw_group_kernel<true>, grid, dim3(THREADS), gsmem, s, S, gbins, n, k,
                   w, idx, mcount, slots);
    launch_end(K_SELECT, s);
    return e;
  }
  if (n <= BOUND_N_MAX && (n & 3) == 0 && w <= THREADS) {
    launch_begin(K_SELECT, s);
    e = launch_pdl(select_topw_bound_kernel, grid, dim3(THREADS), 0, s, S, n, k, w, idx, mcount,
                   slots);
    launch_end(K_SELECT, s);
    return e;
  }
  if (n <= GROUP_N_MAX && (n & 3) == 0) {
    const size_t gsmem = group_smem_bytes(n);
    e = set_smem_limit(reinterpret_cast<const void*>(select_topw_group_kernel<false>), (int)gsmem);
    if (e != cudaSuccess) return e;
    launch_begin(K_SELECT, s);
    e = launch_pdl(select_topw_group_kernel<false>, grid, dim3(THREADS), gsmem, s, S, nullptr, n,
                   k, w, idx, mcount, slots);
    launch_end(K_SELECT, s);
    return e;
  }
  launch_begin(K_SELECT, s);
  e = launch_pdl(select_topw_kernel, grid, dim3(THREADS), smem, s, S, n, k, w, idx, mcount, slots,
                 staged);
  launch_end(K_SELECT, s);
  return e;
}

}  // namespace rt
