// In-cluster softmax attention for clusters of 128 < w <= 256 members (two
// 128-row tiles), bf16 inputs, fp32 accumulation on tcgen05 tensor cores.
//
// "Efficient Content-Based Sparse Attention with Routing Transformers":
// §3 (softmax attention, autoregressive masking) restricted by §4 to the
// query/key pairs of one cluster.  Members are listed in ascending position
// order, so the causal mask on original positions is the lower triangle in
// slot order (diagonal included).  Queries double as keys (shared QK).
//
// One CTA of 256 threads per cluster holds the whole cluster: its (up to) 256
// member rows of Q -- which are also the keys -- and of V are gathered once
// with 16-byte cp.async into 128-byte-swizzled rows ([D/64 blocks][256 rows]
// [128 bytes]), read as the K-major operands of S = Q K^T and the MN-major
// operand of O = P V.  Both row tiles' scores go to TMEM at once (tile 0:
// columns 0.., tile 1: columns 256..; the full 512 columns), so each row's
// softmax sees its whole row: no online rescaling.  Warps 0-3 take tile 0's
// rows, warps 4-7 tile 1's (the TMEM lane quadrant of warp w is w % 4), one
// thread per row: the row's maximum, exp2 of the visible columns, P (bf16)
// into shared memory (tile 1's over Q, which S no longer needs) with the row
// sums of exactly those bf16 weights, then O = P V into the score columns, the
// O rows divided by their sums and staged over Q and V as
// 128-byte-swizzled boxes: one bulk tensor store per 32 features writes the
// cluster's slot rows to `yslot` (fp32), while the warps copy the rows of
// positions in exactly one cluster to `out` (bf16).  Chunks of 16 keys that
// every row of a warp sees skip the mask.  Every mbarrier wait is bounded; one
// that runs out sets the device status word, waits (bounded again) for the
// CTA's own MMAs, gives back TMEM and returns.
#include "attn_common.cuh"

namespace rt {
namespace {

using namespace attn;
constexpr int PR_THREADS = 256;
constexpr int NR = 256;  // rows per cluster (w padded to two tiles)
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000 * 1000;  // 0.2 s

template <int D>
struct PairSmem {
  static constexpr int QB = NR * D * 2;      // Q (= K) rows, swizzled
  static constexpr int VB = NR * D * 2;      // V rows, swizzled
  static constexpr int PB = ROWS * NR * 2;   // P of one tile: 128 rows x 256 keys, bf16
  static constexpr int Q_OFF = 0;
  static constexpr int V_OFF = QB;
  static constexpr int P0_OFF = QB + VB;
  // tile 1's P goes over Q once the scores are done when it fits there
  static constexpr int P1_OFF = QB >= PB ? Q_OFF : P0_OFF + PB;
  static constexpr int BYTES = (QB >= PB ? P0_OFF + PB : P1_OFF + PB);
  static_assert(QB + VB >= NR * D * 4, "the output staging fits over Q and V");
};

// Gather NR rows (positions pos[r], -1 = zero row) of D bf16 into the
// 128-byte-swizzled layout [D/64][NR][128 B]; a warp instruction moves four
// whole 128-byte row pieces.
template <int D>
__device__ __forceinline__ void gather_rows_sw128(uint8_t* dst, const bf16* __restrict__ src,
                                                  const int* pos) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int KB = D / 64;
  constexpr int ITEMS = (NR / 4) * KB;
  const uint32_t base = tc::smem_u32(dst);
  const int jj = lane & 7;
  for (int it = warp; it < ITEMS; it += PR_THREADS / 32) {
    const int kb = it % KB;
    const int r = (it / KB) * 4 + (lane >> 3);
    const int p = pos[r];
    const uint32_t off = kb * (NR * 128) + r * 128 + ((jj ^ (r & 7)) << 4);
    const bf16* g = src + (size_t)(p < 0 ? 0 : p) * D + kb * 64 + jj * 8;
    cp_async16(base + off, g, p >= 0);
  }
}

template <int D>
__global__ void __launch_bounds__(PR_THREADS, 1)
attention_pair_kernel(const __grid_constant__ CUtensorMap ymap, const bf16* __restrict__ q,
                      const bf16* __restrict__ v, int n, int k, int w,
                      int causal, float scale_log2, const int32_t* __restrict__ idx,
                      const int32_t* __restrict__ mcount, bf16* __restrict__ out,
                      float* __restrict__ yslot, unsigned int* __restrict__ err,
                      uint64_t fault_ns) {
  using L = PairSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int pos_s[NR], m_s[NR];

  pdl_trigger();
  pdl_wait();
  // the injected test timeout returns here: nothing is in flight, no TMEM held
  if (injected_wait_timeout(fault_ns, err)) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, bh = blockIdx.y;
  const int32_t* list = idx + ((size_t)bh * k + c) * w;
  const bf16* q_bh = q + (size_t)bh * n * D;
  const bf16* v_bh = v + (size_t)bh * n * D;

  // member positions and membership counts of the cluster's slots
  {
    int p = tid < w ? __ldcg(list + tid) : -1;
    if ((unsigned)p >= (unsigned)n) p = -1;  // defensive
    pos_s[tid] = p;
    m_s[tid] = p >= 0 ? __ldcg(mcount + (size_t)bh * n + p) : 0;
  }
  if (tid == 0) {
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  __syncthreads();
  gather_rows_sw128<D>(sm + L::Q_OFF, q_bh, pos_s);
  gather_rows_sw128<D>(sm + L::V_OFF, v_bh, pos_s);
  cp_async_commit();
  cp_async_wait_all();
  tc::fence_proxy_async_smem();  // the rows are visible to the MMA
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  // keys each tile's rows can see: tile 0 (slots < 128) sees keys < 128 when
  // causal; otherwise every tile sees all 256 (keys >= w are zero rows, masked)
  const int n0 = causal ? ROWS : NR;
  if (tid == 0) {
    const uint32_t qa = tc::smem_u32(sm + L::Q_OFF);
    const uint32_t idesc0 = tc::idesc_f16(ROWS, n0, true, false, false);
    const uint32_t idesc1 = tc::idesc_f16(ROWS, NR, true, false, false);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t kofs = (kk / 4) * (NR * 128) + (kk % 4) * 32;
        const uint64_t ad = tc::smem_desc_sw128(qa + t * (ROWS * 128) + kofs, 1024);
        const uint64_t bd = tc::smem_desc_sw128(qa + kofs, 1024);
        tc::mma_f16_ss(tmem + t * 256, ad, bd, t == 0 ? idesc0 : idesc1, kk > 0 ? 1u : 0u);
      }
    }
    tc::mma_commit(&bar_s);
  }
  __syncwarp();
  bool ok = tc::mbar_wait_bounded(&bar_s, 0, WAIT_LIMIT_NS);
  if (!ok && lane == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
  if (__syncthreads_or(!ok)) {
    // give the MMAs a second bounded wait before TMEM is given back
    tc::mbar_wait_bounded(&bar_s, 0, WAIT_LIMIT_NS);
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
    return;
  }
  tc::tc_fence_after_sync();

  // ---- softmax of this thread's row -----------------------------------------
  const int t = warp >> 2;             // row tile
  const int r = 32 * (warp & 3) + lane;  // row within the tile == TMEM lane
  const int slot = t * ROWS + r;
  const bool row_valid = slot < w && pos_s[slot] >= 0;
  const uint32_t t_row = tmem + t * 256 + ((uint32_t)(32 * (warp & 3)) << 16);
  const int kt = t == 0 ? n0 : NR;  // keys of this tile's P
  int jmax = causal ? slot + 1 : w;
  if (jmax > w) jmax = w;
  if (!row_valid) jmax = 0;
  const int whi = __reduce_max_sync(0xffffffffu, jmax);
  const int ch_hi = (whi + 15) >> 4;
  // keys every valid row of the warp sees: those chunks need no mask (an
  // invalid row's values are never stored)
  const int fhi = __reduce_min_sync(0xffffffffu, row_valid ? jmax : NR);
  float mrow = -INFINITY;
  for (int ch = 0; ch < ch_hi; ch += 2) {
    uint32_t rr[2][16];
    tc::tmem_ld16(t_row + ch * 16, rr[0]);
    if (ch + 1 < ch_hi) tc::tmem_ld16(t_row + (ch + 1) * 16, rr[1]);
    tc::tmem_ld_wait();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int c = ch + hh;
      if (c >= ch_hi) break;
      if (c * 16 + 16 <= fhi) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) mrow = fmaxf(mrow, __uint_as_float(rr[hh][jj]));
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          if (c * 16 + jj < jmax) mrow = fmaxf(mrow, __uint_as_float(rr[hh][jj]));
      }
    }
  }
  const float neg_m = (mrow == -INFINITY) ? 0.0f : -mrow * scale_log2;
  float lsum = 0.0f;  // the sum of this row's bf16 weights
  // P row: K-major core matrices, element (r, key) at (r/8)*(kt*16) +
  // (key/8)*128 + (r%8)*16 + (key%8)*2
  uint8_t* pt = sm + (t == 0 ? L::P0_OFF : L::P1_OFF);
  const uint32_t prow = tc::smem_u32(pt) + (r >> 3) * (kt * 16) + (r & 7) * 16;
  auto store_chunk = [&](int ch, const uint32_t (&pk)[8]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t addr = prow + (2 * ch + h) * 128;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * h]),
                   "r"(pk[4 * h + 1]), "r"(pk[4 * h + 2]), "r"(pk[4 * h + 3])
                   : "memory");
    }
  };
  {
    const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
    for (int ch = ch_hi; ch < kt / 16; ++ch) store_chunk(ch, zero);
  }
  // P = 2^(S*scale*log2e - max), bf16, and the sum of those bf16 values
#pragma unroll 1
  for (int ch = 0; ch < ch_hi; ch += 2) {
    uint32_t rr[2][16];
    tc::tmem_ld16(t_row + ch * 16, rr[0]);
    if (ch + 1 < ch_hi) tc::tmem_ld16(t_row + (ch + 1) * 16, rr[1]);
    tc::tmem_ld_wait();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int c = ch + hh;
      if (c >= ch_hi) break;
      uint32_t pk[8];
      if (c * 16 + 16 <= fhi) {
#pragma unroll
        for (int jj = 0; jj < 16; jj += 2) {
          const float e0 = tc::exp2_approx(fmaf(__uint_as_float(rr[hh][jj]), scale_log2, neg_m));
          const float e1 = tc::exp2_approx(fmaf(__uint_as_float(rr[hh][jj + 1]), scale_log2, neg_m));
          pk[jj >> 1] = pack_bf16(e0, e1);
          lsum += __uint_as_float(pk[jj >> 1] << 16) + __uint_as_float(pk[jj >> 1] & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; jj += 2) {
          const int col = c * 16 + jj;
          const float e0 =
              col < jmax ? tc::exp2_approx(fmaf(__uint_as_float(rr[hh][jj]), scale_log2, neg_m)) : 0.0f;
          const float e1 =
              col + 1 < jmax ? tc::exp2_approx(fmaf(__uint_as_float(rr[hh][jj + 1]), scale_log2, neg_m))
                             : 0.0f;
          pk[jj >> 1] = pack_bf16(e0, e1);
          lsum += __uint_as_float(pk[jj >> 1] << 16) + __uint_as_float(pk[jj >> 1] & 0xffff0000u);
        }
      }
      store_chunk(c, pk);
    }
  }
  tc::fence_proxy_async_smem();  // P (generic writes) before the MMA reads it
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();

  // ---- O = P V into the score columns -----------------------------------------
  if (tid == 0) {
    const uint32_t va = tc::smem_u32(sm + L::V_OFF);
    const uint32_t idesc_o = tc::idesc_f16(ROWS, D, true, false, true);
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const int ktt = tt == 0 ? n0 : NR;
      const uint32_t pa = tc::smem_u32(sm + (tt == 0 ? L::P0_OFF : L::P1_OFF));
      for (int kk = 0; kk < ktt / 16; ++kk) {
        const uint64_t ad = tc::smem_desc_noswizzle(pa + kk * 256, 128, ktt * 16);
        const uint64_t bd = tc::smem_desc_sw128_mn(va + kk * 2048, NR * 128, 1024);
        tc::mma_f16_ss(tmem + tt * 256, ad, bd, idesc_o, kk > 0 ? 1u : 0u);
      }
    }
    tc::mma_commit(&bar_o);
  }
  __syncwarp();
  ok = tc::mbar_wait_bounded(&bar_o, 0, WAIT_LIMIT_NS);
  if (!ok && lane == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
  if (__syncthreads_or(!ok)) {
    tc::mbar_wait_bounded(&bar_o, 0, WAIT_LIMIT_NS);
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
    return;
  }
  tc::tc_fence_after_sync();

  // ---- O rows divided by their sums: TMEM -> fp32 staging over Q and V (free
  //      now) as bulk-store boxes: D/32 segments of [256 rows][128 bytes],
  //      16-byte chunk q of row s at (q ^ (s % 8)) (128-byte swizzle) ----------
  const float inv_l = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t rr[2][16];
    tc::tmem_ld16(t_row + c0, rr[0]);
    tc::tmem_ld16(t_row + c0 + 16, rr[1]);
    tc::tmem_ld_wait();
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      const int chunk = c0 / 4 + q4;
      const uint32_t* x = &rr[q4 >> 2][4 * (q4 & 3)];
      *reinterpret_cast<float4*>(sm + (chunk >> 3) * (NR * 128) + slot * 128 +
                                 (((chunk & 7) ^ (slot & 7)) << 4)) =
          make_float4(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l,
                      __uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l);
    }
  }
  tc::tc_fence_before_sync();
  tc::fence_proxy_async_smem();  // the staged rows, before the bulk store reads them
  __syncthreads();
  // every slot row of the cluster to `yslot` (fp32), one bulk tensor store per
  // 32 features; rows of positions in exactly one cluster also straight to
  // `out` as bf16, a warp per row
  if (tid == 0) {
#pragma unroll
    for (int sg = 0; sg < D / 32; ++sg)
      tc::tma_store_3d(&ymap, sm + sg * (NR * 128), sg * 32, c * w, bh);
    tc::bulk_commit();
  }
  {
    const int my_s = warp * 32 + lane;
    const int my_p = pos_s[my_s];
    unsigned single = __ballot_sync(0xffffffffu, my_s < w && my_p >= 0 && m_s[my_s] == 1);
    bf16* out_bh = out + (size_t)bh * n * D;
    if constexpr (D == 128) {
      while (single) {
        const int i = __ffs(single) - 1;
        single &= single - 1;
        const int row = warp * 32 + i;
        const int p = __shfl_sync(0xffffffffu, my_p, i);
        const float4 val = *reinterpret_cast<const float4*>(
            sm + (lane >> 3) * (NR * 128) + row * 128 + (((lane & 7) ^ (row & 7)) << 4));
        uint2 u;
        u.x = pack_bf16(val.x, val.y);
        u.y = pack_bf16(val.z, val.w);
        reinterpret_cast<uint2*>(out_bh + (size_t)p * D)[lane] = u;
      }
    } else {  // D == 64: 16 chunks a row, two rows a pass
      const int half = lane >> 4, cc = lane & 15;
      while (single) {
        const int i0 = __ffs(single) - 1;
        single &= single - 1;
        int i1 = -1;
        if (single) {
          i1 = __ffs(single) - 1;
          single &= single - 1;
        }
        const int p0 = __shfl_sync(0xffffffffu, my_p, i0);
        const int p1 = __shfl_sync(0xffffffffu, my_p, i1 < 0 ? i0 : i1);
        const int i = half ? i1 : i0;
        if (i >= 0) {
          const int row = warp * 32 + i;
          const int p = half ? p1 : p0;
          const float4 val = *reinterpret_cast<const float4*>(
              sm + (cc >> 3) * (NR * 128) + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
          uint2 u;
          u.x = pack_bf16(val.x, val.y);
          u.y = pack_bf16(val.z, val.w);
          reinterpret_cast<uint2*>(out_bh + (size_t)p * D)[cc] = u;
        }
      }
    }
  }
  if (tid == 0) tc::bulk_wait_all();  // the bulk stores have read the rows and landed
  tc::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int D>
cudaError_t launch_pair_t(const void* q, const void* v, int BH, int n, int k, int w, int causal,
                          float scale, const int32_t* idx, const int32_t* mcount, void* out,
                          float* yslot, unsigned int* err, cudaStream_t s) {
  const size_t smem = 1024 + (size_t)PairSmem<D>::BYTES;
  auto kern = attention_pair_kernel<D>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  // yslot as [BH][k*w slot rows][D] fp32; a box is one cluster's w rows
  CUtensorMap ymap;
  if (!f32_tensor_map_3d(yslot, D, (unsigned long long)k * w, (unsigned)BH, (unsigned)w, &ymap))
    return cudaErrorInvalidValue;
  launch_begin(K_ATTN_TC, s);
  e = launch_pdl(kern, dim3(k, BH), dim3(PR_THREADS), smem, s, ymap, static_cast<const bf16*>(q),
                 static_cast<const bf16*>(v), n, k, w, causal, scale_log2, idx, mcount,
                 static_cast<bf16*>(out), yslot, err, injected_limit_ns(K_ATTN_TC));
  launch_end(K_ATTN_TC, s);
  return e;
}

}  // namespace

cudaError_t launch_attention_pair(const void* q, const void* v, int BH, int n, int d, int k,
                                  int w, int causal, float scale, const int32_t* idx,
                                  const int32_t* mcount, void* out, float* yslot,
                                  unsigned int* err, cudaStream_t s) {
  return d == 64 ? launch_pair_t<64>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s)
                 : launch_pair_t<128>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s);
}

}  // namespace rt
