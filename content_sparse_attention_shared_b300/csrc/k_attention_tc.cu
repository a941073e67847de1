// In-cluster causal softmax attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM), bf16 inputs, fp32 accumulation.
//
// "Efficient Content-Based Sparse Attention with Routing Transformers":
// §3 (softmax attention, autoregressive masking) restricted by §4 to the
// query/key pairs of one cluster.  Members of a cluster are listed in
// ascending position order, so the causal mask on original positions is the
// lower triangle in slot order (diagonal included).  Queries double as keys
// (shared QK).
//
// This kernel serves clusters wider than two 128-row tiles (w > 256; narrower
// clusters go to k_attention_pipe.cu and k_attention_pair.cu), routing with
// separate queries and keys (any w; queries and keys of a cluster come from
// their own lists, the mask compares original positions), and local
// attention.  Work unit: a
// row tile of 128 consecutive slots of one cluster (TMEM lanes); it walks the
// cluster's key blocks of 128 (causal: up to its own block) with an online
// softmax, the partial P V of each block read back from TMEM and accumulated
// in registers.  Each of the 128 threads owns one row: it reads its S row
// from TMEM, applies the mask and the softmax in registers, writes its P row
// (bf16) to shared memory in the MMA operand layout, and after O = P V reads
// its O row back.  Only the 16-column chunks that hold a valid key for some
// row of the warp are read and exponentiated; the other chunks of P are
// written as zeros.  P reuses the shared memory of the key block once
// S = Q K^T is done, and O reuses S's TMEM columns (128 columns per CTA).
// Rows are gathered from HBM by position with 16-byte cp.async straight into
// the no-swizzle core-matrix layouts (Q/K: K-major; V: MN-major).  The MMA
// completions are waited on with a bounded mbarrier wait; a wait that runs
// out sets the device error word and the CTA gives up its tile.
#include "attn_common.cuh"

namespace rt {
namespace {

using bf16 = __nv_bfloat16;
using attn::ROWS;
using attn::cp_async_commit;
using attn::cp_async_wait_all;
using attn::pack_bf16;
constexpr int THREADS = 128;
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000 * 1000;  // 0.2 s

template <int D>
__device__ __forceinline__ void gather_kmajor(uint8_t* dst, const bf16* src, const int* pos) {
  attn::gather_kmajor<D>(dst, src, pos, threadIdx.x >> 5, THREADS / 32);
}
template <int D>
__device__ __forceinline__ void gather_mnmajor(uint8_t* dst, const bf16* src, const int* pos) {
  attn::gather_mnmajor<D>(dst, src, pos, threadIdx.x >> 5, THREADS / 32);
}

// Shared-memory plan (bytes, after 1 KiB alignment slack):
//   [Q] [K then P: max(K, P)] [V]
template <int D>
struct AttnSmem {
  static constexpr int QB = ROWS * D * 2;
  static constexpr int PB = ROWS * ROWS * 2;
  static constexpr int XB = QB > PB ? QB : PB;
  static constexpr int Q_OFF = 0;
  static constexpr int KP_OFF = QB;  // K block, then P
  static constexpr int V_OFF = QB + XB;
  static constexpr int BYTES = V_OFF + QB;
};

// MODE_CLUSTER:  shared QK, clusters wider than one tile (positions from
//                idx, w > 128).
// MODE_LOCAL:    local attention -- tile lt holds positions lt*128 .. +127,
//                w is the window (a row sees the w positions ending at its
//                own), and its key blocks are the 128-position blocks from the
//                one holding lt*128 - w + 1 up to lt; idx, mcount and yslot
//                are not used and every row goes to `out`.
// MODE_SEPARATE: separate queries and keys.  Query rows come from idx (the
//                queries' lists), key and value rows from idx_k (the keys'
//                lists), keys from `kk`; every key block of the cluster is
//                visited, and with causal=1 a key is visible to a query when
//                its position is not after the query's.  A query row with no
//                visible key is written as zeros and is not counted in
//                mvis[position] (the number of visible memberships the
//                scatter divides by).
constexpr int MODE_CLUSTER = 0, MODE_LOCAL = 1, MODE_SEPARATE = 2;

template <int D, int MODE>
__global__ void __launch_bounds__(THREADS, 2)
attention_tc_kernel(const bf16* __restrict__ q, const bf16* __restrict__ kk,
                    const bf16* __restrict__ v, int n, int k, int w,
                    int tiles_per_bh, int R, int causal, float scale_log2,
                    const int32_t* __restrict__ idx, const int32_t* __restrict__ idx_k,
                    const int32_t* __restrict__ mcount, int32_t* __restrict__ mvis,
                    bf16* __restrict__ out, float* __restrict__ yslot,
                    unsigned int* __restrict__ err, uint64_t fault_ns) {
  constexpr bool LOCAL = MODE == MODE_LOCAL;
  constexpr bool SEP = MODE == MODE_SEPARATE;
  using L = AttnSmem<D>;
  pdl_trigger();
  pdl_wait();
  // the injected test timeout returns here: nothing is in flight and no TMEM
  // is held yet
  if (injected_wait_timeout(fault_ns, err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* Qs = sm + L::Q_OFF;   // K-major [128 x D]
  uint8_t* KPs = sm + L::KP_OFF; // K-major keys, then P [128 x 128 keys]
  uint8_t* Vs = sm + L::V_OFF;   // MN-major [128 keys x D]

  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int qpos[ROWS];
  __shared__ int kpos[ROWS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const int bh = tile / tiles_per_bh;
  const int lt = tile % tiles_per_bh;
  const int32_t* idx_bh = LOCAL ? nullptr : idx + (size_t)bh * k * w;
  const int32_t* kidx_bh = SEP ? idx_k + (size_t)bh * k * w : idx_bh;
  const bf16* q_bh = q + (size_t)bh * n * D;
  const bf16* k_bh = (SEP ? kk : q) + (size_t)bh * n * D;
  const bf16* v_bh = v + (size_t)bh * n * D;

  // ---- row mapping (thread tid owns tile row tid) ----------------------------
  // clusters: slot rt*128 + tid of cluster lt / R; local: position lt*128 + tid
  int cluster = 0, rt, slot = 0, nkb, kb0 = 0;
  bool row_valid;
  int my_pos = -1;
  if (LOCAL) {
    rt = lt;
    row_valid = lt * ROWS + tid < n;
    if (row_valid) my_pos = lt * ROWS + tid;
    const int first = lt * ROWS - w + 1;  // first position any row of the tile sees
    kb0 = first > 0 ? first / ROWS : 0;
    nkb = lt - kb0 + 1;
  } else {
    cluster = lt / R;
    rt = lt % R;
    slot = rt * ROWS + tid;
    row_valid = slot < w;
    nkb = (causal && !SEP) ? rt + 1 : R;
    if (row_valid) {
      my_pos = __ldcg(idx_bh + (size_t)cluster * w + slot);
      if ((unsigned)my_pos >= (unsigned)n) { my_pos = -1; row_valid = false; }  // defensive
    }
  }
  // membership count of this row's position, loaded now, used by the epilogue
  const int my_m = (!LOCAL && row_valid) ? __ldcg(mcount + (size_t)bh * n + my_pos) : 1;
  qpos[tid] = my_pos;
  __syncthreads();

  gather_kmajor<D>(Qs, q_bh, qpos);
  cp_async_commit();

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 128);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);  // S, later O: columns [0, 128)

  constexpr uint32_t IDESC_S = tc::idesc_f16(ROWS, ROWS, true, false, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(ROWS, D, true, false, true);
  constexpr uint32_t SBO_QK = (D / 8) * 128;  // 8-row group stride, K-major [rows x D]

  float m_run = -INFINITY, l_run = 0.0f;
  float o_acc[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o_acc[i] = 0.0f;
  uint32_t phase = 0;
  bool failed = false;

  for (int kb = 0; kb < nkb && !failed; ++kb) {
    // key / value rows of key block kbi (the diagonal block's keys are the
    // tile's own rows: Q serves as K there)
    const int kbi = kb0 + kb;
    const uint8_t* Kop = Qs;
    {
      const int ks = kbi * ROWS + tid;
      int p = -1;
      if (LOCAL) {
        if (ks < n) p = ks;
      } else if (ks < w) {
        p = __ldcg(kidx_bh + (size_t)cluster * w + ks);
        if ((unsigned)p >= (unsigned)n) p = -1;
      }
      __syncthreads();  // previous block's buffers are free (all reads done)
      kpos[tid] = p;
      __syncthreads();
      if (SEP || kbi != rt) {
        gather_kmajor<D>(KPs, k_bh, kpos);
        Kop = KPs;
      }
      gather_mnmajor<D>(Vs, v_bh, kpos);
      cp_async_commit();
      cp_async_wait_all();
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();

    // ---- S = Q K^T ------------------------------------------------------
    if (tid == 0) {
      const uint32_t qa = tc::smem_u32(Qs), ka = tc::smem_u32(Kop);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint64_t ad = tc::smem_desc_noswizzle(qa + s * 256, 128, SBO_QK);
        const uint64_t bd = tc::smem_desc_noswizzle(ka + s * 256, 128, SBO_QK);
        tc::mma_f16_ss(tmem, ad, bd, IDESC_S, s > 0 ? 1u : 0u);
      }
      tc::mma_commit(&bar_s);
    }
    __syncwarp();
    if (!tc::mbar_wait_bounded(&bar_s, phase, WAIT_LIMIT_NS)) {
      failed = true;
      if (lane == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
    }
    failed = __syncthreads_or(failed);
    if (failed) break;
    tc::tc_fence_after_sync();

    // ---- softmax on this thread's row -----------------------------------
    // valid key columns [jmin, jmax).  Clusters: key slot < w, and causal:
    // key slot <= own slot.  Local: key position in [pos - w + 1, pos], < n.
    int jmin = 0, jmax;
    if (LOCAL) {
      const int pk0 = kbi * ROWS;
      jmin = max(0, my_pos - w + 1 - pk0);
      jmax = min(min(ROWS, my_pos - pk0 + 1), n - pk0);
    } else if (SEP) {
      // keys of the block in ascending position order: the visible ones are
      // the first `jmax`, those at positions <= this row's
      const int nvalid = min(ROWS, w - kbi * ROWS);
      jmax = nvalid;
      if (causal) {
        int lo = 0, hi = nvalid;  // first key position above my_pos
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (kpos[mid] <= my_pos) lo = mid + 1; else hi = mid;
        }
        jmax = lo;
      }
    } else {
      const int kslot0 = kbi * ROWS;
      jmax = min(ROWS, w - kslot0);
      if (causal) jmax = min(jmax, slot - kslot0 + 1);
    }
    if (!row_valid || jmax <= jmin) { jmin = ROWS; jmax = 0; }
    // chunks of 16 columns that hold a valid column for some row of the warp
    const int wlo = __reduce_min_sync(0xffffffffu, jmin);
    const int whi = __reduce_max_sync(0xffffffffu, jmax);
    const int ch_lo = (whi > wlo) ? (wlo >> 4) : 0;
    const int ch_hi = (whi > wlo) ? ((whi + 15) >> 4) : 0;

    // tcgen05.ld is warp-collective: the chunk range is warp-uniform.
    float mrow = -INFINITY;
    for (int ch = ch_lo; ch < ch_hi; ++ch) {
      uint32_t r[16];
      tc::tmem_ld16(t_row + ch * 16, r);
      tc::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = ch * 16 + j;
        if (col >= jmin && col < jmax) mrow = fmaxf(mrow, __uint_as_float(r[j]));
      }
    }
    const float m_new = fmaxf(m_run, mrow);
    const float mscaled = (m_new == -INFINITY) ? 0.0f : m_new * scale_log2;
    float lsum = 0.0f;
    // P overwrites the key block (on the diagonal block, the otherwise unused
    // K buffer): S = Q K^T is complete.
    uint8_t* Ps = KPs;
    const uint32_t prow = tc::smem_u32(Ps) + (tid >> 3) * 2048 + (tid & 7) * 16;
#pragma unroll 1
    for (int ch = 0; ch < ROWS / 16; ++ch) {
      uint32_t pk[8];
      if (ch >= ch_lo && ch < ch_hi) {
        uint32_t r[16];
        tc::tmem_ld16(t_row + ch * 16, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const int col = ch * 16 + j;
          const bool ok0 = col >= jmin && col < jmax;
          const bool ok1 = col + 1 >= jmin && col + 1 < jmax;
          const float e0 = ok0 ? exp2f(__uint_as_float(r[j]) * scale_log2 - mscaled) : 0.0f;
          const float e1 = ok1 ? exp2f(__uint_as_float(r[j + 1]) * scale_log2 - mscaled) : 0.0f;
          const uint32_t pp = pack_bf16(e0, e1);
          pk[j >> 1] = pp;
          lsum += __uint_as_float(pp << 16) + __uint_as_float(pp & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) pk[j] = 0u;
      }
      // two 16-byte chunks (keys 16ch..16ch+7, 16ch+8..16ch+15)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t addr = prow + (2 * ch + h) * 128;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * h]),
                     "r"(pk[4 * h + 1]), "r"(pk[4 * h + 2]), "r"(pk[4 * h + 3])
                     : "memory");
      }
    }
    const float alpha = (m_run == -INFINITY) ? 0.0f : exp2f((m_run - m_new) * scale_log2);
    l_run = l_run * alpha + lsum;
    m_run = m_new;

    tc::fence_proxy_async_smem();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();

    // ---- O_blk = P V (into S's columns) ---------------------------------
    if (tid == 0) {
      const uint32_t pa = tc::smem_u32(Ps), va = tc::smem_u32(Vs);
#pragma unroll
      for (int s = 0; s < ROWS / 16; ++s) {
        const uint64_t ad = tc::smem_desc_noswizzle(pa + s * 256, 128, 2048);
        const uint64_t bd = tc::smem_desc_noswizzle(va + s * 256, 128, 2048);
        tc::mma_f16_ss(tmem, ad, bd, IDESC_O, s > 0 ? 1u : 0u);
      }
      tc::mma_commit(&bar_o);
    }
    __syncwarp();
    if (!tc::mbar_wait_bounded(&bar_o, phase, WAIT_LIMIT_NS)) {
      failed = true;
      if (lane == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
    }
    failed = __syncthreads_or(failed);
    if (failed) break;
    tc::tc_fence_after_sync();
    phase ^= 1u;

#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t r[16];
      tc::tmem_ld16(t_row + c0, r);
      tc::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) o_acc[c0 + j] = o_acc[c0 + j] * alpha + __uint_as_float(r[j]);
    }
    tc::tc_fence_before_sync();  // O read before the next block's S overwrites it
  }

  // ---- epilogue ------------------------------------------------------------
  // Every MMA is complete, so the operand shared memory is free: each thread
  // stages its normalised O row there as fp32 (16-byte chunks XOR-swizzled by
  // row, conflict-free), then every warp copies its own 32 rows out with
  // row-contiguous stores -- bf16 to `out` for a position in exactly one
  // cluster, fp32 to its slot row in `yslot` otherwise.
  if (!failed) {
    constexpr int CPR = D / 4;        // 16-byte fp32 chunks per row
    constexpr int RPI = 32 / CPR;     // rows per warp instruction
    float4* stage = reinterpret_cast<float4*>(sm);
    const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      float o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = o_acc[c0 + j] * inv_l;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chunk = c0 / 4 + q4;
        stage[tid * CPR + (chunk ^ (tid & 7))] =
            make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
      }
    }
    __syncwarp();
    if (SEP && row_valid && my_m != 1 && l_run > 0.0f) atomicAdd(mvis + (size_t)bh * n + my_pos, 1);
    const int single = (row_valid && (LOCAL || my_m == 1)) ? 1 : 0;
    const int ch = lane % CPR;
#pragma unroll 4
    for (int it = 0; it < 32 / RPI; ++it) {
      const int rr = it * RPI + lane / CPR;  // row of this warp; its owner is lane rr
      const int r = warp * 32 + rr;
      const int t = __shfl_sync(0xffffffffu, my_pos, rr);
      const int ok = __shfl_sync(0xffffffffu, row_valid ? 1 : 0, rr);
      const int sg = __shfl_sync(0xffffffffu, single, rr);
      const int cl = __shfl_sync(0xffffffffu, cluster, rr);
      const int sl = __shfl_sync(0xffffffffu, slot, rr);
      const float4 val = stage[r * CPR + (ch ^ (r & 7))];
      if (!ok) continue;
      if (sg) {
        uint2 u;
        u.x = pack_bf16(val.x, val.y);
        u.y = pack_bf16(val.z, val.w);
        *reinterpret_cast<uint2*>(out + ((size_t)bh * n + t) * D + ch * 4) = u;
      } else {
        *reinterpret_cast<float4*>(yslot + (((size_t)bh * k + cl) * w + sl) * D + ch * 4) = val;
      }
    }

  }

  tc::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

template <int D>
cudaError_t launch_t(const void* q, const void* v, int BH, int n, int k, int w, int causal,
                     float scale, const int32_t* idx, const int32_t* mcount, void* out,
                     float* yslot, unsigned int* err, cudaStream_t s) {
  const int R = (w + ROWS - 1) / ROWS;  // row tiles (and key blocks) per cluster
  const int tiles_per_bh = k * R;
  const size_t smem = 1024 + (size_t)AttnSmem<D>::BYTES;
  auto kern = attention_tc_kernel<D, MODE_CLUSTER>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)BH * tiles_per_bh;
  const float scale_log2 = scale * 1.4426950408889634f;
  launch_begin(K_ATTN_TC, s);
  e = launch_pdl(kern, dim3((unsigned)tiles), dim3(THREADS), smem, s, static_cast<const bf16*>(q),
                 static_cast<const bf16*>(q), static_cast<const bf16*>(v), n, k, w, tiles_per_bh,
                 R, causal, scale_log2, idx, static_cast<const int32_t*>(nullptr), mcount,
                 static_cast<int32_t*>(nullptr), static_cast<bf16*>(out), yslot, err,
                 injected_limit_ns(K_ATTN_TC));
  launch_end(K_ATTN_TC, s);
  return e;
}

template <int D>
cudaError_t launch_sep_t(const void* q, const void* kk, const void* v, int BH, int n, int k,
                         int w, int causal, float scale, const int32_t* idx_q,
                         const int32_t* idx_k, const int32_t* mcount, int32_t* mvis, void* out,
                         float* yslot, unsigned int* err, cudaStream_t s) {
  const int R = (w + ROWS - 1) / ROWS;
  const int tiles_per_bh = k * R;
  const size_t smem = 1024 + (size_t)AttnSmem<D>::BYTES;
  auto kern = attention_tc_kernel<D, MODE_SEPARATE>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)BH * tiles_per_bh;
  const float scale_log2 = scale * 1.4426950408889634f;
  launch_begin(K_ATTN_TC, s);
  e = launch_pdl(kern, dim3((unsigned)tiles), dim3(THREADS), smem, s, static_cast<const bf16*>(q),
                 static_cast<const bf16*>(kk), static_cast<const bf16*>(v), n, k, w, tiles_per_bh,
                 R, causal, scale_log2, idx_q, idx_k, mcount, mvis, static_cast<bf16*>(out),
                 yslot, err, injected_limit_ns(K_ATTN_TC));
  launch_end(K_ATTN_TC, s);
  return e;
}

template <int D>
cudaError_t launch_local_t(const void* q, const void* v, int BH, int n, int window, float scale,
                           void* out, unsigned int* err, cudaStream_t s) {
  const int tiles_per_bh = (n + ROWS - 1) / ROWS;
  const size_t smem = 1024 + (size_t)AttnSmem<D>::BYTES;
  auto kern = attention_tc_kernel<D, MODE_LOCAL>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)BH * tiles_per_bh;
  const float scale_log2 = scale * 1.4426950408889634f;
  launch_begin(K_LOCAL_ATTN, s);
  e = launch_pdl(kern, dim3((unsigned)tiles), dim3(THREADS), smem, s, static_cast<const bf16*>(q),
                 static_cast<const bf16*>(q), static_cast<const bf16*>(v), n, 0, window,
                 tiles_per_bh, 1, 1, scale_log2, static_cast<const int32_t*>(nullptr),
                 static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr),
                 static_cast<int32_t*>(nullptr), static_cast<bf16*>(out),
                 static_cast<float*>(nullptr), err, injected_limit_ns(K_LOCAL_ATTN));
  launch_end(K_LOCAL_ATTN, s);
  return e;
}

}  // namespace

cudaError_t launch_local_attention(const void* q, const void* v, int BH, int n, int d, int window,
                                   float scale, void* out, unsigned int* err, cudaStream_t s) {
  return d == 64 ? launch_local_t<64>(q, v, BH, n, window, scale, out, err, s)
                 : launch_local_t<128>(q, v, BH, n, window, scale, out, err, s);
}

cudaError_t launch_attention_separate_tc(const void* q, const void* kk, const void* v, int BH,
                                         int n, int d, int k, int w, int causal, float scale,
                                         const int32_t* idx_q, const int32_t* idx_k,
                                         const int32_t* mcount, int32_t* mvis, void* out,
                                         float* yslot, unsigned int* err, cudaStream_t s) {
  return d == 64 ? launch_sep_t<64>(q, kk, v, BH, n, k, w, causal, scale, idx_q, idx_k, mcount,
                                    mvis, out, yslot, err, s)
                 : launch_sep_t<128>(q, kk, v, BH, n, k, w, causal, scale, idx_q, idx_k, mcount,
                                     mvis, out, yslot, err, s);
}

bool attention_tc_supported(rt_dtype dt, int d, int w) {
  return dt == RT_BF16 && (d == 64 || d == 128) && w >= 1 && tensor_maps_available();
}

cudaError_t launch_attention_tc(const void* q, const void* v, int BH, int n, int d, int k, int w,
                                int causal, float scale, const int32_t* idx,
                                const int32_t* mcount, void* out, float* yslot,
                                unsigned int* err, cudaStream_t s) {
  if (w <= ROWS)
    return launch_attention_pipe(q, v, BH, n, d, k, w, causal, scale, idx, mcount, out, yslot, err, s);
  if (w <= 2 * ROWS)
    return launch_attention_pair(q, v, BH, n, d, k, w, causal, scale, idx, mcount, out, yslot, err, s);
  return d == 64 ? launch_t<64>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s)
                 : launch_t<128>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s);
}

}  // namespace rt
