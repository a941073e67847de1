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
// Work unit: a tile of 128 query rows (TMEM lanes).
//   * w <= 128 ("packed"): g = floor(128 / w) whole clusters share a tile.
//     With shared QK the keys of the tile are its own rows, so one
//     S = Q Q^T (128 x 128) MMA covers every cluster of the tile and the mask
//     is block-diagonal (same cluster) and causal inside each block.  Padding
//     rows are zero-filled and masked.
//   * w > 128 ("multi"): a cluster spans ceil(w/128) row tiles; each row tile
//     walks its key blocks of 128 (causal: up to its own) with an online
//     softmax, the partial P V of each block read back from TMEM and
//     accumulated in registers.
// Each of the 128 threads owns one row: it reads its S row from TMEM,
// applies the mask and the softmax in registers, writes its P row (bf16) to
// shared memory in the MMA operand layout, and after O = P V reads its O row
// back.  Rows are gathered from HBM by position with 16-byte cp.async straight
// into the no-swizzle core-matrix layouts (Q/K: K-major; V: MN-major).  The
// MMA completions are waited on with a bounded mbarrier wait; a wait that runs
// out sets the device error word and the CTA gives up its tile.
#include "rt_internal.cuh"
#include "tc_ptx.cuh"

namespace rt {
namespace {

using bf16 = __nv_bfloat16;
constexpr int ROWS = 128;
constexpr int THREADS = 128;
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000 * 1000;  // 0.2 s

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: zero fill, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Gather 128 rows (positions pos[r], -1 = zero row) of D bf16 into the K-major
// no-swizzle layout: chunk (r, kc) at (r/8)*(D/8)*128 + kc*128 + (r%8)*16.
// A warp covers 8 rows x 4 chunks per instruction (512 contiguous bytes).
template <int D>
__device__ __forceinline__ void gather_kmajor(uint8_t* dst, const bf16* __restrict__ src,
                                              const int* pos) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int KC = D / 8;                // chunks per row
  constexpr int ITEMS = (ROWS / 8) * (KC / 4);
  const uint32_t base = tc::smem_u32(dst);
  for (int it = warp; it < ITEMS; it += THREADS / 32) {
    const int rg = it / (KC / 4);
    const int kc = (it % (KC / 4)) * 4 + (lane >> 3);
    const int r = rg * 8 + (lane & 7);
    const int p = pos[r];
    const uint32_t off = rg * (KC * 128) + kc * 128 + (lane & 7) * 16;
    const bf16* g = src + (size_t)(p < 0 ? 0 : p) * D + kc * 8;
    cp_async16(base + off, g, p >= 0);
  }
}

// Gather 128 key rows of V (D features) into the MN-major no-swizzle layout
// used as the B operand of O = P V (N = features, K = keys): chunk
// (j, ec) at ec*2048 + (j/8)*128 + (j%8)*16.
template <int D>
__device__ __forceinline__ void gather_mnmajor(uint8_t* dst, const bf16* __restrict__ src,
                                               const int* pos) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int EC = D / 8;
  constexpr int ITEMS = (ROWS / 8) * (EC / 4);
  const uint32_t base = tc::smem_u32(dst);
  for (int it = warp; it < ITEMS; it += THREADS / 32) {
    const int jg = it / (EC / 4);
    const int ec = (it % (EC / 4)) * 4 + (lane >> 3);
    const int j = jg * 8 + (lane & 7);
    const int p = pos[j];
    const uint32_t off = ec * 2048 + jg * 128 + (lane & 7) * 16;
    const bf16* g = src + (size_t)(p < 0 ? 0 : p) * D + ec * 8;
    cp_async16(base + off, g, p >= 0);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D, bool MULTI>
__global__ void __launch_bounds__(THREADS, MULTI ? 1 : 2)
attention_tc_kernel(const bf16* __restrict__ q, const bf16* __restrict__ v, int n, int k, int w,
                    int g, int tiles_per_bh, int R, int causal, float scale_log2,
                    const int32_t* __restrict__ idx, const int32_t* __restrict__ mcount,
                    bf16* __restrict__ out, float* __restrict__ yslot,
                    unsigned int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  constexpr int QB = ROWS * D * 2;
  uint8_t* Qs = sm;                 // K-major [128 x D]
  uint8_t* Vs = Qs + QB;            // MN-major [128 keys x D]
  uint8_t* Ps = Vs + QB;            // K-major [128 x 128 keys]
  uint8_t* Ks = Ps + ROWS * ROWS * 2;  // MULTI only: K-major [128 keys x D]

  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int qpos[ROWS];
  __shared__ int kpos[ROWS];
  __shared__ int vpos[ROWS];

  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int bh = tile / tiles_per_bh;
  const int lt = tile % tiles_per_bh;
  const int32_t* idx_bh = idx + (size_t)bh * k * w;
  const bf16* q_bh = q + (size_t)bh * n * D;
  const bf16* v_bh = v + (size_t)bh * n * D;

  // ---- row mapping (thread tid owns tile row tid) ------------------------
  int cluster, slot, row_lo, row_hi;  // row_lo/hi: valid key columns of this row
  bool row_valid;
  int nkb = 1, rt = 0;
  if (!MULTI) {
    const int ci = tid / w;
    cluster = lt * g + ci;
    slot = tid - ci * w;
    row_valid = (ci < g) && (cluster < k);
    row_lo = ci * w;
    row_hi = row_lo + w;
  } else {
    cluster = lt / R;
    rt = lt % R;
    slot = rt * ROWS + tid;
    row_valid = slot < w;
    nkb = causal ? rt + 1 : R;
    row_lo = 0;
    row_hi = w;
  }
  int my_pos = -1;
  if (row_valid) {
    my_pos = idx_bh[(size_t)cluster * w + slot];
    if ((unsigned)my_pos >= (unsigned)n) { my_pos = -1; row_valid = false; }  // defensive
  }
  qpos[tid] = my_pos;
  if (!MULTI) vpos[tid] = my_pos;
  __syncthreads();

  gather_kmajor<D>(Qs, q_bh, qpos);
  cp_async_commit();
  if (!MULTI) {
    gather_mnmajor<D>(Vs, v_bh, vpos);
    cp_async_commit();
  }

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 256);
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
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const uint32_t t_s = tmem + lane_base;        // S: columns [0, 128)
  const uint32_t t_o = tmem + lane_base + 128;  // O: columns [128, 128 + D)

  constexpr uint32_t IDESC_S = tc::idesc_f16(ROWS, ROWS, true, false, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(ROWS, D, true, false, true);
  constexpr uint32_t SBO_QK = (D / 8) * 128;  // 8-row group stride, K-major [rows x D]

  float m_run = -INFINITY, l_run = 0.0f;
  float o_acc[MULTI ? D : 1];
#pragma unroll
  for (int i = 0; i < (MULTI ? D : 1); ++i) o_acc[i] = 0.0f;
  uint32_t phase = 0;
  bool failed = false;

  for (int kb = 0; kb < nkb && !failed; ++kb) {
    const uint8_t* Kop = Qs;
    if (MULTI) {
      // key / value rows of key block kb
      const int ks = kb * ROWS + tid;
      int p = -1;
      if (ks < w) {
        p = idx_bh[(size_t)cluster * w + ks];
        if ((unsigned)p >= (unsigned)n) p = -1;
      }
      __syncthreads();  // previous block's buffers are free (all reads done)
      kpos[tid] = p;
      vpos[tid] = p;
      __syncthreads();
      if (kb != rt) {
        gather_kmajor<D>(Ks, q_bh, kpos);
        Kop = Ks;
      }
      gather_mnmajor<D>(Vs, v_bh, vpos);
      cp_async_commit();
      cp_async_wait_all();
    } else {
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // Q landed; V may be in flight
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
      if ((tid & 31) == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
    }
    failed = __syncthreads_or(failed);
    if (failed) break;
    tc::tc_fence_after_sync();

    // ---- softmax on this thread's row -----------------------------------
    // valid key column j: inside [row_lo, row_hi) (packed: own cluster),
    // key slot < w, and causal: key slot <= own slot.
    const int kslot0 = MULTI ? kb * ROWS : 0;
    int jmax = ROWS;  // exclusive upper bound on valid key columns
    int jmin = 0;
    if (!MULTI) {
      jmin = row_lo;
      jmax = causal ? tid + 1 : row_hi;
    } else {
      jmax = min(ROWS, w - kslot0);
      if (causal) jmax = min(jmax, slot - kslot0 + 1);
    }
    if (!row_valid) { jmin = 0; jmax = 0; }

    // tcgen05.ld is warp-collective: every thread loads every chunk.
    float mrow = -INFINITY;
#pragma unroll 1
    for (int c0 = 0; c0 < ROWS; c0 += 16) {
      uint32_t r[16];
      tc::tmem_ld16(t_s + c0, r);
      tc::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = c0 + j;
        if (col >= jmin && col < jmax) mrow = fmaxf(mrow, __uint_as_float(r[j]));
      }
    }
    const float m_new = fmaxf(m_run, mrow);
    const float mscaled = (m_new == -INFINITY) ? 0.0f : m_new * scale_log2;
    float lsum = 0.0f;
    const uint32_t prow = tc::smem_u32(Ps) + (tid >> 3) * 2048 + (tid & 7) * 16;
#pragma unroll 1
    for (int c0 = 0; c0 < ROWS; c0 += 16) {
      uint32_t r[16];
      tc::tmem_ld16(t_s + c0, r);
      tc::tmem_ld_wait();
      float p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = c0 + j;
        const bool ok = col >= jmin && col < jmax;
        const float e = ok ? exp2f(__uint_as_float(r[j]) * scale_log2 - mscaled) : 0.0f;
        const bf16 b = __float2bfloat16_rn(e);
        p[j] = __bfloat162float(b);
        lsum += p[j];
      }
      // two 16-byte chunks (keys c0..c0+7, c0+8..c0+15)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t a0 = pack_bf16(p[8 * h + 0], p[8 * h + 1]);
        const uint32_t a1 = pack_bf16(p[8 * h + 2], p[8 * h + 3]);
        const uint32_t a2 = pack_bf16(p[8 * h + 4], p[8 * h + 5]);
        const uint32_t a3 = pack_bf16(p[8 * h + 6], p[8 * h + 7]);
        const uint32_t addr = prow + ((c0 >> 3) + h) * 128;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a0), "r"(a1),
                     "r"(a2), "r"(a3)
                     : "memory");
      }
    }
    const float alpha = (m_run == -INFINITY) ? 0.0f : exp2f((m_run - m_new) * scale_log2);
    l_run = l_run * alpha + lsum;
    m_run = m_new;

    if (!MULTI) cp_async_wait_all();  // V landed
    tc::fence_proxy_async_smem();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();

    // ---- O_blk = P V ----------------------------------------------------
    if (tid == 0) {
      const uint32_t pa = tc::smem_u32(Ps), va = tc::smem_u32(Vs);
#pragma unroll
      for (int s = 0; s < ROWS / 16; ++s) {
        const uint64_t ad = tc::smem_desc_noswizzle(pa + s * 256, 128, 2048);
        const uint64_t bd = tc::smem_desc_noswizzle(va + s * 256, 128, 2048);
        tc::mma_f16_ss(tmem + 128, ad, bd, IDESC_O, s > 0 ? 1u : 0u);
      }
      tc::mma_commit(&bar_o);
    }
    __syncwarp();
    if (!tc::mbar_wait_bounded(&bar_o, phase, WAIT_LIMIT_NS)) {
      failed = true;
      if ((tid & 31) == 0) atomicExch(err, (unsigned)DEV_TIMEOUT);
    }
    failed = __syncthreads_or(failed);
    if (failed) break;
    tc::tc_fence_after_sync();
    phase ^= 1u;

    if (MULTI) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(t_o + c0, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) o_acc[c0 + j] = o_acc[c0 + j] * alpha + __uint_as_float(r[j]);
      }
    }
  }

  // ---- epilogue: this thread's output row --------------------------------
  if (!failed) {
    const int t = my_pos;
    const bool single = row_valid && mcount[(size_t)bh * n + t] == 1;
    const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      float o[16];
      if (MULTI) {
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = o_acc[c0 + j] * inv_l;
      } else {
        uint32_t r[16];
        tc::tmem_ld16(t_o + c0, r);  // warp-collective: every thread loads
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(r[j]) * inv_l;
      }
      if (!row_valid) continue;
      if (single) {
        uint4 a, b;
        a.x = pack_bf16(o[0], o[1]); a.y = pack_bf16(o[2], o[3]);
        a.z = pack_bf16(o[4], o[5]); a.w = pack_bf16(o[6], o[7]);
        b.x = pack_bf16(o[8], o[9]); b.y = pack_bf16(o[10], o[11]);
        b.z = pack_bf16(o[12], o[13]); b.w = pack_bf16(o[14], o[15]);
        uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)bh * n + t) * D + c0);
        dst[0] = a;
        dst[1] = b;
      } else {
        float4* dst = reinterpret_cast<float4*>(
            yslot + (((size_t)bh * k + cluster) * w + slot) * D + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      }
    }
  }

  tc::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

template <int D, bool MULTI>
cudaError_t launch_t(const void* q, const void* v, int BH, int n, int k, int w, int causal,
                     float scale, const int32_t* idx, const int32_t* mcount, void* out,
                     float* yslot, unsigned int* err, cudaStream_t s) {
  int g = 1, R = 1, tiles_per_bh;
  if (!MULTI) {
    g = ROWS / w;
    tiles_per_bh = (k + g - 1) / g;
  } else {
    R = (w + ROWS - 1) / ROWS;
    tiles_per_bh = k * R;
  }
  const size_t smem = 1024 + 2 * (size_t)ROWS * D * 2 + (size_t)ROWS * ROWS * 2 +
                      (MULTI ? (size_t)ROWS * D * 2 : 0);
  auto kern = attention_tc_kernel<D, MULTI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)BH * tiles_per_bh;
  const float scale_log2 = scale * 1.4426950408889634f;
  launch_begin(K_ATTN_TC, s);
  kern<<<(unsigned)tiles, THREADS, smem, s>>>(
      static_cast<const bf16*>(q), static_cast<const bf16*>(v), n, k, w, g, tiles_per_bh, R,
      causal, scale_log2, idx, mcount, static_cast<bf16*>(out), yslot, err);
  e = cudaGetLastError();
  launch_end(K_ATTN_TC, s);
  return e;
}

}  // namespace

bool attention_tc_supported(rt_dtype dt, int d, int w) {
  return dt == RT_BF16 && (d == 64 || d == 128) && w >= 1;
}

cudaError_t launch_attention_tc(const void* q, const void* v, int BH, int n, int d, int k, int w,
                                int causal, float scale, const int32_t* idx,
                                const int32_t* mcount, void* out, float* yslot,
                                unsigned int* err, cudaStream_t s) {
  const bool multi = w > ROWS;
  if (d == 64) {
    return multi ? launch_t<64, true>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s)
                 : launch_t<64, false>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s);
  }
  return multi ? launch_t<128, true>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s)
               : launch_t<128, false>(q, v, BH, n, k, w, causal, scale, idx, mcount, out, yslot, err, s);
}

}  // namespace rt
