// Normalise + score + argmax on the tcgen05 tensor cores, fp32-accurate.
//
// Routing step of "Efficient Content-Based Sparse Attention with Routing
// Transformers" (§4, "Routing attention with clustering"): each shared
// query/key row x_t goes on the unit sphere, r_t = (x_t - mean)/||x_t - mean||,
// and is scored against every centroid, S[c,t] = <r_t, mu_c>; the nearest
// centroid is the argmax (ties to the lower index).
//
// The scores decide integer outcomes (top-w lists, argmax), so they must be
// as good as an fp32 evaluation, while the tensor cores multiply bf16.  The
// rows are bf16 already, so only the fp32 centroids are split:
//   mu = hi + mid + lo   (three bf16 planes; the residual is ~2^-24 |mu|),
// and <x, mu> = <x, lo> + <x, mid> + <x, hi> is three bf16 MMAs whose
// products are exact in fp32, accumulated in fp32 in TMEM.  The epilogue
// applies the centring and normalisation per row:
//   S[c,t] = (<x_t, mu_c> - mean(x_t) * sum_j mu_cj) / ||x_t - mean(x_t)||
// (0 for a row whose centred norm is 0, matching r_t = 0).
//
// Persistent, warp-specialised CTA per (slice of tiles, head): the head's
// centroid planes are built once in shared memory (no-swizzle K-major core
// matrices); warp 0 streams 128-row tiles of Q with TMA (a 2-D tensor map,
// 8-element x 128-row boxes that land directly in the core-matrix layout),
// warp 1 issues the MMAs into one of two TMEM accumulators, warps 2-5 run
// the epilogue (row statistics from the L2-resident row, scores written
// centroid-major [BH,k,n] with coalesced stores, argmax) while the next tile
// is loaded and multiplied.  Every mbarrier wait is bounded; a wait that runs
// out sets the device error word and the CTA stops.
#include <cuda.h>

#include <mutex>

#include "rt_internal.cuh"
#include "tc_ptx.cuh"

namespace rt {
namespace {

using bf16 = __nv_bfloat16;
constexpr int ROWS = 128;
constexpr int THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000 * 1000;
constexpr int MAX_SMEM = 232448;  // 227 KiB opt-in per block

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(tc::smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void set_timeout(unsigned int* err) {
  if (err != nullptr) atomicExch(err, (unsigned)DEV_TIMEOUT);
}

struct ScoreCfg {
  int D, kpad, acc_cols, stages;
  size_t a_bytes, plane_bytes, smem;
};

inline int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap qmap, const bf16* __restrict__ q, int B,
                int H, int n, const float* __restrict__ mu, int k, int kpad, int acc_cols,
                int stages, int ctas_per_head, float* __restrict__ S, int32_t* __restrict__ assign,
                int32_t* __restrict__ mcount, unsigned int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  constexpr int A_BYTES = ROWS * D * 2;
  const int plane_bytes = kpad * D * 2;
  uint8_t* As = sm;                                  // stages x [128 x D] K-major
  uint8_t* Bs = As + (size_t)stages * A_BYTES;       // 3 planes x [kpad x D] K-major
  float* sumu = reinterpret_cast<float*>(Bs + 3 * (size_t)plane_bytes);  // [kpad]

  __shared__ uint64_t full_bar[2], empty_bar[2], accf_bar[2], acce_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int stop_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int tiles_per_bh = (n + ROWS - 1) / ROWS;
  const int ntiles = B * tiles_per_bh;  // tiles of this head (all sequences)

  // ---- centroid planes for head h (all threads) ---------------------------
  // warp per centroid row, each lane D/32 consecutive elements; the loads of
  // several rows are issued before any is used, so the set-up costs a few L2
  // round trips instead of one per element.  Row sums use a fixed order.
  {
    constexpr int PER = D / 32;
    constexpr int ROWS_IN_FLIGHT = 8;
    const float* mu_h = mu + (size_t)h * k * D;
    for (int c0 = warp * ROWS_IN_FLIGHT; c0 < kpad; c0 += (THREADS / 32) * ROWS_IN_FLIGHT) {
      float vals[ROWS_IN_FLIGHT][PER];
#pragma unroll
      for (int rr = 0; rr < ROWS_IN_FLIGHT; ++rr) {
        const int c = c0 + rr;
#pragma unroll
        for (int e = 0; e < PER; ++e)
          vals[rr][e] = (c < k) ? __ldg(mu_h + (size_t)c * D + lane * PER + e) : 0.0f;
      }
#pragma unroll
      for (int rr = 0; rr < ROWS_IN_FLIGHT; ++rr) {
        const int c = c0 + rr;
        if (c >= kpad) break;
        float rowsum = 0.0f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const int j = lane * PER + e;
          const float m = vals[rr][e];
          rowsum += m;
          const bf16 hi = __float2bfloat16_rn(m);
          const float r1 = m - __bfloat162float(hi);
          const bf16 md = __float2bfloat16_rn(r1);
          const float r2 = r1 - __bfloat162float(md);
          const bf16 lo = __float2bfloat16_rn(r2);
          const size_t off = (size_t)(j >> 3) * (kpad * 16) + c * 16 + (j & 7) * 2;
          *reinterpret_cast<bf16*>(Bs + off) = hi;
          *reinterpret_cast<bf16*>(Bs + plane_bytes + off) = md;
          *reinterpret_cast<bf16*>(Bs + 2 * (size_t)plane_bytes + off) = lo;
        }
        rowsum = warp_sum(rowsum);
        if (lane == 0) sumu[c] = rowsum;
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base_sh, 2 * acc_cols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&full_bar[i], 1);
      tc::mbar_init(&empty_bar[i], 1);
      tc::mbar_init(&accf_bar[i], 1);
      tc::mbar_init(&acce_bar[i], 4);
    }
    stop_flag = 0;
    tc::fence_mbar_init();
  }
  tc::fence_proxy_async_smem();  // planes written by threads, read by the MMA
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const int first = blockIdx.x, stride = ctas_per_head;
  if (warp == 0) {
    // ===================== TMA producer =====================================
    if (lane == 0) {
      int i = 0;
      for (int tile = first; tile < ntiles; tile += stride, ++i) {
        const int s = i % stages;
        const uint32_t use = (uint32_t)(i / stages);
        if (!tc::mbar_wait_bounded(&empty_bar[s], (use & 1u) ^ 1u, WAIT_LIMIT_NS) ||
            *(volatile int*)&stop_flag) {
          set_timeout(err);
          stop_flag = 1;
          break;
        }
        const int b = tile / tiles_per_bh, tb = tile - b * tiles_per_bh;
        const int row0 = (b * H + h) * n + tb * ROWS;
        tc::mbar_arrive_expect_tx(&full_bar[s], A_BYTES);
        uint8_t* dst = As + (size_t)s * A_BYTES;
#pragma unroll
        for (int kc = 0; kc < D / 8; ++kc)
          tma_load_2d(dst + kc * 2048, &qmap, kc * 8, row0, &full_bar[s]);
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =======================================
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(ROWS, kpad, true, false, false);
      const uint32_t lbo_b = kpad * 16;
      int i = 0;
      for (int tile = first; tile < ntiles; tile += stride, ++i) {
        const int s = i % stages;
        const uint32_t use = (uint32_t)(i / stages);
        const int ab = i & 1;
        const uint32_t ause = (uint32_t)(i >> 1);
        if (!tc::mbar_wait_bounded(&full_bar[s], use & 1u, WAIT_LIMIT_NS) ||
            !tc::mbar_wait_bounded(&acce_bar[ab], (ause & 1u) ^ 1u, WAIT_LIMIT_NS) ||
            *(volatile int*)&stop_flag) {
          set_timeout(err);
          stop_flag = 1;
          break;
        }
        tc::tc_fence_after_sync();
        const uint32_t a0 = tc::smem_u32(As + (size_t)s * A_BYTES);
        const uint32_t d_tmem = tmem + ab * acc_cols;
        int first_mma = 1;
        for (int p = 2; p >= 0; --p) {  // lo, mid, hi
          const uint32_t b0 = tc::smem_u32(Bs + (size_t)p * plane_bytes);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad = tc::smem_desc_noswizzle(a0 + ks * 4096, 2048, 128);
            const uint64_t bd = tc::smem_desc_noswizzle(b0 + ks * 2 * lbo_b, lbo_b, 128);
            tc::mma_f16_ss(d_tmem, ad, bd, idesc, first_mma ? 0u : 1u);
            first_mma = 0;
          }
        }
        tc::mma_commit(&empty_bar[s]);
        tc::mma_commit(&accf_bar[ab]);
      }
    }
  } else {
    // ===================== epilogue (warps 2..5) ============================
    const int row = 32 * (warp & 3) + lane;  // TMEM lane this thread reads
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int i = 0;
    for (int tile = first; tile < ntiles; tile += stride, ++i) {
      const int ab = i & 1;
      const uint32_t ause = (uint32_t)(i >> 1);
      const int b = tile / tiles_per_bh, tb = tile - b * tiles_per_bh;
      const int bh = b * H + h;
      const int t = tb * ROWS + row;
      const bool valid = t < n;
      // row statistics from the (L2-resident) row: mean, centred norm
      float mean = 0.0f, inv = 0.0f;
      bool zero_row = true;
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)bh * n + t) * D);
        uint4 v[D / 8];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) v[c] = __ldg(src + c);
        float s = 0.0f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
            s += __low2float(p2);
            s += __high2float(p2);
          }
        }
        mean = s / (float)D;
        float ss = 0.0f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
            const float a = __low2float(p2) - mean, bq = __high2float(p2) - mean;
            ss = fmaf(a, a, ss);
            ss = fmaf(bq, bq, ss);
          }
        }
        zero_row = !(ss > 0.0f);
        inv = zero_row ? 0.0f : 1.0f / sqrtf(ss);
      }
      bool ok = tc::mbar_wait_bounded(&accf_bar[ab], ause & 1u, WAIT_LIMIT_NS) &&
                !*(volatile int*)&stop_flag;
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: tcgen05.ld below is collective
      if (!ok) {
        if (lane == 0) set_timeout(err);
        stop_flag = 1;
        break;
      }
      tc::tc_fence_after_sync();
      float best = -INFINITY;
      int best_c = 0;
      float* srow = S + (size_t)bh * k * n + t;
      for (int c0 = 0; c0 < kpad; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tmem + ab * acc_cols + lane_base + c0, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          const float dot = __uint_as_float(r[j]);
          const float sc = zero_row ? 0.0f : (dot - mean * sumu[c]) * inv;
          if (valid && c < k) {
            if (S != nullptr) srow[(size_t)c * n] = sc;
            if (sc > best) { best = sc; best_c = c; }
          }
        }
      }
      tc::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&acce_bar[ab]))
                     : "memory");
      if (valid) {
        if (assign != nullptr) assign[(size_t)bh * n + t] = best_c;
        if (mcount != nullptr) mcount[(size_t)bh * n + t] = 0;
      }
    }
  }

  tc::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * acc_cols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool plan(int d, int k, ScoreCfg& c) {
  c.D = d;
  c.kpad = (k + 15) / 16 * 16;
  if (c.kpad > 256) return false;
  c.acc_cols = pow2_at_least(c.kpad);
  c.a_bytes = (size_t)ROWS * d * 2;
  c.plane_bytes = (size_t)c.kpad * d * 2;
  const size_t fixed = 1024 + 3 * c.plane_bytes + (size_t)c.kpad * 4;
  c.stages = (fixed + 2 * c.a_bytes + 512 <= (size_t)MAX_SMEM) ? 2 : 1;
  c.smem = fixed + c.stages * c.a_bytes;
  return c.smem + 512 <= (size_t)MAX_SMEM;
}

template <int D>
cudaError_t launch_t(const ScoreCfg& c, const void* qk, int B, int H, int n, const float* mu,
                     int k, float* S, int32_t* a, int32_t* mcount, unsigned int* err,
                     cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)B * H * n};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {8, (cuuint32_t)ROWS};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qk), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  auto kern = score_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  if (e != cudaSuccess) return e;
  const int tiles_per_head = B * ((n + ROWS - 1) / ROWS);
  int cph = 148 / H;
  if (cph < 1) cph = 1;
  if (cph > tiles_per_head) cph = tiles_per_head;
  launch_begin(K_SCORE_TC, s);
  kern<<<dim3(cph, H), THREADS, c.smem, s>>>(map, static_cast<const bf16*>(qk), B, H, n, mu, k,
                                             c.kpad, c.acc_cols, c.stages, cph, S, a, mcount,
                                             err);
  e = cudaGetLastError();
  launch_end(K_SCORE_TC, s);
  return e;
}

}  // namespace

bool score_tc_supported(rt_dtype dt, int d, int k) {
  ScoreCfg c;
  return dt == RT_BF16 && (d == 64 || d == 128) && plan(d, k, c) && encode_fn() != nullptr;
}

cudaError_t launch_score(const void* qk, rt_dtype dt, int B, int H, int n, int d, const float* mu,
                         int k, float* S, int32_t* a, int32_t* mcount, unsigned int* err,
                         cudaStream_t s) {
  ScoreCfg c;
  if (dt == RT_BF16 && (d == 64 || d == 128) && plan(d, k, c) && encode_fn() != nullptr &&
      (reinterpret_cast<uintptr_t>(qk) & 15u) == 0) {
    return d == 64 ? launch_t<64>(c, qk, B, H, n, mu, k, S, a, mcount, err, s)
                   : launch_t<128>(c, qk, B, H, n, mu, k, S, a, mcount, err, s);
  }
  return launch_score_simt(qk, dt, B * H, H, n, d, mu, k, S, a, mcount, s);
}

}  // namespace rt
