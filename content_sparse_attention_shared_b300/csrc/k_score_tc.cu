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
// matrices, written 16 bytes per thread, conflict-free); warp 0 streams
// 128-row tiles of Q with TMA (2-D tensor map, 64-element x 128-row boxes,
// 128-byte swizzle) into a ring of stages, warp 1 issues the MMAs into one of
// NG TMEM accumulators, and NG epilogue warpgroups (warps 2-5, 6-9, ...; NG =
// 4 when four accumulators fit in TMEM, else 2) take the tiles in turn: each
// reads its rows' statistics (mean, centred norm) from the staged tile in
// shared memory (while the MMA runs, when the group owns its stage), then
// the scores from TMEM, writes them centroid-major [BH,k,n] with coalesced
// stores and takes the argmax.  With the scores it can write the group bins of the
// select kernel (the bin of the largest score of every 8 consecutive
// positions per centroid): a tile row is a lane, so a group is a lane octet,
// and a shuffle reduce-scatter leaves each lane one centroid's group maximum
// per 8 columns.  Every mbarrier wait is bounded; a wait that runs out
// sets the device error word and the CTA stops.
#include "rt_internal.cuh"
#include "tc_ptx.cuh"

namespace rt {
namespace {

using bf16 = __nv_bfloat16;
constexpr int ROWS = 128;
// warp 0 TMA, warp 1 MMA, then NG epilogue groups of four warps
__host__ __device__ constexpr int score_threads(int ng) { return 64 + 128 * ng; }
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000 * 1000;
constexpr int MAX_SMEM = 232448;  // 227 KiB opt-in per block
constexpr int BOX_K = 64;         // elements per 128-byte swizzled row

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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
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

__device__ __forceinline__ uint32_t pack2_bf16(bf16 a, bf16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Centroid image of one head, as the score kernel holds it in shared memory:
// three bf16 planes [kpad x D] (no-swizzle K-major core matrices: chunk
// (c, jc) at jc*kpad*16 + c*16), then the kpad fp32 row sums.
__host__ __device__ inline size_t prep_image_bytes(int d, int kpad) {
  return 3 * (size_t)kpad * d * 2 + (size_t)kpad * 4;
}

// Split centroid row elements into the three bf16 planes and write one
// 16-byte chunk (8 features of centroid c) of each plane.
__device__ __forceinline__ void split_store8(uint8_t* planes, size_t plane_bytes, size_t off,
                                             const float (&m)[8]) {
  uint32_t ph[4], pm[4], pl[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    bf16 hi[2], md[2], lo[2];
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      hi[v] = __float2bfloat16_rn(m[e + v]);
      const float r1 = m[e + v] - __bfloat162float(hi[v]);
      md[v] = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(md[v]);
      lo[v] = __float2bfloat16_rn(r2);
    }
    ph[e / 2] = pack2_bf16(hi[0], hi[1]);
    pm[e / 2] = pack2_bf16(md[0], md[1]);
    pl[e / 2] = pack2_bf16(lo[0], lo[1]);
  }
  *reinterpret_cast<uint4*>(planes + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
  *reinterpret_cast<uint4*>(planes + plane_bytes + off) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
  *reinterpret_cast<uint4*>(planes + 2 * plane_bytes + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
}

// Builds every head's centroid image once per call (grid: centroid blocks of
// 32 x heads), so each score CTA fetches it with bulk copies instead of
// converting the centroids itself.  Row sums: one warp per centroid row,
// fixed shuffle order.
template <int D>
__global__ void __launch_bounds__(256)
centroid_prep_kernel(const float* __restrict__ mu, int k, int kpad, uint8_t* __restrict__ image) {
  // wait first: the score kernel behind this one reads Q before its own wait
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.y, c0 = blockIdx.x * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t plane_bytes = (size_t)kpad * D * 2;
  uint8_t* img = image + (size_t)h * prep_image_bytes(D, kpad);
  const float* mu_h = mu + (size_t)h * k * D;
  // every global load first (one round trip), then the conversion: item u of
  // this thread is 8 features (chunk warp + 8u) of centroid c0 + lane; the row
  // sums read D/32 consecutive features per lane of rows c0 + 4 warp + u
  constexpr int ITEMS = 32 * (D / 8) / 256;
  float4 ld[ITEMS][2];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int it = tid + 256 * u;
    const int c = c0 + (it & 31), jc = it >> 5;
    if (c < k) {
      const float4* src = reinterpret_cast<const float4*>(mu_h + (size_t)c * D + jc * 8);
      ld[u][0] = __ldcg(src);
      ld[u][1] = __ldcg(src + 1);
    } else {
      ld[u][0] = ld[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  }
  float rv[4][D / 32];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = c0 + warp * 4 + u;
#pragma unroll
    for (int e = 0; e < D / 32; ++e)
      rv[u][e] = c < k ? __ldcg(mu_h + (size_t)c * D + lane * (D / 32) + e) : 0.0f;
  }
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int it = tid + 256 * u;
    const int c = c0 + (it & 31), jc = it >> 5;
    if (c >= kpad) continue;
    const float m[8] = {ld[u][0].x, ld[u][0].y, ld[u][0].z, ld[u][0].w,
                        ld[u][1].x, ld[u][1].y, ld[u][1].z, ld[u][1].w};
    split_store8(img, plane_bytes, (size_t)jc * (kpad * 16) + (size_t)c * 16, m);
  }
  float* sums = reinterpret_cast<float*>(img + 3 * plane_bytes);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = c0 + warp * 4 + u;
    float v = 0.0f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) v += rv[u][e];
    v = warp_sum(v);
    if (lane == 0 && c < kpad) sums[c] = v;
  }
}

template <int D, bool PREP, int NG>
__global__ void __launch_bounds__(score_threads(NG), 1)
score_tc_kernel(const __grid_constant__ CUtensorMap qmap, int B, int H, int n,
                const float* __restrict__ mu, const uint8_t* __restrict__ image, int k, int kpad,
                int acc_cols, int stages, int ctas_per_head, float* __restrict__ S,
                int32_t* __restrict__ assign, int32_t* __restrict__ mcount,
                uint16_t* __restrict__ gbins, int gstride, unsigned int* __restrict__ err,
                uint64_t fault_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  constexpr int A_BYTES = ROWS * D * 2;
  constexpr int KB = D / BOX_K;  // swizzled 128-byte column blocks per row
  const int plane_bytes = kpad * D * 2;
  uint8_t* As = sm;                                  // stages x [KB][128 rows x 128 B] SW128
  uint8_t* Bs = As + (size_t)stages * A_BYTES;       // 3 planes x [kpad x D] K-major
  float* sumu = reinterpret_cast<float*>(Bs + 3 * (size_t)plane_bytes);  // [kpad]

  constexpr int THREADS = score_threads(NG);
  __shared__ uint64_t full_bar[4], empty_bar[4], accf_bar[NG], acce_bar[NG], prep_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int stop_flag;

  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int tiles_per_bh = (n + ROWS - 1) / ROWS;
  const int ntiles = B * tiles_per_bh;  // tiles of this head (all sequences)

  // ---- barriers first, so the first Q tiles stream in during the set-up ---
  const int first = blockIdx.x, stride = ctas_per_head;
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      tc::mbar_init(&full_bar[i], 1);
      tc::mbar_init(&empty_bar[i], 4);  // the 4 warps of the epilogue group that read the tile
    }
    for (int i = 0; i < NG; ++i) {
      tc::mbar_init(&accf_bar[i], 1);
      tc::mbar_init(&acce_bar[i], 4);
    }
    tc::mbar_init(&prep_bar, 1);
    stop_flag = 0;
    tc::fence_mbar_init();
  }
  // the first `stages` tiles need no free slot
  auto issue_first_tiles = [&]() {
    int i = 0;
    for (int tile = first; tile < ntiles && i < stages; tile += stride, ++i) {
      const int b = tile / tiles_per_bh, tb = tile - b * tiles_per_bh;
      const int row0 = (b * H + h) * n + tb * ROWS;
      tc::mbar_arrive_expect_tx(&full_bar[i], A_BYTES);
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d(As + (size_t)i * A_BYTES + kb * (ROWS * 128), &qmap, kb * BOX_K, row0,
                    &full_bar[i]);
    }
  };
  // Behind the prep kernel, Q is complete before this kernel starts: the prep
  // kernel lets it launch only after its own wait for the kernel before it.
  // So the first Q tiles are requested before the wait for the image (not
  // under the injected test timeout, which returns with nothing in flight).
  const bool q_early = PREP && fault_ns == 0;
  if (q_early && tid == 0) issue_first_tiles();
  pdl_wait();  // every other global access below comes after the previous kernel
  // the injected test timeout returns here: nothing is in flight and no TMEM
  // is held yet
  if (injected_wait_timeout(fault_ns, err)) return;
  if (tid == 0) {
    if (PREP) {
      // the head's centroid image, in bulk copies of at most 32 KiB
      const uint32_t total = (uint32_t)prep_image_bytes(D, kpad);
      const uint8_t* src = image + (size_t)h * total;
      tc::mbar_arrive_expect_tx(&prep_bar, total);
      for (uint32_t off = 0; off < total; off += 32768u) {
        const uint32_t bytes = min(32768u, total - off);
        tc::bulk_g2s(Bs + off, src + off, bytes, &prep_bar);
      }
    }
    if (!q_early) issue_first_tiles();
  }

  if (!PREP) {
    // ---- centroid planes for head h, built here (all threads) -------------
    // item (c, jc): 8 consecutive features of centroid c; consecutive threads
    // take consecutive c (conflict-free 16-byte stores).  Four items per
    // thread are loaded before any is converted.
    const float* mu_h = mu + (size_t)h * k * D;
    const int items = kpad * (D / 8);
    constexpr int U = 4;
    for (int it0 = tid; it0 < items; it0 += U * THREADS) {
      float m[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int it = it0 + u * THREADS;
        const int c = it % kpad, jc = it / kpad;
        if (it < items && c < k) {
          const float4* src = reinterpret_cast<const float4*>(mu_h + (size_t)c * D + jc * 8);
          const float4 a = __ldcg(src), b = __ldcg(src + 1);
          m[u][0] = a.x; m[u][1] = a.y; m[u][2] = a.z; m[u][3] = a.w;
          m[u][4] = b.x; m[u][5] = b.y; m[u][6] = b.z; m[u][7] = b.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) m[u][e] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int it = it0 + u * THREADS;
        if (it >= items) break;
        const int c = it % kpad, jc = it / kpad;
        split_store8(Bs, (size_t)plane_bytes, (size_t)jc * (kpad * 16) + (size_t)c * 16, m[u]);
      }
    }
    // row sums of the fp32 centroids: one warp per row (fixed shuffle
    // order), eight rows in flight per warp
    constexpr int NW = THREADS / 32;
    constexpr int RU = 8;
    for (int c0 = warp; c0 < kpad; c0 += NW * RU) {
      float v[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int c = c0 + u * NW;
        v[u] = 0.0f;
        if (c < k) {
          const float* r = mu_h + (size_t)c * D + lane * (D / 32);
#pragma unroll
          for (int e = 0; e < D / 32; ++e) v[u] += __ldcg(r + e);
        }
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const float rs = warp_sum(v[u]);
        const int c = c0 + u * NW;
        if (lane == 0 && c < kpad) sumu[c] = rs;
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base_sh, NG * acc_cols);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();  // planes written by threads, read by the MMA
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ===================== TMA producer =====================================
    if (lane == 0) {
      int i = stages;  // tiles 0 .. stages-1 were issued before the set-up
      for (int tile = first + stages * stride; tile < ntiles; tile += stride, ++i) {
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
        for (int kb = 0; kb < KB; ++kb)
          tma_load_2d(dst + kb * (ROWS * 128), &qmap, kb * BOX_K, row0, &full_bar[s]);
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =======================================
    if (lane == 0) {
      if (PREP && !tc::mbar_wait_bounded(&prep_bar, 0, WAIT_LIMIT_NS)) {
        set_timeout(err);
        stop_flag = 1;
      }
      const uint32_t idesc = tc::idesc_f16(ROWS, kpad, true, false, false);
      const uint32_t lbo_b = kpad * 16;
      int i = 0;
      for (int tile = first; tile < ntiles; tile += stride, ++i) {
        const int s = i % stages;
        const uint32_t use = (uint32_t)(i / stages);
        const int ab = i % NG;
        const uint32_t ause = (uint32_t)(i / NG);
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
            const uint32_t a_addr = a0 + (ks / 4) * (ROWS * 128) + (ks % 4) * 32;
            const uint64_t ad = tc::smem_desc_sw128(a_addr, 1024);
            const uint64_t bd = tc::smem_desc_noswizzle(b0 + ks * 2 * lbo_b, lbo_b, 128);
            tc::mma_f16_ss(d_tmem, ad, bd, idesc, first_mma ? 0u : 1u);
            first_mma = 0;
          }
        }
        tc::mma_commit(&accf_bar[ab]);
      }
    }
  } else {
    // ===================== epilogue groups (warps 2 .. 4 NG + 1) =============
    const int grp = (warp - 2) >> 2;         // takes tiles i with i % NG == grp
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int row = 32 * quad + lane;        // tile row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    if (PREP) {
      // the row sums arrive with the bulk copies
      bool okp = tc::mbar_wait_bounded(&prep_bar, 0, WAIT_LIMIT_NS);
      okp = __all_sync(0xffffffffu, okp);
      if (!okp) {
        if (lane == 0) set_timeout(err);
        stop_flag = 1;
      }
    }
    int i = grp;
    for (int tile = first + grp * stride; tile < ntiles; tile += NG * stride, i += NG) {
      const int s = i % stages;
      const uint32_t use = (uint32_t)(i / stages);
      const uint32_t ause = (uint32_t)(i / NG);
      const int b = tile / tiles_per_bh, tb = tile - b * tiles_per_bh;
      const int bh = b * H + h;
      const int t = tb * ROWS + row;
      const bool valid = t < n;
      // The row statistics need only the staged tile.  When the stage's
      // previous use was this group's own tile (NG divides the stage count),
      // the group waits for the TMA alone, computes them while the MMA runs
      // and waits for the MMA afterwards: the full barrier cannot be a phase
      // behind or ahead, since the stage is refilled only after this group
      // releases it, which follows the MMA's completion.  Otherwise it waits
      // for the MMA first, which implies the tile's TMA phase (the MMA waited
      // for it); that phase cannot advance before this group releases the
      // stage, so the full-barrier wait returns at once and only orders the
      // staged bytes for this thread.
      const bool early = stages % NG == 0;
      bool ok = (early || tc::mbar_wait_bounded(&accf_bar[grp], ause & 1u, WAIT_LIMIT_NS)) &&
                tc::mbar_wait_bounded(&full_bar[s], use & 1u, WAIT_LIMIT_NS) &&
                !*(volatile int*)&stop_flag;
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: tcgen05.ld below is collective
      if (!ok) {
        if (lane == 0) set_timeout(err);
        stop_flag = 1;
        break;
      }
      // row statistics from the staged tile: mean and centred norm
      float mean = 0.0f, inv = 0.0f;
      bool zero_row = true;
      {
        // two passes over the row in shared memory (sum, then centred
        // squares), QB 16-byte chunks in flight (all of them when the
        // registers allow), four partial sums each
        const uint8_t* arow = As + (size_t)s * A_BYTES + row * 128;
        auto chunk = [&](int q) {  // chunk q: features 8q..8q+7
          return *reinterpret_cast<const uint4*>(arow + (q >> 3) * (ROWS * 128) +
                                                 (((q & 7) ^ (row & 7)) << 4));
        };
        constexpr int QB = NG == 2 ? D / 8 : 8;
        float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
        for (int q0 = 0; q0 < D / 8; q0 += QB) {
          uint4 v[QB];
#pragma unroll
          for (int u = 0; u < QB; ++u) v[u] = chunk(q0 + u);
#pragma unroll
          for (int u = 0; u < QB; ++u) {
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
              p4[e] += __low2float(p2);
              p4[e] += __high2float(p2);
            }
          }
        }
        mean = ((p4[0] + p4[1]) + (p4[2] + p4[3])) / (float)D;
        float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
        for (int q0 = 0; q0 < D / 8; q0 += QB) {
          uint4 v[QB];
#pragma unroll
          for (int u = 0; u < QB; ++u) v[u] = chunk(q0 + u);
#pragma unroll
          for (int u = 0; u < QB; ++u) {
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
              const float a = __low2float(p2) - mean, bq = __high2float(p2) - mean;
              s4[e] = fmaf(a, a, s4[e]);
              s4[e] = fmaf(bq, bq, s4[e]);
            }
          }
        }
        const float sxx = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        zero_row = !(sxx > 0.0f);
        inv = zero_row ? 0.0f : 1.0f / sqrtf(sxx);
      }
      if (early) {
        bool okm = tc::mbar_wait_bounded(&accf_bar[grp], ause & 1u, WAIT_LIMIT_NS) &&
                   !*(volatile int*)&stop_flag;
        okm = __all_sync(0xffffffffu, okm);
        if (!okm) {
          if (lane == 0) set_timeout(err);
          stop_flag = 1;
          break;
        }
      }
      // stage free: rows read and the MMA done (the MMA reads the stage too,
      // so it is released only after the accumulator barrier)
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      tc::tc_fence_after_sync();
      float best = -INFINITY;
      int best_c = 0;
      const float nmean = -mean;
      float* sp = (S != nullptr && valid) ? S + (size_t)bh * k * n + t : nullptr;
      // group bins: the lane octet holding positions 8m..8m+7 of this tile
      // reduces each centroid's column, and lane 8m+j writes centroid j's bin
      const int gi = tb * (ROWS / GROUP_SIZE) + (row >> 3);
      uint16_t* gp = (gbins != nullptr && gi * GROUP_SIZE < n)
                         ? gbins + (size_t)bh * k * gstride + gi + (size_t)(lane & 7) * gstride
                         : nullptr;
      const uint32_t tacc = tmem + grp * acc_cols + lane_base;
      const bool tile_full = (tb + 1) * ROWS <= n;  // the same for the whole tile
      for (int c0 = 0; c0 < kpad; c0 += 32) {
        uint32_t r[2][16];
        tc::tmem_ld16(tacc + c0, r[0]);
        if (c0 + 16 < kpad) tc::tmem_ld16(tacc + c0 + 16, r[1]);
        tc::tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int cb = c0 + 16 * hh;
          if (cb >= kpad) break;
          float sc[16];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 su = *reinterpret_cast<const float4*>(sumu + cb + 4 * q4);
            sc[4 * q4 + 0] = fmaf(nmean, su.x, __uint_as_float(r[hh][4 * q4 + 0])) * inv;
            sc[4 * q4 + 1] = fmaf(nmean, su.y, __uint_as_float(r[hh][4 * q4 + 1])) * inv;
            sc[4 * q4 + 2] = fmaf(nmean, su.z, __uint_as_float(r[hh][4 * q4 + 2])) * inv;
            sc[4 * q4 + 3] = fmaf(nmean, su.w, __uint_as_float(r[hh][4 * q4 + 3])) * inv;
          }
          // (a row with a zero centred norm has inv = 0, so its scores are 0)
          if (gbins != nullptr) {  // warp-uniform: the shuffles need every lane
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
              float m[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                m[j] = (tile_full || valid) ? sc[8 * hv + j] : -INFINITY;
              const float gm = octet_column_max(m, lane);
              const int cg = cb + 8 * hv + (lane & 7);
              if (gp != nullptr && cg < k)
                gp[(size_t)(cb + 8 * hv) * gstride] = (uint16_t)score_bin(gm);
            }
          }
          if (cb + 16 <= k) {
            // argmax of the 16 columns as a pairwise tree (the left one wins
            // ties, so each node holds the first maximum of its range), then
            // against the running best: five dependent steps, not sixteen
            float tv[8];
            int ti[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool right = sc[2 * j + 1] > sc[2 * j];
              tv[j] = right ? sc[2 * j + 1] : sc[2 * j];
              ti[j] = 2 * j + (right ? 1 : 0);
            }
#pragma unroll
            for (int span = 4; span >= 1; span >>= 1) {
#pragma unroll
              for (int j = 0; j < span; ++j) {
                const bool right = tv[2 * j + 1] > tv[2 * j];
                tv[j] = right ? tv[2 * j + 1] : tv[2 * j];
                ti[j] = right ? ti[2 * j + 1] : ti[2 * j];
              }
            }
            if (tv[0] > best) { best = tv[0]; best_c = cb + ti[0]; }
            if (sp != nullptr) {
              // (column offsets are the same for the whole warp)
#pragma unroll
              for (int j = 0; j < 16; ++j) sp[(size_t)(cb + j) * n] = sc[j];
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (cb + j < k) {
                if (sc[j] > best) { best = sc[j]; best_c = cb + j; }
                if (sp != nullptr) sp[(size_t)(cb + j) * n] = sc[j];
              }
            }
          }
        }
      }
      tc::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[grp]);
      if (valid) {
        if (assign != nullptr) assign[(size_t)bh * n + t] = best_c;
        if (mcount != nullptr) mcount[(size_t)bh * n + t] = 0;
      }
    }
  }

  tc::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, NG * acc_cols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Tensor map of Q viewed as [rows, D] bf16 with 64-element x 128-row boxes,
// 128-byte swizzle.
bool q_tensor_map(const void* qk, unsigned long long rows, int D, CUtensorMap* out) {
  return bf16_tensor_map_2d(qk, rows, (unsigned)D, BOX_K, ROWS, out);
}

// Shared-memory plan: 1 KiB alignment slack, A stages (1024-byte aligned
// swizzle atoms), the three centroid planes, the centroid row sums; as many
// A stages (up to 4) as fit beside the planes.  Static shared memory (the
// barriers) takes well under 256 bytes.
bool plan(int d, int k, ScoreCfg& c) {
  c.D = d;
  c.kpad = (k + 15) / 16 * 16;
  if (c.kpad > 256) return false;
  c.acc_cols = pow2_at_least(c.kpad);
  c.a_bytes = (size_t)ROWS * d * 2;
  c.plane_bytes = (size_t)c.kpad * d * 2;
  const size_t fixed = 1024 + 3 * c.plane_bytes + (size_t)c.kpad * 4;
  const size_t budget = (size_t)MAX_SMEM - 256;
  c.stages = 0;
  for (int st = 4; st >= 1; --st)
    if (fixed + st * c.a_bytes <= budget) { c.stages = st; break; }
  if (c.stages == 0) return false;
  c.smem = fixed + c.stages * c.a_bytes;
  return true;
}

template <int D>
cudaError_t launch_t(const ScoreCfg& c, const void* qk, int B, int H, int n, const float* mu,
                     int k, float* S, int32_t* a, int32_t* mcount, uint16_t* gbins, void* prep,
                     unsigned int* err, cudaStream_t s) {
  CUtensorMap map;
  if (!q_tensor_map(qk, (unsigned long long)B * H * n, D, &map)) return cudaErrorInvalidValue;
  cudaError_t e;
  if (prep != nullptr) {
    launch_begin(K_CENTROID_PREP, s);
    e = launch_pdl(centroid_prep_kernel<D>, dim3((c.kpad + 31) / 32, H), dim3(256), 0, s, mu, k,
                   c.kpad, static_cast<uint8_t*>(prep));
    launch_end(K_CENTROID_PREP, s);
    if (e != cudaSuccess) return e;
  }
  // four epilogue groups (four tiles in flight) when four accumulators fit
  // in the 512 TMEM columns, else two
  const int ng = 4 * c.acc_cols <= 512 ? 4 : 2;
  auto kern = prep != nullptr ? (ng == 4 ? score_tc_kernel<D, true, 4> : score_tc_kernel<D, true, 2>)
                              : (ng == 4 ? score_tc_kernel<D, false, 4> : score_tc_kernel<D, false, 2>);
  e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)c.smem);
  if (e != cudaSuccess) return e;
  const int tiles_per_head = B * ((n + ROWS - 1) / ROWS);
  int cph = 148 / H;
  if (cph < 1) cph = 1;
  if (cph > tiles_per_head) cph = tiles_per_head;
  launch_begin(K_SCORE_TC, s);
  e = launch_pdl(kern, dim3(cph, H), dim3(score_threads(ng)), c.smem, s, map, B, H, n, mu,
                 static_cast<const uint8_t*>(prep), k, c.kpad, c.acc_cols, c.stages, cph, S, a,
                 mcount, S != nullptr ? gbins : nullptr, gbin_stride(n), err,
                 injected_limit_ns(K_SCORE_TC));
  launch_end(K_SCORE_TC, s);
  return e;
}

}  // namespace

bool score_tc_supported(rt_dtype dt, int d, int k) {
  ScoreCfg c;
  return dt == RT_BF16 && (d == 64 || d == 128) && plan(d, k, c) && tensor_maps_available();
}

size_t score_prep_bytes(int H, int d, int k) {
  ScoreCfg c;
  if (!plan(d, k, c)) return 0;
  return (size_t)H * prep_image_bytes(d, c.kpad);
}

cudaError_t launch_score(const void* qk, rt_dtype dt, int B, int H, int n, int d, const float* mu,
                         int k, float* S, int32_t* a, int32_t* mcount, uint16_t* gbins,
                         void* prep, unsigned int* err, cudaStream_t s) {
  ScoreCfg c;
  if (dt == RT_BF16 && (d == 64 || d == 128) && plan(d, k, c) && tensor_maps_available() &&
      (reinterpret_cast<uintptr_t>(qk) & 15u) == 0) {
    return d == 64 ? launch_t<64>(c, qk, B, H, n, mu, k, S, a, mcount, gbins, prep, err, s)
                   : launch_t<128>(c, qk, B, H, n, mu, k, S, a, mcount, gbins, prep, err, s);
  }
  return launch_score_simt(qk, dt, B * H, H, n, d, mu, k, S, a, mcount, gbins, s);
}

}  // namespace rt
