// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "../../include/routing_attention.h"

namespace rt {

// ---------------------------------------------------------------------------
// kernel kinds (for launch counting and the per-launch timing hook)
// ---------------------------------------------------------------------------
enum KernelId {
  K_SCORE_SIMT = 0,
  K_SCORE_TC = 1,
  K_SELECT = 2,
  K_ATTN_SIMT = 3,
  K_ATTN_TC = 4,
  K_SCATTER = 5,
  K_EMA_TOPW = 6,
  K_EMA_UPDATE = 7,
  K_CENTROID_PREP = 8,
  K_LOCAL_ATTN = 9,
  K_EMA_BUCKET = 10,
  K_BACKWARD = 11,
  K_MEMBERSHIP = 12,
  K_NUM_KINDS = 13
};

// Error detail for the calling host thread (rt_last_error_detail) and the
// shape checks shared by the entry points.
rt_status record_error(rt_status s, const char* msg);
rt_status validate_shape(rt_dtype dt, int B, int H, int n, int d, int k, int w);
// Reads and clears the status word of rt_route_assign_noalloc in the current
// context (synchronises `s`).
rt_status noalloc_check_status(cudaStream_t s);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute call is made only the first time a kernel
// needs more than it was given before on that device, so launches pay a map
// lookup instead of a driver call.
cudaError_t set_smem_limit(const void* func, int bytes);

// 2-D tensor map of a row-major bf16 matrix [rows, cols] (cols contiguous)
// with boxes of box_cols x box_rows elements and 128-byte swizzle (box_cols *
// 2 must be 128).  Encoding is host work; recent maps are cached (keyed by
// base pointer, shape and box) so repeated calls on the same tensors skip it.
bool tensor_maps_available();
bool bf16_tensor_map_2d(const void* base, unsigned long long rows, unsigned cols,
                        unsigned box_cols, unsigned box_rows, CUtensorMap* out);
// 3-D tensor map of fp32 rows [batches][rows][cols] (cols contiguous, a
// multiple of 32) with boxes of 32 columns x box_rows rows x 1 batch and
// 128-byte swizzle, for bulk stores of staged row tiles (cached the same way).
bool f32_tensor_map_3d(const void* base, unsigned cols, unsigned long long rows,
                       unsigned batches, unsigned box_rows, CUtensorMap* out);

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialization allowed, tells the runtime at its start
// that its dependents may be scheduled (pdl_trigger), and waits for its
// predecessor grid to complete, with its memory visible (pdl_wait), before it
// reads or writes any global memory.  Only shared-memory / TMEM set-up comes
// before pdl_wait, so the set-up overlaps the predecessor's tail.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Called by every launcher around its launch.
void launch_begin(int kind, cudaStream_t s);
void launch_end(int kind, cudaStream_t s);

// ---------------------------------------------------------------------------
// device error word (first bytes of every workspace)
// ---------------------------------------------------------------------------
enum DeviceError : unsigned int {
  DEV_OK = 0,
  DEV_TIMEOUT = 1,
};

// Test aid for the device-side timeout path (rt_debug_inject_wait_timeout):
// with limit_ns > 0, thread 0 waits on an mbarrier that nothing arrives on,
// bounded by limit_ns, before the kernel issues any asynchronous copy or MMA;
// the wait runs out, the status word is set, and the caller returns -- with
// nothing in flight.  Every thread of the CTA calls it (it contains block
// barriers); returns true when the kernel must return.
__device__ __forceinline__ bool injected_wait_timeout(uint64_t limit_ns, unsigned int* err) {
  if (limit_ns == 0) return false;
  __shared__ uint64_t fault_bar;
  __shared__ int s_out;
  if (threadIdx.x == 0) {
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&fault_bar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    bool done = false;
    while (true) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(bar)
          : "memory");
      if (ok) { done = true; break; }
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > limit_ns) break;
    }
    if (!done && err != nullptr) atomicExch(err, (unsigned)DEV_TIMEOUT);
    s_out = done ? 0 : 1;
  }
  __syncthreads();
  return s_out != 0;
}

// Host side of the test aid: the limit to pass to a kernel of the given kind
// (0 unless rt_debug_inject_wait_timeout selected that kind).
uint64_t injected_limit_ns(int kind);

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exclusive prefix sum over the NT threads of a block (one int each) and the
// block total.  wsum: NT/32 ints of shared memory.  Contains two barriers, so
// every thread of the block must call it.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int x = wsum[i];
    before += (i < warp) ? x : 0;
    total += x;
  }
  __syncthreads();  // wsum may be reused at once
  return before + incl - v;
}

// Order-preserving map of an fp32 score to an unsigned key (larger score,
// larger key).  -0 is folded onto +0 so that equal scores give equal keys.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// group bins: a by-product of the score kernels for the select kernel
// ---------------------------------------------------------------------------
// Scores are cosines of unit vectors, so they lie in [-1, 1].  A score's bin is
// its interval in a partition of [-1, 1] into SCORE_BINS equal parts (clamped;
// non-decreasing in the score, so every score of a higher bin is strictly
// larger; NaN -> 0).  For every run of GROUP_SIZE consecutive positions of a
// (batch*head, centroid) row the score kernels can also write the bin of the
// run's largest score ("group bin") to gbins [BH, k, gbin_stride(n)] u16; the
// entries past ceil(n / GROUP_SIZE) of a row are padding and never written.
// Since the bin is monotone, a group's bin is the largest bin of its members.
constexpr int SCORE_BINS = 2048;
constexpr int GROUP_SIZE = 8;

__host__ __device__ inline int gbin_stride(int n) {
  const int ng = (n + GROUP_SIZE - 1) / GROUP_SIZE;
  return (ng + 7) & ~7;  // rows start on 16-byte boundaries
}

__device__ __forceinline__ int score_bin(float s) {
  float f = (s + 1.0f) * (0.5f * SCORE_BINS);
  f = fminf(fmaxf(f, 0.0f), (float)(SCORE_BINS - 1));
  return (int)f;
}

// Column maxima over the 8 lanes of each aligned lane octet (lanes 8m..8m+7):
// v holds a lane's value for 8 columns; lane l returns the maximum over its
// octet of column (l & 7).  A reduce-scatter in three exchange steps (4, 2,
// then 1 value per lane), 7 shuffles for 8 columns.  Every lane of the warp
// must call it.
__device__ __forceinline__ float octet_column_max(const float (&v)[8], int lane) {
  const bool b2 = (lane & 4) != 0, b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
  float u[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = b2 ? v[j + 4] : v[j], give = b2 ? v[j] : v[j + 4];
    u[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 4));
  }
  float u2[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = b1 ? u[j + 2] : u[j], give = b1 ? u[j] : u[j + 2];
    u2[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 2));
  }
  const float keep = b0 ? u2[1] : u2[0], give = b0 ? u2[0] : u2[1];
  return fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 1));
}

// ---------------------------------------------------------------------------
// launchers (one per kernel family); all asynchronous on `s`
// ---------------------------------------------------------------------------

// normalise + score + argmax.  S: [BH,k,n] fp32 (may be null), a: [BH,n]
// (may be null), mcount: [BH,n] zeroed here when non-null, gbins: the group
// bins [BH,k,gbin_stride(n)] (may be null; written only with S).
cudaError_t launch_score_simt(const void* qk, rt_dtype dt, int BH, int H, int n, int d,
                              const float* mu, int k, float* S, int32_t* a,
                              int32_t* mcount, uint16_t* gbins, cudaStream_t s);

// dispatcher: tcgen05 scoring for bf16 with k <= 256 (fp32-accurate via a
// three-plane split of the centroids), the SIMT kernel otherwise.  prep: device
// scratch of score_prep_bytes(H, d, k) bytes for the per-head centroid image
// (null: every score CTA builds the image itself).  err: device error word
// (may be null).
bool score_tc_supported(rt_dtype dt, int d, int k);
size_t score_prep_bytes(int H, int d, int k);
cudaError_t launch_score(const void* qk, rt_dtype dt, int B, int H, int n, int d, const float* mu,
                         int k, float* S, int32_t* a, int32_t* mcount, uint16_t* gbins,
                         void* prep, unsigned int* err, cudaStream_t s);

// top-w per centroid in ascending position order; counts memberships into
// mcount (atomic integer increments; may be null) and records up to
// SLOTS_PER_ROW global slot ids (c*w + slot) per position in `slots`
// [BH, n, SLOTS_PER_ROW] (may be null; entry order is arbitrary).  gbins:
// the group bins the score kernel wrote with S (may be null: the select then
// derives everything from S).
constexpr int SLOTS_PER_ROW = 8;

// Whether the forward asks the score kernel for group bins: only for rows long
// enough that streaming them costs the select more than the bins cost the
// score epilogue.
bool select_wants_group_bins(int n);
cudaError_t launch_select(const float* S, const uint16_t* gbins, int BH, int n, int k, int w,
                          int32_t* idx, int32_t* mcount, int32_t* slots, cudaStream_t s);

// in-cluster attention.  Rows of positions with mcount == 1 go straight to
// `out`; rows of positions in several clusters go to yslot [BH,k,w,d] fp32.
// idx_k: the keys' own lists (separate queries and keys; null when queries
// double as keys); mvis then counts every position's memberships with a
// visible key (zeroed beforehand).
cudaError_t launch_attention_simt(const void* q, const void* kk, const void* v, rt_dtype dt,
                                  int BH, int n, int d, int k, int w, int causal,
                                  float scale, const int32_t* idx, const int32_t* idx_k,
                                  const int32_t* mcount, int32_t* mvis, void* out, float* yslot,
                                  cudaStream_t s);

// the same on tcgen05 tensor cores (bf16 only): the pipelined kernel for
// w <= 128, the two-tile kernel for w <= 256, the key-block kernel above
// that; err: device error word.
bool attention_tc_supported(rt_dtype dt, int d, int w);
cudaError_t launch_attention_tc(const void* q, const void* v, int BH, int n, int d, int k, int w,
                                int causal, float scale, const int32_t* idx,
                                const int32_t* mcount, void* out, float* yslot,
                                unsigned int* err, cudaStream_t s);

// separate queries and keys on tcgen05 (bf16, any w): query rows from idx_q,
// key/value rows from idx_k, causal on original positions; mvis (zeroed
// beforehand) counts every position's memberships with a visible key.
cudaError_t launch_attention_separate_tc(const void* q, const void* kk, const void* v, int BH,
                                         int n, int d, int k, int w, int causal, float scale,
                                         const int32_t* idx_q, const int32_t* idx_k,
                                         const int32_t* mcount, int32_t* mvis, void* out,
                                         float* yslot, unsigned int* err, cudaStream_t s);

// local (sliding-window) causal attention, shared QK, bf16: every position
// attends to the `window` positions ending at it; out [BH, n, d].
cudaError_t launch_local_attention(const void* q, const void* v, int BH, int n, int d, int window,
                                   float scale, void* out, unsigned int* err, cudaStream_t s);

// clusters of 128 < w <= 256 (two row tiles): one CTA per cluster, both
// tiles' scores in TMEM at once (bf16 only).
cudaError_t launch_attention_pair(const void* q, const void* v, int BH, int n, int d, int k,
                                  int w, int causal, float scale, const int32_t* idx,
                                  const int32_t* mcount, void* out, float* yslot,
                                  unsigned int* err, cudaStream_t s);

// the same, persistent and pipelined, for w <= 128 (bf16 only).
cudaError_t launch_attention_pipe(const void* q, const void* v, int BH, int n, int d, int k,
                                  int w, int causal, float scale, const int32_t* idx,
                                  const int32_t* mcount, void* out, float* yslot,
                                  unsigned int* err, cudaStream_t s);

// zero rows (mcount == 0) and the mean over clusters (mcount >= 2); mdiv
// (may be null) replaces mcount as the divisor (0: zero row).
cudaError_t launch_scatter(rt_dtype dt, int BH, int n, int d, int k, int w,
                           const int32_t* idx, const int32_t* mcount, const int32_t* mdiv,
                           const int32_t* slots, const float* yslot, void* out, cudaStream_t s);

// backward of a5..a6 with the routing held fixed: per-slot gradient rows of
// every cluster (dq_slot, dv_slot [BH,k,w,d] fp32), from the lists idx and
// the membership counts mcount; dout [BH,n,d] fp32.
cudaError_t launch_backward_clusters(const void* q, const void* v, rt_dtype dt, int BH, int n,
                                     int d, int k, int w, int causal, float scale,
                                     const int32_t* idx, const int32_t* mcount, const float* dout,
                                     float* dq_slot, float* dv_slot, cudaStream_t s);
// membership counts and the first SLOTS_PER_ROW slot ids of every position,
// rebuilt from the lists (mcount is cleared first)
cudaError_t launch_membership(const int32_t* idx, int BH, int n, int k, int w, int32_t* mcount,
                              int32_t* slots, cudaStream_t s);
// every position's sum of its slot rows (fp32; zero for no membership)
cudaError_t launch_gather_sum(int BH, int n, int d, int k, int w, const int32_t* idx,
                              const int32_t* mcount, const int32_t* slots, const float* yslot,
                              float* out, cudaStream_t s);

// centroid update (argmax assignment), a segmented reduction: a bucketing
// kernel sorts every chunk's rows by centroid, then one CTA per (head,
// centroid) sums its rows.  ws: device scratch of
// ema_workspace_bytes(B, H, n, d, k, dt) bytes.
size_t ema_workspace_bytes(int B, int H, int n, int d, int k, rt_dtype dt);
cudaError_t launch_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                       const int32_t* assign, float* mu, int k, float decay,
                       void* ws, cudaStream_t s);
// the same reduction stopped before the blend: sums [H][k][d+1] receives every
// centroid's sum of normalised rows and (as a float) its count
cudaError_t launch_ema_sums(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                            const int32_t* assign, int k, float* sums, void* ws, cudaStream_t s);
// the blend from such sums (possibly added over shards of the batch)
cudaError_t launch_ema_apply(const float* sums, int H, int d, float* mu, int k, float decay,
                             cudaStream_t s);
// the centroid step driven by the top-w lists idx [B,H,k,w] instead of an
// assignment (entries outside [0, n) are skipped)
cudaError_t launch_ema_topw(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                            const int32_t* idx, int w, float* mu, int k, float decay,
                            cudaStream_t s);

}  // namespace rt
