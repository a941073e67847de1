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
  K_NUM_KINDS = 10
};

// Error detail for the calling host thread (rt_last_error_detail) and the
// shape checks shared by the entry points.
rt_status record_error(rt_status s, const char* msg);
rt_status validate_shape(rt_dtype dt, int B, int H, int n, int d, int k, int w);

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
// launchers (one per kernel family); all asynchronous on `s`
// ---------------------------------------------------------------------------

// normalise + score + argmax.  S: [BH,k,n] fp32 (may be null), a: [BH,n]
// (may be null), mcount: [BH,n] zeroed here when non-null.
cudaError_t launch_score_simt(const void* qk, rt_dtype dt, int BH, int H, int n, int d,
                              const float* mu, int k, float* S, int32_t* a,
                              int32_t* mcount, cudaStream_t s);

// dispatcher: tcgen05 scoring for bf16 with k <= 256 (fp32-accurate via a
// three-plane split of the centroids), the SIMT kernel otherwise.  prep: device
// scratch of score_prep_bytes(H, d, k) bytes for the per-head centroid image
// (null: every score CTA builds the image itself).  err: device error word
// (may be null).
bool score_tc_supported(rt_dtype dt, int d, int k);
size_t score_prep_bytes(int H, int d, int k);
cudaError_t launch_score(const void* qk, rt_dtype dt, int B, int H, int n, int d, const float* mu,
                         int k, float* S, int32_t* a, int32_t* mcount, void* prep,
                         unsigned int* err, cudaStream_t s);

// top-w per centroid in ascending position order; counts memberships into
// mcount (atomic integer increments; may be null) and records up to
// SLOTS_PER_ROW global slot ids (c*w + slot) per position in `slots`
// [BH, n, SLOTS_PER_ROW] (may be null; entry order is arbitrary).
constexpr int SLOTS_PER_ROW = 8;
cudaError_t launch_select(const float* S, int BH, int n, int k, int w, int32_t* idx,
                          int32_t* mcount, int32_t* slots, cudaStream_t s);

// in-cluster attention.  Rows of positions with mcount == 1 go straight to
// `out`; rows of positions in several clusters go to yslot [BH,k,w,d] fp32.
cudaError_t launch_attention_simt(const void* q, const void* kk, const void* v, rt_dtype dt,
                                  int BH, int n, int d, int k, int w, int causal,
                                  float scale, const int32_t* idx, const int32_t* mcount,
                                  void* out, float* yslot, cudaStream_t s);

// the same on tcgen05 tensor cores (bf16 only): the pipelined kernel below
// for w <= 128, the key-block kernel above that; err: device error word.
bool attention_tc_supported(rt_dtype dt, int d, int w);
cudaError_t launch_attention_tc(const void* q, const void* v, int BH, int n, int d, int k, int w,
                                int causal, float scale, const int32_t* idx,
                                const int32_t* mcount, void* out, float* yslot,
                                unsigned int* err, cudaStream_t s);

// local (sliding-window) causal attention, shared QK, bf16: every position
// attends to the `window` positions ending at it; out [BH, n, d].
cudaError_t launch_local_attention(const void* q, const void* v, int BH, int n, int d, int window,
                                   float scale, void* out, unsigned int* err, cudaStream_t s);

// the same, persistent and pipelined, for w <= 128 (bf16 only).
cudaError_t launch_attention_pipe(const void* q, const void* v, int BH, int n, int d, int k,
                                  int w, int causal, float scale, const int32_t* idx,
                                  const int32_t* mcount, void* out, float* yslot,
                                  unsigned int* err, cudaStream_t s);

// zero rows (mcount == 0) and the mean over clusters (mcount >= 2).
cudaError_t launch_scatter(rt_dtype dt, int BH, int n, int d, int k, int w,
                           const int32_t* idx, const int32_t* mcount, const int32_t* slots,
                           const float* yslot, void* out, cudaStream_t s);

// centroid update: one CTA per (head, centroid) lists its rows, sums them
// normalised in a fixed order, blends and renormalises (no workspace needed
// beyond the status word: ema_workspace_bytes returns 0).
size_t ema_workspace_bytes(int B, int H, int n, int k);
cudaError_t launch_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                       const int32_t* assign, float* mu, int k, float decay,
                       void* ws, cudaStream_t s);
// the centroid step driven by the top-w lists idx [B,H,k,w] instead of an
// assignment (entries outside [0, n) are skipped)
cudaError_t launch_ema_topw(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                            const int32_t* idx, int w, float* mu, int k, float decay,
                            cudaStream_t s);

}  // namespace rt
