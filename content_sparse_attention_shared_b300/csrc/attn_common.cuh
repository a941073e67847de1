// Helpers shared by the tensor-core attention kernels: 16-byte cp.async row
// gathers into the no-swizzle core-matrix layouts the MMA operands use, and
// bf16 packing.
#pragma once

#include "rt_internal.cuh"
#include "tc_ptx.cuh"

namespace rt {
namespace attn {

using bf16 = __nv_bfloat16;
constexpr int ROWS = 128;  // tile rows = TMEM lanes = MMA M

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
__device__ __forceinline__ void cp_async_wait_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Gather 128 rows (positions pos[r], -1 = zero row) of D bf16 into the K-major
// no-swizzle layout: chunk (r, kc) at (r/8)*(D/8)*128 + kc*128 + (r%8)*16.
// `nwarps` warps share the work (warp = this warp's index among them); a warp
// covers 8 rows x 4 chunks per instruction (512 contiguous bytes).
template <int D>
__device__ __forceinline__ void gather_kmajor(uint8_t* dst, const bf16* __restrict__ src,
                                              const int* pos, int warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  constexpr int KC = D / 8;  // chunks per row
  constexpr int ITEMS = (ROWS / 8) * (KC / 4);
  const uint32_t base = tc::smem_u32(dst);
  for (int it = warp; it < ITEMS; it += nwarps) {
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
                                               const int* pos, int warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  constexpr int EC = D / 8;
  constexpr int ITEMS = (ROWS / 8) * (EC / 4);
  const uint32_t base = tc::smem_u32(dst);
  for (int it = warp; it < ITEMS; it += nwarps) {
    const int jg = it / (EC / 4);
    const int ec = (it % (EC / 4)) * 4 + (lane >> 3);
    const int j = jg * 8 + (lane & 7);
    const int p = pos[j];
    const uint32_t off = ec * 2048 + jg * 128 + (lane & 7) * 16;
    const bf16* g = src + (size_t)(p < 0 ? 0 : p) * D + ec * 8;
    cp_async16(base + off, g, p >= 0);
  }
}

// Gather 128 rows (positions pos[r], -1 = zero row) of D bf16 into the
// 128-byte-swizzled row layout: D/64 blocks of [128 rows x 128 bytes], row r
// of block kb at kb*16384 + r*128, its 16-byte chunk j XOR-permuted to
// (j ^ (r % 8)).  Read as the K-major operand of S = Q K^T and as the MN-major
// operand of O = P V.  A warp instruction moves four whole 128-byte row pieces
// (eight lanes per row: full-line global reads, conflict-free shared writes).
template <int D>
__device__ __forceinline__ void gather_sw128(uint8_t* dst, const bf16* __restrict__ src,
                                             const int* pos, int warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  constexpr int KB = D / 64;
  constexpr int ITEMS = (ROWS / 4) * KB;
  const uint32_t base = tc::smem_u32(dst);
  const int jj = lane & 7;
  for (int it = warp; it < ITEMS; it += nwarps) {
    const int kb = it % KB;
    const int r = (it / KB) * 4 + (lane >> 3);
    const int p = pos[r];
    const uint32_t off = kb * (ROWS * 128) + r * 128 + ((jj ^ (r & 7)) << 4);
    const bf16* g = src + (size_t)(p < 0 ? 0 : p) * D + kb * 64 + jj * 8;
    cp_async16(base + off, g, p >= 0);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace attn
}  // namespace rt
